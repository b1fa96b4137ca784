"""GPU path vs the CPU oracle, byte for byte, through the C ABI.

Tolerance: 0 ULP everywhere (bytes compared); the canonical order fixes every
bit, so any difference is a bug.  Covers the five workloads (small sizes in
full, full sizes in full too), the grid / segment-size / replay /
shard invariances, and the edge cases.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_bytes_equal, case_np, gpu_scatter, np_bits, oracle_dtype, oracle_scatter
from invariant_gradient_reduction_gb300 import detreduce as dr
from invariant_gradient_reduction_gb300 import workloads as wl
from invariant_gradient_reduction_gb300.workloads import ScatterCase

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from invariant_gradient_reduction_gb300 import build
    build.build()
    dr.lib()
    oracle.build()


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def small_case(name):
    return wl.make(name, "small", device=DEV)


SCATTER_SMALL = ["tiny_moe", "moe_combine", "ep_invariance", "sparse_key_scatter"]


# --------------------------------------------------------------------------
# plan: destination lists are integer-exact
# --------------------------------------------------------------------------

def cluster_plan_applies(N, M, src):
    """Mirror of the single-cluster plan's size rule (1024 threads, slices of ~2048, <= 16 CTAs)."""
    if src or N <= 0 or N > 16 * 8192:
        return False
    C = min(16, max(1, -(-N // 2048)))
    return -(-(-(-M // C)) // 1024) <= 8


def owner_plan_possible(N, M, src):
    """The owner plan's hard limits (clusters of 8, 4 or 2 CTAs, each owning <= 1024 destinations, a
    full histogram of M counts per CTA): outside them it must refuse.  Inside, whether it runs
    also depends on how many clusters the device runs at once."""
    return not src and 0 < N <= (1 << 18) and 0 < M <= (1 << 15)


def owner_plan_sure(N, M, src):
    """Inside the limits with at most 1024 destinations: one cluster is enough, so it may not refuse."""
    return owner_plan_possible(N, M, src) and M <= 1024


def radix_plan_applies(N, M, src):
    """Mirror of the radix plan's size rule (packed 24-bit source positions, one or two 8-bit digits)."""
    return not src and 0 < N < (1 << 24) and 0 < M <= 65536


def plan_path_applies(path, N, M, src):
    if path == 2:
        return cluster_plan_applies(N, M, src)
    if path == 3:
        return owner_plan_possible(N, M, src)
    if path == 4:
        return radix_plan_applies(N, M, src)
    return True


@pytest.mark.parametrize("plan_path", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("N,M,src", [(0, 7, False), (1, 1, False), (1000, 1, False), (5000, 37, False),
                                     (70000, 300, False), (20000, 70000, False), (9000, 600, True),
                                     (100000, 65536, False), (40000, 5, True), (31, 3, False),
                                     (4097, 4096, False), (131072, 16384, False), (131072, 131072, False),
                                     (65536 + 17, 2, False), (65536, 4096, False), (65537, 4096, False),
                                     (2, 2, False), (100, 4096, False), (131072, 4097, False),
                                     (1 << 18, 1 << 15, False), ((1 << 18) + 1, 5, False), (3, 1 << 15, False),
                                     (200000, 20000, False), (77777, 151, False), (32768, 4096, False)])
def test_plan_lists_match_oracle(N, M, src, plan_path):
    g = torch.Generator().manual_seed(N * 31 + M)
    idx = torch.randint(0, M, (N,), generator=g, dtype=torch.int32)
    sid = None
    if src:
        sid = (torch.randperm(N, generator=g) * 5 - 100).to(torch.int64)
    opts = {"plan_path": plan_path}
    if not plan_path_applies(plan_path, N, M, src):
        with pytest.raises(dr.DetError) as e:
            dr.det_reduce_plan(idx.to(DEV), M, src_id=None if sid is None else sid.to(DEV), opts=opts)
        assert e.value.code == dr.DET_ERR_UNSUPPORTED
        return
    try:
        plan = dr.det_reduce_plan(idx.to(DEV), M, src_id=None if sid is None else sid.to(DEV), opts=opts)
    except dr.DetError as e:
        # only the owner plan may refuse inside its limits, and only where the
        # device runs too few clusters at once for this many destinations
        assert plan_path == 3 and e.code == dr.DET_ERR_UNSUPPORTED and not owner_plan_sure(N, M, src), (N, M)
        return
    rp, perm = dr.plan_lists(plan)
    want_rp, want_perm = oracle.build_lists(idx.numpy(), M, src_id=None if sid is None else sid.numpy())
    assert np.array_equal(rp.cpu().numpy().astype(np.int64), want_rp)
    assert np.array_equal(perm.cpu().numpy().astype(np.int64), want_perm)
    d = plan.describe()
    counts = np.diff(want_rp)
    assert d["max_row_len"] == (counts.max() if M else 0)


def test_plan_zipf_hot_rows_and_work_list():
    case = small_case("sparse_key_scatter")
    plan = dr.det_reduce_plan(case.idx, case.M)
    rp, perm = dr.plan_lists(plan)
    want_rp, want_perm = oracle.build_lists(case.idx.cpu().numpy(), case.M)
    assert np.array_equal(rp.cpu().numpy(), want_rp)
    assert np.array_equal(perm.cpu().numpy(), want_perm)
    d = plan.describe()
    counts = np.diff(want_rp)
    nch = (counts + 31) // 32
    G = 1 << d["seg_chunks_log2"]
    hot = nch > G
    assert d["n_hot_rows"] == int(hot.sum())
    assert d["n_segments"] == int(((nch[hot] + G - 1) // G).sum())
    assert d["n_units"] == d["n_segments"] + int((~hot).sum())
    assert d["n_hot_rows"] > 0


@pytest.mark.parametrize("plan_path", [0, 1, 3, 4])
def test_plan_errors(plan_path):
    o = {"plan_path": plan_path}
    idx = torch.tensor([0, 1, 5, 2], dtype=torch.int32, device=DEV)
    with pytest.raises(dr.DetError) as e:
        dr.det_reduce_plan(idx, 5, opts=o)
    assert e.value.code == dr.DET_ERR_INDEX_RANGE
    with pytest.raises(dr.DetError) as e:
        dr.det_reduce_plan(torch.tensor([0, -1], dtype=torch.int32, device=DEV), 5, opts=o)
    assert e.value.code == dr.DET_ERR_INDEX_RANGE
    # an out-of-range index in a later CTA of the cluster
    big = torch.zeros(50000, dtype=torch.int32, device=DEV)
    big[-1] = 9
    with pytest.raises(dr.DetError) as e:
        dr.det_reduce_plan(big, 9, opts=o)
    assert e.value.code == dr.DET_ERR_INDEX_RANGE
    # 2^18 sources: the owner plan's warps sweep full rounds (1024 sources each)
    full = torch.zeros(1 << 18, dtype=torch.int32, device=DEV)
    full[123457] = -5
    with pytest.raises(dr.DetError) as e:
        dr.det_reduce_plan(full, 9, opts=o)
    assert e.value.code == dr.DET_ERR_INDEX_RANGE
    with pytest.raises(dr.DetError) as e:
        dr.det_reduce_plan(idx, 5, opts={"plan_path": 7})
    assert e.value.code == dr.DET_ERR_ARG
    with pytest.raises(dr.DetError) as e:
        dr.det_reduce_plan(torch.tensor([1, 1, 0], dtype=torch.int32, device=DEV), 3,
                           src_id=torch.tensor([7, 7, 7], dtype=torch.int64, device=DEV))
    assert e.value.code == dr.DET_ERR_ORDER_KEY
    # equal keys in different destinations are fine
    dr.det_reduce_plan(torch.tensor([1, 2, 0], dtype=torch.int32, device=DEV), 3,
                       src_id=torch.tensor([7, 7, 7], dtype=torch.int64, device=DEV))
    with pytest.raises(dr.DetError) as e:
        dr.det_reduce_plan(idx[:2], 5, workspace=torch.empty(64, dtype=torch.uint8, device=DEV))
    assert e.value.code == dr.DET_ERR_WORKSPACE


# --------------------------------------------------------------------------
# scatter-reduce parity
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", SCATTER_SMALL)
def test_scatter_small_matches_oracle(name):
    case = small_case(name)
    out, plan = gpu_scatter(case)
    assert_bytes_equal(np_bits(out), oracle_scatter(case), name)


@pytest.mark.parametrize("name", SCATTER_SMALL)
def test_plan_paths_give_same_bytes(name):
    """The multi-kernel, single-cluster, owner and radix plans feed the reduce the same lists and work counts."""
    case = small_case(name)
    want = oracle_scatter(case)
    counts = {}
    for path in (1, 2, 3, 4):
        if not plan_path_applies(path, case.N, case.M, case.src_id is not None):
            continue
        for seg in (3, 5):
            out, plan = gpu_scatter(case, opts={"plan_path": path, "seg_chunks_log2": seg})
            assert_bytes_equal(np_bits(out), want, f"{name} plan_path={path} g={seg}")
            d = plan.describe()
            c = (d["n_units"], d["n_segments"], d["n_hot_rows"], d["max_row_len"])
            assert counts.setdefault(seg, c) == c, (path, seg, c, counts[seg])


def test_cluster_plan_hot_rows():
    """Zipf-like destinations with rows far longer than a segment, through the single-cluster plan."""
    g = torch.Generator().manual_seed(77)
    N, M, H = 60000, 300, 40
    r = torch.rand(N, generator=g, dtype=torch.float64)
    idx = torch.minimum((M * r ** 4).floor(), torch.tensor(M - 1.0)).to(torch.int32)
    x = torch.randn(N, H, generator=g)
    w = torch.rand(N, generator=g)
    case = _case(idx, x, M, w=w)
    want = oracle_scatter(case)
    for path in (1, 2, 3, 4):
        out, plan = gpu_scatter(case, opts={"plan_path": path})
        d = plan.describe()
        assert d["n_hot_rows"] > 0 and d["n_segments"] > d["n_hot_rows"]
        assert_bytes_equal(np_bits(out), want, f"hot rows plan_path={path}")


@pytest.mark.parametrize("name", ["moe_combine", "sparse_key_scatter"])
@pytest.mark.parametrize("seg", [3, 4, 5, 6])
def test_segment_size_changes_no_bit(name, seg):
    case = small_case(name)
    base, _ = gpu_scatter(case)
    out, plan = gpu_scatter(case, opts={"seg_chunks_log2": seg})
    assert_bytes_equal(np_bits(out), np_bits(base), f"{name} g={seg}")


@pytest.mark.parametrize("name", ["moe_combine", "sparse_key_scatter", "tiny_moe"])
def test_grid_size_changes_no_bit(name):
    case = small_case(name)
    base, plan = gpu_scatter(case)
    want = np_bits(base)
    for grid in (1, 3, sms() - 1, sms(), 4 * sms(), 0):
        out = torch.empty_like(base)
        dr.det_scatter_reduce(plan, case.x, out, w=case.w, opts={"grid_ctas": grid})
        assert_bytes_equal(np_bits(out), want, f"{name} grid={grid}")


@pytest.mark.parametrize("name", ["moe_combine", "sparse_key_scatter", "tiny_moe", "ep_invariance"])
def test_gather_path_changes_no_bit(name):
    """Every gather kernel (register-staged, cp.async ring, TMA bulk ring) gives the same bytes."""
    case = small_case(name)
    base, plan = gpu_scatter(case)
    want = np_bits(base)
    for path in (1, 2, 3):
        out = torch.empty_like(base)
        try:
            dr.det_scatter_reduce(plan, case.x, out, w=case.w, opts={"gather_path": path})
        except dr.DetError as e:
            assert path == 3 and e.code == dr.DET_ERR_UNSUPPORTED
            continue
        assert_bytes_equal(np_bits(out), want, f"{name} path={path}")


def test_replays_identical_under_contention(replay):
    """R replays give identical bytes and identical fingerprints while a side
    stream runs matmuls (the pages' contention replay), for the scatter-reduce,
    index_add, split-K and an unwaited plan + reduce."""
    case = small_case("sparse_key_scatter")
    base, plan = gpu_scatter(case)
    out = replay.identical(lambda: dr.det_scatter_reduce(plan, case.x, torch.empty_like(base), w=case.w),
                           name="scatter_reduce")
    assert_bytes_equal(np_bits(out), np_bits(base), "replay")
    init = torch.randn_like(base)
    replay.identical(lambda: dr.det_index_add(plan, case.x, init.clone(), w=case.w), name="index_add")

    def unwaited():
        p = dr.det_reduce_plan(case.idx, case.M, opts={"async_plan": 1})
        o = dr.det_scatter_reduce(p, case.x, torch.empty_like(base), w=case.w, opts={"async_plan": 1})
        dr.det_plan_status(p)
        return o
    assert_bytes_equal(np_bits(replay.identical(unwaited, name="plan+reduce")), np_bits(base), "unwaited")
    P = wl.make("splitk", "small", device=DEV)  # 56 splits: the two-chunk kernel
    replay.identical(lambda: dr.det_splitk_reduce(P, torch.empty(P.shape[1], device=DEV)), name="splitk")
    # a waited plan with <= 32 terms per destination and 2 KB rows: the TMA bulk kernel
    mc = small_case("moe_combine")
    mbase, mplan = gpu_scatter(mc)
    mout = replay.identical(lambda: dr.det_scatter_reduce(mplan, mc.x, torch.empty_like(mbase), w=mc.w),
                            name="moe_combine waited")
    assert_bytes_equal(np_bits(mout), np_bits(mbase), "moe replay")
    # the split-K GEMM: two MMA-issuing warps, the fold in the epilogue
    A, W = wl.splitk_gemm_inputs(384, 56 * 128, 24, seed=3, device=DEV)

    def gemm():
        o = torch.empty(384, 24, device=DEV)
        dr.det_splitk_gemm_reduce(A, W, 56, o)
        return o
    replay.identical(gemm, name="splitk_gemm")
    # the ring kernel (dynamic claims from the plan's counter, reset by its
    # last CTA) with the register-staged kernel beside it: index_add and the
    # scatter-reduce behind an unwaited plan, the same plan reused each time
    ec = small_case("embedding_backward")
    eplan = dr.det_reduce_plan(ec.idx, ec.M)
    einit = torch.randn(ec.M, ec.H, device=DEV)
    ering = replay.identical(lambda: dr.det_index_add(eplan, ec.x, einit.clone(), opts={"gather_path": 3}),
                             name="index_add ring")
    eref = dr.det_index_add(eplan, ec.x, einit.clone(), opts={"gather_path": 1})
    assert_bytes_equal(np_bits(ering), np_bits(eref), "ring replay")
    aplan = dr.det_reduce_plan(ec.idx, ec.M, opts={"async_plan": 1})
    dr.det_plan_status(aplan)

    def ring_scatter():
        return dr.det_scatter_reduce(aplan, ec.x, torch.empty(ec.M, ec.H, device=DEV),
                                     opts={"async_plan": 1, "gather_path": 3})
    sring = replay.identical(ring_scatter, name="scatter ring")
    sref = dr.det_scatter_reduce(eplan, ec.x, torch.empty(ec.M, ec.H, device=DEV), opts={"gather_path": 1})
    assert_bytes_equal(np_bits(sring), np_bits(sref), "ring scatter replay")


def test_ring_kernel_edge_cases():
    """The ring kernel at its limits: destinations of exactly 32 terms and of
    1 term in one plan (the widest and the narrowest items), H that leaves a
    ragged last tile, a grid larger than the units, and many calls on one plan
    (the claim counter must be back at 0 after each call)."""
    M, H = 300, 1048  # bf16 rows of 2096 bytes: 32-term items are split into tiles, the last one ragged
    lens = np.where(np.arange(M) % 3 == 0, 32, np.where(np.arange(M) % 3 == 1, 1, 0))
    idx_np = np.repeat(np.arange(M, dtype=np.int32), lens)
    np.random.default_rng(7).shuffle(idx_np)
    g = torch.Generator(device=DEV).manual_seed(8)
    x = torch.randn(idx_np.size, H, generator=g, device=DEV).to(torch.bfloat16)
    idx = torch.from_numpy(idx_np).to(DEV)
    plan = dr.det_reduce_plan(idx, M)
    want = oracle.scatter_reduce(idx_np, np_bits(x), M)
    for grid in (0, 1, 7, 1000):
        for rep in range(3):
            out = torch.full((M, H), 5.0, device=DEV)
            dr.det_scatter_reduce(plan, x, out, opts={"gather_path": 3, "grid_ctas": grid, "debug_checks": 1})
            assert_bytes_equal(np_bits(out), want, f"ring grid={grid} rep={rep}")
    init = torch.randn(M, H, generator=g, device=DEV)
    want_a = oracle.scatter_reduce(idx_np, np_bits(x), M, out_init=np_bits(init))
    for rep in range(3):
        out = init.clone()
        dr.det_index_add(plan, x, out, opts={"gather_path": 3, "debug_checks": 1})
        assert_bytes_equal(np_bits(out), want_a, f"ring index_add rep={rep}")


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_ep_shards_identical(P):
    """Sources split into P separate expert-shard buffers give identical bytes."""
    case = small_case("ep_invariance")
    base, plan = gpu_scatter(case)
    rows = wl.ep_shard_rows(case, P)
    shards = wl.split_rows(case.x, rows)
    out, _ = gpu_scatter(case, shards=shards, plan=plan)
    assert_bytes_equal(np_bits(out), np_bits(base), f"P={P}")
    assert_bytes_equal(np_bits(out), oracle_scatter(case), f"P={P} vs oracle")


def test_physical_row_permutation_with_src_id():
    case = small_case("moe_combine")
    base, _ = gpu_scatter(case)
    g = torch.Generator().manual_seed(5)
    pr = torch.randperm(case.N, generator=g)
    prd = pr.to(DEV)
    perm_case = ScatterCase(name="permuted", idx=case.idx[prd].contiguous(), x=case.x[prd].contiguous(),
                            w=case.w[prd].contiguous(), M=case.M, out_dtype=case.out_dtype,
                            src_id=prd.to(torch.int64))
    out, _ = gpu_scatter(perm_case)
    assert_bytes_equal(np_bits(out), np_bits(base), "permuted rows with src_id")


def test_batch_invariance():
    """One token's 8 rows combined alone and inside batches of other sizes, at other
    positions: identical output row (property A of the DeepSeek-V4 chapter)."""
    H = 4096
    g = torch.Generator(device=DEV).manual_seed(3)
    tok = torch.randn(8, H, generator=g, device=DEV).to(torch.bfloat16)
    tw = torch.rand(8, generator=g, device=DEV)
    alone = ScatterCase("alone", torch.zeros(8, dtype=torch.int32, device=DEV), tok, tw, 1, torch.bfloat16)
    want = np_bits(gpu_scatter(alone)[0])[0]
    for T in (3, 64, 1000):
        big = wl.moe_combine(T, 16, 8, H, seed=T, device=DEV)
        pos = T // 2
        keep = big.idx != pos
        others_idx, others_x, others_w = big.idx[keep], big.x[keep], big.w[keep]
        n = others_idx.numel()
        slots = torch.sort(torch.randperm(n + 8, generator=torch.Generator().manual_seed(T))[:8]).values.to(DEV)
        mask = torch.zeros(n + 8, dtype=torch.bool, device=DEV)
        mask[slots] = True
        idx = torch.empty(n + 8, dtype=torch.int32, device=DEV)
        x = torch.empty(n + 8, H, dtype=torch.bfloat16, device=DEV)
        w = torch.empty(n + 8, device=DEV)
        idx[mask], x[mask], w[mask] = pos, tok, tw
        idx[~mask], x[~mask], w[~mask] = others_idx, others_x, others_w
        out, _ = gpu_scatter(ScatterCase("batch", idx, x, w, T, torch.bfloat16))
        assert np_bits(out)[pos].tobytes() == want.tobytes()


# --------------------------------------------------------------------------
# full-size workloads (every destination checked against the oracle)
# --------------------------------------------------------------------------

@pytest.mark.slow
@pytest.mark.parametrize("name", ["tiny_moe", "moe_combine", "ep_invariance", "sparse_key_scatter"])
def test_full_size_parity(name):
    """The full-size workloads, every destination compared with the oracle (the
    EP-invariance workload with the sources in one buffer and in 8 shards)."""
    case = wl.make(name, "full", device=DEV)
    out, plan = gpu_scatter(case)
    want = oracle_scatter(case)
    assert_bytes_equal(np_bits(out), want, name)
    if name == "ep_invariance":
        for P in (2, 4, 8):
            shards = wl.split_rows(case.x, wl.ep_shard_rows(case, P))
            o2, _ = gpu_scatter(case, shards=shards, plan=plan)
            if P == 8:
                assert_bytes_equal(np_bits(o2), want, f"{name} P={P}")
            assert torch.equal(o2.view(torch.int16), out.view(torch.int16)), P
            del shards, o2
    if name == "sparse_key_scatter":
        for grid in (sms(), 3 * sms() + 1):
            o3 = torch.empty_like(out)
            dr.det_scatter_reduce(plan, case.x, o3, w=case.w, opts={"grid_ctas": grid})
            assert torch.equal(o3.view(torch.int32), out.view(torch.int32)), grid


# --------------------------------------------------------------------------
# edge cases
# --------------------------------------------------------------------------

def _case(idx, x, M, w=None, out_dtype=torch.float32, src_id=None):
    return ScatterCase("edge", torch.as_tensor(idx, dtype=torch.int32).to(DEV), x.to(DEV),
                       None if w is None else w.to(DEV), M, out_dtype,
                       None if src_id is None else src_id.to(DEV))


@pytest.mark.parametrize("n", [1, 2, 31, 32, 33, 63, 64, 65, 255, 256, 257, 1000, 4097, 16384, 20001])
@pytest.mark.parametrize("H,xdt", [(128, torch.bfloat16), (24, torch.float32), (13, torch.bfloat16)])
def test_row_lengths(n, H, xdt):
    g = torch.Generator().manual_seed(n + H)
    M = 3
    idx = torch.full((n,), 1, dtype=torch.int32)
    idx[::7] = 0
    x = (torch.randn(n, H, generator=g) * torch.exp2(torch.randint(-12, 12, (n, 1), generator=g).float())).to(xdt)
    w = torch.rand(n, generator=g)
    for od in (torch.float32, torch.bfloat16):
        case = _case(idx, x, M, w, od)
        out, _ = gpu_scatter(case)
        assert_bytes_equal(np_bits(out), oracle_scatter(case), f"n={n} H={H} {xdt} -> {od}")


def test_empty_inputs():
    x = torch.zeros(0, 16, dtype=torch.bfloat16)
    case = _case([], x, 5)
    out = torch.full((5, 16), 7.0, device=DEV)
    gpu_scatter(case, out=out)
    assert torch.equal(out, torch.zeros_like(out)) and not torch.signbit(out).any()
    # M = 0, N = 0
    case0 = _case([], x, 0)
    gpu_scatter(case0)
    # H = 0
    casen = _case([0, 1], torch.zeros(2, 0), 3)
    gpu_scatter(casen)


def test_negative_zero_and_specials():
    """All -0.0 terms give -0.0; empty rows give +0.0; inf, subnormals and NaN propagate."""
    n = 70
    H = 8
    x = torch.full((n, H), -0.0)
    x[:, 1] = torch.tensor(float("inf"))
    x[5, 2] = float("-inf")
    x[7, 2] = float("inf")  # inf - inf: NaN
    x[:, 3] = 1e-40  # subnormal
    x[:, 4] = -1e-45
    x[3, 5] = float("nan")
    x[:, 6] = 3.4e38
    idx = torch.zeros(n, dtype=torch.int32)
    case = _case(idx, x, 2)
    out = np_bits(gpu_scatter(case)[0])
    want = oracle_scatter(case)
    assert out[0, 0].view(np.uint32) == 0x80000000
    assert out[1].view(np.uint32).tolist() == [0] * H
    assert np.isnan(out[0, 2]) and np.isnan(out[0, 5])
    fin = [0, 1, 3, 4, 6, 7]
    assert_bytes_equal(out[:, fin], want[:, fin], "specials")
    assert np.isinf(out[0, 6])  # overflow to +inf


def test_padded_and_unaligned_rows():
    """Row strides that are not a multiple of 16 bytes take the scalar path: same bits."""
    g = torch.Generator().manual_seed(9)
    N, M, H = 3000, 40, 96
    idx = torch.randint(0, M, (N,), generator=g, dtype=torch.int32)
    base = torch.randn(N, H + 3, generator=g).to(torch.bfloat16)
    w = torch.rand(N, generator=g)
    padded = _case(idx, base[:, :H], M, w, torch.bfloat16)  # ldx = 99 elements: scalar loads
    dense = _case(idx, base[:, :H].contiguous(), M, w, torch.bfloat16)
    a = np_bits(gpu_scatter(padded)[0])
    b = np_bits(gpu_scatter(dense)[0])
    assert_bytes_equal(a, b, "padded vs dense")
    assert_bytes_equal(a, oracle_scatter(dense), "vs oracle")
    # padded output rows: columns beyond H untouched
    out = torch.full((M, H + 5), 3.0, dtype=torch.bfloat16, device=DEV)[:, :H]
    gpu_scatter(dense, out=out)
    full = out.as_strided((M, H + 5), (H + 5, 1))
    assert torch.all(full[:, H:] == 3.0)
    assert_bytes_equal(np_bits(out), b, "padded out")


def test_no_fused_multiply_add_on_gpu():
    """Same construction as the oracle pin: a fused multiply-add would give 2^-24."""
    xs = torch.tensor([[1.0 + 2.0 ** -7] * 8, [-(1.0 + 2.0 ** -7)] * 8]).to(torch.bfloat16)
    w = torch.tensor([1.0 + 2.0 ** -17] * 2)
    case = _case([0, 0], xs, 1, w, src_id=torch.tensor([1, 0], dtype=torch.int64))
    out = np_bits(gpu_scatter(case)[0])
    assert np.all(out.view(np.uint32) == 0)


def test_scatter_argument_errors():
    case = small_case("tiny_moe")
    plan = dr.det_reduce_plan(case.idx, case.M)
    out = torch.empty(case.M, case.H, device=DEV)
    with pytest.raises(dr.DetError) as e:  # out aliases x
        dr.det_scatter_reduce(plan, case.x, case.x[:case.M], w=case.w)
    assert e.value.code == dr.DET_ERR_ARG
    with pytest.raises(dr.DetError) as e:  # shards do not add up to N
        dr.det_scatter_reduce(plan, [case.x[:10]], out, w=case.w)
    assert e.value.code == dr.DET_ERR_ARG


# --------------------------------------------------------------------------
# split-K
# --------------------------------------------------------------------------

@pytest.mark.parametrize("size", ["small", "full"])
@pytest.mark.parametrize("odt", [torch.float32, torch.bfloat16])
def test_splitk_matches_oracle(size, odt):
    P = wl.make("splitk", size, device=DEV)
    out = torch.empty(P.shape[1], dtype=odt, device=DEV)
    dr.det_splitk_reduce(P, out)
    want = oracle.splitk_reduce(P.cpu().numpy(), out_dtype=oracle.F32 if odt == torch.float32 else oracle.BF16)
    assert_bytes_equal(np_bits(out), want, f"splitk {size} {odt}")
    for grid in (1, 7, sms(), 5 * sms()):
        o2 = torch.empty_like(out)
        dr.det_splitk_reduce(P, o2, opts={"grid_ctas": grid})
        assert_bytes_equal(np_bits(o2), want, f"grid {grid}")


@pytest.mark.parametrize("S", [0, 1, 2, 31, 32, 33, 56, 64, 65, 100, 257, 1000, 4000])
def test_splitk_split_counts(S):
    g = torch.Generator().manual_seed(S)
    count = 4 * 37
    P = (torch.randn(S, count, generator=g) * torch.exp2(torch.rand(S, count, generator=g) * 16 - 8))
    want = oracle.splitk_reduce(P.numpy()) if S > 0 else np.zeros(count, np.float32)
    out = torch.empty(count, device=DEV)
    dr.det_splitk_reduce(P.to(DEV), out)
    assert_bytes_equal(np_bits(out), want, f"S={S}")
    # unaligned count / stride: scalar path
    P2 = P[:, :count - 1].to(DEV)
    o2 = torch.empty(count - 1, device=DEV)
    dr.det_splitk_reduce(P2, o2)
    assert_bytes_equal(np_bits(o2), want[:count - 1], f"S={S} scalar")


# --------------------------------------------------------------------------
# fingerprint
# --------------------------------------------------------------------------

@pytest.mark.parametrize("nbytes", [0, 1, 7, 8, 9, 15, 16, 17, 31, 33, 1000, 4096, 65537, 10_000_019])
def test_hash_matches_oracle(nbytes):
    g = torch.Generator().manual_seed(nbytes)
    buf = torch.randint(0, 256, (nbytes + 16,), generator=g, dtype=torch.uint8)
    dbuf = buf.to(DEV)
    for off in (0, 1, 3, 8, 12):
        got = dr.det_hash(dbuf, nbytes=nbytes, byte_offset=off).item() & (2 ** 64 - 1)
        want = oracle.hash_bytes(buf[off:off + nbytes].numpy())
        assert got == want, (nbytes, off)


# --------------------------------------------------------------------------
# the atomic baseline: close to the exact sum, and (on hot keys) not repeatable
# --------------------------------------------------------------------------

def test_atomic_baseline_close_to_oracle():
    case = small_case("sparse_key_scatter")
    out = torch.empty(case.M, case.H, device=DEV)
    dr.det_atomic_scatter_reduce(case.idx, case.M, case.x, out, w=case.w, opts={"debug_checks": 1})
    want = oracle_scatter(case).astype(np.float64)
    counts = np.bincount(case.idx.cpu().numpy(), minlength=case.M)[:, None]
    xs = np.abs(np_bits(case.x.float()).astype(np.float64))
    absum = np.zeros((case.M, case.H))
    np.add.at(absum, case.idx.cpu().numpy(), xs)
    bound = 2 * (counts + 1) * 2.0 ** -24 * absum + 1e-30
    assert np.all(np.abs(np_bits(out).astype(np.float64) - want) <= bound)


def test_atomic_baseline_bf16_and_index_errors():
    case = small_case("moe_combine")
    out = torch.empty(case.M, case.H, dtype=torch.bfloat16, device=DEV)
    dr.det_atomic_scatter_reduce(case.idx, case.M, case.x, out, w=case.w)
    want = oracle.bf16_to_f32(oracle_scatter(case)).astype(np.float64)
    got = np_bits(out.float()).astype(np.float64)
    assert np.all(np.abs(got - want) <= 2.0 ** -7 * np.abs(want) + 1e-6)
    bad = case.idx.clone()
    bad[3] = case.M + 5
    with pytest.raises(dr.DetError) as e:
        dr.det_atomic_scatter_reduce(bad, case.M, case.x, out, w=case.w, opts={"debug_checks": 1})
    assert e.value.code == dr.DET_ERR_INDEX_RANGE


def test_atomic_negative_control_differs_across_replays(replay):
    """The pages' negative control: the atomic path on hot keys is not byte-repeatable,
    which shows the replay check is sensitive; the deterministic path on the same
    input is."""
    case = wl.sparse_key_scatter(2048, 512, 8192, 128, device=DEV, seed=77)
    replay.runs = 6
    assert replay.differing(lambda: dr.det_atomic_scatter_reduce(
        case.idx, case.M, case.x, torch.empty(case.M, case.H, device=DEV)), name="atomic") > 0
    plan = dr.det_reduce_plan(case.idx, case.M)
    replay.identical(lambda: dr.det_scatter_reduce(plan, case.x, torch.empty(case.M, case.H, device=DEV)),
                     name="deterministic")


# --------------------------------------------------------------------------
# plan without a host wait: counts read on the device
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", SCATTER_SMALL)
def test_async_plan_same_bytes(name):
    """A plan that does not wait gives the same bytes, on every gather kernel that accepts it."""
    case = small_case(name)
    want = oracle_scatter(case)
    out, plan = gpu_scatter(case, opts={"async_plan": 1})
    assert_bytes_equal(np_bits(out), want, f"{name} async")
    assert plan.describe()["n_units"] == -1
    for path, grid in ((1, 0), (1, 3), (2, 0), (0, sms())):
        out2 = torch.full_like(out, 7.0)
        dr.det_scatter_reduce(plan, case.x, out2, w=case.w, opts={"async_plan": 1, "gather_path": path,
                                                                   "grid_ctas": grid})
        assert_bytes_equal(np_bits(out2), want, f"{name} async path={path} grid={grid}")
    dr.det_plan_status(plan)
    d = plan.describe()
    want_rp, _ = oracle.build_lists(case.idx.cpu().numpy(), case.M)
    assert d["max_row_len"] == int(np.diff(want_rp).max())
    # once the counts are on the host the plan behaves like a waited one
    out3, _ = gpu_scatter(case, plan=plan)
    assert_bytes_equal(np_bits(out3), want, f"{name} after status")


def test_async_plan_full_size():
    case = wl.make("sparse_key_scatter", "full", device=DEV)
    out, plan = gpu_scatter(case, opts={"async_plan": 1})
    dr.det_plan_status(plan)
    assert_bytes_equal(np_bits(out), oracle_scatter(case), "sparse_key_scatter full async")


def test_async_plan_errors_reported_and_nothing_written():
    M, H = 6, 64
    x = torch.randn(4, H, device=DEV)
    for idx, sid, code in (([0, 1, 6, 2], None, dr.DET_ERR_INDEX_RANGE),
                           ([0, -3, 1, 1], None, dr.DET_ERR_INDEX_RANGE),
                           ([1, 1, 0, 2], [4, 4, 1, 2], dr.DET_ERR_ORDER_KEY)):
        it = torch.tensor(idx, dtype=torch.int32, device=DEV)
        st = None if sid is None else torch.tensor(sid, dtype=torch.int64, device=DEV)
        plan = dr.det_reduce_plan(it, M, src_id=st, opts={"async_plan": 1})
        out = torch.full((M, H), 3.5, device=DEV)
        dr.det_scatter_reduce(plan, x, out, opts={"async_plan": 1})
        # index_add through the ring kernel and the register-staged kernel beside it
        dr.det_index_add(plan, x, out, opts={"async_plan": 1, "gather_path": 3})
        with pytest.raises(dr.DetError) as e:
            dr.det_plan_status(plan)
        assert e.value.code == code
        assert bool((out == 3.5).all()), "a failed plan must leave the output untouched"
    # a waited plan reports OK from det_plan_status
    plan = dr.det_reduce_plan(torch.tensor([0, 1], dtype=torch.int32, device=DEV), 2)
    dr.det_plan_status(plan)


# --------------------------------------------------------------------------
# det_index_add: index_add_ semantics, out += canonical sum
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", SCATTER_SMALL + ["embedding_backward"])
def test_index_add_matches_oracle(name):
    case = small_case(name)
    g = torch.Generator(device=DEV).manual_seed(99)
    init = (torch.randn(case.M, case.H, generator=g, device=DEV) * 3).to(case.out_dtype)
    init[case.M - 1] = -0.0  # an empty destination (if any) must keep its bits
    out = init.clone()
    plan = dr.det_reduce_plan(case.idx, case.M, src_id=case.src_id)
    dr.det_index_add(plan, case.x, out, w=case.w)
    idx, x, w, sid = case_np(case)
    want = oracle.scatter_reduce(idx, x, case.M, w=w, src_id=sid, out_dtype=oracle_dtype(case.out_dtype),
                                 out_init=np_bits(init))
    assert_bytes_equal(np_bits(out), want, f"{name} index_add")
    # a second call adds the same sums once more, on any grid and with an unwaited plan
    plan2 = dr.det_reduce_plan(case.idx, case.M, src_id=case.src_id, opts={"async_plan": 1})
    dr.det_index_add(plan2, case.x, out, w=case.w, opts={"async_plan": 1, "grid_ctas": 5})
    dr.det_plan_status(plan2)
    want2 = oracle.scatter_reduce(idx, x, case.M, w=w, src_id=sid, out_dtype=oracle_dtype(case.out_dtype),
                                  out_init=want)
    assert_bytes_equal(np_bits(out), want2, f"{name} index_add twice")


def test_index_add_empty_rows_untouched_and_paths():
    idx = torch.tensor([0, 2, 2, 5], dtype=torch.int32, device=DEV)
    M, H = 8, 16
    x = torch.randn(4, H, device=DEV)
    init = torch.randn(M, H, device=DEV)
    init[0] = -0.0
    init[1] = float("nan")  # untouched rows keep any bit pattern
    init[3] = -0.0
    out = init.clone()
    plan = dr.det_reduce_plan(idx, M)
    dr.det_index_add(plan, x, out)
    untouched = [1, 3, 4, 6, 7]
    assert out[untouched].view(torch.int32).equal(init[untouched].view(torch.int32))
    want = oracle.scatter_reduce(idx.cpu().numpy(), x.cpu().numpy(), M, out_init=init.cpu().numpy())
    assert_bytes_equal(np_bits(out), want, "index_add small")
    with pytest.raises(dr.DetError) as e:
        dr.det_index_add(plan, x, out, opts={"gather_path": 2})
    assert e.value.code == dr.DET_ERR_UNSUPPORTED
    # the TMA-staged ring kernel takes 64-byte rows when asked for (auto keeps them on the register kernel)
    out3 = init.clone()
    dr.det_index_add(plan, x, out3, opts={"gather_path": 3, "debug_checks": 1})
    assert_bytes_equal(np_bits(out3), want, "index_add small, ring kernel")


def _mixed_lengths_idx(M, seed):
    """Destination ids of a mix of row lengths in a shuffled source order: empty
    rows, many of 1..3 terms, some of 4..32 (all one chunk), some of 33..300
    (long rows) and one of 700 (a hot row cut into segments); row 0 is empty."""
    rng = np.random.default_rng(seed)
    u = rng.random(M)
    lens = np.where(u < 0.3, 0, np.where(u < 0.7, 1, np.where(u < 0.85, rng.integers(2, 4, M),
                    np.where(u < 0.97, rng.integers(4, 33, M), rng.integers(33, 301, M)))))
    lens[M // 2] = 700
    lens[0] = 0
    idx = np.repeat(np.arange(M, dtype=np.int32), lens)
    rng.shuffle(idx)
    return idx


@pytest.mark.parametrize("accumulate", [True, False])
@pytest.mark.parametrize("H,xdt,odt,weighted", [(4096, torch.bfloat16, torch.float32, False),
                                                (1000, torch.bfloat16, torch.float32, True),
                                                (520, torch.bfloat16, torch.bfloat16, False),
                                                (300, torch.float32, torch.float32, True),
                                                (264, torch.float32, torch.bfloat16, False)])
def test_index_add_bulk_ring_matches_oracle(H, xdt, odt, weighted, accumulate):
    """The TMA-staged ring kernel for the destinations of at most one chunk
    (gather_path 3, and auto where it applies), with the long and hot rows on
    the register-staged kernel beside it and the finish pass: det_index_add
    (accumulate) and det_scatter_reduce (empty rows written as +0.0) give the
    same bytes as the oracle and as the register-staged kernel alone
    (gather_path 1), for row widths that give one tile or several per
    destination and ragged last tiles, bf16 and fp32 outputs, weights, plans
    that did and did not wait, two shards and a small grid."""
    M = 700
    idx_np = _mixed_lengths_idx(M, seed=H)
    N = idx_np.size
    g = torch.Generator(device=DEV).manual_seed(H)
    x = (torch.randn(N, H, generator=g, device=DEV) * 2).to(xdt)
    w = torch.rand(N, generator=g, device=DEV) if weighted else None
    init = (torch.randn(M, H, generator=g, device=DEV) * 3).to(odt)
    init[0] = float("nan")  # untouched rows keep any bits (index_add); overwritten by the scatter-reduce
    idx = torch.from_numpy(idx_np).to(DEV)
    plan = dr.det_reduce_plan(idx, M)
    d = plan.describe()
    assert d["n_hot_rows"] >= 1
    call = dr.det_index_add if accumulate else dr.det_scatter_reduce
    want = oracle.scatter_reduce(idx_np, np_bits(x), M, w=None if w is None else w.cpu().numpy(),
                                 out_dtype=oracle_dtype(odt), out_init=np_bits(init) if accumulate else None)
    what = f"{'index_add' if accumulate else 'scatter'} H={H}"
    outs = {}
    for path in (0, 1, 3):
        out = init.clone()
        call(plan, x, out, w=w, opts={"gather_path": path, "debug_checks": 1})
        assert_bytes_equal(np_bits(out), want, f"{what} path {path}")
        outs[path] = out
    # a plan that did not wait: the ring kernel reads its unit count on the device
    plan2 = dr.det_reduce_plan(idx, M, opts={"async_plan": 1})
    for path in (0, 3):
        out = init.clone()
        call(plan2, x, out, w=w, opts={"async_plan": 1, "gather_path": path})
        dr.det_plan_status(plan2)
        assert_bytes_equal(np_bits(out), want, f"{what} unwaited plan, path {path}")
    # two shards (the ring kernel when asked for it), and a small grid
    cut = N // 3
    out = init.clone()
    call(plan, [x[:cut], x[cut:]], out, w=w, opts={"gather_path": 3, "grid_ctas": 3, "debug_checks": 1})
    assert_bytes_equal(np_bits(out), want, f"{what} two shards")
    if accumulate:  # the empty destination rows are untouched, bit for bit
        empty = np.setdiff1d(np.arange(M), idx_np)
        assert np_bits(outs[0])[empty].tobytes() == np_bits(init)[empty].tobytes()


def test_index_add_bulk_ring_unsupported_layouts():
    """The ring kernel's 16-byte copies need H a multiple of the quantum and
    16-byte output rows: otherwise gather_path 3 is refused and auto takes the
    register-staged kernel, with the oracle's bytes."""
    M, H = 64, 1028  # bf16 x, fp32 out: the quantum is 8 elements
    idx_np = _mixed_lengths_idx(M, seed=3)
    g = torch.Generator(device=DEV).manual_seed(3)
    x = torch.randn(idx_np.size, H, generator=g, device=DEV).to(torch.bfloat16)
    init = torch.randn(M, H, generator=g, device=DEV)
    plan = dr.det_reduce_plan(torch.from_numpy(idx_np).to(DEV), M)
    out = init.clone()
    with pytest.raises(dr.DetError) as e:
        dr.det_index_add(plan, x, out, opts={"gather_path": 3})
    assert e.value.code == dr.DET_ERR_UNSUPPORTED
    dr.det_index_add(plan, x, out)
    want = oracle.scatter_reduce(idx_np, np_bits(x), M, out_init=np_bits(init))
    assert_bytes_equal(np_bits(out), want, "index_add H=1028")


def test_embedding_backward_index_add():
    """Token-embedding backward (Zipf token ids, hot rows): det_index_add into an
    fp32 gradient, twice, against the oracle; the atomic twin stays within the
    reordering bound."""
    case = small_case("embedding_backward")
    g = torch.Generator(device=DEV).manual_seed(5)
    grad = torch.randn(case.M, case.H, generator=g, device=DEV) * 1e-3
    init = grad.clone()
    plan = dr.det_reduce_plan(case.idx, case.M)
    assert plan.describe()["n_hot_rows"] >= 1
    dr.det_index_add(plan, case.x, grad)
    idx, x, w, sid = case_np(case)
    want = oracle.scatter_reduce(idx, x, case.M, out_init=init.cpu().numpy())
    assert_bytes_equal(np_bits(grad), want, "embedding index_add")
    dr.det_index_add(plan, case.x, grad)
    want2 = oracle.scatter_reduce(idx, x, case.M, out_init=want)
    assert_bytes_equal(np_bits(grad), want2, "embedding index_add twice")
    # the atomic twin adds in scheduler order: close, not bit-equal in general
    ga = init.clone()
    dr.det_atomic_index_add(case.idx, case.M, case.x, ga, opts={"debug_checks": 1})
    counts = np.bincount(idx, minlength=case.M)[:, None]
    absum = np.abs(init.cpu().numpy().astype(np.float64))
    np.add.at(absum, idx, np.abs(np_bits(case.x.float()).astype(np.float64)))
    bound = 2 * (counts + 2) * 2.0 ** -24 * absum + 1e-30
    assert np.all(np.abs(np_bits(ga).astype(np.float64) - want.astype(np.float64)) <= bound)
    with pytest.raises(dr.DetError) as e:
        dr.det_atomic_index_add(case.idx, case.M, case.x, grad.to(torch.bfloat16))
    assert e.value.code == dr.DET_ERR_UNSUPPORTED
