"""Sorted router top-k and the MoE route plan on the GPU vs the CPU oracle, byte for byte.

Everything here is selection and integer work (plus one renormalising
division per weight), so the tolerance is 0: ids, offsets, rows, lists and
weights must have the same bytes as the oracle's, and the combine run on the
route plan must give the oracle's output bits.  Cases cover the MoE shapes
(T=4096/E=128/top-8 and T=16384/E=256/top-8), both plan methods (one cluster
kernel; the destination-list plan over the expert ids), ragged expert counts,
empty experts, repeated choices, long and hot lists (k > 32 and k > 256), the
empty problem, bad ids and replays.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_bytes_equal, np_bits
from invariant_gradient_reduction_gb300 import detreduce as dr
from invariant_gradient_reduction_gb300 import workloads as wl

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


def cluster_route_applies(T, k, E):
    """Mirror of the route cluster kernel's size rule (E <= 256, <= 16 CTAs of <= 8192 slots of whole tokens)."""
    N = T * k
    if T <= 0 or k <= 0 or E > 256 or N > 16 * 8192:
        return False
    c = min(16, max(1, -(-N // 2048)))
    return -(-T // c) * k <= 8192


def distinct_ids(T, k, E, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.argsort(torch.rand(T, E, generator=g), dim=1)[:, :k].to(torch.int32).contiguous()


def repeated_ids(T, k, E, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)


def weights(T, k, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.rand(T, k, generator=g, dtype=torch.float32)


# --------------------------------------------------------------------------
# sorted router top-k
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (4096, 128, 8), (16384, 256, 8), (1000, 33, 5), (300, 1024, 32),
                                   (77, 7, 7), (513, 64, 1), (1, 512, 16), (0, 8, 2)])
@pytest.mark.parametrize("renormalize", [False, True])
def test_router_topk_matches_oracle(T, E, k, renormalize):
    s = wl.router_scores(T, E, seed=T + E + k)
    ids, w = dr.det_router_topk(s.to(DEV), k, renormalize=renormalize)
    want_ids, want_w = oracle.router_topk(s.numpy(), k, renormalize=renormalize)
    assert_bytes_equal(ids.cpu().numpy(), want_ids, "ids")
    assert_bytes_equal(w.cpu().numpy(), want_w, "w")


def test_router_topk_ties_and_special_values():
    """Scores from a small pool with infinities, signed zeros, subnormals and NaN (ids and chosen
    scores compared bit for bit; NaN payloads never pass through an add here)."""
    rng = np.random.default_rng(21)
    pool = np.array([np.nan, -np.nan, np.inf, -np.inf, 0.0, -0.0, 1e-45, -1e-45, 0.25, 0.25, 0.5, -3.0],
                    dtype=np.float32)
    for T, E, k in [(500, 40, 6), (200, 256, 32), (64, 1000, 9)]:
        s = pool[rng.integers(0, pool.size, size=(T, E))]
        ids, w = dr.det_router_topk(torch.from_numpy(s).to(DEV), k)
        want_ids, want_w = oracle.router_topk(s, k)
        assert_bytes_equal(ids.cpu().numpy(), want_ids, "ids")
        assert_bytes_equal(w.cpu().numpy().view(np.uint32), want_w.view(np.uint32), "w")


def test_router_topk_padded_rows_and_ids_only():
    s = wl.router_scores(999, 160, seed=3)
    padded = torch.full((999, 200), 7.0)
    padded[:, :160] = s
    ids, w = dr.det_router_topk(padded.to(DEV)[:, :160], 8, renormalize=True)
    want_ids, want_w = oracle.router_topk(s.numpy(), 8, renormalize=True)
    assert_bytes_equal(ids.cpu().numpy(), want_ids, "ids")
    assert_bytes_equal(w.cpu().numpy(), want_w, "w")
    ids2, none = dr.det_router_topk(s.to(DEV), 8, with_weights=False)
    assert none is None
    assert_bytes_equal(ids2.cpu().numpy(), want_ids, "ids only")


# --------------------------------------------------------------------------
# route plan: dispatch arrays and combine lists
# --------------------------------------------------------------------------

ROUTE_SHAPES = [(64, 2, 8, "distinct"), (4096, 8, 128, "distinct"), (16384, 8, 256, "distinct"),
                (3000, 6, 300, "distinct"), (1000, 40, 64, "distinct"), (100, 300, 512, "distinct"),
                (2049, 3, 5, "repeated"), (5000, 4, 256, "repeated"), (20000, 8, 64, "distinct"),
                (1, 1, 1, "distinct"), (7, 3, 250, "distinct"), (0, 4, 8, "distinct"), (9, 0, 8, "distinct")]


def route_inputs(T, k, E, kind, seed=1):
    ids = distinct_ids(T, k, E, seed) if kind == "distinct" else repeated_ids(T, k, E, seed)
    return ids.reshape(T, k).contiguous(), weights(T, k, seed + 1)


def check_route(T, k, E, ids, w, plan, arrays, what):
    want_off, want_tok, want_w, want_slot = oracle.moe_route(ids.numpy(), E, w.numpy())
    assert_bytes_equal(arrays["expert_offsets"].cpu().numpy().astype(np.int64), want_off, what + " offsets")
    assert_bytes_equal(arrays["row_token"].cpu().numpy(), want_tok, what + " row_token")
    assert_bytes_equal(arrays["row_w"].cpu().numpy(), want_w, what + " row_w")
    assert_bytes_equal(arrays["slot_row"].cpu().numpy(), want_slot, what + " slot_row")
    row_ptr, perm = dr.plan_lists(plan)
    want_rp, want_perm = oracle.build_lists(want_tok, T)
    assert_bytes_equal(row_ptr.cpu().numpy().astype(np.int64), want_rp, what + " row_ptr")
    assert_bytes_equal(perm.cpu().numpy().astype(np.int64), want_perm, what + " perm")
    return want_tok, want_w


@pytest.mark.parametrize("plan_path", [0, 1, 2])
@pytest.mark.parametrize("T,k,E,kind", ROUTE_SHAPES)
def test_route_plan_matches_oracle(T, k, E, kind, plan_path):
    if plan_path == 2 and not cluster_route_applies(T, k, E):
        with pytest.raises(dr.DetError) as e:
            ids, w = route_inputs(T, k, E, kind)
            dr.det_moe_route_plan(ids.to(DEV), E, w.to(DEV), opts={"plan_path": 2})
        assert e.value.code == dr.DET_ERR_UNSUPPORTED
        return
    ids, w = route_inputs(T, k, E, kind)
    plan, arrays = dr.det_moe_route_plan(ids.to(DEV), E, w.to(DEV), opts={"plan_path": plan_path})
    want_tok, _ = check_route(T, k, E, ids, w, plan, arrays, f"path {plan_path}")
    # same work counts as the destination-list plan over row_token
    ref = dr.det_reduce_plan(torch.from_numpy(want_tok).to(DEV), T)
    d, r = plan.describe(), ref.describe()
    for key in ("n_units", "n_segments", "n_hot_rows", "max_row_len"):
        assert d[key] == r[key], key


@pytest.mark.parametrize("g", [3, 4, 6])
@pytest.mark.parametrize("T,k,E", [(50, 300, 512), (40, 1000, 1024), (300, 257, 300)])
def test_route_hot_lists_segment_sizes(T, k, E, g):
    """Lists longer than 32 * 2^g terms become hot segments; every segment size gives the same combine."""
    ids, w = route_inputs(T, k, E, "distinct", seed=g)
    opts = {"seg_chunks_log2": g}
    plan, arrays = dr.det_moe_route_plan(ids.to(DEV), E, w.to(DEV), opts=opts)
    want_tok, want_w = check_route(T, k, E, ids, w, plan, arrays, f"g={g}")
    H = 40
    x = torch.randn(T * k, H, generator=torch.Generator().manual_seed(g))
    out = dr.det_scatter_reduce(plan, x.to(DEV), torch.empty(T, H, device=DEV), w=arrays["row_w"], opts=opts)
    want = oracle.scatter_reduce(want_tok, x.numpy(), T, w=want_w)
    assert_bytes_equal(out.cpu().numpy(), want, f"combine g={g}")


@pytest.mark.parametrize("x_dtype,out_dtype", [(torch.bfloat16, torch.bfloat16), (torch.float32, torch.float32),
                                               (torch.bfloat16, torch.float32)])
@pytest.mark.parametrize("T,k,E,H", [(64, 2, 8, 128), (1000, 8, 128, 712), (3000, 6, 300, 96), (600, 40, 64, 64)])
@pytest.mark.parametrize("async_plan", [0, 1])
def test_route_combine_matches_oracle(T, k, E, H, x_dtype, out_dtype, async_plan):
    """The combine on the route plan gives the oracle's bits, and the bits of the combine on the
    destination-list plan built from row_token."""
    ids, w = route_inputs(T, k, E, "distinct", seed=H)
    opts = {"async_plan": async_plan}
    plan, arrays = dr.det_moe_route_plan(ids.to(DEV), E, w.to(DEV), opts=opts, with_slot_row=False)
    x = torch.randn(T * k, H, generator=torch.Generator().manual_seed(T)).to(x_dtype).to(DEV)
    out = dr.det_scatter_reduce(plan, x, torch.empty(T, H, dtype=out_dtype, device=DEV), w=arrays["row_w"],
                                opts=opts)
    if async_plan:
        dr.det_plan_status(plan)
    _, want_tok, want_w, _ = oracle.moe_route(ids.numpy(), E, w.numpy())
    od = oracle.F32 if out_dtype == torch.float32 else oracle.BF16
    want = oracle.scatter_reduce(want_tok, np_bits(x), T, w=want_w, out_dtype=od)
    assert_bytes_equal(np_bits(out), want, "route combine")
    ref_plan = dr.det_reduce_plan(arrays["row_token"], T)
    ref = dr.det_scatter_reduce(ref_plan, x, torch.empty_like(out), w=arrays["row_w"])
    assert_bytes_equal(np_bits(out), np_bits(ref), "route plan vs destination-list plan")


def test_route_end_to_end_from_scores():
    """scores -> sorted top-k (renormalised) -> route plan -> combine, against the oracle's chain, at the
    MoE combine shape with a narrow row."""
    T, E, k, H = 4096, 128, 8, 256
    s = wl.router_scores(T, E, seed=9)
    ids, w = dr.det_router_topk(s.to(DEV), k, renormalize=True)
    plan, arrays = dr.det_moe_route_plan(ids, E, w)
    x = torch.randn(T * k, H, generator=torch.Generator().manual_seed(10)).to(torch.bfloat16).to(DEV)
    out = dr.det_scatter_reduce(plan, x, torch.empty(T, H, dtype=torch.bfloat16, device=DEV), w=arrays["row_w"])
    o_ids, o_w = oracle.router_topk(s.numpy(), k, renormalize=True)
    _, o_tok, o_roww, _ = oracle.moe_route(o_ids, E, o_w)
    want = oracle.scatter_reduce(o_tok, np_bits(x), T, w=o_roww, out_dtype=oracle.BF16)
    assert_bytes_equal(np_bits(out), want, "end to end")


@pytest.mark.parametrize("plan_path", [1, 2])
@pytest.mark.parametrize("bad", [-1, 128, 1 << 20])
def test_route_rejects_bad_ids(plan_path, bad):
    """An id outside [0, E): the waited plan fails with DET_ERR_INDEX_RANGE and writes no output; the
    unwaited plan reports it from det_plan_status, and the combine on it writes nothing."""
    T, k, E = 1000, 8, 128
    ids, w = route_inputs(T, k, E, "distinct")
    ids[517, 3] = bad
    idd, wd = ids.to(DEV), w.to(DEV)
    sentinel = {"expert_offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=DEV),
                "row_token": torch.full((T * k,), -7, dtype=torch.int32, device=DEV),
                "row_w": torch.full((T * k,), -7.0, device=DEV),
                "slot_row": torch.full((T * k,), -7, dtype=torch.int32, device=DEV)}
    with pytest.raises(dr.DetError) as e:
        dr.det_moe_route_plan(idd, E, wd, opts={"plan_path": plan_path}, out=sentinel)
    assert e.value.code == dr.DET_ERR_INDEX_RANGE
    for name, t in sentinel.items():
        assert bool((t == -7).all()), name
    plan, arrays = dr.det_moe_route_plan(idd, E, wd, opts={"plan_path": plan_path, "async_plan": 1})
    out = torch.full((T, 64), 3.0, device=DEV)
    dr.det_scatter_reduce(plan, torch.randn(T * k, 64, device=DEV), out, w=arrays["row_w"],
                          opts={"async_plan": 1})
    with pytest.raises(dr.DetError) as e:
        dr.det_plan_status(plan)
    assert e.value.code == dr.DET_ERR_INDEX_RANGE
    assert bool((out == 3.0).all())


def test_route_plan_replays_identical(replay):
    """Replays of route plan + combine under contention give identical bytes, on both methods."""
    T, k, E, H = 4096, 8, 128, 512
    ids, w = route_inputs(T, k, E, "distinct", seed=4)
    idd, wd = ids.to(DEV), w.to(DEV)
    x = torch.randn(T * k, H, device=DEV).to(torch.bfloat16)
    outs = []
    for path in (1, 2):
        def run():
            plan, arrays = dr.det_moe_route_plan(idd, E, wd, opts={"plan_path": path, "async_plan": 1})
            o = dr.det_scatter_reduce(plan, x, torch.empty(T, H, dtype=torch.bfloat16, device=DEV),
                                      w=arrays["row_w"], opts={"async_plan": 1})
            dr.det_plan_status(plan)
            return torch.cat([o.view(torch.int16).reshape(-1).to(torch.int32), arrays["row_token"],
                              arrays["slot_row"], arrays["expert_offsets"]])
        outs.append(replay.identical(run, name=f"route path {path}"))
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("T,k,E", [(3000, 8, 128), (100, 1, 1), (5000, 1, 16), (40000, 3, 512)])
def test_route_plan_without_weights(T, k, E):
    """No top-k weights: the dispatch arrays still match the oracle, row_w is not produced, and the
    combine without a multiply gives the oracle's bits."""
    ids, _ = route_inputs(T, k, E, "distinct" if k <= E else "repeated", seed=T + k)
    plan, arrays = dr.det_moe_route_plan(ids.to(DEV), E)
    assert arrays["row_w"] is None
    want_off, want_tok, _, want_slot = oracle.moe_route(ids.numpy(), E)
    assert_bytes_equal(arrays["expert_offsets"].cpu().numpy().astype(np.int64), want_off, "offsets")
    assert_bytes_equal(arrays["row_token"].cpu().numpy(), want_tok, "row_token")
    assert_bytes_equal(arrays["slot_row"].cpu().numpy(), want_slot, "slot_row")
    H = 48
    x = torch.randn(T * k, H, generator=torch.Generator().manual_seed(k)).to(DEV)
    out = dr.det_scatter_reduce(plan, x, torch.empty(T, H, device=DEV))
    assert_bytes_equal(out.cpu().numpy(), oracle.scatter_reduce(want_tok, x.cpu().numpy(), T), "combine")
