"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties one part of the oracle to something it cannot simply repeat:
the pages' BF16 worked example, IEEE single-operation results computed by
numpy, torch's bf16 conversion, an independent recursive formulation of the
tree, exact integer sums, published SplitMix64 outputs, and invariants the
pages require.  A plausible slip in the oracle (a dropped term, a truncating
cast, a fused multiply-add, a different tree shape, a swapped index) fails at
least one of them.
"""
import os
import random

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
f32 = np.float32


def bits32(v) -> int:
    return int(np.array(v, dtype=np.float32).view(np.uint32))


def fadd(a, b):
    """One IEEE binary32 add (numpy single op, round to nearest even)."""
    return f32(f32(a) + f32(b))


# --------------------------------------------------------------------------
# bf16 rounding: the pages' worked example and torch's conversion
# --------------------------------------------------------------------------

def _golden(name):
    vals = {}
    with open(os.path.join(HERE, "golden", name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, hexv, dec = line.split()
            vals[key] = (int(hexv, 16), float(dec))
    return vals


def test_bf16_worked_example(oracle_mod):
    """Ch 09 worked example: (1+x)+x = 1.0 but 1+(x+x) = 1.0078125 in bf16, x = 3*2^-10.

    A bf16 add is a binary32 add of the two widened values rounded once to
    bf16; that equals a correctly rounded bf16 add because 24 >= 2*8 + 2
    (double rounding is innocuous for that ratio).
    """
    g = _golden("bf16_worked_example.txt")
    o = oracle_mod
    x = g["x"][0]
    one = g["one"][0]
    assert o.bf16_to_f32(np.array([x], np.uint16))[0] == g["x"][1]
    assert o.bf16_to_f32(np.array([one], np.uint16))[0] == 1.0

    def bf16_add(a, b):
        fa, fb = o.bf16_to_f32(np.array([a, b], np.uint16))
        return int(o.f32_to_bf16(np.array([fadd(fa, fb)], np.float32))[0])

    assert bf16_add(x, x) == g["x_plus_x"][0]
    order_a = bf16_add(bf16_add(one, x), x)
    order_b = bf16_add(one, bf16_add(x, x))
    assert order_a == g["order_a"][0]
    assert order_b == g["order_b"][0]
    assert o.bf16_to_f32(np.array([order_b], np.uint16))[0] == g["order_b"][1]


def _edge_f32_patterns():
    pats = [0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7F7FFFFF, 0xFF7FFFFF,
            0x7F7F8000, 0x7F7F7FFF, 0x7F7F8001, 0x00000001, 0x80000001, 0x007FFFFF, 0x00008000,
            0x00018000, 0x00010000, 0x3F808000, 0x3F818000, 0x3F807FFF, 0x3F808001, 0x3F80FFFF]
    rng = np.random.default_rng(7)
    hi = rng.integers(0, 1 << 16, size=20000, dtype=np.uint64)
    # exact ties (low half 0x8000) with odd and even kept halves, and neighbours of ties
    for low in (0x8000, 0x7FFF, 0x8001, 0x0000, 0xFFFF):
        pats.extend(((hi << np.uint64(16)) | np.uint64(low)).astype(np.uint32).tolist())
    return np.array(pats, dtype=np.uint32)


def test_rne_cast_matches_torch(oracle_mod):
    """Host fp32->bf16 rounding equals torch's CPU conversion (round to nearest even)."""
    rng = np.random.default_rng(1234)
    rand = rng.integers(0, 1 << 32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    pats = np.concatenate([rand, _edge_f32_patterns()])
    vals = pats.view(np.float32)
    ours = oracle_mod.f32_to_bf16(vals)
    ref = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(vals)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN stays NaN with its sign; the payload is kept only in its high bits.
    back = oracle_mod.bf16_to_f32(ours[nan])
    assert np.all(np.isnan(back))
    assert np.array_equal(np.signbit(back), np.signbit(vals[nan]))


def test_bf16_widen_matches_torch(oracle_mod):
    allp = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.bf16_to_f32(allp)
    ref = torch.from_numpy(allp.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    finite = ~np.isnan(ref)
    assert np.array_equal(ours[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.all(np.isnan(ours[~finite]))


# --------------------------------------------------------------------------
# the fold inside one chunk
# --------------------------------------------------------------------------

def test_chunk_fold_is_sequential_left_to_right(oracle_mod):
    """n <= 32: the canonical sum is the textbook left-to-right binary32 loop."""
    rng = np.random.default_rng(5)
    for n in range(1, 33):
        for _ in range(20):
            p = (rng.standard_normal(n) * np.exp2(rng.uniform(-20, 20, n))).astype(np.float32)
            acc = p[0]
            for v in p[1:]:
                acc = fadd(acc, v)
            assert bits32(oracle_mod.canonical_sum(p)) == bits32(acc)


def test_chunk_fold_order_special_case(oracle_mod):
    """[1, 2^-24 x 31]: left to right every add ties back to 1.0; small-first would give 1 + 2^-19."""
    p = np.array([1.0] + [2.0 ** -24] * 31, dtype=np.float32)
    assert bits32(oracle_mod.canonical_sum(p)) == 0x3F800000
    rev = f32(0.0)
    for v in p[::-1]:
        rev = fadd(rev, v)
    assert bits32(rev) == bits32(1.0 + 2.0 ** -19)  # the test can tell the two orders apart


def test_fold_starts_from_first_term_and_empty_is_positive_zero(oracle_mod):
    """All terms -0.0 give -0.0 (a fold seeded with +0.0 would give +0.0); no terms give +0.0."""
    for n in (1, 5, 32, 33, 64, 100):
        assert bits32(oracle_mod.canonical_sum(np.full(n, -0.0, np.float32))) == 0x80000000
    assert bits32(oracle_mod.canonical_sum(np.zeros(0, np.float32))) == 0x00000000


# --------------------------------------------------------------------------
# the tree over chunk sums
# --------------------------------------------------------------------------

def _terms_with_chunk_sums(chunk_sums, last_len=32):
    """Terms whose chunk folds are exactly the given values: chunk = [c, 0, 0, ...]."""
    out = []
    for i, c in enumerate(chunk_sums):
        ln = 32 if i < len(chunk_sums) - 1 else last_len
        out.extend([c] + [0.0] * (ln - 1))
    return np.array(out, dtype=np.float32)


def test_tree_five_chunks_hand_derived(oracle_mod):
    """Five chunk sums c0 = 1, c1..c4 = 2^-24 (ulp(1) = 2^-23; 2^-24 is half an ulp).

    Level-wise tree:  L1 = [1 + 2^-24 -> 1 (tie to even), 2^-23, 2^-24 (carried)]
                      L2 = [1 + 2^-23, 2^-24 (carried)]
                      L3 = [1 + 2^-23 + 2^-24 -> 1 + 2^-22 (tie to even)]   = 0x3F800002
    Recursive halving ((c0+c1)+c2)+(c3+c4) would give 1 + 2^-23 = 0x3F800001 and
    the sequential sum 1.0 = 0x3F800000, so the three readings are told apart.
    """
    c = [1.0] + [2.0 ** -24] * 4
    p = _terms_with_chunk_sums(c, last_len=7)
    assert bits32(oracle_mod.canonical_sum(p)) == 0x3F800002
    halving = fadd(fadd(fadd(c[0], c[1]), c[2]), fadd(c[3], c[4]))
    seq = fadd(fadd(fadd(fadd(c[0], c[1]), c[2]), c[3]), c[4])
    assert bits32(halving) == 0x3F800001 and bits32(seq) == 0x3F800000


def _node_recursive(cs, t, k):
    """Value of the aligned node covering chunks [k*2^t, min((k+1)*2^t, nc)), top-down."""
    nc = len(cs)
    lo = k << t
    if t == 0:
        return cs[lo]
    right_lo = (2 * k + 1) << (t - 1)
    left = _node_recursive(cs, t - 1, 2 * k)
    if right_lo >= nc:
        return left
    return fadd(left, _node_recursive(cs, t - 1, 2 * k + 1))


def _chunk_sums_sequential(p):
    cs = []
    for lo in range(0, len(p), 32):
        acc = p[lo]
        for v in p[lo + 1:lo + 32]:
            acc = fadd(acc, v)
        cs.append(acc)
    return cs


def test_tree_matches_recursive_definition(oracle_mod):
    """Level-wise tree with odd carry == top-down recursion over aligned power-of-two ranges."""
    rng = np.random.default_rng(11)
    for nc in list(range(1, 70)) + [127, 128, 129, 255, 256, 257, 300]:
        tail = int(rng.integers(1, 33))
        n = (nc - 1) * 32 + tail
        p = (rng.standard_normal(n) * np.exp2(rng.uniform(-30, 30, n))).astype(np.float32)
        cs = _chunk_sums_sequential(p)
        top = max(0, (nc - 1).bit_length())
        expect = _node_recursive(cs, top, 0)
        assert bits32(oracle_mod.canonical_sum(p)) == bits32(expect), nc


def test_tree_is_not_sequential_for_some_inputs(oracle_mod):
    """Order sensitivity: on mixed-magnitude data the tree differs from one long fold."""
    rng = np.random.default_rng(3)
    differs = 0
    for _ in range(50):
        p = (rng.standard_normal(200) * np.exp2(rng.uniform(-12, 12, 200))).astype(np.float32)
        acc = p[0]
        for v in p[1:]:
            acc = fadd(acc, v)
        differs += bits32(oracle_mod.canonical_sum(p)) != bits32(acc)
    assert differs > 0


def _levelwise(vals):
    vals = list(vals)
    while len(vals) > 1:
        nxt = [fadd(vals[2 * k], vals[2 * k + 1]) for k in range(len(vals) // 2)]
        if len(vals) % 2:
            nxt.append(vals[-1])
        vals = nxt
    return vals[0]


def test_tree_node_locality(oracle_mod):
    """Splitting a destination into aligned 2^g-chunk segments and finishing with the same
    level-wise tree over the segment values gives the same bits (the hot-destination split)."""
    rng = np.random.default_rng(17)
    for nc in (9, 16, 17, 33, 100, 512, 515):
        n = (nc - 1) * 32 + int(rng.integers(1, 33))
        p = (rng.standard_normal(n) * np.exp2(rng.uniform(-16, 16, n))).astype(np.float32)
        whole = oracle_mod.canonical_sum(p)
        for g in (0, 1, 2, 3, 4):
            seg = 32 << g
            parts = [oracle_mod.canonical_sum(p[s:s + seg]) for s in range(0, n, seg)]
            assert bits32(_levelwise(parts)) == bits32(whole), (nc, g)


def test_exact_integer_sums(oracle_mod):
    """Small integers: every partial sum is exact, so any order gives the exact integer sum."""
    rng = np.random.default_rng(23)
    for n in (1, 2, 31, 32, 33, 64, 65, 1000, 4097, 16384):
        bound = max(1, (1 << 24) // (n + 1) // 2)
        ints = rng.integers(-bound, bound + 1, size=n)
        p = ints.astype(np.float32)
        assert oracle_mod.canonical_sum(p) == float(int(ints.sum()))
        q = p.copy()
        rng.shuffle(q)
        assert oracle_mod.canonical_sum(q) == float(int(ints.sum()))


def test_power_of_two_terms_exact(oracle_mod):
    """Terms 2^e with a bounded exponent spread sum exactly; the result is the exact value."""
    rng = np.random.default_rng(29)
    for n in (40, 300, 2000):
        e = rng.integers(-10, 10, size=n)
        s = rng.choice([-1.0, 1.0], size=n)
        p = (s * np.exp2(e)).astype(np.float32)
        exact = float(np.sum(p.astype(np.float64)))
        assert oracle_mod.canonical_sum(p) == exact


def test_demo_four_orders(oracle_mod):
    """Ch 09 Demo: 16 mixed-magnitude fp32 values summed four ways (A sequential, B pairwise
    tree, C split-K simulation with 4 blocks then a reduce, D shuffled) can differ by ULPs.
    With 16 <= 32 terms the canonical sum is order A exactly."""
    rng = random.Random(99)
    any_diff = 0
    for _ in range(200):
        v = [f32(rng.gauss(0, 1) * 2.0 ** rng.randint(-12, 12)) for _ in range(16)]
        a = v[0]
        for t in v[1:]:
            a = fadd(a, t)
        b = _levelwise(v)
        blocks = []
        for q in range(4):
            s = v[4 * q]
            for t in v[4 * q + 1:4 * q + 4]:
                s = fadd(s, t)
            blocks.append(s)
        c = blocks[0]
        for s in blocks[1:]:
            c = fadd(c, s)
        w = v[:]
        rng.shuffle(w)
        d = w[0]
        for t in w[1:]:
            d = fadd(d, t)
        any_diff += len({bits32(a), bits32(b), bits32(c), bits32(d)}) > 1
        assert bits32(oracle_mod.canonical_sum(np.array(v, np.float32))) == bits32(a)
    assert any_diff > 0


# --------------------------------------------------------------------------
# products, the multiply/add split, the scatter definition
# --------------------------------------------------------------------------

def test_product_is_single_rounded_multiply(oracle_mod):
    """One term per destination: out = fl32(w * x) for fp32 and bf16 x; bf16 out = RNE of it."""
    rng = np.random.default_rng(31)
    M, H = 50, 24
    idx = np.arange(M, dtype=np.int32)
    w = rng.standard_normal(M).astype(np.float32)
    x = rng.standard_normal((M, H)).astype(np.float32)
    out = oracle_mod.scatter_reduce(idx, x, M, w=w)
    assert np.array_equal(out.view(np.uint32), (w[:, None] * x).astype(np.float32).view(np.uint32))
    xb = oracle_mod.f32_to_bf16(x)
    out_b = oracle_mod.scatter_reduce(idx, xb, M, w=w, out_dtype=oracle_mod.BF16)
    xw = oracle_mod.bf16_to_f32(xb)
    ref = torch.from_numpy(w[:, None] * xw).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out_b, ref)


def test_no_fused_multiply_add(oracle_mod):
    """Terms p0 = -(1 + 2^-7 + 2^-17) and p1 = (1 + 2^-17) * (1 + 2^-7) (bf16 x).

    The exact product is 1 + 2^-7 + 2^-17 + 2^-24; rounded to binary32 it loses the
    2^-24 (a tie, kept part even), so p0 + p1 = 0.  A fused multiply-add would
    return 2^-24.
    """
    o = oracle_mod
    xs = np.array([[1.0 + 2.0 ** -7], [-(1.0 + 2.0 ** -7)]], dtype=np.float32)  # exact in bf16
    w = np.array([1.0 + 2.0 ** -17, 1.0 + 2.0 ** -17], dtype=np.float32)
    idx = np.array([0, 0], dtype=np.int32)
    # order: row 1 (negative) first via src_id
    out = o.scatter_reduce(idx, o.f32_to_bf16(xs), 1, w=w, src_id=np.array([1, 0], np.int64))
    assert bits32(out[0, 0]) == 0
    p0 = float(f32(w[1] * xs[1, 0]))                       # first term, rounded
    fused = float(np.float64(w[0]) * np.float64(xs[0, 0]) + p0)  # exact product + p0: one rounding
    assert p0 == -(1.0 + 2.0 ** -7 + 2.0 ** -17)
    assert fused == 2.0 ** -24


def test_scatter_within_error_bound_of_exact_sum(oracle_mod):
    """|out - exact| <= n * 2^-24 * sum|p| per element (a backward-error bound on any order),
    plus the rounding of the product; a dropped term, sign slip or transposed index fails it."""
    rng = np.random.default_rng(37)
    N, M, H = 3000, 97, 40
    idx = rng.integers(0, M, N).astype(np.int32)
    x = rng.standard_normal((N, H)).astype(np.float32)
    w = rng.uniform(0.1, 1.0, N).astype(np.float32)
    out = oracle_mod.scatter_reduce(idx, x, M, w=w).astype(np.float64)
    prod = w[:, None].astype(np.float64) * x.astype(np.float64)
    exact = np.zeros((M, H))
    absum = np.zeros((M, H))
    np.add.at(exact, idx, prod)
    np.add.at(absum, idx, np.abs(prod))
    cnt = np.bincount(idx, minlength=M)[:, None]
    bound = (cnt + 1) * 2.0 ** -24 * absum + 1e-300
    assert np.all(np.abs(out - exact) <= bound)
    # the bound is tight enough to catch a dropped term
    assert np.any(np.abs(prod[idx == 0][0]) > bound[0])


def test_csr_matches_stable_argsort(oracle_mod):
    rng = np.random.default_rng(41)
    for N, M in ((0, 5), (1, 1), (100, 7), (5000, 300), (20000, 1)):
        idx = rng.integers(0, M, N).astype(np.int32)
        rp, perm = oracle_mod.build_lists(idx, M)
        assert np.array_equal(perm, np.argsort(idx, kind="stable"))
        assert np.array_equal(rp, np.concatenate([[0], np.cumsum(np.bincount(idx, minlength=M))]))
        sid = rng.permutation(N).astype(np.int64) * 3 - 7
        rp2, perm2 = oracle_mod.build_lists(idx, M, src_id=sid)
        assert np.array_equal(perm2, np.lexsort((sid, idx)))
        assert np.array_equal(rp2, rp)


def test_csr_rejects_bad_index_and_duplicate_keys(oracle_mod):
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.build_lists(np.array([0, 3], np.int32), 3)
    assert e.value.code == -2
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.build_lists(np.array([1, 1], np.int32), 3, src_id=np.array([5, 5], np.int64))
    assert e.value.code == -3
    # equal keys in different destinations are fine
    oracle_mod.build_lists(np.array([0, 1], np.int32), 3, src_id=np.array([5, 5], np.int64))


# --------------------------------------------------------------------------
# invariants the pages require
# --------------------------------------------------------------------------

def _random_case(rng, N=4000, M=53, H=33):
    idx = rng.integers(0, M, N).astype(np.int32)
    x = oracle_mod_bf16(rng.standard_normal((N, H)).astype(np.float32))
    w = rng.uniform(0.0, 1.0, N).astype(np.float32)
    return idx, x, w


def oracle_mod_bf16(a):
    import oracle
    return oracle.f32_to_bf16(a)


def test_invariant_to_physical_row_permutation(oracle_mod):
    """Permuting the physical rows while keeping each row's order key gives the same bytes."""
    rng = np.random.default_rng(43)
    idx, x, w = _random_case(rng)
    base = oracle_mod.scatter_reduce(idx, x, 53, w=w, out_dtype=oracle_mod.BF16)
    for _ in range(3):
        pr = rng.permutation(len(idx))
        out = oracle_mod.scatter_reduce(idx[pr], x[pr], 53, w=w[pr], out_dtype=oracle_mod.BF16,
                                        src_id=pr.astype(np.int64))
        assert out.tobytes() == base.tobytes()


def test_batch_invariance(oracle_mod):
    """A token's output row is the same bits alone, in a small batch and in a large one,
    at any position, as long as its own terms keep their relative order (Ch 09, property A)."""
    rng = np.random.default_rng(47)
    H = 64
    k = 8
    tok_rows = rng.standard_normal((k, H)).astype(np.float32)
    tok_w = rng.uniform(0, 1, k).astype(np.float32)
    alone = oracle_mod.scatter_reduce(np.zeros(k, np.int32), tok_rows, 1, w=tok_w)[0]
    for T in (2, 17, 300):
        pos = int(rng.integers(0, T))
        other_idx = rng.integers(0, T, size=k * T).astype(np.int32)
        other_idx[other_idx == pos] = (pos + 1) % T
        other = rng.standard_normal((k * T, H)).astype(np.float32)
        ow = rng.uniform(0, 1, k * T).astype(np.float32)
        slots = np.sort(rng.choice(k * T + k, size=k, replace=False))
        N = k * T + k
        idx = np.empty(N, np.int32)
        x = np.empty((N, H), np.float32)
        w = np.empty(N, np.float32)
        mask = np.zeros(N, bool)
        mask[slots] = True
        idx[mask], x[mask], w[mask] = pos, tok_rows, tok_w
        idx[~mask], x[~mask], w[~mask] = other_idx, other, ow
        out = oracle_mod.scatter_reduce(idx, x, T, w=w)
        assert out[pos].tobytes() == alone.tobytes()


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_invariant_to_shard_split(oracle_mod, P):
    """Splitting the sources into P shards (separate buffers) gives identical bytes (EP-size invariance)."""
    rng = np.random.default_rng(53)
    idx, x, w = _random_case(rng)
    base = oracle_mod.scatter_reduce(idx, x, 53, w=w, out_dtype=oracle_mod.BF16)
    cuts = np.sort(rng.choice(np.arange(1, len(idx)), size=P - 1, replace=False)) if P > 1 else []
    bounds = [0, *list(cuts), len(idx)]
    shards = [x[bounds[q]:bounds[q + 1]].copy() for q in range(P)]
    out = oracle_mod.scatter_reduce(idx, shards, 53, w=w, out_dtype=oracle_mod.BF16)
    assert out.tobytes() == base.tobytes()


# --------------------------------------------------------------------------
# split-K
# --------------------------------------------------------------------------

def test_splitk_56_is_two_chunks(oracle_mod):
    """S = 56: chunk 0 folds s = 0..31, chunk 1 folds s = 32..55, out = c0 + c1."""
    rng = np.random.default_rng(59)
    P = (rng.standard_normal((56, 300)) * np.exp2(rng.uniform(-8, 8, (56, 300)))).astype(np.float32)
    out = oracle_mod.splitk_reduce(P)
    for e in range(300):
        c0 = P[0, e]
        for s in range(1, 32):
            c0 = fadd(c0, P[s, e])
        c1 = P[32, e]
        for s in range(33, 56):
            c1 = fadd(c1, P[s, e])
        assert bits32(out[e]) == bits32(fadd(c0, c1))
    outb = oracle_mod.splitk_reduce(P, out_dtype=oracle_mod.BF16)
    assert np.array_equal(outb, oracle_mod.f32_to_bf16(out))


def test_splitk_matches_recursive_definition(oracle_mod):
    rng = np.random.default_rng(61)
    for S in (1, 2, 31, 32, 33, 64, 65, 97, 200):
        P = (rng.standard_normal((S, 8)) * np.exp2(rng.uniform(-8, 8, (S, 8)))).astype(np.float32)
        out = oracle_mod.splitk_reduce(P)
        for e in range(8):
            cs = _chunk_sums_sequential(P[:, e])
            top = max(0, (len(cs) - 1).bit_length())
            assert bits32(out[e]) == bits32(_node_recursive(cs, top, 0))


# --------------------------------------------------------------------------
# fingerprint
# --------------------------------------------------------------------------

def test_mix_is_splitmix64(oracle_mod):
    """SplitMix64 with seed 0 (state advanced by 0x9E3779B97F4A7C15 before each output)
    yields 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F (published outputs of
    the reference generator)."""
    gamma = 0x9E3779B97F4A7C15
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    got = [oracle_mod.mix64((gamma * (k + 1)) & (2 ** 64 - 1)) for k in range(3)]
    assert got == want


def test_hash_structure(oracle_mod):
    o = oracle_mod
    C0 = 0x6A09E667F3BCC909
    C1 = 0x9E3779B97F4A7C15
    assert o.hash_bytes(b"") == o.mix64(0 ^ C0)
    rng = np.random.default_rng(67)
    a = rng.integers(0, 256, size=803, dtype=np.uint8)
    ha = o.hash_bytes(a)
    # changing one word changes the hash by exactly the difference of that word's term
    b = a.copy()
    b[8 * 13 + 2] ^= 0x5A
    wa = int(a[104:112].view("<u8")[0])
    wb = int(b[104:112].view("<u8")[0])
    diff = (o.mix64(wb ^ (13 * C1 % 2 ** 64)) - o.mix64(wa ^ (13 * C1 % 2 ** 64))) % 2 ** 64
    assert (o.hash_bytes(b) - ha) % 2 ** 64 == diff
    # the padded tail is little-endian with zero fill: a trailing zero byte still changes nbytes
    assert o.hash_bytes(np.concatenate([a, [0]]).astype(np.uint8)) != ha
    # swapping two words changes the hash
    c = a.copy()
    c[0:8], c[8:16] = a[8:16], a[0:8]
    assert o.hash_bytes(c) != ha
    # byte order inside a word: bytes b0..b7 form the word sum b_k 256^k
    one = np.array([1, 0, 0, 0, 0, 0, 0, 0], np.uint8)
    assert o.hash_bytes(one) == (o.mix64(8 ^ C0) + o.mix64(1)) % 2 ** 64


# --------------------------------------------------------------------------
# index_add_ semantics (Megatron-LM determinism developer reference, section
# 3.1 op catalog: index_add_ replaces the atomic scatter_add_)
# --------------------------------------------------------------------------

def test_index_add_exact_integers(oracle_mod):
    """Small integers: every add is exact, so the result is the integer sum
    out_init + sum of terms, and destinations without terms keep their bits."""
    rng = np.random.default_rng(11)
    N, M, H = 500, 40, 6
    idx = rng.integers(0, M - 5, size=N).astype(np.int32)  # the last 5 destinations get no term
    x = rng.integers(-8, 9, size=(N, H)).astype(np.float32)
    w = rng.integers(-3, 4, size=N).astype(np.float32)
    init = rng.integers(-1000, 1001, size=(M, H)).astype(np.float32)
    init[-1, 0] = -0.0
    init[-2, 1] = np.float32(np.nan)
    got = oracle_mod.scatter_reduce(idx, x, M, w=w, out_init=init)
    want = init.astype(np.float64).copy()
    for i in range(N):
        want[idx[i]] += float(w[i]) * x[i]
    touched = np.zeros(M, bool)
    touched[idx] = True
    assert np.array_equal(got[touched], want[touched].astype(np.float32))
    assert got[~touched].tobytes() == init[~touched].tobytes()  # -0.0 and the NaN pattern kept


def test_index_add_is_one_add_of_the_canonical_sum(oracle_mod):
    """From +0.0 it equals the plain scatter-reduce on touched destinations; a
    second call adds the same canonical sums once more (x + S, not a refold)."""
    rng = np.random.default_rng(12)
    N, M, H = 700, 9, 5
    idx = rng.integers(0, M, size=N).astype(np.int32)
    x = (rng.standard_normal((N, H)) * 2.0 ** rng.integers(-8, 8, size=(N, 1))).astype(np.float32)
    S = oracle_mod.scatter_reduce(idx, x, M)
    zero = np.zeros((M, H), np.float32)
    first = oracle_mod.scatter_reduce(idx, x, M, out_init=zero)
    assert first.tobytes() == S.tobytes()
    second = oracle_mod.scatter_reduce(idx, x, M, out_init=first)
    assert second.tobytes() == (S + S).astype(np.float32).tobytes()  # numpy float32 add: one rounding
    refold = oracle_mod.scatter_reduce(np.concatenate([idx, idx]), np.concatenate([x, x]), M)
    assert not np.array_equal(second, refold)  # folding 2N terms is a different order


def test_index_add_bf16_out_rounds_once(oracle_mod):
    """bf16 out: the old value widens exactly, the binary32 add rounds, then one
    RNE cast to bf16; checked against torch's CPU bf16 conversion."""
    rng = np.random.default_rng(13)
    N, M, H = 300, 7, 4
    idx = rng.integers(0, M, size=N).astype(np.int32)
    x = rng.standard_normal((N, H)).astype(np.float32)
    init_f = rng.standard_normal((M, H)).astype(np.float32) * 100
    init_b = torch.from_numpy(init_f).to(torch.bfloat16)
    init_bits = init_b.view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.scatter_reduce(idx, x, M, out_dtype=oracle_mod.BF16, out_init=init_bits)
    S = oracle_mod.scatter_reduce(idx, x, M)
    want = (torch.from_numpy(init_b.float().numpy() + S)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert got.tobytes() == want.tobytes()


# --------------------------------------------------------------------------
# sorted router top-k and the MoE dispatch layout
# --------------------------------------------------------------------------

def _golden_cases(name):
    """Blocks of `key value...` lines; `case <name>` starts a new block."""
    cases, cur = [], {}
    with open(os.path.join(HERE, "golden", name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
                cases.append(cur)
            else:
                cur[key] = vals
    return cases or [cur]


def _hexf(vals):
    return np.array([int(v, 16) for v in vals], dtype=np.uint32).view(np.float32)


@pytest.mark.parametrize("case", _golden_cases("router_topk_hand.txt"), ids=lambda c: c["name"])
def test_router_topk_hand_cases(oracle_mod, case):
    """Hand-derived order, tie and renormalisation cases (totalOrder, lower id first, left-to-right sum)."""
    s = _hexf(case["scores"]).reshape(1, -1)
    k = int(case["k"][0])
    ids, w = oracle_mod.router_topk(s, k, renormalize=case["renormalize"][0] == "1")
    assert ids.reshape(-1).tolist() == [int(v) for v in case["ids"]]
    assert w.reshape(-1).view(np.uint32).tolist() == _hexf(case["w"]).view(np.uint32).tolist()


def test_router_topk_is_torch_stable_sort(oracle_mod):
    """Without signed zeros and NaN, totalOrder is the numeric order: the selection is the head of
    torch's stable descending sort (equal scores keep ascending expert order), also checked with
    Python's sorted().  Scores come from a small set so that ties are everywhere."""
    rng = np.random.default_rng(11)
    for T, E, k in [(64, 8, 2), (200, 128, 8), (33, 256, 8), (5, 7, 7), (40, 96, 1)]:
        s = (rng.integers(-12, 13, size=(T, E)).astype(np.float32) / f32(8))
        s[rng.random((T, E)) < 0.05] = np.inf
        s[rng.random((T, E)) < 0.05] = -np.inf
        s[s == 0] = f32(0.0)  # +0.0 only
        ids, w = oracle_mod.router_topk(s, k)
        ref = torch.sort(torch.from_numpy(s), dim=1, descending=True, stable=True).indices[:, :k].numpy()
        assert np.array_equal(ids, ref.astype(np.int32))
        for t in range(0, T, 7):
            order = sorted(range(E), key=lambda e: (-float(s[t, e]), e))[:k]
            assert ids[t].tolist() == order
        assert np.array_equal(w.view(np.uint32), np.take_along_axis(s, ids.astype(np.int64), 1).view(np.uint32))


def test_router_topk_renormalise_exact_sums(oracle_mod):
    """Dyadic scores with few bits: the binary32 sum is exact, so each weight is the correctly
    rounded quotient, which a binary64 quotient rounded once to binary32 gives (double rounding is
    innocuous for division when 53 >= 2*24 + 2)."""
    rng = np.random.default_rng(12)
    s = rng.integers(1, 256, size=(300, 64)).astype(np.float32) * f32(2.0 ** -10)
    ids, w = oracle_mod.router_topk(s, 8, renormalize=True)
    top = np.take_along_axis(s, ids.astype(np.int64), 1).astype(np.float64)
    expect = (top / top.sum(axis=1, keepdims=True)).astype(np.float32)
    assert np.array_equal(w.view(np.uint32), expect.view(np.uint32))
    # general inputs: the weights sum to 1 within a few ulp
    s = rng.random((300, 64), dtype=np.float32)
    _, w = oracle_mod.router_topk(s, 8, renormalize=True)
    assert np.all(np.abs(w.astype(np.float64).sum(axis=1) - 1.0) < 8 * 2.0 ** -24 * 8)


def test_router_topk_special_values_dominate(oracle_mod):
    """With NaN, infinities, signed zeros and subnormals mixed in: the list is strictly decreasing in
    (totalOrder key, -expert), and every chosen key beats every unchosen one.  The key here is built
    from the sign and magnitude bits by comparisons, not by the oracle's bit trick."""
    rng = np.random.default_rng(13)
    T, E, k = 64, 40, 6
    pool = np.array([np.nan, -np.nan, np.inf, -np.inf, 0.0, -0.0, 1e-45, -1e-45, 1.0, -1.0, 0.5, 3.0],
                    dtype=np.float32)
    s = pool[rng.integers(0, pool.size, size=(T, E))]
    ids, _ = oracle_mod.router_topk(s, k)
    u = s.view(np.uint32).astype(np.int64)
    neg = u >= 2 ** 31
    mag = u & 0x7FFFFFFF
    key = np.where(neg, -mag - 1, mag)  # negatives below positives, larger magnitude lower
    for t in range(T):
        chosen = [(key[t, e], -e) for e in ids[t]]
        assert chosen == sorted(chosen, reverse=True) and len(set(ids[t])) == k
        rest = [(key[t, e], -e) for e in range(E) if e not in set(ids[t].tolist())]
        assert min(chosen) > max(rest)


def test_moe_route_hand_example(oracle_mod):
    """The hand-derived T=3, k=2, E=6 layout (two experts without tokens) and its combine lists."""
    g = _golden_cases("moe_route_hand.txt")[0]
    T, k, E = int(g["T"][0]), int(g["k"][0]), int(g["E"][0])
    ids = np.array([int(v) for v in g["ids"]], np.int32).reshape(T, k)
    w = np.array([float(v) for v in g["w"]], np.float32).reshape(T, k)
    off, row_token, row_w, slot_row = oracle_mod.moe_route(ids, E, w)
    assert off.tolist() == [int(v) for v in g["expert_offsets"]]
    assert row_token.tolist() == [int(v) for v in g["row_token"]]
    assert slot_row.tolist() == [int(v) for v in g["slot_row"]]
    row_slot = [int(v) for v in g["row_slot"]]
    assert np.array_equal(row_w.view(np.uint32), w.reshape(-1)[row_slot].view(np.uint32))
    row_ptr, perm = oracle_mod.build_lists(row_token, T)
    assert row_ptr.tolist() == [int(v) for v in g["combine_row_ptr"]]
    assert perm.tolist() == [int(v) for v in g["combine_perm"]]


def test_moe_route_rank_formula(oracle_mod):
    """Row of slot i = (slots with a lower expert) + (earlier slots with the same expert), computed
    all-pairs; for distinct choices per token it is also the rank of the key e*T + t, the (expert id,
    token id) order the workload generator uses."""
    rng = np.random.default_rng(14)
    for T, k, E, distinct in [(64, 2, 8, True), (50, 8, 16, True), (40, 3, 5, False), (1, 4, 4, True),
                              (7, 1, 300, True)]:
        if distinct:
            ids = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
        else:
            ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
        w = rng.random((T, k), dtype=np.float32)
        off, row_token, row_w, slot_row = oracle_mod.moe_route(ids, E, w)
        f = ids.reshape(-1).astype(np.int64)
        N = f.size
        lower = (f[None, :] < f[:, None]).sum(axis=1)
        same_before = np.tril(f[None, :] == f[:, None], k=-1).sum(axis=1)
        assert np.array_equal(slot_row, (lower + same_before).astype(np.int32))
        assert np.array_equal(off, np.array([(f < e).sum() for e in range(E + 1)]))
        assert sorted(slot_row.tolist()) == list(range(N))
        inv = np.empty(N, np.int64)
        inv[slot_row] = np.arange(N)
        assert np.array_equal(row_token, (inv // k).astype(np.int32))
        assert np.array_equal(row_w.view(np.uint32), w.reshape(-1)[inv].view(np.uint32))
        if distinct:
            t = np.repeat(np.arange(T), k)
            assert np.array_equal(inv, np.argsort(f * T + t, kind="stable"))


def test_moe_route_rejects_bad_ids(oracle_mod):
    for bad in (-1, 6):
        ids = np.array([[0, 1], [2, bad]], np.int32)
        with pytest.raises(oracle_mod.OracleError) as ei:
            oracle_mod.moe_route(ids, 6)
        assert ei.value.code == -2


# --------------------------------------------------------------------------
# split-K GEMM partials (the producer of the split-K reduce)
# --------------------------------------------------------------------------

def _bf16_ints(oracle, rng, shape, lo=-4, hi=5):
    return oracle.f32_to_bf16(rng.integers(lo, hi, size=shape).astype(np.float32))


def test_splitk_gemm_partials_brute_force(oracle_mod):
    oracle = oracle_mod
    """Each partial is the plain triple loop over its own K slice (rows of A
    against rows of W), on tiny shapes with non-integer values."""
    rng = np.random.default_rng(41)
    for R, C, K, S in [(3, 2, 8, 2), (1, 1, 4, 4), (5, 3, 12, 3)]:
        a = oracle.f32_to_bf16(rng.normal(size=(R, K)).astype(np.float32))
        w = oracle.f32_to_bf16(rng.normal(size=(C, K)).astype(np.float32))
        got = oracle.splitk_gemm_partials(a, w, S)
        af = oracle.bf16_to_f32(a).astype(np.float64)
        wf = oracle.bf16_to_f32(w).astype(np.float64)
        ks = K // S
        for s in range(S):
            for r in range(R):
                for c in range(C):
                    v = 0.0
                    for k in range(s * ks, (s + 1) * ks):
                        v += af[r, k] * wf[c, k]
                    assert got[s, r, c] == v


def test_splitk_gemm_partials_sum_to_the_whole_product(oracle_mod):
    oracle = oracle_mod
    """Small integers: every partial and the whole product are exact, and the
    partials add up to A @ W.T (a dropped or doubled K slice would not)."""
    rng = np.random.default_rng(42)
    a = _bf16_ints(oracle, rng, (7, 96))
    w = _bf16_ints(oracle, rng, (5, 96))
    p = oracle.splitk_gemm_partials(a, w, 6)
    whole = oracle.bf16_to_f32(a).astype(np.float64) @ oracle.bf16_to_f32(w).astype(np.float64).T
    assert p.shape == (6, 7, 5)
    assert np.array_equal(p.sum(axis=0), whole)
    # each split really is its own slice: zeroing one slice of A zeroes exactly that partial
    a2 = a.copy()
    a2[:, 16:32] = 0
    p2 = oracle.splitk_gemm_partials(a2, w, 6)
    assert np.all(p2[1] == 0) and np.array_equal(np.delete(p2, 1, 0), np.delete(p, 1, 0))


def test_splitk_gemm_partials_orientation(oracle_mod):
    oracle = oracle_mod
    """W is [C, K] (the transposed right operand): a [K, C] array of the same
    values gives other numbers or is rejected."""
    rng = np.random.default_rng(43)
    a = _bf16_ints(oracle, rng, (4, 6))
    w = _bf16_ints(oracle, rng, (6, 6))  # square, so a transposed W is accepted but differs
    p = oracle.splitk_gemm_partials(a, w, 2)
    pt = oracle.splitk_gemm_partials(a, np.ascontiguousarray(w.T), 2)
    assert not np.array_equal(p, pt)
    with pytest.raises(ValueError):
        oracle.splitk_gemm_partials(a, w, 4)  # K = 6 is not a multiple of 4
