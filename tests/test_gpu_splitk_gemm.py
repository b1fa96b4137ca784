"""Split-K GEMM with the fold over split ids in its epilogue (det_splitk_gemm_reduce).

Two checks pin it: (1) each split's partial, which the call can also write
out, against a binary64 GEMM of the same split (exactly, for small-integer
inputs, whose every partial is exact in binary32; within the binary32
rounding bound for normal inputs); (2) the output, byte for byte, against
the oracle's canonical fold of those partials, and against det_splitk_reduce
over them.  Every output is also the same bits with and without writing the
partials, and from run to run.
"""
import numpy as np
import pytest
import torch

import oracle
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


def _bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _run(A, W, S, out_dtype=torch.float32, dump=True, opts=None):
    R, C = A.shape[0], W.shape[0]
    out = torch.full((R, C), 7.0, dtype=out_dtype, device=DEV)
    P = torch.full((S, R * C), 9.0, device=DEV) if dump else None
    dr.det_splitk_gemm_reduce(A, W, S, out, partials=P, opts=opts or {"debug_checks": 1})
    return out, P


def _fold_bytes(P, R, C, out_dtype):
    od = oracle.F32 if out_dtype == torch.float32 else oracle.BF16
    return oracle.splitk_reduce(P.cpu().numpy()[:, :R * C], od).tobytes()


def _out_bytes(out):
    t = out.detach().cpu().contiguous()
    return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t).numpy().tobytes()


@pytest.mark.parametrize("R,K,C,S", [(128, 64, 8, 1), (128, 128, 24, 2), (200, 256, 24, 4), (1, 64, 1, 1),
                                     (129, 64 * 33, 32, 33), (300, 64 * 40, 24, 40), (517, 128 * 56, 24, 56)])
def test_splitk_gemm_partials_exact_on_integers(R, K, C, S):
    """Small-integer inputs: every product and every partial sum is an integer
    below 2^24, exact in binary32 whatever the accumulation order, so each
    split's partial must equal the binary64 reference exactly (a wrong K slice,
    row, column or transpose cannot pass)."""
    g = torch.Generator().manual_seed(R * 7 + K + C + S)
    A = torch.randint(-3, 4, (R, K), generator=g).to(torch.bfloat16).to(DEV)
    W = torch.randint(-3, 4, (C, K), generator=g).to(torch.bfloat16).to(DEV)
    out, P = _run(A, W, S)
    want = oracle.splitk_gemm_partials(_bits16(A), _bits16(W), S)
    got = P.cpu().numpy()[:, :R * C].reshape(S, R, C).astype(np.float64)
    assert np.array_equal(got, want)
    assert _out_bytes(out) == _fold_bytes(P, R, C, torch.float32)
    # the exact integer sum, for a fold whose every add is exact
    total = want.sum(axis=0).astype(np.float32)
    assert np.array_equal(out.cpu().numpy(), total)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("R,C,S,ks", [(256, 24, 56, 128), (1000, 24, 56, 128), (384, 32, 100, 64), (130, 5, 7, 64),
                                      (640, 16, 256, 64), (128, 24, 32, 128), (128, 24, 64, 64), (128, 24, 65, 64),
                                      (256, 24, 8, 256), (200, 24, 9, 192), (128, 24, 3, 320)])
def test_splitk_gemm_fold_matches_oracle(R, C, S, ks, out_dtype):
    """Normal inputs: the partials within the binary32 bound of the binary64
    GEMM; the output the oracle's canonical fold of those partials, byte for
    byte; the same bits without writing the partials and on a second run; and
    det_splitk_reduce over the partials gives the same output."""
    K = S * ks
    A, W = wl.splitk_gemm_inputs(R, K, C, seed=R + S, device=DEV)
    out, P = _run(A, W, S, out_dtype)
    want = oracle.splitk_gemm_partials(_bits16(A), _bits16(W), S)
    got = P.cpu().numpy()[:, :R * C].reshape(S, R, C).astype(np.float64)
    a = oracle.bf16_to_f32(_bits16(A)).astype(np.float64)
    w = oracle.bf16_to_f32(_bits16(W)).astype(np.float64)
    mag = np.stack([np.abs(a[:, s * ks:(s + 1) * ks]) @ np.abs(w[:, s * ks:(s + 1) * ks]).T for s in range(S)])
    # binary32 accumulation of ks exact products: |error| <= ks * 2^-24 * sum|a*w| (a loose bound)
    assert np.all(np.abs(got - want) <= ks * 2.0 ** -24 * mag + 1e-30)
    assert _out_bytes(out) == _fold_bytes(P, R, C, out_dtype)
    o2, _ = _run(A, W, S, out_dtype, dump=False)
    o3, _ = _run(A, W, S, out_dtype, dump=False, opts={})
    assert _out_bytes(o2) == _out_bytes(out) and _out_bytes(o3) == _out_bytes(out)
    o4 = torch.empty(R * C, dtype=out_dtype, device=DEV)
    dr.det_splitk_reduce(P[:, :R * C], o4)
    assert _out_bytes(o4) == _out_bytes(out)


def test_splitk_gemm_full_size_mhc_shape():
    """The mHC-like shape: 16384 rows, K = 7168 in 56 splits, 24 columns."""
    R, K, C, S = 16384, 7168, 24, 56
    A, W = wl.splitk_gemm_inputs(R, K, C, seed=5, device=DEV)
    out, P = _run(A, W, S)
    assert _out_bytes(out) == _fold_bytes(P, R, C, torch.float32)
    o2, _ = _run(A, W, S, dump=False, opts={})
    assert _out_bytes(o2) == _out_bytes(out)
    # sampled partials against the binary64 GEMM
    rows = np.array([0, 1, 127, 128, 5000, 16383])
    want = oracle.splitk_gemm_partials(_bits16(A[rows]), _bits16(W), S)
    got = P.cpu().numpy().reshape(S, R, C)[:, rows, :].astype(np.float64)
    a = oracle.bf16_to_f32(_bits16(A[rows])).astype(np.float64)
    w = oracle.bf16_to_f32(_bits16(W)).astype(np.float64)
    ks = K // S
    mag = np.stack([np.abs(a[:, s * ks:(s + 1) * ks]) @ np.abs(w[:, s * ks:(s + 1) * ks]).T for s in range(S)])
    assert np.all(np.abs(got - want) <= ks * 2.0 ** -24 * mag + 1e-30)


def test_splitk_gemm_argument_errors():
    A = torch.zeros(128, 128, dtype=torch.bfloat16, device=DEV)
    W = torch.zeros(40, 128, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(128, 40, device=DEV)
    with pytest.raises(dr.DetError) as e:
        dr.det_splitk_gemm_reduce(A, W, 2, out)  # C > 32
    assert e.value.code == dr.DET_ERR_UNSUPPORTED
    W = torch.zeros(24, 128, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(128, 24, device=DEV)
    with pytest.raises(dr.DetError) as e:
        dr.det_splitk_gemm_reduce(A, W, 3, out)  # K not a multiple of S
    assert e.value.code == dr.DET_ERR_UNSUPPORTED
    with pytest.raises(dr.DetError) as e:
        dr.det_splitk_gemm_reduce(A, W, 4, out)  # K/S = 32, not a multiple of 64
    assert e.value.code == dr.DET_ERR_UNSUPPORTED
    A2 = torch.zeros(128, 129, dtype=torch.bfloat16, device=DEV)[:, 1:]  # 2-byte offset rows
    with pytest.raises(dr.DetError) as e:
        dr.det_splitk_gemm_reduce(A2, W, 2, out)
    assert e.value.code == dr.DET_ERR_ARG
    with pytest.raises(dr.DetError) as e:
        dr.det_splitk_gemm_reduce(A, W, 2, out.to(torch.bfloat16), partials=torch.empty(2, 10, device=DEV))
    assert e.value.code == dr.DET_ERR_ARG
