"""det_scatter_reduce_noalloc: the scatter-reduce for callers that cannot allocate
device memory when they call in (an embedding runtime that owns the allocator, a
path that must not allocate after start-up, an interface with no way to pass a
workspace).  Its scratch is a fixed 16 MiB array in the library's device image.

Called straight through the C ABI (ctypes), twice in a row, and compared byte
for byte with the CPU oracle and with det_scatter_reduce given a caller
workspace (the same 0-ULP tolerance as every other parity test).  Collected
last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from helpers import oracle_scatter

pytestmark = pytest.mark.gpu

DEV = "cuda"
LIMIT = 16 << 20


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from invariant_gradient_reduction_gb300 import build
    build.build()
    oracle.build()
    from invariant_gradient_reduction_gb300 import detreduce as dr
    L = dr.lib()
    f = L.det_scatter_reduce_noalloc
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(i64), i32, i32, i64, i64, vp, vp, i64, i32,
                  ctypes.POINTER(dr.det_opts), vp]
    f.restype = i32
    return L


def _noalloc(L, plan, case, out):
    from invariant_gradient_reduction_gb300 import detreduce as dr
    ptrs = (ctypes.c_void_p * 1)(case.x.data_ptr())
    rows = (ctypes.c_int64 * 1)(case.N)
    xdt = dr.DET_BF16 if case.x.dtype == torch.bfloat16 else dr.DET_F32
    odt = dr.DET_BF16 if out.dtype == torch.bfloat16 else dr.DET_F32
    return L.det_scatter_reduce_noalloc(plan.handle, ptrs, rows, 1, xdt, case.x.stride(0), case.H,
                                        None if case.w is None else case.w.data_ptr(), out.data_ptr(), out.stride(0),
                                        odt, None, torch.cuda.current_stream().cuda_stream)


def _bits(t):
    t = t.cpu()
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.view(torch.int32).numpy()


@pytest.mark.parametrize("name", ["sparse_key_scatter", "moe_combine"])
def test_noalloc_matches_workspace_entry_point_twice(lib, name):
    from invariant_gradient_reduction_gb300 import detreduce as dr
    from invariant_gradient_reduction_gb300 import workloads as wl
    case = wl.make(name, "small", device=DEV)
    plan = dr.det_reduce_plan(case.idx, case.M)
    if name == "sparse_key_scatter":
        assert plan.describe()["n_segments"] > 0  # the scratch is really used
    want = torch.empty(case.M, case.H, dtype=case.out_dtype, device=DEV)
    dr.det_scatter_reduce(plan, case.x, want, w=case.w)
    ref = oracle_scatter(case)
    for _ in range(2):
        got = torch.full_like(want, 7)
        assert _noalloc(lib, plan, case, got) == dr.DET_OK
        torch.cuda.synchronize()
        assert np.array_equal(_bits(got), _bits(want))
        assert _bits(got).tobytes() == ref.tobytes()


def test_noalloc_with_an_unwaited_plan(lib):
    """A plan that does not wait: its counts stay on the device, the size check takes
    the upper bound, and the hot destinations' finish pass reads its counts there."""
    from invariant_gradient_reduction_gb300 import detreduce as dr
    from invariant_gradient_reduction_gb300 import workloads as wl
    oracle.build()
    case = wl.make("sparse_key_scatter", "small", device=DEV)
    plan = dr.det_reduce_plan(case.idx, case.M, opts={"async_plan": 1})
    ref = oracle_scatter(case)
    for _ in range(2):
        got = torch.full((case.M, case.H), 7.0, dtype=case.out_dtype, device=DEV)
        assert _noalloc(lib, plan, case, got) == dr.DET_OK
        torch.cuda.synchronize()
        assert _bits(got).tobytes() == ref.tobytes()
    dr.det_plan_status(plan)
    assert plan.describe()["n_segments"] > 0  # hot segments went through the shared array


def test_noalloc_rejects_an_unwaited_plan_whose_bound_is_too_large(lib):
    """An unwaited plan over 65536 sources bounds its partial slots by 513; at a
    width of 8192 that is 513 x 32 KB > 16 MiB, so the call is refused before any
    launch, whatever the data."""
    from invariant_gradient_reduction_gb300 import detreduce as dr
    from invariant_gradient_reduction_gb300.workloads import ScatterCase
    N, H = 65536, 8192
    x = torch.zeros(N, H, dtype=torch.bfloat16, device=DEV)
    case = ScatterCase("bound", torch.arange(N, dtype=torch.int32, device=DEV) % 7, x, None, 7, torch.float32)
    plan = dr.det_reduce_plan(case.idx, case.M, opts={"async_plan": 1})
    assert dr.det_scatter_workspace_size(plan, H) > LIMIT
    out = torch.empty(case.M, H, device=DEV)
    assert _noalloc(lib, plan, case, out) == dr.DET_ERR_UNSUPPORTED
    dr.det_plan_status(plan)
    del x
    torch.cuda.empty_cache()


def test_noalloc_scratch_reuse_between_different_problems(lib):
    """The shared array keeps the previous call's partials; a following call with other
    inputs must not see them."""
    from invariant_gradient_reduction_gb300 import detreduce as dr
    from invariant_gradient_reduction_gb300 import workloads as wl
    a = wl.sparse_key_scatter(640, 128, 4096, 128, seed=31, device=DEV)
    b = wl.sparse_key_scatter(700, 96, 2048, 64, seed=32, device=DEV)
    for case in (a, b, a):
        plan = dr.det_reduce_plan(case.idx, case.M)
        want = torch.empty(case.M, case.H, device=DEV)
        dr.det_scatter_reduce(plan, case.x, want, w=case.w)
        got = torch.empty_like(want)
        assert _noalloc(lib, plan, case, got) == dr.DET_OK
        torch.cuda.synchronize()
        assert np.array_equal(_bits(got), _bits(want))
        assert _bits(got).tobytes() == oracle_scatter(case).tobytes()


def test_noalloc_rejects_scratch_beyond_limit(lib):
    """Two hot segments of a 2,097,160-wide fp32 row need 2 x 8,388,640 bytes > 16 MiB."""
    from invariant_gradient_reduction_gb300 import detreduce as dr
    from invariant_gradient_reduction_gb300.workloads import ScatterCase
    H = 2_097_160
    n = 300  # 300 terms = 10 chunks > 8: one hot destination, two segments
    x = torch.zeros(n, H, dtype=torch.bfloat16, device=DEV)
    case = ScatterCase("big", torch.zeros(n, dtype=torch.int32, device=DEV), x, None, 1, torch.float32)
    plan = dr.det_reduce_plan(case.idx, case.M)
    assert dr.det_scatter_workspace_size(plan, H) > LIMIT
    out = torch.empty(1, H, device=DEV)
    assert _noalloc(lib, plan, case, out) == dr.DET_ERR_UNSUPPORTED
    del x
    torch.cuda.empty_cache()
