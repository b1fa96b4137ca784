"""The C-ABI library builds, loads and exports every declared entry point; host-side
argument checks fail closed.  No GPU is touched: every call here returns before the
library makes its first CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

from invariant_gradient_reduction_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for fn in sorted(os.listdir(inc)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(inc, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+char\s*\*|det_status|int32_t|int64_t|void)\s*\**\s*(det_\w+)\s*\(", text,
                            flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    path = build_mod.build()
    from invariant_gradient_reduction_gb300 import detreduce
    return detreduce.lib()


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for must in ("det_reduce_plan", "det_scatter_reduce", "det_splitk_reduce", "det_hash",
                 "det_atomic_scatter_reduce", "det_plan_workspace_size", "det_status_str"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", build_mod.LIB], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT\s+(\w+)$", out.stdout, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing


def test_status_strings_and_version(lib):
    from invariant_gradient_reduction_gb300 import detreduce as dr
    for code in range(0, 9):
        s = dr.det_status_str(code)
        assert s and s != "unknown status"
    assert dr.det_status_str(99) == "unknown status"
    assert dr.det_version() >> 16 == 1


def test_plan_workspace_size_host_logic(lib):
    from invariant_gradient_reduction_gb300 import detreduce as dr
    a = dr.det_plan_workspace_size(1000, 100)
    b = dr.det_plan_workspace_size(100000, 100)
    c = dr.det_plan_workspace_size(100000, 100, with_src_id=True)
    assert 0 < a < b < c
    assert dr.det_plan_workspace_size(0, 0) > 0
    assert dr.det_plan_workspace_size(1 << 20, 1 << 10, opts={"seg_chunks_log2": 6}) <= \
        dr.det_plan_workspace_size(1 << 20, 1 << 10, opts={"seg_chunks_log2": 3})
    with pytest.raises(dr.DetError) as e:
        dr.det_plan_workspace_size(-1, 5)
    assert e.value.code == dr.DET_ERR_ARG
    with pytest.raises(dr.DetError) as e:
        dr.det_plan_workspace_size(1 << 31, 5)
    assert e.value.code == dr.DET_ERR_UNSUPPORTED
    with pytest.raises(dr.DetError) as e:
        dr.det_plan_workspace_size(10, 5, opts={"seg_chunks_log2": 2})
    assert e.value.code == dr.DET_ERR_ARG


def test_entry_points_fail_closed_before_any_cuda_call(lib):
    from invariant_gradient_reduction_gb300 import detreduce as dr
    vp = ctypes.c_void_p
    h = vp(None)
    # det_reduce_plan: missing out-param, negative sizes, missing workspace
    assert lib.det_reduce_plan(None, None, 10, 10, None, 0, None, None, None) == dr.DET_ERR_ARG
    assert lib.det_reduce_plan(None, None, -1, 10, None, 0, None, None, ctypes.byref(h)) == dr.DET_ERR_ARG
    assert lib.det_reduce_plan(vp(256), None, 10, 10, None, 0, None, None, ctypes.byref(h)) == dr.DET_ERR_WORKSPACE
    assert lib.det_reduce_plan(vp(256), None, 10, 10, vp(4096 * 1024), 16, None, None,
                               ctypes.byref(h)) == dr.DET_ERR_WORKSPACE
    assert lib.det_reduce_plan(vp(258), None, 10, 10, vp(1 << 30), 1 << 30, None, None,
                               ctypes.byref(h)) == dr.DET_ERR_ARG  # misaligned idx
    assert lib.det_reduce_plan(vp(256), None, 10, 0, vp(1 << 30), 1 << 30, None, None,
                               ctypes.byref(h)) == dr.DET_ERR_INDEX_RANGE  # sources but no destination
    assert h.value is None
    # det_scatter_reduce without a plan
    assert lib.det_scatter_reduce(None, None, None, 1, 0, 8, 8, None, None, 8, 0, None, 0, None, None) == dr.DET_ERR_ARG
    # det_splitk_reduce: bad dtype, bad stride, NULL out
    assert lib.det_splitk_reduce(vp(256), 4, 16, 16, vp(1 << 20), 7, None, None) == dr.DET_ERR_DTYPE
    assert lib.det_splitk_reduce(vp(256), 4, 16, 8, vp(1 << 20), 0, None, None) == dr.DET_ERR_ARG
    assert lib.det_splitk_reduce(vp(256), 4, 16, 16, None, 0, None, None) == dr.DET_ERR_ARG
    assert lib.det_splitk_reduce(vp(256), 4, 16, 16, vp(256 + 64), 0, None, None) == dr.DET_ERR_ARG  # aliasing
    # det_hash: NULL or misaligned out, NULL data with bytes
    assert lib.det_hash(vp(256), 16, None, None) == dr.DET_ERR_ARG
    assert lib.det_hash(vp(256), 16, vp(1 << 20 | 4), None) == dr.DET_ERR_ARG
    assert lib.det_hash(None, 16, vp(1 << 20), None) == dr.DET_ERR_ARG
    # det_atomic_scatter_reduce: too many shards, bad dtype
    rows = (ctypes.c_int64 * 1)(10)
    ptrs = (vp * 1)(1 << 20)
    assert lib.det_atomic_scatter_reduce(vp(256), 10, 4, ptrs, rows, 17, 0, 8, 8, None, vp(1 << 24), 8, 0,
                                         vp(1 << 26), 1 << 20, None, None) == dr.DET_ERR_UNSUPPORTED
    assert lib.det_atomic_scatter_reduce(vp(256), 10, 4, ptrs, rows, 1, 5, 8, 8, None, vp(1 << 24), 8, 0,
                                         vp(1 << 26), 1 << 20, None, None) == dr.DET_ERR_DTYPE
    # shard rows that do not add up to N
    assert lib.det_atomic_scatter_reduce(vp(256), 11, 4, ptrs, rows, 1, 0, 8, 8, None, vp(1 << 24), 8, 0,
                                         vp(1 << 26), 1 << 20, None, None) == dr.DET_ERR_ARG
    # out overlapping x
    assert lib.det_atomic_scatter_reduce(vp(256), 10, 4, ptrs, rows, 1, 0, 8, 8, None, vp((1 << 20) + 64), 8, 0,
                                         vp(1 << 26), 1 << 20, None, None) == dr.DET_ERR_ARG


def test_product_path_fails_loudly_without_library(tmp_path, monkeypatch):
    """No silent fallback: a missing library raises on first use."""
    from invariant_gradient_reduction_gb300 import detreduce as dr
    monkeypatch.setattr(dr, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(dr, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        dr.lib()


def test_route_host_logic(lib):
    """Sizes and fail-closed argument checks of the router top-k and the route plan (no CUDA call)."""
    from invariant_gradient_reduction_gb300 import detreduce as dr
    a = dr.det_moe_route_workspace_size(64, 2, 8)
    b = dr.det_moe_route_workspace_size(4096, 8, 128)
    c = dr.det_moe_route_workspace_size(16384, 8, 256)
    assert 0 < a < b < c
    assert dr.det_moe_route_workspace_size(0, 8, 8) > 0
    assert dr.det_moe_route_workspace_size(100, 0, 8) > 0
    # a long list (k > 32 * 2^g) needs segment units
    assert dr.det_moe_route_workspace_size(100, 300, 512) > dr.det_moe_route_workspace_size(100, 300, 512, {"seg_chunks_log2": 6})
    for args, code in [((-1, 2, 8), dr.DET_ERR_ARG), ((4, -1, 8), dr.DET_ERR_ARG), ((4, 2, 0), dr.DET_ERR_ARG),
                       ((1 << 30, 4, 8), dr.DET_ERR_UNSUPPORTED)]:
        with pytest.raises(dr.DetError) as e:
            dr.det_moe_route_workspace_size(*args)
        assert e.value.code == code
    L = dr.lib()
    h = ctypes.c_void_p(None)
    fake = 1 << 20  # never dereferenced: every call below fails before its first CUDA call
    # no workspace
    assert L.det_moe_route_plan(fake, None, 4, 2, 8, fake * 2, fake * 3, None, None, None, 0, None, None,
                                ctypes.byref(h)) == dr.DET_ERR_WORKSPACE
    # row_w without topk_w; no expert_offsets; out_plan NULL
    assert L.det_moe_route_plan(fake, None, 4, 2, 8, fake * 2, fake * 3, fake * 4, None, fake * 8, 1 << 20, None,
                                None, ctypes.byref(h)) == dr.DET_ERR_ARG
    assert L.det_moe_route_plan(fake, None, 4, 2, 8, None, fake * 3, None, None, fake * 8, 1 << 20, None, None,
                                ctypes.byref(h)) == dr.DET_ERR_ARG
    assert L.det_moe_route_plan(fake, None, 4, 2, 8, fake * 2, fake * 3, None, None, fake * 8, 1 << 20, None, None,
                                None) == dr.DET_ERR_ARG
    # an output overlapping the ids
    assert L.det_moe_route_plan(fake, None, 4, 2, 8, fake * 2, fake + 16, None, None, fake * 8, 1 << 20, None, None,
                                ctypes.byref(h)) == dr.DET_ERR_ARG
    assert h.value is None
    # top-k: k outside [1, E], E or k beyond the kernel's limits, renormalise without weights, overlap
    for T, E, lds, k, ren, w, code in [(4, 8, 8, 0, 0, fake * 4, dr.DET_ERR_ARG), (4, 8, 8, 9, 0, fake * 4, dr.DET_ERR_ARG),
                                       (4, 8, 7, 2, 0, fake * 4, dr.DET_ERR_ARG),
                                       (4, 2048, 2048, 2, 0, fake * 4, dr.DET_ERR_UNSUPPORTED),
                                       (4, 64, 64, 33, 0, fake * 4, dr.DET_ERR_UNSUPPORTED),
                                       (4, 8, 8, 2, 1, None, dr.DET_ERR_ARG), (4, 8, 8, 2, 0, fake + 8, dr.DET_ERR_ARG)]:
        assert L.det_router_topk(fake, T, E, lds, k, ren, fake * 2, w, None) == code
    assert L.det_router_topk(None, 0, 8, 8, 2, 0, None, None, None) == dr.DET_OK  # nothing to do


def test_route_binding_checks_arguments(lib):
    """The binding rejects wrong dtypes and shapes before it calls the library (no GPU needed)."""
    import torch
    from invariant_gradient_reduction_gb300 import detreduce as dr
    with pytest.raises(ValueError):
        dr.det_moe_route_plan(torch.zeros((4, 2), dtype=torch.int64), 8)   # ids must be int32
    with pytest.raises(ValueError):
        dr.det_moe_route_plan(torch.zeros(8, dtype=torch.int32), 8)        # ids must be [T, k]
    with pytest.raises(ValueError):
        dr.det_moe_route_plan(torch.zeros((4, 2), dtype=torch.int32), 8,
                              topk_w=torch.zeros((4, 3)))                  # weights shaped like the ids
    with pytest.raises(ValueError):
        dr.det_router_topk(torch.zeros((4, 8), dtype=torch.float64), 2)    # scores must be float32
