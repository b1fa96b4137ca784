"""Thin ctypes binding of libdetreduce.so, under the C names.

Argument marshalling only: tensors become device pointers, strides become
leading dimensions, the current torch CUDA stream becomes the cudaStream_t.
Every step of the computation runs in the library's kernels; there is no
fallback.  If the library is missing or fails to load, every call raises.

Workspaces the C functions take from their caller are allocated here with
torch (the caching allocator), unless the caller passes one.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence, Union

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdetreduce.so")

DET_OK = 0
DET_ERR_ARG = 1
DET_ERR_DTYPE = 2
DET_ERR_INDEX_RANGE = 3
DET_ERR_ORDER_KEY = 4
DET_ERR_WORKSPACE = 5
DET_ERR_CUDA = 6
DET_ERR_TIMEOUT = 7
DET_ERR_UNSUPPORTED = 8
DET_F32 = 0
DET_BF16 = 1
DET_MAX_SHARDS = 16

_TORCH_TO_DET = {torch.float32: DET_F32, torch.bfloat16: DET_BF16}


class DetError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        msg = _lib_or_none().det_status_str(code).decode() if _lib_or_none() else str(code)
        if code == DET_ERR_CUDA and _lib_or_none():
            msg += f" (cudaError {_lib_or_none().det_last_cuda_error()})"
        super().__init__(f"{what}: {msg} [{code}]")


class det_opts(ctypes.Structure):
    _fields_ = [("grid_ctas", ctypes.c_int32), ("seg_chunks_log2", ctypes.c_int32),
                ("debug_checks", ctypes.c_int32), ("gather_path", ctypes.c_int32),
                ("tiles_per_task", ctypes.c_int32), ("async_plan", ctypes.c_int32),
                ("plan_path", ctypes.c_int32), ("reserved", ctypes.c_int32 * 1)]


class det_plan_desc(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("M", ctypes.c_int64), ("seg_chunks_log2", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("row_ptr", ctypes.c_void_p), ("perm", ctypes.c_void_p),
                ("n_units", ctypes.c_int64), ("n_segments", ctypes.c_int64), ("n_hot_rows", ctypes.c_int64),
                ("max_row_len", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def _declare(lib):
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    P = ctypes.POINTER
    sigs = {
        "det_status_str": ([i32], ctypes.c_char_p),
        "det_last_cuda_error": ([], i32),
        "det_version": ([], i32),
        "det_kernel_launches": ([], i64),
        "det_plan_workspace_size": ([i64, i64, i32, P(det_opts), P(sz)], i32),
        "det_reduce_plan": ([vp, vp, i64, i64, vp, sz, P(det_opts), vp, P(vp)], i32),
        "det_plan_destroy": ([vp], i32),
        "det_plan_describe": ([vp, P(det_plan_desc)], i32),
        "det_plan_status": ([vp, vp], i32),
        "det_scatter_workspace_size": ([vp, i64, P(sz)], i32),
        "det_scatter_reduce": ([vp, P(vp), P(i64), i32, i32, i64, i64, vp, vp, i64, i32, vp, sz,
                                P(det_opts), vp], i32),
        "det_index_add": ([vp, P(vp), P(i64), i32, i32, i64, i64, vp, vp, i64, i32, vp, sz, P(det_opts), vp], i32),
        "det_splitk_reduce": ([vp, i32, i64, i64, vp, i32, P(det_opts), vp], i32),
        "det_splitk_gemm_reduce": ([vp, i64, vp, i64, i64, i32, i64, i32, i32, vp, i64, i32, vp, i64, P(det_opts),
                                    vp], i32),
        "det_hash": ([vp, ctypes.c_uint64, vp, vp], i32),
        "det_atomic_workspace_size": ([i64, i64, i32, P(sz)], i32),
        "det_atomic_scatter_reduce": ([vp, i64, i64, P(vp), P(i64), i32, i32, i64, i64, vp, vp, i64, i32, vp,
                                       sz, P(det_opts), vp], i32),
        "det_atomic_index_add": ([vp, i64, i64, P(vp), P(i64), i32, i32, i64, i64, vp, vp, i64, i32, vp,
                                  sz, P(det_opts), vp], i32),
        "det_router_topk": ([vp, i64, i32, i64, i32, i32, vp, vp, vp], i32),
        "det_moe_route_workspace_size": ([i64, i32, i32, P(det_opts), P(sz)], i32),
        "det_moe_route_plan": ([vp, vp, i64, i32, i32, vp, vp, vp, vp, vp, sz, P(det_opts), vp, P(vp)], i32),
    }
    for name, (args, res) in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


def _lib_or_none():
    return _lib


def lib():
    """The loaded library.  Raises if libdetreduce.so has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libdetreduce.so is not built ({LIB_PATH}); run "
                                   "invariant_gradient_reduction_gb300.build.build() first")
            _lib = _declare(ctypes.CDLL(LIB_PATH))
        return _lib


def _check(code: int, what: str):
    if code != DET_OK:
        raise DetError(code, what)


def _opts(opts: Optional[dict]):
    if opts is None:
        return None
    o = det_opts(grid_ctas=int(opts.get("grid_ctas", 0)), seg_chunks_log2=int(opts.get("seg_chunks_log2", -1)),
                 debug_checks=int(opts.get("debug_checks", 0)), gather_path=int(opts.get("gather_path", 0)),
                 tiles_per_task=int(opts.get("tiles_per_task", 0)), async_plan=int(opts.get("async_plan", 0)),
                 plan_path=int(opts.get("plan_path", 0)))
    return ctypes.byref(o)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _rows(x: torch.Tensor):
    """(ldx, H) of a 2-D row-major tensor whose rows may be padded."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("row tensors must be 2-D with unit stride along a row")
    return (x.stride(0) if x.shape[0] > 1 else max(x.shape[1], x.stride(0))), x.shape[1]


def _workspace(nbytes: int, device, given: Optional[torch.Tensor]):
    if given is not None:
        return given
    return torch.empty(max(nbytes, 1) + 256, dtype=torch.uint8, device=device)


def _aligned_ptr(t: torch.Tensor) -> int:
    p = t.data_ptr()
    return (p + 255) // 256 * 256


def _aligned_bytes(t: torch.Tensor) -> int:
    return t.numel() - (_aligned_ptr(t) - t.data_ptr())


def det_status_str(code: int) -> str:
    return lib().det_status_str(code).decode()


def det_version() -> int:
    return lib().det_version()


def det_kernel_launches() -> int:
    return lib().det_kernel_launches()


def det_plan_workspace_size(N: int, M: int, with_src_id: bool = False, opts: Optional[dict] = None) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().det_plan_workspace_size(N, M, int(bool(with_src_id)), _opts(opts), ctypes.byref(out)),
           "det_plan_workspace_size")
    return out.value


class Plan:
    """A built plan: the C handle plus the torch buffer holding its device arrays."""

    def __init__(self, handle, workspace: torch.Tensor, N: int, M: int):
        self._h = handle
        self.workspace = workspace
        self.N, self.M = N, M

    @property
    def handle(self):
        if self._h is None:
            raise RuntimeError("plan destroyed")
        return self._h

    def describe(self) -> dict:
        return det_plan_describe(self)

    def destroy(self):
        if self._h is not None and _lib is not None:
            _lib.det_plan_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def det_reduce_plan(idx: torch.Tensor, M: int, src_id: Optional[torch.Tensor] = None, opts: Optional[dict] = None,
                    stream=None, workspace: Optional[torch.Tensor] = None) -> Plan:
    """Destination lists + work list for idx (int32 [N], device)."""
    if idx.dtype != torch.int32 or not idx.is_contiguous():
        raise ValueError("idx must be a contiguous int32 tensor")
    if src_id is not None and (src_id.dtype != torch.int64 or not src_id.is_contiguous()):
        raise ValueError("src_id must be a contiguous int64 tensor")
    N = idx.numel()
    need = det_plan_workspace_size(N, M, src_id is not None, opts)
    ws = _workspace(need, idx.device, workspace)
    h = ctypes.c_void_p(None)
    _check(lib().det_reduce_plan(_ptr(idx), _ptr(src_id), N, M, _aligned_ptr(ws), _aligned_bytes(ws), _opts(opts),
                                 _stream(stream), ctypes.byref(h)), "det_reduce_plan")
    return Plan(h, ws, N, M)


def det_plan_status(plan: Plan, stream=None) -> None:
    """Wait for the plan's kernels and raise DetError if they found an error (async plans)."""
    _check(lib().det_plan_status(plan.handle, _stream(stream)), "det_plan_status")


def det_plan_describe(plan: Plan) -> dict:
    d = det_plan_desc()
    _check(lib().det_plan_describe(plan.handle, ctypes.byref(d)), "det_plan_describe")
    return {f: getattr(d, f) for f, _ in det_plan_desc._fields_ if f != "reserved"}


def plan_lists(plan: Plan):
    """(row_ptr int32 [M+1], perm int32 [N]) as device tensors viewing the plan workspace."""
    d = det_plan_describe(plan)
    ws = plan.workspace
    base = ws.data_ptr()
    rp_off = d["row_ptr"] - base
    pm_off = d["perm"] - base
    row_ptr = ws[rp_off:rp_off + 4 * (plan.M + 1)].view(torch.int32)
    perm = ws[pm_off:pm_off + 4 * plan.N].view(torch.int32)
    return row_ptr, perm


def det_router_topk(scores: torch.Tensor, k: int, renormalize: bool = False, with_weights: bool = True,
                    stream=None, out: Optional[tuple] = None):
    """(ids int32 [T, k], w float32 [T, k] or None): each token's k greatest scores, greatest first.

    ``scores`` float32 [T, E] (rows may be padded).  Order and renormalisation
    as in det_router_topk of det_reduce.h.  ``out`` = (ids, w) to write into.
    """
    if scores.dtype != torch.float32:
        raise ValueError("scores must be float32")
    lds, E = _rows(scores)
    T = scores.shape[0]
    if out is not None:
        ids, w = out
    else:
        ids = torch.empty((T, k), dtype=torch.int32, device=scores.device)
        w = torch.empty((T, k), dtype=torch.float32, device=scores.device) if (with_weights or renormalize) else None
    _check(lib().det_router_topk(_ptr(scores), T, E, lds, k, int(bool(renormalize)), _ptr(ids), _ptr(w),
                                 _stream(stream)), "det_router_topk")
    return ids, w


def det_moe_route_workspace_size(T: int, k: int, E: int, opts: Optional[dict] = None) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().det_moe_route_workspace_size(T, k, E, _opts(opts), ctypes.byref(out)),
           "det_moe_route_workspace_size")
    return out.value


def det_moe_route_plan(topk_ids: torch.Tensor, E: int, topk_w: Optional[torch.Tensor] = None,
                       opts: Optional[dict] = None, stream=None, workspace: Optional[torch.Tensor] = None,
                       with_slot_row: bool = True, out: Optional[dict] = None):
    """Dispatch layout + combine plan of top-k routing (``topk_ids`` int32 [T, k], device).

    Returns (plan, arrays): ``plan`` is the combine's Plan over M = T tokens;
    ``arrays`` holds the device tensors expert_offsets int32 [E+1], row_token
    int32 [T*k], row_w float32 [T*k] (None without topk_w) and slot_row int32
    [T*k] (None unless with_slot_row).  ``out`` may give these tensors to
    write into (same keys).
    """
    if topk_ids.dtype != torch.int32 or not topk_ids.is_contiguous() or topk_ids.dim() != 2:
        raise ValueError("topk_ids must be a contiguous int32 [T, k] tensor")
    if topk_w is not None and (topk_w.dtype != torch.float32 or not topk_w.is_contiguous()
                               or topk_w.shape != topk_ids.shape):
        raise ValueError("topk_w must be a contiguous float32 tensor shaped like topk_ids")
    T, k = topk_ids.shape
    N = T * k
    dev = topk_ids.device
    o = dict(out or {})
    if "expert_offsets" not in o:
        o["expert_offsets"] = torch.empty(E + 1, dtype=torch.int32, device=dev)
    if "row_token" not in o:
        o["row_token"] = torch.empty(N, dtype=torch.int32, device=dev)
    if "row_w" not in o:
        o["row_w"] = torch.empty(N, dtype=torch.float32, device=dev) if topk_w is not None else None
    if "slot_row" not in o:
        o["slot_row"] = torch.empty(N, dtype=torch.int32, device=dev) if with_slot_row else None
    need = det_moe_route_workspace_size(T, k, E, opts)
    ws = _workspace(need, dev, workspace)
    h = ctypes.c_void_p(None)
    _check(lib().det_moe_route_plan(_ptr(topk_ids), _ptr(topk_w), T, k, E, _ptr(o["expert_offsets"]),
                                    _ptr(o["row_token"]), _ptr(o["row_w"]), _ptr(o["slot_row"]), _aligned_ptr(ws),
                                    _aligned_bytes(ws), _opts(opts), _stream(stream), ctypes.byref(h)),
           "det_moe_route_plan")
    return Plan(h, ws, N, T), o


def det_scatter_workspace_size(plan: Plan, H: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().det_scatter_workspace_size(plan.handle, H, ctypes.byref(out)), "det_scatter_workspace_size")
    return out.value


def _shards(x: Union[torch.Tensor, Sequence[torch.Tensor]]):
    xs = [x] if isinstance(x, torch.Tensor) else list(x)
    if not xs:
        raise ValueError("need at least one shard")
    dt = xs[0].dtype
    if dt not in _TORCH_TO_DET or any(s.dtype != dt for s in xs):
        raise ValueError("shards must all be float32 or all bfloat16")
    lds = [_rows(s) for s in xs]
    H = lds[0][1]
    nonempty = [ld for (ld, h), s in zip(lds, xs) if s.shape[0] > 1]
    ldx = nonempty[0] if nonempty else max(ld for ld, _ in lds)
    if any(h != H for _, h in lds) or any(ld != ldx for ld in nonempty):
        raise ValueError("shards must share the row width and row stride")
    ptrs = (ctypes.c_void_p * len(xs))(*[s.data_ptr() for s in xs])
    rows = (ctypes.c_int64 * len(xs))(*[s.shape[0] for s in xs])
    return ptrs, rows, len(xs), _TORCH_TO_DET[dt], ldx, H


def det_index_add(plan: Plan, x, out: torch.Tensor, w: Optional[torch.Tensor] = None,
                  opts: Optional[dict] = None, stream=None, workspace: Optional[torch.Tensor] = None):
    """out[m] += canonical sum of w[i] * x[i] over the sources of m (one fp32 add; rows without sources untouched)."""
    return _reduce_call("det_index_add", plan, x, out, w, opts, stream, workspace)


def det_scatter_reduce(plan: Plan, x, out: torch.Tensor, w: Optional[torch.Tensor] = None,
                       opts: Optional[dict] = None, stream=None, workspace: Optional[torch.Tensor] = None):
    """out[m] = canonical sum of w[i] * x[i] over the sources of m (x: tensor or list of shards)."""
    return _reduce_call("det_scatter_reduce", plan, x, out, w, opts, stream, workspace)


def _reduce_call(name, plan, x, out, w, opts, stream, workspace):
    ptrs, rows, P, xdt, ldx, H = _shards(x)
    ldo, Ho = _rows(out)
    if Ho != H or out.shape[0] != plan.M:
        raise ValueError("out must be [M, H]")
    if out.dtype not in _TORCH_TO_DET:
        raise ValueError("out must be float32 or bfloat16")
    if w is not None and (w.dtype != torch.float32 or not w.is_contiguous()):
        raise ValueError("w must be a contiguous float32 tensor")
    need = det_scatter_workspace_size(plan, H)
    ws = _workspace(need, out.device, workspace) if need > 0 else None
    _check(getattr(lib(), name)(plan.handle, ptrs, rows, P, xdt, ldx, H, _ptr(w), _ptr(out), ldo,
                                _TORCH_TO_DET[out.dtype], _aligned_ptr(ws) if ws is not None else None,
                                _aligned_bytes(ws) if ws is not None else 0, _opts(opts), _stream(stream)), name)
    return out


def det_splitk_reduce(partials: torch.Tensor, out: torch.Tensor, opts: Optional[dict] = None, stream=None):
    """out[e] = canonical sum over s of partials[s, e] (partials float32 [S, count])."""
    if partials.dtype != torch.float32:
        raise ValueError("partials must be float32")
    ldp, count = _rows(partials)
    S = partials.shape[0]
    if out.numel() != count or not out.is_contiguous() or out.dtype not in _TORCH_TO_DET:
        raise ValueError("out must be a contiguous float32/bfloat16 tensor of `count` elements")
    _check(lib().det_splitk_reduce(_ptr(partials), S, count, ldp, _ptr(out), _TORCH_TO_DET[out.dtype],
                                   _opts(opts), _stream(stream)), "det_splitk_reduce")
    return out


def det_splitk_gemm_reduce(A: torch.Tensor, W: torch.Tensor, S: int, out: torch.Tensor,
                           partials: Optional[torch.Tensor] = None, opts: Optional[dict] = None, stream=None):
    """out[r, c] = canonical sum over s of P_s[r, c], P_s = the split-s K-slice of A @ W.T.

    ``A`` bf16 [R, K] and ``W`` bf16 [C, K] (rows may be padded: K contiguous),
    K = S * (a multiple of 64), C <= 32; ``out`` float32/bfloat16 [R, C] (rows
    may be padded).  ``partials``: None, or float32 [S, >= R*C] to receive each
    split's partial as well (row-major [R, C] per split).
    """
    if A.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise ValueError("A and W must be bfloat16")
    lda, K = _rows(A)
    ldw, Kw = _rows(W)
    if Kw != K:
        raise ValueError("A and W need the same K")
    R, C = A.shape[0], W.shape[0]
    ldo, oc = _rows(out)
    if out.shape[0] != R or oc != C or out.dtype not in _TORCH_TO_DET:
        raise ValueError("out must be float32/bfloat16 [R, C]")
    ldp = 0
    if partials is not None:
        if partials.dtype != torch.float32 or partials.dim() != 2 or partials.shape[0] != S:
            raise ValueError("partials must be float32 [S, >= R*C]")
        ldp = _rows(partials)[0]
    _check(lib().det_splitk_gemm_reduce(_ptr(A), lda, _ptr(W), ldw, R, C, K, S, DET_BF16, _ptr(out), ldo,
                                        _TORCH_TO_DET[out.dtype], _ptr(partials), ldp, _opts(opts), _stream(stream)),
           "det_splitk_gemm_reduce")
    return out


def det_hash(t: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None, nbytes: Optional[int] = None,
             byte_offset: int = 0) -> torch.Tensor:
    """u64 fingerprint of a contiguous tensor's bytes, into a 1-element int64 device tensor."""
    if not t.is_contiguous():
        raise ValueError("det_hash needs a contiguous tensor")
    if out is None:
        out = torch.empty(1, dtype=torch.int64, device=t.device)
    n = t.numel() * t.element_size() if nbytes is None else nbytes
    _check(lib().det_hash(t.data_ptr() + byte_offset if n > 0 else None, n, _ptr(out), _stream(stream)), "det_hash")
    return out


def det_atomic_workspace_size(M: int, H: int, out_dtype: torch.dtype) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().det_atomic_workspace_size(M, H, _TORCH_TO_DET[out_dtype], ctypes.byref(out)),
           "det_atomic_workspace_size")
    return out.value


def det_atomic_scatter_reduce(idx: torch.Tensor, M: int, x, out: torch.Tensor, w: Optional[torch.Tensor] = None,
                              opts: Optional[dict] = None, stream=None, workspace: Optional[torch.Tensor] = None):
    """NOT deterministic: the atomicAdd scatter-add baseline (same arguments as det_scatter_reduce)."""
    return _atomic_call("det_atomic_scatter_reduce", idx, M, x, out, w, opts, stream, workspace)


def det_atomic_index_add(idx: torch.Tensor, M: int, x, out: torch.Tensor, w: Optional[torch.Tensor] = None,
                         opts: Optional[dict] = None, stream=None, workspace: Optional[torch.Tensor] = None):
    """NOT deterministic: atomicAdd into out as it is (the twin of det_index_add); fp32 out only."""
    return _atomic_call("det_atomic_index_add", idx, M, x, out, w, opts, stream, workspace)


def _atomic_call(name, idx, M, x, out, w, opts, stream, workspace):
    ptrs, rows, P, xdt, ldx, H = _shards(x)
    ldo, Ho = _rows(out)
    if Ho != H or out.shape[0] != M:
        raise ValueError("out must be [M, H]")
    need = det_atomic_workspace_size(M, H, out.dtype)
    ws = _workspace(need, out.device, workspace)
    _check(getattr(lib(), name)(_ptr(idx), idx.numel(), M, ptrs, rows, P, xdt, ldx, H, _ptr(w), _ptr(out), ldo,
                                _TORCH_TO_DET[out.dtype], _aligned_ptr(ws), _aligned_bytes(ws), _opts(opts),
                                _stream(stream)), name)
    return out


__all__ = [n for n in dir() if n.startswith("det_") or n.startswith("DET_")] + ["Plan", "DetError", "lib",
                                                                                   "plan_lists", "LIB_PATH"]


def det_scatter_reduce_noalloc(plan: Plan, x, out: torch.Tensor, w: Optional[torch.Tensor] = None,
                               opts: Optional[dict] = None, stream=None):
    """det_scatter_reduce for callers that cannot allocate: its scratch is the
    library's fixed 16 MiB device array (see the C header for the limits)."""
    f = lib().det_scatter_reduce_noalloc
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(i64), i32, i32, i64, i64, vp, vp, i64, i32,
                  ctypes.POINTER(det_opts), vp]
    f.restype = i32
    ptrs, rows, P, xdt, ldx, H = _shards(x)
    ldo, Ho = _rows(out)
    if Ho != H or out.shape[0] != plan.M or out.dtype not in _TORCH_TO_DET:
        raise ValueError("out must be a float32/bfloat16 [M, H] tensor")
    _check(f(plan.handle, ptrs, rows, P, xdt, ldx, H, _ptr(w), _ptr(out), ldo, _TORCH_TO_DET[out.dtype], _opts(opts),
             _stream(stream)), "det_scatter_reduce_noalloc")
    return out
