"""CPU oracle for the deterministic multi-writer reduction (ctypes over oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use it.  The GPU library never imports, links or calls it and
it shares no code with the GPU library.

Every function takes and returns numpy arrays.  bf16 data travels as
``np.uint16`` bit patterns.  The arithmetic itself lives in ``oracle.c``,
which documents the canonical order it implements.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

F32 = 0
BF16 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, no fused multiply-add)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        i32, i64, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
        vp, fp = ctypes.c_void_p, ctypes.c_float
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = fp
        lib.oracle_f32_to_bf16.argtypes = [fp]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_f32_to_bf16_array.argtypes = [vp, vp, i64]
        lib.oracle_f32_to_bf16_array.restype = None
        lib.oracle_bf16_to_f32_array.argtypes = [vp, vp, i64]
        lib.oracle_bf16_to_f32_array.restype = None
        lib.oracle_canonical_sum.argtypes = [vp, i64, ctypes.POINTER(i32)]
        lib.oracle_canonical_sum.restype = fp
        lib.oracle_build_lists.argtypes = [vp, vp, i64, i64, vp, vp]
        lib.oracle_build_lists.restype = ctypes.c_int
        lib.oracle_scatter_reduce.argtypes = [vp, vp, i64, i64, vp, vp, i32, i32, i64, i64, vp, vp, i64, i32]
        lib.oracle_scatter_reduce.restype = ctypes.c_int
        lib.oracle_index_add.argtypes = [vp, vp, i64, i64, vp, vp, i32, i32, i64, i64, vp, vp, i64, i32]
        lib.oracle_index_add.restype = ctypes.c_int
        lib.oracle_splitk_reduce.argtypes = [vp, i32, i64, i64, vp, i32]
        lib.oracle_splitk_reduce.restype = ctypes.c_int
        lib.oracle_mix64.argtypes = [u64]
        lib.oracle_mix64.restype = u64
        lib.oracle_hash.argtypes = [vp, u64]
        lib.oracle_hash.restype = u64
        lib.oracle_router_topk.argtypes = [vp, i64, i32, i64, i32, i32, vp, vp]
        lib.oracle_router_topk.restype = ctypes.c_int
        lib.oracle_moe_route.argtypes = [vp, vp, i64, i32, i32, vp, vp, vp, vp]
        lib.oracle_moe_route.restype = ctypes.c_int
        _lib = lib
        return lib


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        names = {-1: "bad argument", -2: "index out of range", -3: "duplicate order key", -4: "out of memory"}
        super().__init__(f"oracle {what}: {names.get(code, code)}")
        self.code = code


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"x must be float32 or uint16 (bf16 bits), got {a.dtype}")


def f32_to_bf16(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_f32_to_bf16_array(_ptr(a), _ptr(out), a.size)
    return out


def bf16_to_f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.uint16)
    out = np.empty(a.shape, dtype=np.float32)
    _load().oracle_bf16_to_f32_array(_ptr(a), _ptr(out), a.size)
    return out


def canonical_sum(terms) -> np.float32:
    """Canonical fold of a 1-D sequence of binary32 terms."""
    t = np.ascontiguousarray(terms, dtype=np.float32).reshape(-1)
    ok = ctypes.c_int32(0)
    r = _load().oracle_canonical_sum(_ptr(t), t.size, ctypes.byref(ok))
    if not ok.value:
        raise MemoryError("oracle canonical_sum")
    return np.float32(r)


def build_lists(idx, M: int, src_id=None):
    """(row_ptr[M+1] int64, perm[N] int64): sources of each destination in order-key order."""
    idx = np.ascontiguousarray(idx, dtype=np.int32).reshape(-1)
    sid = None if src_id is None else np.ascontiguousarray(src_id, dtype=np.int64).reshape(-1)
    N = idx.size
    row_ptr = np.empty(M + 1, dtype=np.int64)
    perm = np.empty(max(N, 1), dtype=np.int64)
    rc = _load().oracle_build_lists(_ptr(idx), _ptr(sid), N, M, _ptr(row_ptr), _ptr(perm))
    if rc != 0:
        raise OracleError(rc, "build_lists")
    return row_ptr, perm[:N]


def scatter_reduce(idx, x_shards, M: int, w=None, out_dtype: int = F32, src_id=None, H: int | None = None,
                   out_init=None):
    """out[m] = canonical sum over {i : idx[i] = m} of w[i] * x[i] (rows in order-key order).

    With ``out_init`` (float32 or uint16 bf16 bits [M, H]) the call has
    index_add_ semantics: every destination with terms becomes
    out_init[m] + sum (one binary32 add), the others keep out_init[m].

    ``x_shards`` is one 2-D array or a list of 2-D arrays (rows of consecutive
    global source ranges), all float32 or all uint16 (bf16 bits), rows
    possibly padded (the row stride is taken from the array).  Returns float32
    [M, H] or uint16 [M, H] (bf16 bits).
    """
    if isinstance(x_shards, np.ndarray):
        x_shards = [x_shards]
    shards = [np.ascontiguousarray(s) for s in x_shards]
    code = _dtype_code(shards[0])
    if any(_dtype_code(s) != code for s in shards):
        raise TypeError("all shards must share one dtype")
    ldx = shards[0].shape[1]
    if any(s.ndim != 2 or s.shape[1] != ldx for s in shards):
        raise ValueError("shards must be 2-D with equal row length")
    H = ldx if H is None else H
    idx = np.ascontiguousarray(idx, dtype=np.int32).reshape(-1)
    N = idx.size
    rows = np.array([s.shape[0] for s in shards], dtype=np.int64)
    ptrs = (ctypes.c_void_p * len(shards))(*[s.ctypes.data for s in shards])
    wv = None if w is None else np.ascontiguousarray(w, dtype=np.float32).reshape(-1)
    sid = None if src_id is None else np.ascontiguousarray(src_id, dtype=np.int64).reshape(-1)
    odt = np.float32 if out_dtype == F32 else np.uint16
    if out_init is None:
        out = np.empty((M, H), dtype=odt)
        fn = _load().oracle_scatter_reduce
    else:
        out = np.array(out_init, dtype=odt, copy=True).reshape(M, H)
        fn = _load().oracle_index_add
    rc = fn(_ptr(idx), _ptr(sid), N, M, ctypes.cast(ptrs, ctypes.c_void_p), _ptr(rows), len(shards), code, ldx, H,
            _ptr(wv), _ptr(out), H, out_dtype)
    if rc != 0:
        raise OracleError(rc, "scatter_reduce")
    return out


def splitk_reduce(partials, out_dtype: int = F32):
    """out[e] = canonical sum over s of partials[s, e] (partials float32 [S, count])."""
    p = np.ascontiguousarray(partials, dtype=np.float32)
    S, count = p.shape
    out = np.empty(count, dtype=np.float32 if out_dtype == F32 else np.uint16)
    rc = _load().oracle_splitk_reduce(_ptr(p), S, count, count, _ptr(out), out_dtype)
    if rc != 0:
        raise OracleError(rc, "splitk_reduce")
    return out


def splitk_gemm_partials(a_bits, w_bits, S: int) -> np.ndarray:
    """Exact (binary64) per-split partial sums of a split-K GEMM: P[s][r][c] =
    sum over the K/S values of k in split s of A[r][k] * W[c][k].

    A is [R, K] and W is [C, K], both bf16 bit patterns (K contiguous); the K
    dimension is cut into S equal consecutive splits, each producing its own
    partial ("DeepSeek-V4 book, Ch 09", section 3.3: every K-split writes its
    own buffer).  A bf16 times bf16 product is exact in binary64 and the sums
    are taken in binary64, so this is the reference the GPU's binary32
    tensor-core partials are compared with (within a rounding bound), not a
    bit-exact one.  Returns float64 [S, R, C].
    """
    a = bf16_to_f32(a_bits).astype(np.float64)
    w = bf16_to_f32(w_bits).astype(np.float64)
    R, K = a.shape
    C = w.shape[0]
    if K % S:
        raise ValueError("K must be a multiple of S")
    ks = K // S
    out = np.empty((S, R, C), dtype=np.float64)
    for s in range(S):
        out[s] = a[:, s * ks:(s + 1) * ks] @ w[:, s * ks:(s + 1) * ks].T
    return out


def mix64(z: int) -> int:
    return int(_load().oracle_mix64(z & 0xFFFFFFFFFFFFFFFF))


def hash_bytes(buf) -> int:
    """u64 fingerprint of a byte buffer (numpy array of any dtype, or bytes)."""
    if isinstance(buf, (bytes, bytearray)):
        a = np.frombuffer(bytes(buf), dtype=np.uint8)
    else:
        a = np.ascontiguousarray(buf).view(np.uint8).reshape(-1)
    if a.size == 0:
        a = np.zeros(1, dtype=np.uint8)
        return int(_load().oracle_hash(_ptr(a), 0))
    return int(_load().oracle_hash(_ptr(a), a.size))


def router_topk(scores, k: int, renormalize: bool = False):
    """(ids int32 [T, k], w float32 [T, k]): each token's k greatest scores, greatest first.

    Order: IEEE 754 totalOrder of the binary32 scores, the lower expert id
    first among equal bit patterns.  ``renormalize``: w[r] / (w[0] + ... +
    w[k-1]), the sum taken left to right in binary32 (oracle.c states the
    definition).
    """
    s = np.ascontiguousarray(scores, dtype=np.float32)
    T, E = s.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    rc = _load().oracle_router_topk(_ptr(s), T, E, E, k, 1 if renormalize else 0, _ptr(ids), _ptr(w))
    if rc != 0:
        raise OracleError(rc, "router_topk")
    return ids, w


def moe_route(ids, E: int, w=None):
    """Dispatch layout of top-k routing (stable counting sort of the slots by expert).

    ``ids`` int32 [T, k], ``w`` float32 [T, k] or None.  Returns
    (expert_offsets int64 [E+1], row_token int32 [T*k], row_w float32 [T*k] or
    None, slot_row int32 [T*k]).
    """
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    N = T * k
    wv = None if w is None else np.ascontiguousarray(w, dtype=np.float32).reshape(-1)
    off = np.empty(E + 1, dtype=np.int64)
    row_token = np.empty(max(N, 1), dtype=np.int32)
    slot_row = np.empty(max(N, 1), dtype=np.int32)
    row_w = None if wv is None else np.empty(max(N, 1), dtype=np.float32)
    rc = _load().oracle_moe_route(_ptr(ids), _ptr(wv), T, k, E, _ptr(off), _ptr(row_token), _ptr(row_w),
                                  _ptr(slot_row))
    if rc != 0:
        raise OracleError(rc, "moe_route")
    return off, row_token[:N], None if row_w is None else row_w[:N], slot_row[:N]
