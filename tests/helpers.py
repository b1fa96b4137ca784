"""Shared test helpers: move seeded cases between torch (GPU path) and numpy (oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from invariant_gradient_reduction_gb300 import detreduce as dr
from invariant_gradient_reduction_gb300.workloads import ScatterCase


def np_bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy; bf16 as uint16 bit patterns, float32 as float32."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def case_np(case: ScatterCase):
    x = np_bits(case.x[:, :case.H])
    w = None if case.w is None else case.w.detach().cpu().numpy()
    idx = case.idx.detach().cpu().numpy().astype(np.int32)
    sid = None if case.src_id is None else case.src_id.detach().cpu().numpy()
    return idx, x, w, sid


def oracle_dtype(t: torch.dtype) -> int:
    return oracle.F32 if t == torch.float32 else oracle.BF16


def oracle_scatter(case: ScatterCase, rows=None) -> np.ndarray:
    """Oracle output, for all destinations or only for the sorted destination list `rows`.

    Sampling keeps only the sources of the chosen destinations, in their
    original relative order, and renumbers the destinations; the result rows
    are the full problem's rows because each destination depends only on its
    own terms in their order (batch invariance).
    """
    idx, x, w, sid = case_np(case)
    od = oracle_dtype(case.out_dtype)
    if rows is None:
        return oracle.scatter_reduce(idx, x, case.M, w=w, out_dtype=od, src_id=sid)
    rows = np.asarray(sorted(set(int(r) for r in rows)), dtype=np.int64)
    pos = np.full(case.M, -1, dtype=np.int64)
    pos[rows] = np.arange(rows.size)
    keep = pos[idx] >= 0
    sub_idx = pos[idx[keep]].astype(np.int32)
    sub_w = None if w is None else w[keep]
    sub_sid = None if sid is None else sid[keep]
    return oracle.scatter_reduce(sub_idx, x[keep], rows.size, w=sub_w, out_dtype=od, src_id=sub_sid)


def gpu_scatter(case: ScatterCase, opts=None, shards=None, out=None, plan=None, stream=None):
    dev = case.x.device
    if plan is None:
        plan = dr.det_reduce_plan(case.idx.to(dev), case.M, src_id=None if case.src_id is None else case.src_id.to(dev),
                                  opts=opts, stream=stream)
    if out is None:
        out = torch.empty((case.M, case.H), dtype=case.out_dtype, device=dev)
    x = case.x if shards is None else shards
    dr.det_scatter_reduce(plan, x, out, w=None if case.w is None else case.w.to(dev), opts=opts, stream=stream)
    return out, plan


def assert_bytes_equal(got: np.ndarray, want: np.ndarray, what: str = ""):
    got = np.ascontiguousarray(got)
    want = np.ascontiguousarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if got.tobytes() == want.tobytes():
        return
    g = got.view(np.uint8).reshape(got.shape + (-1,))
    wv = want.view(np.uint8).reshape(want.shape + (-1,))
    bad = np.argwhere(np.any(g != wv, axis=-1))
    first = tuple(bad[0])
    raise AssertionError(f"{what}: {len(bad)} elements differ; first at {first}: got {got[first]!r} "
                         f"want {want[first]!r}")
