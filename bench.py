#!/usr/bin/env python3
"""Benchmark of the deterministic multi-writer reduction on one node.

Metric: deterministic scatter-reduce HBM GB/s (compulsory bytes: sources read
once, outputs written once, indices and weights read once), its fraction of
the measured HBM peak, and the overhead against the in-repo atomicAdd kernel.

One step = the whole hot path over one batch of the workload: the plan
(destination histogram, scan, stable sort of sources, work list) followed by
the gather-reduce (and the hot-destination second pass when the workload has
hot destinations).  Inputs are resident in HBM when the timed region starts;
L2 is flushed before every timed step, outside the step's CUDA events: a
256 MiB write, then a 256 MiB read of a second buffer, so that the write's
dirty lines go back to HBM during the flush and not inside the timed step
(with the write alone that write-back costs the MoE step about 10 us).
Every step is timed with CUDA events on the launching stream.

Default workload: the MoE combine/unpermute, T=4096 tokens, E=128 experts,
top-8, H=4096, bf16 expert outputs with fp32 routing weights, bf16 out.  The
sparse-attention key scatter and the split-K reduce are measured alongside
and reported under "also" (same timing rules).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (single thread, the machine's host cores)
on a bounded sample of the same workload and prints the same JSON line with
"impl": "reference".  With N > 1 (torchrun) every rank runs an independent
replica of the workload on its own GPU (the path has no exchange step on one
node): value = all ranks' bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "deterministic scatter-reduce HBM GB/s (% of peak) and overhead vs atomicAdd"
UNIT = "GB/s"
ASYNC = {"async_plan": 1}  # plans enqueue without a host wait
# the reduce-only measurement takes the library's choice for a waited plan,
# which is the kernel the step's unwaited plan gets too: the fixed-stage TMA
# kernel for the MoE and EP shapes (every destination <= 32 terms, wide rows,
# one shard), the register-staged kernel for the sparse scatter's 256-byte rows
STEP_KERNEL = {}
REGISTER_KERNEL = {"gather_path": 1}
ROOFLINE_KERNEL = {"moe_combine": ("gather_bulk_kernel", "gather_bulk.cu"),
                   "ep_invariance": ("gather_bulk_kernel", "gather_bulk.cu"),
                   "sparse_key_scatter": ("gather_reduce_kernel", "gather.cu")}
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
WORKLOADS = {
    "moe_combine": "moe_combine T=4096 E=128 top-k=8 H=4096 bf16 x, fp32 w -> bf16 out",
    "sparse_key_scatter": "sparse_key_scatter Q=16384 K=512 S=65536 zipf=1.1 H=128 bf16 x -> fp32 out",
    "ep_invariance": "ep_invariance T=16384 E=256 top-k=8 H=7168 bf16 x, fp32 w -> bf16 out",
    "splitk": "splitk S=56 R=16384 C=24 fp32 -> fp32",
    "splitk_gemm": "split-K GEMM with the split-ordered fold in its epilogue (16384 x 7168 x 24, 56 splits)",
    "embedding_backward": "embedding_backward T=32768 tokens V=131072 zipf=1.0 H=4096 bf16 dY, index_add into fp32 grad",
    "moe_route": "moe_route T=4096 E=128 top-k=8 H=4096: softmax scores -> sorted top-k -> route plan -> combine, "
                 "bf16 x -> bf16 out",
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["moe_combine", "sparse_key_scatter", "ep_invariance"],
                    default="moe_combine")
    ap.add_argument("--size", choices=["full", "medium"], default="full",
                    help="medium: a quarter-size case of the same shape (for profiler captures only)")
    ap.add_argument("--no-also", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--also", default="sparse_key_scatter,ep_invariance,moe_route,splitk,splitk_gemm,embedding_backward",
                    help="comma-separated secondary workloads to measure (default: all)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-dir", default=os.path.join(ROOT, "bench_out"),
                    help="where the nvidia-smi clock samples of the timed region are written")
    ap.add_argument("--no-e2e", action="store_true")
    a = ap.parse_args(argv)
    a.warmup = max(3, a.warmup)
    a.steps = max(1, a.steps)
    return a


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


def read_traffic(kernel_file: str, workload: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on the current source."""
    import hashlib
    src = os.path.join(ROOT, "invariant_gradient_reduction_gb300", "csrc", kernel_file)
    summ = os.path.join(ROOT, "profiles", f"{os.path.splitext(kernel_file)[0]}_{workload}.md")
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        fields = {}
        for line in open(summ):
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
        if fields.get("source_sha256_16") != digest:
            return None
        return float(fields["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, out_dir: str):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(out_dir, f"clocks_rank{gpu_index}.csv")
        self.windows = []

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "nvidia-smi unavailable"}
        rows = []
        import datetime
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        inwin = [r for r in rows if t0 - 0.02 <= r[0] <= t1 + 0.02]
        window = "timed"
        if len(inwin) < 3:
            inwin = [r for r in rows if r[0] <= t1 + 0.02]
            window = "warmup+timed (timed region shorter than the sampling interval)"
        if not inwin:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": window}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in inwin for k, v in enumerate(r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in inwin), "sm_max_mhz": max(r[2] for r in inwin),
                "reasons": reasons, "samples": len(inwin), "window": window}


# --------------------------------------------------------------------------
# timing helpers
# --------------------------------------------------------------------------

class Timer:
    """Per-step CUDA events on the current stream; an L2 flush before each step, outside the events."""

    def __init__(self, torch, device):
        self.torch = torch
        self.flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.clean_buf = torch.ones(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)

    def flush(self):
        self.flush_buf.zero_()   # evicts everything the last step left in L2
        self.clean_buf.amax()    # evicts the write's dirty lines (written back here, outside the events)

    def run(self, fn, steps: int, warmup: int, flush: bool = True):
        torch = self.torch
        for _ in range(warmup):
            if flush:
                self.flush()
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        from invariant_gradient_reduction_gb300 import detreduce as dr
        l0 = dr.det_kernel_launches()
        for s, e in ev:
            if flush:
                self.flush()
            s.record()
            fn()
            e.record()
        torch.cuda.synchronize()
        launches = dr.det_kernel_launches() - l0
        return [s.elapsed_time(e) for s, e in ev], launches


def gbs(nbytes: float, ms: float) -> float:
    return nbytes / (ms * 1e-3) / 1e9


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

def make_case(name, device, size="full"):
    from invariant_gradient_reduction_gb300 import workloads as wl
    return wl.make(name, size, device=device)


def scatter_step_fns(case, torch):
    from invariant_gradient_reduction_gb300 import detreduce as dr
    dev = case.x.device
    ws_plan = torch.empty(dr.det_plan_workspace_size(case.N, case.M) + 256, dtype=torch.uint8, device=dev)
    out = torch.empty(case.M, case.H, dtype=case.out_dtype, device=dev)
    state = {}

    # The step's plan does not wait for its counts (they stay on the device);
    # its error status is read once after the timed region (check_last_plan).
    def plan_and_reduce():
        p = dr.det_reduce_plan(case.idx, case.M, workspace=ws_plan, opts=ASYNC)
        dr.det_scatter_reduce(p, case.x, out, w=case.w, workspace=state.get("ws_red"), opts=ASYNC)
        state["plan"] = p

    plan0 = dr.det_reduce_plan(case.idx, case.M, workspace=ws_plan, opts=ASYNC)
    need = dr.det_scatter_workspace_size(plan0, case.H)  # the bound for an unwaited plan covers a waited one
    state["ws_red"] = torch.empty(need + 256, dtype=torch.uint8, device=dev) if need else None
    ws_plan_fixed = torch.empty_like(ws_plan)
    plan_fixed = dr.det_reduce_plan(case.idx, case.M, workspace=ws_plan_fixed)

    # the step's own gather kernel, for the roofline
    def reduce_only():
        dr.det_scatter_reduce(plan_fixed, case.x, out, w=case.w, workspace=state.get("ws_red"), opts=STEP_KERNEL)

    # the register-staged kernel on the same plan, for comparison
    def reduce_only_register():
        dr.det_scatter_reduce(plan_fixed, case.x, out, w=case.w, workspace=state.get("ws_red"), opts=REGISTER_KERNEL)

    ws_atomic = torch.empty(dr.det_atomic_workspace_size(case.M, case.H, case.out_dtype) + 256, dtype=torch.uint8,
                            device=dev)
    out_atomic = torch.empty_like(out)

    def atomic():
        dr.det_atomic_scatter_reduce(case.idx, case.M, case.x, out_atomic, w=case.w, workspace=ws_atomic)

    def check_last_plan():
        dr.det_plan_status(state.get("plan", plan0))

    state["reduce_only_register"] = reduce_only_register
    return plan_and_reduce, reduce_only, atomic, out, plan_fixed, check_last_plan, state


def measure_scatter(case, timer, steps, warmup, torch, with_e2e=True):
    from invariant_gradient_reduction_gb300 import detreduce as dr
    cb = case.compulsory_bytes()
    full, red, atom, out, plan, check_last_plan, st = scatter_step_fns(case, torch)
    t_full, l_full = timer.run(full, steps, warmup)
    check_last_plan()
    t_red, _ = timer.run(red, steps, warmup)
    t_atom, _ = timer.run(atom, steps, warmup)
    ms_full, ms_red, ms_atom = statistics.mean(t_full), statistics.mean(t_red), statistics.mean(t_atom)
    res = {
        "compulsory_bytes": cb,
        "plan_reduce": {"ms": ms_full, "gbs": gbs(cb, ms_full), "ms_median": statistics.median(t_full)},
        "reduce_only": {"ms": ms_red, "gbs": gbs(cb, ms_red), "ms_median": statistics.median(t_red)},
        "atomic": {"ms": ms_atom, "gbs": gbs(cb, ms_atom)},
        "overhead_vs_atomic": {"reduce_only": ms_red / ms_atom - 1.0, "plan_reduce": ms_full / ms_atom - 1.0},
        "launches_per_step": l_full / max(1, steps),
        "plan": {k: v for k, v in plan.describe().items() if k not in ("row_ptr", "perm")},
        "times_full": t_full,
        "launches_total": l_full,
    }
    h = dr.det_hash(out).item() & (2 ** 64 - 1)
    res["out_fingerprint"] = f"{h:016x}"
    if with_e2e:
        res["e2e"] = measure_e2e(case, timer, max(3, min(steps, 20)), warmup, torch)
    return res


def measure_e2e(case, timer, steps, warmup, torch):
    """Same step through the public API from pinned HOST buffers: H2D of x, idx, w, the
    plan and reduce, and the D2H of out, all inside each step's events."""
    from invariant_gradient_reduction_gb300 import detreduce as dr
    dev = case.x.device
    x_h = case.x.cpu().pin_memory()
    idx_h = case.idx.cpu().pin_memory()
    w_h = None if case.w is None else case.w.cpu().pin_memory()
    x_d, idx_d = torch.empty_like(case.x), torch.empty_like(case.idx)
    w_d = None if case.w is None else torch.empty_like(case.w)
    out_d = torch.empty(case.M, case.H, dtype=case.out_dtype, device=dev)
    out_h = torch.empty(out_d.shape, dtype=out_d.dtype).pin_memory()
    ws_plan = torch.empty(dr.det_plan_workspace_size(case.N, case.M) + 256, dtype=torch.uint8, device=dev)
    p0 = dr.det_reduce_plan(case.idx, case.M, opts=ASYNC)
    need = dr.det_scatter_workspace_size(p0, case.H)
    ws_red = torch.empty(need + 256, dtype=torch.uint8, device=dev) if need else None
    last = {"plan": p0}

    def step():
        x_d.copy_(x_h, non_blocking=True)
        idx_d.copy_(idx_h, non_blocking=True)
        if w_h is not None:
            w_d.copy_(w_h, non_blocking=True)
        p = dr.det_reduce_plan(idx_d, case.M, workspace=ws_plan, opts=ASYNC)
        dr.det_scatter_reduce(p, x_d, out_d, w=w_d, workspace=ws_red, opts=ASYNC)
        out_h.copy_(out_d, non_blocking=True)
        last["plan"] = p

    t, _ = timer.run(step, steps, warmup)
    dr.det_plan_status(last["plan"])
    ms = statistics.mean(t)
    bi = x_h.numel() * x_h.element_size() + idx_h.numel() * 4 + (0 if w_h is None else w_h.numel() * 4)
    bo = out_h.numel() * out_h.element_size()
    return {"value": gbs(case.compulsory_bytes(), ms), "unit": UNIT, "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "ms_per_step": ms, "steps": steps}


def measure_ep_invariance(timer, steps, warmup, torch, device, shard_counts=(1, 8)):
    """The EP-invariance MoE combine (T=16384, E=256, top-8, H=7168) with the
    sources split into P simulated expert shards (separate allocations): the
    step (unwaited plan + reduce) and the reduce alone per P, and each P's
    output fingerprint, which must all be equal."""
    from invariant_gradient_reduction_gb300 import detreduce as dr
    from invariant_gradient_reduction_gb300 import workloads as wl
    case = make_case("ep_invariance", device)
    cb = case.compulsory_bytes()
    out = torch.empty(case.M, case.H, dtype=case.out_dtype, device=device)
    ws_plan = torch.empty(dr.det_plan_workspace_size(case.N, case.M) + 256, dtype=torch.uint8, device=device)
    plan0 = dr.det_reduce_plan(case.idx, case.M, workspace=ws_plan, opts=ASYNC)
    need = dr.det_scatter_workspace_size(plan0, case.H)
    ws_red = torch.empty(need + 256, dtype=torch.uint8, device=device) if need else None
    plan_fixed = dr.det_reduce_plan(case.idx, case.M, workspace=torch.empty_like(ws_plan))
    res = {"compulsory_bytes": cb, "plan": {k: v for k, v in plan_fixed.describe().items()
                                            if k not in ("row_ptr", "perm")}}
    fps = {}
    for P in shard_counts:
        xs = case.x if P == 1 else wl.split_rows(case.x, wl.ep_shard_rows(case, P))
        state = {"plan": plan0}

        def step():
            p = dr.det_reduce_plan(case.idx, case.M, workspace=ws_plan, opts=ASYNC)
            dr.det_scatter_reduce(p, xs, out, w=case.w, workspace=ws_red, opts=ASYNC)
            state["plan"] = p

        t_full, l_full = timer.run(step, steps, warmup)
        dr.det_plan_status(state["plan"])
        t_red, _ = timer.run(lambda: dr.det_scatter_reduce(plan_fixed, xs, out, w=case.w, workspace=ws_red),
                             steps, warmup)
        torch.cuda.synchronize()
        fps[P] = dr.det_hash(out).item() & (2 ** 64 - 1)
        ms_full, ms_red = statistics.mean(t_full), statistics.mean(t_red)
        res[f"P{P}"] = {"plan_reduce": {"ms": ms_full, "gbs": gbs(cb, ms_full)},
                        "reduce_only": {"ms": ms_red, "gbs": gbs(cb, ms_red)},
                        "launches_per_step": l_full / max(1, steps), "out_fingerprint": f"{fps[P]:016x}"}
        del xs
    res["fingerprints_equal"] = len(set(fps.values())) == 1
    del case
    torch.cuda.empty_cache()
    return res


def measure_index_add(case, timer, steps, warmup, torch):
    """The embedding backward: det_index_add of dY rows into an fp32 gradient.
    Compulsory bytes: dY read once, idx once, each touched gradient row read
    and written once."""
    from invariant_gradient_reduction_gb300 import detreduce as dr
    dev = case.x.device
    touched = int((torch.bincount(case.idx.long(), minlength=case.M) > 0).sum().item())
    cb = case.N * case.H * case.x.element_size() + case.N * 4 + 2 * touched * case.H * 4
    grad = torch.zeros(case.M, case.H, dtype=torch.float32, device=dev)
    ws_plan = torch.empty(dr.det_plan_workspace_size(case.N, case.M) + 256, dtype=torch.uint8, device=dev)
    plan0 = dr.det_reduce_plan(case.idx, case.M, workspace=ws_plan, opts=ASYNC)
    need = dr.det_scatter_workspace_size(plan0, case.H)
    ws_red = torch.empty(need + 256, dtype=torch.uint8, device=dev) if need else None
    state = {"plan": plan0}

    def full():
        p = dr.det_reduce_plan(case.idx, case.M, workspace=ws_plan, opts=ASYNC)
        dr.det_index_add(p, case.x, grad, workspace=ws_red, opts=ASYNC)
        state["plan"] = p

    ws_fixed = torch.empty_like(ws_plan)
    plan_fixed = dr.det_reduce_plan(case.idx, case.M, workspace=ws_fixed)
    ws_atomic = torch.empty(dr.det_atomic_workspace_size(case.M, case.H, torch.float32) + 256, dtype=torch.uint8,
                            device=dev)
    t_full, l_full = timer.run(full, steps, warmup)
    dr.det_plan_status(state["plan"])
    t_red, _ = timer.run(lambda: dr.det_index_add(plan_fixed, case.x, grad, workspace=ws_red), steps, warmup)
    t_atom, _ = timer.run(lambda: dr.det_atomic_index_add(case.idx, case.M, case.x, grad, workspace=ws_atomic),
                          steps, warmup)
    ms_full, ms_red, ms_atom = statistics.mean(t_full), statistics.mean(t_red), statistics.mean(t_atom)
    d = plan_fixed.describe()
    return {"compulsory_bytes": cb, "touched_rows": touched,
            "plan_index_add": {"ms": ms_full, "gbs": gbs(cb, ms_full)},
            "index_add_only": {"ms": ms_red, "gbs": gbs(cb, ms_red)},
            "atomic_index_add": {"ms": ms_atom, "gbs": gbs(cb, ms_atom)},
            "overhead_vs_atomic": {"index_add_only": ms_red / ms_atom - 1.0, "plan_index_add": ms_full / ms_atom - 1.0},
            "launches_per_step": l_full / max(1, steps),
            "plan": {k: v for k, v in d.items() if k not in ("row_ptr", "perm")}}


def measure_moe_route(timer, steps, warmup, torch, device):
    """The MoE combine driven by the route plan: router scores (T=4096, E=128) ->
    sorted top-8 (renormalised) -> dispatch layout + combine plan from the ids
    -> the combine of bf16 expert outputs [32768, 4096] in dispatch order.
    Compulsory bytes as for the MoE combine (x, out, ids, weights); the
    top-k leg adds the scores."""
    from invariant_gradient_reduction_gb300 import detreduce as dr
    from invariant_gradient_reduction_gb300 import workloads as wl
    T, E, k, H = 4096, 128, 8, 4096
    N = T * k
    scores = wl.router_scores(T, E, seed=2, device=device)
    ids, tw = dr.det_router_topk(scores, k, renormalize=True)
    x = wl._fill_normal((N, H), torch.bfloat16, 1.0, 2 * 7919 + 1, device)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=device)
    ws = torch.empty(dr.det_moe_route_workspace_size(T, k, E, ASYNC) + 256, dtype=torch.uint8, device=device)
    arrays = {"expert_offsets": torch.empty(E + 1, dtype=torch.int32, device=device),
              "row_token": torch.empty(N, dtype=torch.int32, device=device),
              "row_w": torch.empty(N, dtype=torch.float32, device=device), "slot_row": None}
    topk_out = (torch.empty_like(ids), torch.empty_like(tw))
    state = {}

    def route():
        p, _ = dr.det_moe_route_plan(ids, E, tw, opts=ASYNC, workspace=ws, out=arrays)
        state["plan"] = p
        return p

    def route_combine():
        dr.det_scatter_reduce(route(), x, out, w=arrays["row_w"], opts=ASYNC)

    def topk_route_combine():
        dr.det_router_topk(scores, k, renormalize=True, out=topk_out)
        p, _ = dr.det_moe_route_plan(topk_out[0], E, topk_out[1], opts=ASYNC, workspace=ws, out=arrays)
        state["plan"] = p
        dr.det_scatter_reduce(p, x, out, w=arrays["row_w"], opts=ASYNC)

    ws_dest = torch.empty(dr.det_plan_workspace_size(N, T) + 256, dtype=torch.uint8, device=device)

    def dest_combine():
        p = dr.det_reduce_plan(arrays["row_token"], T, workspace=ws_dest, opts=ASYNC)
        state["plan"] = p
        dr.det_scatter_reduce(p, x, out, w=arrays["row_w"], opts=ASYNC)

    res = {}
    cb = N * H * 2 + T * H * 2 + N * 4 + N * 4
    for name, fn, nbytes in (("route_plan_combine", route_combine, cb),
                             ("topk_route_plan_combine", topk_route_combine, cb + T * E * 4),
                             ("destination_plan_combine", dest_combine, cb),
                             ("route_plan_only", route, None),
                             ("route_plan_only_multi_kernel",
                              lambda: state.__setitem__("plan", dr.det_moe_route_plan(
                                  ids, E, tw, opts={**ASYNC, "plan_path": 1}, workspace=ws, out=arrays)[0]), None),
                             ("router_topk_only", lambda: dr.det_router_topk(scores, k, renormalize=True,
                                                                             out=topk_out), None)):
        t, launches = timer.run(fn, steps, warmup)
        if "plan" in state:
            dr.det_plan_status(state.pop("plan"))
        ms = statistics.mean(t)
        r = {"ms": ms, "launches_per_step": launches / max(1, steps)}
        if nbytes:
            r["gbs"] = gbs(nbytes, ms)
        res[name] = r
    fp = dr.det_hash(out).item() & (2 ** 64 - 1)
    return {"compulsory_bytes": cb, "fingerprint": f"{fp:016x}", **res}


def measure_splitk(timer, steps, warmup, torch, device):
    from invariant_gradient_reduction_gb300 import detreduce as dr
    from invariant_gradient_reduction_gb300 import workloads as wl
    P = wl.make("splitk", "full", device=device)
    res = {}
    for name, odt in (("f32_out", torch.float32), ("bf16_out", torch.bfloat16)):
        out = torch.empty(P.shape[1], dtype=odt, device=device)
        t, l = timer.run(lambda: dr.det_splitk_reduce(P, out), steps, warmup)
        cb = P.numel() * 4 + out.numel() * out.element_size()
        ms = statistics.mean(t)
        res[name] = {"ms": ms, "gbs": gbs(cb, ms), "compulsory_bytes": cb, "launches_per_step": l / steps}
    return res


def measure_splitk_gemm(timer, steps, warmup, torch, device, peaks):
    """The split-K producer with the fold in its epilogue (mHC-like shape: 16384
    rows, K = 7168 in 56 splits of 128, 24 columns), against the same producer
    writing its 56 partials to memory followed by det_splitk_reduce over them.
    Compulsory bytes of the fused step: A and W read once, out written once."""
    from invariant_gradient_reduction_gb300 import detreduce as dr
    from invariant_gradient_reduction_gb300 import workloads as wl
    R, K, C, S = 16384, 7168, 24, 56
    A, W = wl.splitk_gemm_inputs(R, K, C, seed=5, device=device)
    out = torch.empty(R, C, dtype=torch.float32, device=device)
    out2 = torch.empty(R * C, dtype=torch.float32, device=device)
    scratch = torch.empty(R, C, dtype=torch.float32, device=device)
    P = torch.empty(S, R * C, dtype=torch.float32, device=device)
    t_f, l_f = timer.run(lambda: dr.det_splitk_gemm_reduce(A, W, S, out), steps, warmup)

    def unfused():
        dr.det_splitk_gemm_reduce(A, W, S, scratch, partials=P)
        dr.det_splitk_reduce(P, out2)

    t_u, l_u = timer.run(unfused, steps, warmup)
    torch.cuda.synchronize()
    same = bool(torch.equal(out.view(-1).view(torch.int32), out2.view(torch.int32)))
    cb = R * K * 2 + C * K * 2 + R * C * 4
    ms_f, ms_u = statistics.mean(t_f), statistics.mean(t_u)
    flops = 2.0 * R * K * C
    return {"workload": f"split-K GEMM A bf16 [{R},{K}] x W bf16 [{C},{K}]^T, K in {S} splits of {K // S}, "
                        f"fold over splits in the epilogue, fp32 out [{R},{C}]",
            "compulsory_bytes": cb,
            "fused": {"ms": ms_f, "gbs": gbs(cb, ms_f), "frac_hbm": gbs(cb, ms_f) / peaks["hbm_gbs"],
                      "tflops": flops / (ms_f * 1e-3) / 1e12, "launches_per_step": l_f / max(1, steps)},
            "partials_then_reduce": {"ms": ms_u, "gbs": gbs(cb, ms_u), "launches_per_step": l_u / max(1, steps),
                                     "partial_bytes": S * R * C * 4},
            "same_output_bits": same}


def oracle_sample_seconds(case, max_rows: int):
    """Run the CPU oracle once on the first max_rows destinations and all their sources.
    Returns (seconds, compulsory bytes of the sample, description)."""
    import numpy as np
    import torch

    import oracle
    idx = case.idx.cpu().numpy().astype(np.int32)
    rows = min(case.M, max_rows)
    keep = idx < rows
    xs = case.x.cpu()[torch.from_numpy(keep)]
    x_np = xs.view(torch.int16).numpy().view(np.uint16) if xs.dtype == torch.bfloat16 else xs.numpy()
    w_np = None if case.w is None else case.w.cpu().numpy()[keep]
    od = oracle.F32 if case.out_dtype == torch.float32 else oracle.BF16
    sub_idx = idx[keep]
    t0 = time.perf_counter()
    oracle.scatter_reduce(sub_idx, x_np, rows, w=w_np, out_dtype=od)
    dt = time.perf_counter() - t0
    n = int(keep.sum())
    cb = n * case.H * case.x.element_size() + n * 4 + (0 if case.w is None else n * 4) + \
        rows * case.H * (4 if case.out_dtype == torch.float32 else 2)
    return dt, cb, f"first {rows} of {case.M} destinations and their {n} sources ({cb} compulsory bytes)"


def host_cpu():
    """The host CPU model and the number of CPUs this process may run on."""
    model = platform.processor() or platform.machine()
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                k, _, v = line.partition(":")
                if k.strip() in ("model name", "Model Name", "CPU part") and v.strip():
                    model = v.strip()
                    if k.strip() != "CPU part":
                        break
    except OSError:
        pass
    try:
        ncpu = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        ncpu = os.cpu_count() or 1
    return {"model": model, "machine": platform.machine(), "nproc": ncpu}


def pinned_to_one_core():
    """Pin this thread to the first CPU it may run on (the oracle is single-threaded);
    returns (that CPU, the previous affinity) or (None, None) where pinning is not available."""
    try:
        prev = os.sched_getaffinity(0)
        cpu = min(prev)
        os.sched_setaffinity(0, {cpu})
        return cpu, prev
    except (AttributeError, OSError, ValueError):
        return None, None


def cpu_baseline(case, budget_s: float = 20.0):
    import oracle
    oracle.build()
    host = host_cpu()
    cpu, prev = pinned_to_one_core()
    try:
        res = _cpu_baseline_runs(case, budget_s)
    finally:
        if prev is not None:
            os.sched_setaffinity(0, prev)
    res["host"] = dict(host, pinned_cpu=cpu)
    return res


def _cpu_baseline_runs(case, budget_s):
    import oracle
    rows = min(case.M, 256)
    dt, cb, desc = oracle_sample_seconds(case, rows)
    # grow the sample towards ~1/3 of the budget per run, then take the median of 3 runs
    if dt < budget_s / 9 and rows < case.M:
        rows = min(case.M, int(rows * max(1.0, (budget_s / 9) / max(dt, 1e-3))))
    runs = []
    for _ in range(3):
        dt, cb, desc = oracle_sample_seconds(case, rows)
        runs.append(dt)
        if sum(runs) > budget_s:
            break
    s = statistics.median(runs)
    return {"value": gbs(cb, s * 1e3), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{desc}; median of {len(runs)} run(s), single thread", "seconds": s}


def run_ours(args):
    import torch
    import torch.distributed as tdist

    rank, local_rank, world = dist_env()
    if world > 1:
        tdist.init_process_group(backend="nccl", init_method="env://")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)

    from invariant_gradient_reduction_gb300 import build as libbuild
    libbuild.build()
    from invariant_gradient_reduction_gb300 import detreduce as dr
    dr.lib()

    peaks = read_peaks()
    timer = Timer(torch, device)
    case = make_case(args.workload, device, args.size)
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank, args.clocks_dir).start()
    time.sleep(0.1)
    # warm-up, then exactly K timed steps bracketed by barrier + synchronize
    full, red, atom, out, plan, check_last_plan, st = scatter_step_fns(case, torch)
    for _ in range(args.warmup):
        timer.flush()
        full()
    if world > 1:
        tdist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    l0 = dr.det_kernel_launches()
    for s, e in ev:
        timer.flush()
        s.record()
        full()
        e.record()
    torch.cuda.synchronize()
    launches = dr.det_kernel_launches() - l0
    check_last_plan()
    if world > 1:
        tdist.barrier()
    t_wall1 = time.time()
    times = [s.elapsed_time(e) for s, e in ev]
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    ms_step = sum(times) / len(times)

    # reduce-only (the dominant kernel, for the roofline) and the atomic baseline
    t_red, _ = timer.run(red, args.steps, args.warmup)
    t_reg, _ = timer.run(st["reduce_only_register"], args.steps, args.warmup)
    t_atom, _ = timer.run(atom, args.steps, args.warmup)
    ms_red, ms_atom = statistics.mean(t_red), statistics.mean(t_atom)
    ms_reg = statistics.mean(t_reg)
    cb = case.compulsory_bytes()
    fingerprint = dr.det_hash(out).item() & (2 ** 64 - 1)

    local = {"ms_step": ms_step, "ms_red": ms_red, "ms_reg": ms_reg, "ms_atom": ms_atom, "launches": launches,
             "wall_ms_per_step": (t_wall1 - t_wall0) * 1e3 / args.steps, "fingerprint": fingerprint}
    if world > 1:
        gathered = [None] * world
        tdist.all_gather_object(gathered, local)
    else:
        gathered = [local]
    agg = combine_ranks(gathered)

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(case, timer, max(3, min(args.steps, 20)), args.warmup, torch)
        if world > 1:
            ge = [None] * world
            tdist.all_gather_object(ge, e2e["ms_per_step"])
            e2e["ms_per_step"] = max(ge)
            e2e["value"] = world * gbs(cb, e2e["ms_per_step"])

    also = {}
    wanted = set(a for a in args.also.split(",") if a)
    if not args.no_also and rank == 0:
        if "sparse_key_scatter" in wanted and args.workload != "sparse_key_scatter":
            c2 = make_case("sparse_key_scatter", device)
            r2 = measure_scatter(c2, timer, max(5, min(args.steps, 30)), args.warmup, torch, with_e2e=False)
            r2.pop("times_full", None)
            r2["frac_reduce_only"] = r2["reduce_only"]["gbs"] / peaks["hbm_gbs"]
            r2["workload"] = WORKLOADS["sparse_key_scatter"]
            also["sparse_key_scatter"] = r2
            del c2
            torch.cuda.empty_cache()
        if "ep_invariance" in wanted and args.workload != "ep_invariance":
            r5 = measure_ep_invariance(timer, max(5, min(args.steps, 20)), args.warmup, torch, device)
            for P in (1, 8):
                r5[f"P{P}"]["frac_plan_reduce"] = r5[f"P{P}"]["plan_reduce"]["gbs"] / peaks["hbm_gbs"]
                r5[f"P{P}"]["frac_reduce_only"] = r5[f"P{P}"]["reduce_only"]["gbs"] / peaks["hbm_gbs"]
            r5["workload"] = WORKLOADS["ep_invariance"]
            also["ep_invariance"] = r5
        if "moe_route" in wanted:
            r4 = measure_moe_route(timer, max(5, min(args.steps, 30)), args.warmup, torch, device)
            r4["frac_route_plan_combine"] = r4["route_plan_combine"]["gbs"] / peaks["hbm_gbs"]
            r4["workload"] = WORKLOADS["moe_route"]
            also["moe_route"] = r4
            torch.cuda.empty_cache()
        if "splitk" in wanted:
            also["splitk"] = measure_splitk(timer, max(10, min(args.steps, 50)), args.warmup, torch, device)
            also["splitk"]["workload"] = WORKLOADS["splitk"]
        if "splitk_gemm" in wanted:
            also["splitk_gemm"] = measure_splitk_gemm(timer, max(10, min(args.steps, 50)), args.warmup, torch, device,
                                                      peaks)
            torch.cuda.empty_cache()
        if "embedding_backward" in wanted:
            c3 = make_case("embedding_backward", device)
            r3 = measure_index_add(c3, timer, max(5, min(args.steps, 30)), args.warmup, torch)
            r3["frac_index_add_only"] = r3["index_add_only"]["gbs"] / peaks["hbm_gbs"]
            r3["workload"] = WORKLOADS["embedding_backward"]
            also["embedding_backward"] = r3
            del c3
            torch.cuda.empty_cache()

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        cpu = cpu_baseline(case)

    if rank == 0:
        red_gbs = gbs(cb, agg["ms_red"])
        rk_name, rk_file = ROOFLINE_KERNEL[args.workload]
        traffic = read_traffic(rk_file, args.workload)
        line = {
            "metric": METRIC,
            "value": world * gbs(cb, agg["ms_step"]),
            "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": agg["ms_step"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOADS[args.workload] + ("" if args.size == "full" else f" [{args.size}]"),
                       "step": "plan (histogram+scan+stable sort+work list) + gather-reduce",
                       "l2": "flushed before every timed step, outside the step events: 256 MiB write, then 256 MiB read "
                             "of another buffer (the write-back of the dirty lines happens before the events)",
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "compulsory_bytes_per_step": cb},
            "roofline": {"kernel": rk_name, "bound": "hbm",
                         "achieved": red_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": red_gbs / peaks["hbm_gbs"], "traffic": traffic,
                         "peak_source": peaks["source"] + " copy bandwidth (burst)",
                         "algorithmic_bytes_per_launch": cb, "launch_ms": agg["ms_red"]},
            "reduce_only": {"value": world * red_gbs, "ms": agg["ms_red"], "kernel": rk_name},
            "reduce_only_register": {"value": world * gbs(cb, agg["ms_reg"]), "ms": agg["ms_reg"],
                                     "kernel": "gather_reduce_kernel (the register-staged kernel, gather_path 1)"},
            "atomic": {"ms": agg["ms_atom"], "value": world * gbs(cb, agg["ms_atom"]),
                       "overhead_reduce_only": agg["ms_red"] / agg["ms_atom"] - 1.0,
                       "overhead_plan_reduce": agg["ms_step"] / agg["ms_atom"] - 1.0},
            "e2e": e2e,
            "gpu_launches": agg["launches"],
            "clocks": clocks,
            "wall_ms_per_step": agg["wall_ms_per_step"],
            "out_fingerprint": f"{agg['fingerprint']:016x}",
            "cpu_baseline": cpu,
            "also": also or None,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        tdist.barrier()
        tdist.destroy_process_group()


def combine_ranks(per_rank):
    """Max over ranks of the timed quantities; launches summed; fingerprints must agree."""
    fps = {r["fingerprint"] for r in per_rank}
    if len(fps) != 1:
        raise RuntimeError(f"replicas disagree on the output fingerprint: {sorted(fps)}")
    return {"ms_step": max(r["ms_step"] for r in per_rank), "ms_red": max(r["ms_red"] for r in per_rank),
            "ms_reg": max(r["ms_reg"] for r in per_rank),
            "ms_atom": max(r["ms_atom"] for r in per_rank), "launches": sum(r["launches"] for r in per_rank),
            "wall_ms_per_step": max(r["wall_ms_per_step"] for r in per_rank), "fingerprint": fps.pop()}


# --------------------------------------------------------------------------
# reference arm: the CPU oracle
# --------------------------------------------------------------------------

def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    host = host_cpu()
    cpu, _prev = pinned_to_one_core()
    from invariant_gradient_reduction_gb300 import workloads as wl
    case = wl.make(args.workload, "full", device="cpu")
    # each step: the oracle on a bounded sample (a prefix of the destinations and their sources)
    rows = 128
    dt, cb, desc = oracle_sample_seconds(case, rows)
    target = 2.0  # seconds per step
    rows = max(1, min(case.M, int(rows * target / max(dt, 1e-3))))
    for _ in range(args.warmup):
        dt, cb, desc = oracle_sample_seconds(case, rows)
    times = []
    for _ in range(args.steps):
        dt, cb, desc = oracle_sample_seconds(case, rows)
        times.append(dt)
    ms = statistics.mean(times) * 1e3
    v = gbs(cb, ms)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload], "step": "CPU oracle (lists + canonical fold) on a sample",
                   "parallelism": "single thread"},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc,
                         "host": dict(host, pinned_cpu=cpu)},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
