"""Host logic of bench.py without a GPU: argument defaults, the max-over-ranks
aggregation (also across two gloo ranks), and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_args_defaults_and_minimum_warmup():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1 and a.impl == "ours"
    assert bench.parse_args(["--warmup", "1"]).warmup == 3
    # every secondary workload runs by default and has a description; the clock samples stay in the repo
    assert set(a.also.split(",")) == {"sparse_key_scatter", "ep_invariance", "moe_route", "splitk", "splitk_gemm",
                                      "embedding_backward"}
    assert all(w in bench.WORKLOADS for w in a.also.split(","))
    assert a.clocks_dir.startswith(ROOT)
    assert bench.parse_args(["--also", "moe_route"]).also == "moe_route"


def test_cpu_baseline_host_record_and_pinning():
    """The CPU baseline records the host CPU and runs pinned to one core, then restores the affinity."""
    h = bench.host_cpu()
    assert h["model"] and h["nproc"] >= 1 and h["machine"]
    before = os.sched_getaffinity(0)
    cpu, prev = bench.pinned_to_one_core()
    try:
        assert cpu in before and os.sched_getaffinity(0) == {cpu}
    finally:
        os.sched_setaffinity(0, prev)
    assert os.sched_getaffinity(0) == before


def _rank(n, ms, fp=7):
    return {"ms_step": ms, "ms_red": ms / 2, "ms_reg": ms / 2, "ms_atom": ms / 3, "launches": n, "wall_ms_per_step": ms * 1.1,
            "fingerprint": fp}


def test_combine_ranks_takes_the_slowest_rank():
    agg = bench.combine_ranks([_rank(10, 1.0), _rank(10, 2.0)])
    assert agg["ms_step"] == 2.0 and agg["ms_red"] == 1.0 and agg["launches"] == 20
    with pytest.raises(RuntimeError):
        bench.combine_ranks([_rank(10, 1.0, fp=1), _rank(10, 1.0, fp=2)])


def _worker(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    local = _rank(11, 1.0 + rank)
    gathered = [None] * world
    tdist.all_gather_object(gathered, local)
    agg = bench.combine_ranks(gathered)
    if rank == 0:
        with open(out_path, "w") as fh:
            json.dump(agg, fh)
    tdist.barrier()
    tdist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_aggregate(tmp_path):
    out = tmp_path / "agg.json"
    mp.start_processes(_worker, args=(2, _free_port(), str(out)), nprocs=2, start_method="spawn")
    agg = json.load(open(out))
    assert agg["ms_step"] == 2.0 and agg["launches"] == 22


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["metric"] == bench.METRIC


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"], capture_output=True,
                       text=True, timeout=120, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""
