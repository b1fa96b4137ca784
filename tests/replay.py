"""Replay harness: the pages' determinism tests as one reusable tool.

The Megatron-LM determinism developer reference (sections 4.4 and 4.5) checks
a kernel by replaying it and comparing bytes: R runs on the same inputs must
give identical bytes, also while other work contends for the GPU, and a
negative control (an order-dependent kernel on the same inputs) must show that
the comparison is able to see a difference.  Fingerprints of every call are
logged so that runs on different days or machines can be compared.

    def test_x(replay):
        out = replay.identical(lambda: run_kernel(...), name="x")   # asserts
        assert replay.differing(lambda: run_atomic(...)) > 0       # control
"""
from __future__ import annotations

import json
import os
from typing import Callable, List, Optional

import torch


class Replay:
    def __init__(self, runs: int = 5, contention: bool = True, matmul_size: int = 2048):
        self.runs = runs
        self.contention = contention
        self.matmul_size = matmul_size
        self.log: List[dict] = []
        self._side = None
        self._a = None

    def _contend(self):
        """Queue matmuls on a side stream, so that they run while the call under test runs."""
        if not self.contention:
            return
        if self._side is None:
            self._side = torch.cuda.Stream()
            self._a = torch.randn(self.matmul_size, self.matmul_size, device="cuda")
        with torch.cuda.stream(self._side):
            for _ in range(4):
                self._a = self._a @ self._a.T * 1e-3

    @staticmethod
    def _bytes(t: torch.Tensor) -> bytes:
        return t.detach().contiguous().view(torch.uint8).cpu().numpy().tobytes()

    def _fingerprint(self, t: torch.Tensor) -> int:
        from invariant_gradient_reduction_gb300 import detreduce as dr
        return int(dr.det_hash(t.detach().contiguous()).item()) & (2 ** 64 - 1)

    def identical(self, fn: Callable[[], torch.Tensor], name: str = "call") -> torch.Tensor:
        """Run fn() `runs` times (with contention); every result must have the same
        bytes and the same fingerprint.  Returns the first result."""
        first = None
        first_bytes = None
        for r in range(self.runs):
            self._contend()
            out = fn()
            torch.cuda.synchronize()
            fp = self._fingerprint(out)
            self.log.append({"call": name, "run": r, "fingerprint": f"{fp:016x}"})
            b = self._bytes(out)
            if first is None:
                first, first_bytes, first_fp = out.clone(), b, fp
            else:
                assert fp == first_fp, f"{name}: replay {r} fingerprint {fp:016x} != {first_fp:016x}"
                assert b == first_bytes, f"{name}: replay {r} differs in its bytes"
        return first

    def differing(self, fn: Callable[[], torch.Tensor], name: str = "control") -> int:
        """Negative control: the number of runs of fn() whose bytes differ from the first run."""
        first = None
        n = 0
        for r in range(self.runs):
            self._contend()
            out = fn()
            torch.cuda.synchronize()
            b = self._bytes(out)
            self.log.append({"call": name, "run": r, "fingerprint": f"{self._fingerprint(out):016x}"})
            if first is None:
                first = b
            elif b != first:
                n += 1
        return n

    def write_log(self, path: Optional[str], test: str):
        if not path or not self.log:
            return
        with open(path, "a") as fh:
            for e in self.log:
                fh.write(json.dumps(dict(e, test=test)) + "\n")
