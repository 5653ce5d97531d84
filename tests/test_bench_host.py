"""Host-side measurement logic of bench.py that needs no GPU: the e2e loop's
median-of-blocks timing and the GPU line's cpu_baseline taken from the
reference arm run as a subprocess."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_host_loop_median_ignores_one_stalled_block(monkeypatch):
    import time

    import torch

    import bench
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a, **k: None)
    calls = []

    def step(i):
        calls.append(i)
        # warm-up calls are 0..4; the first timed block (steps 0..9) stalls
        if len(calls) == 5 + 3:
            time.sleep(0.05)

    us = bench._host_loop_us(None, 50, step, warmup=5, blocks=5)
    assert len(calls) == 5 + 50
    assert calls[5:] == list(range(50))          # the timed steps see indices 0..49
    assert us < 2000.0, us                       # a 50 ms stall would add 5000 us per step to its block


def test_host_loop_uses_whole_blocks(monkeypatch):
    import torch

    import bench
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a, **k: None)
    calls = []
    bench._host_loop_us(None, 7, calls.append, warmup=0, blocks=5)
    assert calls == list(range(5))               # 7 steps in 5 blocks: one step per block


def test_cpu_baseline_comes_from_the_reference_arm():
    import bench
    w = bench.make_workload("tiny_fp32", "cpu", copies=False)
    cb = bench.cpu_baseline_ref_arm(w, "tiny_fp32")
    assert cb["kind"] == "oracle" and cb["unit"] == "us/call"
    assert "measured by the reference arm in a separate process" in cb["sample"]
    assert cb["value"] > 0 and cb["cores"] >= 1


def test_cpu_baseline_falls_back_in_process(monkeypatch):
    import subprocess

    import bench

    def broken(*a, **k):
        raise subprocess.TimeoutExpired(cmd="bench.py", timeout=1)

    monkeypatch.setattr(bench.subprocess, "run", broken)
    w = bench.make_workload("tiny_fp32", "cpu", copies=False)
    cb = bench.cpu_baseline_ref_arm(w, "tiny_fp32")
    assert "the reference arm subprocess gave no line" in cb["sample"]
    assert cb["value"] > 0
