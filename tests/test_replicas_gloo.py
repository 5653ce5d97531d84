"""Host logic of the benchmark on the CPU.  Multi-replica (gloo, world size
2): the timings reduce to their maximum over ranks, and only rank 0 of the
reference arm does any work; the data path has no collective (replicas
only), so this is the whole multi-process surface.  Also the source hash
that decides whether a committed DRAM-traffic record still applies."""

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        v = torch.tensor([10.0 + rank, 5.0 - rank, 1.5], dtype=torch.float64)
        out = bench.max_over_ranks(v, world)
        q.put((rank, [float(x) for x in out.tolist()]))
    finally:
        dist.destroy_process_group()


def test_timings_reduce_to_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(2):
        rank, vals = q.get(timeout=120)
        got[rank] = vals
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0] == got[1] == [11.0, 5.0, 1.5]


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import torch
    import bench
    v = torch.tensor([3.0, 4.0], dtype=torch.float64)
    assert bench.max_over_ranks(v, 1) is v


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    args = bench.argparse.Namespace(workload="b1_64k", steps=1, warmup=0, gpus=2, num_splits=0)
    assert bench.run_reference(args, rank=1, world=2) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_the_gpu_arm_config(capsys):
    """The oracle arm's `config` is the object the GPU arm prints for the same
    workload: the library heuristic's split count (its oracle mirror), the
    same rotating-copy count, parallelism and L2 note; its cpu_baseline is the
    best step over the same fixed sample."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    from decode_attention_20_b300 import _lib
    args = bench.argparse.Namespace(workload="tiny_fp32", steps=2, warmup=1, gpus=1, num_splits=0)
    assert bench.run_reference(args, rank=0, world=1) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    w = bench.make_workload("tiny_fp32", "cpu")          # as the GPU arm builds it (with copies)
    ns = _lib.lib().fd_choose_num_splits(w.B, w.Hkv, w.Lcap, bench.num_sms_for_config())
    assert line["config"] == bench.line_config(w, ns, 1)
    assert line["steps"] == 2 and line["impl"] == "reference"
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "us/call", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_rotation_copies_exceed_l2():
    """Rotating input copies always span more than twice L2 (up to the cap),
    so a timed call never finds its K/V resident."""
    sys.path.insert(0, ROOT)
    import bench
    for per_copy in [1 << 20, 2 << 20, 50 << 20, 126 << 20, 268 << 20, 2 << 30]:
        n = bench.rotation_copies(per_copy)
        assert n * per_copy > 2 * bench.L2_BYTES or n == 512
        assert n >= 1


def test_traffic_hash_ignores_comments_not_code():
    """The DRAM-traffic records stay valid across comment edits of a kernel's
    sources and lapse on any code edit."""
    import bench
    src = {n: "int a = 1;  // one\n/* block\n comment */ int b = 2;\n" for n in
           bench.KERNEL_SOURCES[bench.FD_KERNEL_SPLIT]}
    h0 = bench.kernel_source_hash(bench.FD_KERNEL_SPLIT, src.__getitem__)
    recommented = {n: "int a = 1;   // another comment\nint b = 2;  /* x */\n" for n in src}
    assert bench.kernel_source_hash(bench.FD_KERNEL_SPLIT, recommented.__getitem__) == h0
    changed = {n: "int a = 1;\nint b = 3;\n" for n in src}
    assert bench.kernel_source_hash(bench.FD_KERNEL_SPLIT, changed.__getitem__) != h0
