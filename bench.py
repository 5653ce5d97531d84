"""Benchmark of the decode-attention hot path on one B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fd|reference]
                    [--workload b1_64k|ragged_b32|long_b4|bif_mqa|paged_b1_64k|
                                int8_b1_64k|e4m3_b1_64k|verify4_b1_64k]
                    [--num-splits S] [--bif-sweep]

Default workload: split-KV decode attention at batch 1 over a 65536-token
history of a CodeLlama-34B-shaped layer (64 query heads, 8 kv heads, head
dim 128, bf16 K/V, fp32 out + LSE).  One call = split kernel + log-sum-exp
combine over the whole history; a timed step replays a graph of such calls.
Other workloads:
  ragged_b32  batch 32, 32/8 heads, padded [32, 32768, 8, 128] cache, lengths
              uniform in [1024, 32768]
  long_b4     batch 4, 131072 tokens, 32/8 heads, 1% of keys scaled by 8
  bif_mqa     bifurcated attention: 64 samples share an 8192-token context,
              256 own decode tokens each, 32 query heads on 1 kv head; the
              line also carries the replicated-context decode time
  paged_b1_64k the batch-1 64K layer with its history in 64-token pages
              scattered by a seeded permutation (paged KV cache)
  int8_b1_64k, e4m3_b1_64k
              the batch-1 64K layer over an 8-bit cache (int8 or e4m3 codes,
              one fp32 scale per kv head for K and for V)
  verify4_b1_64k
              the batch-1 64K layer verifying 4 new query positions per
              sequence (causal among them)
  --bif-sweep bifurcated vs replicated-context timings over samples,
              context lengths and kv heads (a measurement aid, not a line)
Prints ONE JSON line (rank 0):
  value        device-timed microseconds per call.  Exactly --steps timed
               steps (after --warmup untimed ones); a step is one replay of a
               CUDA graph of C back-to-back calls over rotating input copies
               that together exceed L2 (C sized so that the steps span about
               --window-ms); CUDA events on the launching stream, a barrier
               and a synchronise on both sides.  ms_per_step is one step.
  e2e          microseconds per step through the Python API: one H2D from
               pinned host memory of the step's new inputs (query, one new K/V
               row per sequence, packed in one buffer), the rows written into
               the cache, the call, one D2H of out + lse (one buffer),
               synchronised per step; host wall clock, the median of five
               equal blocks of steps
  roofline     the dominant kernel's algorithmic bytes (or FLOPs) per launch /
               its mean CUDA-event duration (launches queued back to back,
               without programmatic dependent launch), against the peak
  configs      (default workload, one GPU) the other workloads measured the
               same way: the tiny fp32 case, the batch-1 layer at 512..32K
               tokens (graph and direct-call microseconds), the ragged batch,
               bifurcated sampling with its replicated-context comparison, and
               the long peaked context
  cpu_baseline the fp64 CPU oracle, best of 3 timings of a fixed sample of
               the same workload on the host cores (rank 0, N = 1)
With --gpus N > 1 (torchrun), every rank runs an independent replica (the
method has no cross-GPU exchange); value is the max over ranks.

--impl reference times the fp64 CPU oracle instead (each step one timing of
the same fixed sample, extrapolated to one full call; value the best step),
with the same config object.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "split-KV decode attention µs/call and achieved HBM GB/s vs ~8 TB/s peak"
L2_BYTES = 126 << 20
FD_KERNEL_SPLIT, FD_KERNEL_COMBINE, FD_KERNEL_BIF_CTX = 0, 1, 2
KERNEL_NAMES = {FD_KERNEL_SPLIT: "split_mma_kernel (mma.sync bf16, TMA ring)",
                FD_KERNEL_BIF_CTX: "bif_ctx_kernel (tcgen05.mma, TMEM accumulators)"}


# Cycles of torch.cuda._sleep per microsecond: the maximum SM clock of a
# B300 (2032 MHz), rounded up, so a delay is at least as long as asked.
SLEEP_CYCLES_PER_US = 2100


def rotation_copies(per_copy_bytes):
    """Input copies a timed loop rotates over so that no call finds its K/V
    in L2: enough copies to cover twice the L2 size, plus one when a copy is
    smaller than four times L2 (its tail may still be resident); at most 512
    (a 512-token batch-1 layer is 2 MiB, so 127 copies)."""
    n = math.ceil(2 * L2_BYTES / max(1, per_copy_bytes))
    n += 1 if per_copy_bytes < 4 * L2_BYTES else 0
    return max(1, min(512, n))

# Source files each roofline kernel is built from: a DRAM-traffic figure in
# profiles/traffic.json is used only while their code (comments and
# whitespace aside) hashes to the value it was captured with; otherwise the
# kernel has changed and traffic is null.
# The kernel's code and the host code that picks its instance (tiling,
# split count): a capture stays valid only while both are unchanged.
KERNEL_SOURCES = {
    FD_KERNEL_SPLIT: ["fd_split_mma.cuh", "fd_split.cuh", "fd_device.cuh", "fd_kernels.cu",
                      "fd_api.cu"],
    FD_KERNEL_BIF_CTX: ["fd_bif_ctx.cuh", "fd_tcgen05.cuh", "fd_split.cuh", "fd_device.cuh",
                        "fd_kernels.cu", "fd_api.cu"],
}


def _code_only(text):
    """Source text without its comments and with whitespace runs collapsed,
    so that editing a comment does not count as changing the kernel."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kind, read=None):
    """Hash of the code of the kind's source files; `read(name)` returns a
    file's text (default: the files under csrc/)."""
    import hashlib
    if read is None:
        def read(name):
            with open(os.path.join(ROOT, "decode_attention_20_b300", "csrc", name)) as f:
                return f.read()
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        h.update(_code_only(read(name)).encode())
    return h.hexdigest()[:16]


def measured_traffic(kind, workload):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None when none matches this workload and source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        table = json.load(f)
    e = table.get(f"{kind}:{workload}")
    if not e or e.get("source_hash") != kernel_source_hash(kind):
        return None
    return int(e["dram_bytes_per_launch"])


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "kind": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "kind": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd_, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd_)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(self.gpu_id)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        num = lambda x: x.replace(".", "", 1).isdigit()
        sm = [float(r[1]) for r in rows if num(r[1])]
        smax = [float(r[2]) for r in rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, n in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [x["num_threads"] for x in threadpool_info() if x.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def f64(t):
    import numpy as np
    import torch
    import oracle
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return oracle.bf16_bits_to_f64(t.view(torch.uint16).numpy())
    return t.numpy().astype(np.float64)


# ------------------------------------------------------------------ workloads

class Workload:
    """One benchmark workload: device inputs, the timed call, its byte / FLOP
    accounting, an end-to-end step and a bounded oracle sample."""

    short = ""
    name = ""
    dominant = FD_KERNEL_SPLIT

    def config(self):
        raise NotImplementedError


def _rows(t, n):
    """t viewed as n rows (8-bit floats as bytes, which indexing kernels take)."""
    import torch
    if t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    return t.view(n, -1)


def _staging(device, specs):
    """One pinned host buffer and one device buffer holding tensors of the
    given (shape, dtype) specs at 256-byte aligned offsets, so that a step
    moves all its inputs (or all its results) in one copy.  Returns (host
    buffer, device buffer, host views, device views)."""
    import numpy as np
    import torch
    sizes = [int(np.prod(shape)) * torch.empty((), dtype=dt).element_size() for shape, dt in specs]
    offs, off = [], 0
    for n in sizes:
        offs.append(off)
        off = (off + n + 255) // 256 * 256
    h = torch.empty(off, dtype=torch.uint8).pin_memory()
    d = torch.empty(off, dtype=torch.uint8, device=device)

    def views(buf):
        return [buf[o:o + n].view(dt).view(shape) for (shape, dt), o, n in zip(specs, offs, sizes)]

    return h, d, views(h), views(d)


def _host_loop_us(stream, steps, step, warmup=5, blocks=5):
    """Wall-clock microseconds per call of step(i) on `stream`, after
    `warmup` untimed calls (first-use costs: lazy kernel loading, pinned
    staging, pool growth): the steps run as `blocks` equal blocks, each
    timed on its own, and the median block gives the value, so that one
    stall of the shared host cores does not set it."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
    torch.cuda.synchronize()
    per = max(1, steps // blocks)
    times = []
    i = 0
    with torch.cuda.stream(stream):
        for _ in range(blocks):
            t0 = time.perf_counter()
            for _ in range(per):
                step(i)
                i += 1
            times.append((time.perf_counter() - t0) * 1e6 / per)
    return statistics.median(times)


class DecodeWorkload(Workload):
    dominant = FD_KERNEL_SPLIT

    def __init__(self, short, builder, device, copies=True):
        import torch
        self.short = short
        self.case = builder(device)
        c = self.case
        self.name = c.name
        if c.q.dim() == 4:                     # multi-token decode: q [B, Tq, Hq, D]
            self.B, self.Tq, self.Hq, self.D = c.q.shape
        else:
            (self.B, self.Hq, self.D), self.Tq = c.q.shape, 1
        self.Lcap, self.Hkv = c.k.shape[1], c.k.shape[2]
        self.lens = c.lens
        self.seqlens_dev = c.seqlens.to(device) if c.seqlens is not None else None
        kv_bytes = c.k.numel() * c.k.element_size() * 2
        self.nbuf = rotation_copies(kv_bytes)
        extra = self.nbuf - 1 if copies else 0
        self.ks = [c.k] + [c.k.clone() for _ in range(extra)]
        self.vs = [c.v] + [c.v.clone() for _ in range(extra)]
        tok = (self.Tq,) if self.Tq > 1 else ()
        self.out = torch.empty((self.B,) + tok + (self.Hq, self.D), dtype=torch.float32, device=device)
        self.lse = torch.empty((self.B,) + tok + (self.Hq,), dtype=torch.float32, device=device)
        esz = c.k.element_size()
        tokens = sum(self.lens)
        self.kv_req = tokens * self.Hkv * self.D * esz * 2
        self.required = (self.kv_req + c.q.numel() * c.q.element_size()
                         + self.out.numel() * 4 + self.lse.numel() * 4)
        self.dominant_units = self.kv_req + c.q.numel() * c.q.element_size()   # split kernel bytes
        self.bound, self.unit = "hbm", "GB/s"

    def config(self, ns):
        return {"workload": self.name, "batch": self.B, "q_heads": self.Hq, "kv_heads": self.Hkv,
                "head_dim": self.D, "kv_capacity": self.Lcap,
                "kv_tokens": sum(self.lens), "num_splits": ns}

    def prepare(self, L, stream, ns):
        from decode_attention_20_b300.api import _desc
        c = self.case
        self.ns = ns
        self.dq, self.do, self.dl = _desc(c.q, "q"), _desc(self.out, "out"), _desc(self.lse, "lse")
        self.ds = _desc(self.seqlens_dev, "seqlens")
        self.dks = [_desc(x, "k") for x in self.ks]
        self.dvs = [_desc(x, "v") for x in self.vs]
        self.L = L
        self.sptr = ctypes.c_void_p(stream.cuda_stream)

    def call(self, i):
        r = ctypes.byref
        st = self.L.fd_decode_attention(r(self.dq), r(self.dks[i % self.nbuf]), r(self.dvs[i % self.nbuf]),
                                        r(self.ds) if self.ds is not None else None, self.ns,
                                        ctypes.c_float(self.case.scale), r(self.do), r(self.dl), self.sptr)
        if st:
            raise RuntimeError(self.L.fd_last_error().decode())

    def api_call(self, q, k, v, stream, out=None, lse=None):
        import decode_attention_20_b300 as fd
        fd.decode_attention(q, k, v, self.seqlens_dev, self.ns, self.case.scale,
                            out=self.out if out is None else out,
                            lse=self.lse if lse is None else lse, stream=stream)

    def e2e(self, stream, steps):
        """Per step: one H2D of the new query and one new K/V row per
        sequence (packed in one pinned buffer; the rows are then written at
        position len_b - 1), the call, one D2H of out + lse (one buffer)."""
        import torch
        c = self.case
        dev = c.q.device
        # the Tq newest rows of every sequence (positions len_b - Tq .. len_b - 1)
        pos = [(b, j) for b, n in enumerate(self.lens) for j in range(max(0, n - self.Tq), max(n, 1))]
        nr = len(pos)
        row = (nr, self.Hkv * self.D)
        h_in, d_in, (hq, hk, hv), (dq, dk, dv) = _staging(
            dev, [(tuple(c.q.shape), c.q.dtype), (row, c.k.dtype), (row, c.k.dtype)])
        hq.copy_(c.q.cpu())
        for i, (b, j) in enumerate(pos):
            hk[i].copy_(c.k[b, j].reshape(-1).cpu())
            hv[i].copy_(c.v[b, j].reshape(-1).cpu())
        h_res, d_res, _, (dout, dlse) = _staging(
            dev, [(tuple(self.out.shape), torch.float32), (tuple(self.lse.shape), torch.float32)])
        rows = torch.tensor([b * self.Lcap + j for b, j in pos], dtype=torch.int64, device=dev)

        def step(i):
            kb, vb = self.ks[i % self.nbuf], self.vs[i % self.nbuf]
            d_in.copy_(h_in, non_blocking=True)
            _rows(kb, self.B * self.Lcap).index_copy_(0, rows, _rows(dk, nr))
            _rows(vb, self.B * self.Lcap).index_copy_(0, rows, _rows(dv, nr))
            self.api_call(dq, kb, vb, stream, out=dout, lse=dlse)
            h_res.copy_(d_res, non_blocking=True)
            stream.synchronize()

        us = _host_loop_us(stream, steps, step)
        return us, h_in.numel(), h_res.numel()

    def _oracle_inputs(self, n0):
        c = self.case
        return f64(c.q[0:1]), f64(c.k[0:1, :n0]), f64(c.v[0:1, :n0])

    def _oracle_call(self, q, k, v, T):
        import oracle
        oracle.decode_attention_ref(q, k[:, :T], v[:, :T], None, self.case.scale)

    def oracle_sample(self):
        """Time the oracle once on a fixed sample: sequence 0's whole history
        with all its kv heads (the whole call at batch 1).  Returns (us per
        full call, extrapolated linearly by tokens when the batch holds more
        than sequence 0; sample text; seconds of the sample).  The inputs'
        float64 conversion is done once and not timed."""
        T = max(self.lens[0], 1)
        if not hasattr(self, "_of"):
            self._of = self._oracle_inputs(T)
        q, k, v = self._of
        t0 = time.perf_counter()
        self._oracle_call(q, k, v, T)
        dt = time.perf_counter() - t0
        total = sum(self.lens)
        full = dt * (total / T)
        text = f"sequence 0: {T} tokens x all {self.Hkv} kv heads"
        if total != T:
            text += f", extrapolated linearly to {total} tokens x {self.B} sequences"
        return full * 1e6, text, dt


class BifWorkload(Workload):
    dominant = FD_KERNEL_BIF_CTX

    def __init__(self, device, copies=True):
        import torch
        from decode_attention_20_b300 import inputs
        self.short = "bif_mqa"
        c = self.case = inputs.bifurcated_mqa(device=device)
        self.name = c.name
        self.n, self.Hq, self.D = c.q.shape
        self.Lc, self.Hkv = c.k_ctx.shape[0], c.k_ctx.shape[1]
        self.Ld = c.k_dec.shape[1]
        self.dec_dev = c.dec_lens.to(device) if c.dec_lens is not None else None
        per_copy = sum(x.numel() * 2 for x in [c.k_ctx, c.v_ctx, c.k_dec, c.v_dec, c.q])
        self.nbuf = rotation_copies(per_copy)
        self.bufs = [(c.q, c.k_ctx, c.v_ctx, c.k_dec, c.v_dec)] + [
            tuple(x.clone() for x in (c.q, c.k_ctx, c.v_ctx, c.k_dec, c.v_dec))
            for _ in range(self.nbuf - 1 if copies else 0)]
        self.out = torch.empty((self.n, self.Hq, self.D), dtype=torch.float32, device=device)
        self.lse = torch.empty((self.n, self.Hq), dtype=torch.float32, device=device)
        kv_ctx = c.k_ctx.numel() * 2 * 2
        kv_dec = sum(self.case.lens) * self.Hkv * self.D * 2 * 2
        self.required = kv_ctx + kv_dec + c.q.numel() * 2 + self.out.numel() * 4 + self.lse.numel() * 4
        # The context kernel also streams every sample's own decode tokens
        # (folded into it for groups of 16+ query heads), so its FLOPs are
        # QK^T and PV over the context plus each sample's decode history.
        self.dominant_units = 4.0 * self.Hq * self.D * (self.n * self.Lc + sum(self.case.lens))
        self.bound, self.unit = "tensor", "TFLOP/s"

    def config(self, ns):
        return {"workload": self.name, "samples": self.n, "q_heads": self.Hq, "kv_heads": self.Hkv,
                "head_dim": self.D, "context_len": self.Lc, "decode_len": self.Ld,
                "ctx_splits": ns}

    def prepare(self, L, stream, ns):
        from decode_attention_20_b300.api import _desc
        self.ns = ns
        self.L = L
        self.sptr = ctypes.c_void_p(stream.cuda_stream)
        self.dbufs = [[_desc(x, "t") for x in b] for b in self.bufs]
        self.ddl = _desc(self.dec_dev, "dec_lens")
        self.do, self.dl = _desc(self.out, "out"), _desc(self.lse, "lse")

    def call(self, i):
        r = ctypes.byref
        d = self.dbufs[i % self.nbuf]
        st = self.L.fd_bifurcated_attention_lse(r(d[0]), r(d[1]), r(d[2]), r(d[3]), r(d[4]),
                                                r(self.ddl) if self.ddl is not None else None,
                                                ctypes.c_float(self.case.scale), self.ns, r(self.do),
                                                r(self.dl), self.sptr)
        if st:
            raise RuntimeError(self.L.fd_last_error().decode())

    def replicated_us(self, stream, steps, ns):
        """The same inputs with the context materialised per sample, through
        the split-KV decode path (the comparison the method is measured
        against)."""
        import torch
        import decode_attention_20_b300 as fd
        from decode_attention_20_b300 import inputs
        rep = inputs.replicate_context(self.case)
        reps = [rep.k, rep.v]
        nb = max(1, math.ceil(2 * L2_BYTES / (rep.k.numel() * 4)))
        ks = [rep.k] + [rep.k.clone() for _ in range(nb - 1)]
        vs = [rep.v] + [rep.v.clone() for _ in range(nb - 1)]
        sl = rep.seqlens.to(rep.k.device)
        with torch.cuda.stream(stream):
            for i in range(3):
                fd.decode_attention(rep.q, ks[i % nb], vs[i % nb], sl, 0, rep.scale, out=self.out,
                                    lse=self.lse, stream=stream)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(steps):
                fd.decode_attention(rep.q, ks[i % nb], vs[i % nb], sl, 0, rep.scale, out=self.out,
                                    lse=self.lse, stream=stream)
            e1.record(stream)
        stream.synchronize()
        kv = sum(rep.lens) * self.Hkv * self.D * 2 * 2
        del ks, vs, reps
        return e0.elapsed_time(e1) * 1e3 / steps, kv

    def e2e(self, stream, steps):
        """Per step: one H2D of the queries and one new decode K/V row per
        sample (one pinned buffer; the rows are then written into the decode
        caches), the call, one D2H of out + lse (one buffer)."""
        import torch
        import decode_attention_20_b300 as fd
        c = self.case
        dev = c.q.device
        rshape = (self.n, self.Hkv * self.D)
        h_in, d_in, (hq, hk, hv), (dq, dk, dv) = _staging(
            dev, [(tuple(c.q.shape), c.q.dtype), (rshape, c.k_dec.dtype), (rshape, c.k_dec.dtype)])
        hq.copy_(c.q.cpu())
        pos = [max(0, x - 1) for x in c.lens]
        for b in range(self.n):
            hk[b].copy_(c.k_dec[b, pos[b]].reshape(-1).cpu())
            hv[b].copy_(c.v_dec[b, pos[b]].reshape(-1).cpu())
        h_res, d_res, _, (dout, dlse) = _staging(
            dev, [(tuple(self.out.shape), torch.float32), (tuple(self.lse.shape), torch.float32)])
        rows = torch.tensor([b * self.Ld + pos[b] for b in range(self.n)], dtype=torch.int64,
                            device=dev)

        def step(i):
            _, kc, vc, kd, vd = self.bufs[i % self.nbuf]
            d_in.copy_(h_in, non_blocking=True)
            kd.view(self.n * self.Ld, -1).index_copy_(0, rows, dk)
            vd.view(self.n * self.Ld, -1).index_copy_(0, rows, dv)
            fd.bifurcated_attention(dq, kc, vc, kd, vd, self.dec_dev, c.scale, out=dout,
                                    lse=dlse, ctx_splits=self.ns, return_lse=True,
                                    stream=stream)
            h_res.copy_(d_res, non_blocking=True)
            stream.synchronize()

        us = _host_loop_us(stream, steps, step)
        return us, h_in.numel(), h_res.numel()

    def oracle_sample(self):
        """Time the oracle once on a fixed sample: sample 0 over the whole
        context and its own decode tokens.  Returns (us per full call,
        extrapolated linearly to all samples; sample text; seconds)."""
        import oracle
        c = self.case
        lens = c.lens
        if not hasattr(self, "_of"):
            self._of = (f64(c.q[:1]), f64(c.k_ctx), f64(c.v_ctx), f64(c.k_dec[:1]), f64(c.v_dec[:1]))
        q, kc, vc, kd, vd = self._of
        t0 = time.perf_counter()
        oracle.bifurcated_attention_ref(q, kc, vc, kd, vd, [lens[0]], c.scale)
        dt = time.perf_counter() - t0
        full_tokens = sum(self.Lc + x for x in lens)
        return dt * full_tokens / (self.Lc + lens[0]) * 1e6, (
            f"sample 0: {self.Lc} context tokens and its {lens[0]} decode tokens, "
            f"extrapolated linearly to {self.n} samples"), dt


class PagedWorkload(DecodeWorkload):
    """The batch-1 64K layer with its history in scattered 64-token pages
    (fd_decode_attention_paged)."""

    def __init__(self, device, copies=True):
        import torch
        from decode_attention_20_b300 import inputs
        self.short = "paged_b1_64k"
        c = self.pcase = inputs.paged_flash_decoding_b1(65536, 64, device=device)
        self.name = c.name
        self.B, self.Hq, self.D = c.q.shape
        self.Hkv = c.k_pages.shape[2]
        self.page_size = c.page_size
        self.Lcap = c.block_table.shape[1] * c.page_size
        self.lens = c.lens
        self.seqlens_dev = None
        self.bt_dev = c.block_table.to(device)
        kv_bytes = c.k_pages.numel() * c.k_pages.element_size() * 2
        self.nbuf = rotation_copies(kv_bytes)
        self.ks = [c.k_pages] + [c.k_pages.clone() for _ in range(self.nbuf - 1 if copies else 0)]
        self.vs = [c.v_pages] + [c.v_pages.clone() for _ in range(self.nbuf - 1 if copies else 0)]
        self.out = torch.empty((self.B, self.Hq, self.D), dtype=torch.float32, device=device)
        self.lse = torch.empty((self.B, self.Hq), dtype=torch.float32, device=device)
        self.kv_req = sum(self.lens) * self.Hkv * self.D * 2 * 2
        self.required = self.kv_req + c.q.numel() * 2 + self.out.numel() * 4 + self.lse.numel() * 4
        self.dominant_units = self.kv_req + c.q.numel() * 2
        self.bound, self.unit = "hbm", "GB/s"
        # the oracle sample and e2e reuse the contiguous view of the same tokens
        from decode_attention_20_b300.inputs import DecodeCase
        bt = c.block_table.to(c.k_pages.device).long()
        kc = c.k_pages[bt].reshape(1, self.Lcap, self.Hkv, self.D)
        vc = c.v_pages[bt].reshape(1, self.Lcap, self.Hkv, self.D)
        self.case = DecodeCase(name=c.name, q=c.q, k=kc, v=vc, seqlens=None, scale=c.scale)

    def config(self, ns):
        cfg = super().config(ns)
        cfg["page_size"] = self.page_size
        return cfg

    def prepare(self, L, stream, ns):
        from decode_attention_20_b300.api import _desc
        c = self.pcase
        self.ns = ns
        self.dq, self.do, self.dl = _desc(c.q, "q"), _desc(self.out, "out"), _desc(self.lse, "lse")
        self.dbt = _desc(self.bt_dev, "block_table")
        self.dks = [_desc(x, "k") for x in self.ks]
        self.dvs = [_desc(x, "v") for x in self.vs]
        self.L = L
        self.sptr = ctypes.c_void_p(stream.cuda_stream)

    def call(self, i):
        r = ctypes.byref
        st = self.L.fd_decode_attention_paged(r(self.dq), r(self.dks[i % self.nbuf]),
                                              r(self.dvs[i % self.nbuf]), r(self.dbt), None,
                                              self.ns, ctypes.c_float(self.pcase.scale), r(self.do),
                                              r(self.dl), self.sptr)
        if st:
            raise RuntimeError(self.L.fd_last_error().decode())

    def e2e(self, stream, steps):
        """Per step: one H2D of the new query and the newest token's K/V row
        (one pinned buffer; the row is then written into its page), the paged
        call, one D2H of out + lse (one buffer)."""
        import torch
        import decode_attention_20_b300 as fd
        c = self.pcase
        dev = c.q.device
        last = self.Lcap - 1
        pid = int(c.block_table[0, last // self.page_size])
        row = pid * self.page_size + last % self.page_size
        rshape = (1, self.Hkv * self.D)
        h_in, d_in, (hq, hk, hv), (dq, dk, dv) = _staging(
            dev, [(tuple(c.q.shape), c.q.dtype), (rshape, c.k_pages.dtype), (rshape, c.k_pages.dtype)])
        hq.copy_(c.q.cpu())
        hk.copy_(c.k_pages.view(-1, self.Hkv * self.D)[row:row + 1].cpu())
        hv.copy_(c.v_pages.view(-1, self.Hkv * self.D)[row:row + 1].cpu())
        h_res, d_res, _, (dout, dlse) = _staging(
            dev, [(tuple(self.out.shape), torch.float32), (tuple(self.lse.shape), torch.float32)])

        def step(i):
            kb, vb = self.ks[i % self.nbuf], self.vs[i % self.nbuf]
            d_in.copy_(h_in, non_blocking=True)
            kb.view(-1, self.Hkv * self.D)[row:row + 1].copy_(dk, non_blocking=True)
            vb.view(-1, self.Hkv * self.D)[row:row + 1].copy_(dv, non_blocking=True)
            fd.decode_attention_paged(dq, kb, vb, self.bt_dev, None, self.ns, c.scale,
                                      out=dout, lse=dlse, stream=stream)
            h_res.copy_(d_res, non_blocking=True)
            stream.synchronize()

        us = _host_loop_us(stream, steps, step)
        return us, h_in.numel(), h_res.numel()


class MultiWorkload(DecodeWorkload):
    """The batch-1 64K-token layer verifying Tq new tokens at once
    (fd_decode_attention_multi)."""

    def __init__(self, short, tq, device, copies=True):
        from decode_attention_20_b300 import inputs
        super().__init__(short, lambda d: inputs.speculative_b1(65536, tq=tq, device=d), device,
                         copies)

    def config(self, ns):
        cfg = super().config(ns)
        cfg["query_tokens"] = self.Tq
        return cfg

    def call(self, i):
        r = ctypes.byref
        st = self.L.fd_decode_attention_multi(r(self.dq), r(self.dks[i % self.nbuf]),
                                              r(self.dvs[i % self.nbuf]),
                                              r(self.ds) if self.ds is not None else None, self.ns,
                                              ctypes.c_float(self.case.scale), r(self.do),
                                              r(self.dl), self.sptr)
        if st:
            raise RuntimeError(self.L.fd_last_error().decode())

    def api_call(self, q, k, v, stream, out=None, lse=None):
        import decode_attention_20_b300 as fd
        fd.decode_attention_multi(q, k, v, self.seqlens_dev, self.ns, self.case.scale,
                                  out=self.out if out is None else out,
                                  lse=self.lse if lse is None else lse, stream=stream)

    def _oracle_call(self, q, k, v, T):
        import oracle
        oracle.multi_token_decode_ref(q, k[:, :T], v[:, :T], None, self.case.scale)


class QuantWorkload(DecodeWorkload):
    """The batch-1 64K-token layer over an 8-bit cache (int8 or e4m3 codes,
    one scale per kv head): fd_decode_attention_quant."""
    dtype = "f16"
    kernel_name = "split_mma_kernel (mma.sync f16 over 8-bit codes, TMA ring)"

    def __init__(self, short, kind, device, copies=True):
        from decode_attention_20_b300 import inputs
        super().__init__(short, lambda d: inputs.quant_flash_decoding_b1(65536, kind=kind, device=d),
                         device, copies)
        self.kind = kind

    def config(self, ns):
        cfg = super().config(ns)
        cfg["kv_codes"] = self.kind
        return cfg

    def prepare(self, L, stream, ns):
        from decode_attention_20_b300.api import _desc
        super().prepare(L, stream, ns)
        self.dkscale = _desc(self.case.k_scale, "k_scale")
        self.dvscale = _desc(self.case.v_scale, "v_scale")

    def call(self, i):
        r = ctypes.byref
        st = self.L.fd_decode_attention_quant(r(self.dq), r(self.dks[i % self.nbuf]),
                                              r(self.dvs[i % self.nbuf]), r(self.dkscale),
                                              r(self.dvscale),
                                              r(self.ds) if self.ds is not None else None, self.ns,
                                              ctypes.c_float(self.case.scale), r(self.do),
                                              r(self.dl), self.sptr)
        if st:
            raise RuntimeError(self.L.fd_last_error().decode())

    def api_call(self, q, k, v, stream, out=None, lse=None):
        import decode_attention_20_b300 as fd
        c = self.case
        fd.decode_attention_quant(q, k, v, c.k_scale, c.v_scale, self.seqlens_dev, self.ns,
                                  c.scale, out=self.out if out is None else out,
                                  lse=self.lse if lse is None else lse, stream=stream)

    def _oracle_inputs(self, n0):
        import torch
        c = self.case
        codes = lambda t: (t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t).cpu().numpy()
        return (f64(c.q[0:1]), codes(c.k[0:1, :n0]), codes(c.v[0:1, :n0]))

    def _oracle_call(self, q, k, v, T):
        import oracle
        c = self.case
        oracle.quant_decode_attention_ref(q, k[:, :T], v[:, :T], c.k_scale.cpu().numpy(),
                                          c.v_scale.cpu().numpy(), self.kind, None, c.scale)


def make_workload(short, device, copies=True):
    """The named workload on `device`; copies=False keeps one copy of the
    inputs (the CPU oracle arm rotates nothing)."""
    from decode_attention_20_b300 import inputs
    if short == "b1_64k":
        return DecodeWorkload(short, lambda d: inputs.flash_decoding_b1(65536, seed=0, device=d),
                              device, copies)
    if short.startswith("b1_L"):                      # the batch-1 layer at another length
        L = int(short[4:])
        return DecodeWorkload(short, lambda d: inputs.flash_decoding_b1(L, seed=0, device=d),
                              device, copies)
    if short == "tiny_fp32":
        return DecodeWorkload(short, lambda d: inputs.tiny_mha(device=d), device, copies)
    if short == "ragged_b32":
        return DecodeWorkload(short, lambda d: inputs.ragged_batch(device=d), device, copies)
    if short == "long_b4":
        return DecodeWorkload(short, lambda d: inputs.long_context_peaked(device=d), device, copies)
    if short == "bif_mqa":
        return BifWorkload(device, copies)
    if short == "paged_b1_64k":
        return PagedWorkload(device, copies)
    if short == "verify4_b1_64k":
        return MultiWorkload(short, 4, device, copies)
    if short == "int8_b1_64k":
        return QuantWorkload(short, "int8", device, copies)
    if short == "e4m3_b1_64k":
        return QuantWorkload(short, "e4m3", device, copies)
    raise SystemExit(f"unknown workload {short}")


# ------------------------------------------------------------------ shared pieces

def num_sms_for_config():
    """SM count the split heuristic is given: the visible GPU's, else a
    B300's 148 (the CPU oracle arm may run where no GPU is visible)."""
    try:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.get_device_properties(0).multi_processor_count
    except Exception:
        pass
    return 148


def line_config(w, ns, world):
    """The `config` object of a line: the same in the GPU arm and the oracle
    arm (workload shapes, split count, parallelism, L2 handling)."""
    return dict(w.config(ns), parallelism="replicas" if world > 1 else "single",
                l2=f"inputs larger than L2: {w.nbuf} rotating input copies")


def workload_splits(w, num_sms):
    """Split count the line reports: the library heuristic's for the decode
    workloads (its host mirror in the oracle, equal bit for bit), 0 for the
    bifurcated call (the library chooses its context splits itself)."""
    import oracle
    if isinstance(w, DecodeWorkload):
        return int(oracle.choose_num_splits_ref(w.B, w.Hkv, w.Lcap, num_sms))
    return 0


def cpu_baseline(w, budget_s=3.0, min_reps=3, max_reps=20):
    """Best of repeated timings of the fp64 oracle on the workload's fixed
    sample, on the host cores: at least `min_reps`, then more while the
    samples so far stay within `budget_s` seconds, at most `max_reps` (the
    reference arm takes the best of its steps the same way).  The host is
    shared, so the best of many is the stable figure."""
    best = None
    sample = ""
    spent = 0.0
    reps = 0
    while reps < max_reps and (reps < min_reps or spent < budget_s):
        us, sample, dt = w.oracle_sample()
        spent += dt
        reps += 1
        best = us if best is None else min(best, us)
    return {"value": round(best, 1), "unit": "us/call", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{sample}; best of {reps}"}


def cpu_baseline_ref_arm(w, short):
    """The reference arm's own measurement of this workload, run as a
    separate process (`bench.py --impl reference`), so that the GPU line's
    cpu_baseline and the reference line come from the same code under the
    same process conditions (a host-memory-bound fp64 oracle is sensitive to
    what else the process did before).  Steps: 20 for a sample under 0.2 s,
    5 under 1.5 s, else 3.  Falls back to timing in this process."""
    one = cpu_baseline(w, budget_s=0.0, min_reps=1, max_reps=1)
    per_s = one["value"] * 1e-6
    steps = 20 if per_s < 0.2 else 5 if per_s < 1.5 else 3
    cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--workload", short,
           "--steps", str(steps), "--warmup", "1"]
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env)
        line = next(json.loads(l) for l in r.stdout.splitlines() if l.startswith("{"))
        cb = dict(line["cpu_baseline"])
        cb["sample"] += "; measured by the reference arm in a separate process"
        return cb
    except Exception:                                   # noqa: BLE001 (fall back to this process)
        cb = cpu_baseline(w)
        cb["sample"] += "; timed in this process (the reference arm subprocess gave no line)"
        return cb


# ------------------------------------------------------------------ reference arm

def run_reference(args, rank, world):
    """--impl reference: the fp64 oracle on host cores, same workload and
    config as the GPU arm; each step one timing of the fixed sample, value
    the best step."""
    if rank != 0:
        return 0
    w = make_workload(args.workload, "cpu", copies=False)
    ns = args.num_splits or workload_splits(w, num_sms_for_config())
    us = []
    step_s = []
    sample = ""
    for i in range(args.warmup + args.steps):
        u, sample, dt = w.oracle_sample()
        if i >= args.warmup:
            us.append(u)
            step_s.append(dt)
    value = min(us)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "us/call",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.median(step_s) * 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": line_config(w, ns, world),
        "timing": {"kind": "host wall clock of the fp64 oracle, one fixed sample per step",
                   "reduction": f"best of {args.steps} steps"},
        "cpu_baseline": {"value": round(value, 1), "unit": "us/call", "cores": blas_threads(),
                         "kind": "oracle", "sample": f"{sample}; best of {args.steps}"},
        "e2e": {"value": round(value, 1), "unit": "us/call", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "achieved_gbs": round(w.required / (value * 1e-6) / 1e9, 3),
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

def max_over_ranks(vals, world):
    """Element-wise maximum of a tensor of timings over all ranks: every
    replica runs the same calls independently, and the slowest one sets the
    job's time.  One all-reduce of the (already measured) timings; no data of
    the attention path crosses ranks."""
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(vals, op=dist.ReduceOp.MAX)
    return vals


def _events():
    import torch
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def time_direct(w, stream, n):
    """Device microseconds per call of n direct (not graph) calls issued back
    to back on `stream`: host issue cost included where it exceeds the
    device time."""
    import torch
    e0, e1 = _events()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(n):
            w.call(i)
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) * 1e3 / n


def capture_calls(w, stream, ncalls):
    """A CUDA graph of `ncalls` consecutive calls over the rotating input
    copies, replayed once; None where capture fails."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(ncalls):
                w.call(i)
        g.replay()
        torch.cuda.synchronize()
        return g
    except Exception:
        torch.cuda.synchronize()
        return None


def time_steps(w, stream, steps, warmup, window_s, barrier=None, sampler=None):
    """Exactly `steps` timed steps after `warmup` untimed ones.  A step is
    one replay of a CUDA graph of C back-to-back calls over the rotating
    input copies (C a multiple of the copies, sized so that the steps span
    about `window_s` seconds); CUDA events on the launching stream bracket
    the steps, with a barrier and a device synchronise on both sides.
    Returns microseconds per call, C, milliseconds per step, the timing
    description and the clocks sampled during the steps."""
    import torch
    est = time_direct(w, stream, max(w.nbuf, 8))
    cps = max(16, math.ceil(window_s * 1e6 / (steps * max(est, 1e-3))))
    cps = min(max(w.nbuf, 4096), w.nbuf * math.ceil(cps / w.nbuf))
    g = capture_calls(w, stream, cps)
    if g is not None:
        timing = f"each step one replay of a CUDA graph of {cps} calls"

        def run():
            g.replay()
    else:
        timing = f"each step {cps} direct calls (graph capture failed)"

        def run():
            for i in range(cps):
                w.call(i)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            run()
    stream.synchronize()
    if sampler is not None:
        sampler.start()
    if barrier is not None:
        barrier()
    torch.cuda.synchronize()
    e0, e1 = _events()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            run()
        e1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    if barrier is not None:
        barrier()
    clk = sampler.stop() if sampler is not None else None
    ms = e0.elapsed_time(e1)
    del g
    return {"us_per_call": ms * 1e3 / (steps * cps), "calls_per_step": cps,
            "ms_per_step": ms / steps, "timing": timing, "clocks": clk}


KERNEL_LABELS = [(FD_KERNEL_SPLIT, "split"), (FD_KERNEL_COMBINE, "combine"),
                 (FD_KERNEL_BIF_CTX, "bif_ctx")]


def kernel_times(w, stream, n, us_direct):
    """Per-kernel device time of n calls: CUDA events around each launch on
    its stream (the library's timing hooks).  The calls are queued behind a
    device-side delay longer than the host takes to issue them, so the GPU
    runs them back to back and each event pair brackets its kernel, not the
    host's time to issue the next call.  Returns {label_us,
    label_launches_per_call} and the launches per call."""
    import torch
    import decode_attention_20_b300 as fd
    delay_us = 2.0 * n * us_direct + 5000.0
    fd.profile_enable(True)
    sleep = getattr(torch.cuda, "_sleep", None)       # a device-side spin of N clock cycles
    with torch.cuda.stream(stream):
        if sleep is not None:
            sleep(int(delay_us * SLEEP_CYCLES_PER_US))
        for i in range(n):
            w.call(i)
    stream.synchronize()
    kern = {}
    launches = 0
    for kind, label in KERNEL_LABELS:
        cnt, ms = fd.profile_read(kind)
        launches += cnt
        if cnt:
            kern[label + "_us"] = round(ms * 1e3 / cnt, 3)
            kern[label + "_launches_per_call"] = cnt / n
    fd.profile_enable(False)
    return kern, launches / n


def dominant_roofline(w, dom_us, peaks):
    """(achieved, peak, per-launch units) of the workload's dominant kernel."""
    if w.bound == "hbm":
        return w.dominant_units / (dom_us * 1e-6) / 1e9, peaks["hbm_gbs"], int(w.dominant_units)
    return w.dominant_units / (dom_us * 1e-6) / 1e12, peaks["bf16_tflops"], w.dominant_units


def measure_config(short, dev, stream, L, peaks, window_s=0.15, ns=0):
    """One of the other workloads measured the way the headline is (graph steps
    over rotating copies, direct calls, per-kernel events), as a compact
    record for the line's `configs` object."""
    import torch
    import decode_attention_20_b300 as fd
    w = make_workload(short, dev)
    if isinstance(w, DecodeWorkload) and ns == 0:
        ns = fd.choose_num_splits(w.B, w.Hkv, w.Lcap,
                                  torch.cuda.get_device_properties(dev).multi_processor_count)
    w.prepare(L, stream, ns)
    with torch.cuda.stream(stream):
        for i in range(3):
            w.call(i)
    stream.synchronize()
    fd.check_device_error(stream)
    t = time_steps(w, stream, 5, 2, window_s)
    us_direct = time_direct(w, stream, max(32, min(500, w.nbuf * 2)))
    kern, _ = kernel_times(w, stream, 64, us_direct)
    dom_label = {FD_KERNEL_SPLIT: "split", FD_KERNEL_BIF_CTX: "bif_ctx"}[w.dominant]
    dom_us = kern[dom_label + "_us"]
    achieved, peak, _ = dominant_roofline(w, dom_us, peaks)
    gbs = w.required / (t["us_per_call"] * 1e-6) / 1e9
    rec = {"workload": w.name, "num_splits": ns, "us": round(t["us_per_call"], 3),
           "direct_us": round(us_direct, 3), "required_bytes": int(w.required),
           "achieved_gbs": round(gbs, 1), "frac_of_nominal_8tbs": round(gbs / 8000.0, 4),
           "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 4),
           "dominant_kernel_us": dom_us, "dominant_achieved": round(achieved, 1),
           "dominant_unit": w.unit, "dominant_frac": round(achieved / peak, 4),
           "rotating_copies": w.nbuf}
    if isinstance(w, BifWorkload):
        rep = DecodeWorkload("bif_replicated", lambda d: _replicated_case(w), dev)
        rns = fd.choose_num_splits(rep.B, rep.Hkv, rep.Lcap,
                                   torch.cuda.get_device_properties(dev).multi_processor_count)
        rep.prepare(L, stream, rns)
        with torch.cuda.stream(stream):
            for i in range(3):
                rep.call(i)
        stream.synchronize()
        rt = time_steps(rep, stream, 5, 2, window_s)
        rec["replicated_context_us"] = round(rt["us_per_call"], 3)
        rec["speedup_vs_replicated"] = round(rt["us_per_call"] / t["us_per_call"], 3)
        kv_bif = w.case.k_ctx.numel() * 4 + sum(w.case.lens) * w.Hkv * w.D * 4
        rec["kv_byte_ratio_replicated_over_bifurcated"] = round(rep.kv_req / kv_bif, 3)
        rec["h_over_g"] = w.Hq // w.Hkv
        del rep
    fd.check_device_error(stream)
    del w
    torch.cuda.empty_cache()
    return rec


def _replicated_case(w):
    from decode_attention_20_b300 import inputs
    return inputs.replicate_context(w.case)


SWEEP_LENGTHS = [512, 1024, 2048, 4096, 8192, 16384, 32768]


def run_fd(args, rank, world):
    import torch
    import torch.distributed as dist
    import decode_attention_20_b300 as fd
    from decode_attention_20_b300 import _lib

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    L = _lib.lib()
    props = torch.cuda.get_device_properties(dev)
    w = make_workload(args.workload, dev)
    if isinstance(w, DecodeWorkload):
        ns = args.num_splits or fd.choose_num_splits(w.B, w.Hkv, w.Lcap, props.multi_processor_count)
    else:
        ns = args.num_splits     # 0: the library's context split choice
    stream = torch.cuda.Stream(device=dev)
    w.prepare(L, stream, ns)

    def barrier():
        if world > 1:
            dist.barrier()

    warm = max(3, args.warmup)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(max(warm, w.nbuf)):
            w.call(i)
    stream.synchronize()
    fd.check_device_error(stream)

    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    gpu_id = vis.split(",")[dev.index] if vis else str(dev.index)
    t = time_steps(w, stream, args.steps, warm, args.window_ms / 1e3, barrier=barrier,
                   sampler=ClockSampler(gpu_id))
    us_per_call, clk = t["us_per_call"], t["clocks"]

    # Direct calls (no graph), same rotation: launch overhead included.
    dsteps = max(w.nbuf, min(t["calls_per_step"] * args.steps, 2000))
    us_direct = time_direct(w, stream, dsteps)

    kern, launches_per_call = kernel_times(w, stream, min(dsteps, 128), us_direct)
    dom_label = {FD_KERNEL_SPLIT: "split", FD_KERNEL_BIF_CTX: "bif_ctx"}[w.dominant]
    dom_us = kern[dom_label + "_us"]

    extra = {}
    if isinstance(w, BifWorkload):
        rep = DecodeWorkload("bif_replicated", lambda d: _replicated_case(w), dev)
        rns = fd.choose_num_splits(rep.B, rep.Hkv, rep.Lcap, props.multi_processor_count)
        rep.prepare(L, stream, rns)
        with torch.cuda.stream(stream):
            for i in range(3):
                rep.call(i)
        stream.synchronize()
        rt = time_steps(rep, stream, 5, 2, 0.15)
        extra["replicated_context_us"] = round(rt["us_per_call"], 3)
        extra["speedup_vs_replicated"] = round(rt["us_per_call"] / us_per_call, 3)
        kv_bif = w.case.k_ctx.numel() * 4 + sum(w.case.lens) * w.Hkv * w.D * 4
        extra["kv_byte_ratio_replicated_over_bifurcated"] = round(rep.kv_req / kv_bif, 3)
        extra["h_over_g"] = w.Hq // w.Hkv
        del rep
        torch.cuda.empty_cache()

    e2e_us, h2d, d2h = w.e2e(stream, max(1, min(t["calls_per_step"] * args.steps, 1000)))
    fd.check_device_error(stream)

    vals = torch.tensor([us_per_call, e2e_us, dom_us], dtype=torch.float64, device=dev)
    vals = max_over_ranks(vals, world)
    us_per_call, e2e_us, dom_us = [float(x) for x in vals.tolist()]

    # The other workloads and the batch-1 length sweep, measured the
    # same way (rank 0 of a single-GPU run, default workload only).
    configs = {}
    if world == 1 and args.workload == "b1_64k" and not args.no_configs:
        peaks = load_peaks()
        configs["tiny_fp32_mha_L256"] = {}
        for tns in (1, 4):
            configs["tiny_fp32_mha_L256"][f"ns{tns}"] = measure_config(
                "tiny_fp32", dev, stream, L, peaks, 0.05, ns=tns)
        configs["flash_decoding_b1_sweep"] = {
            str(n): measure_config(f"b1_L{n}", dev, stream, L, peaks, 0.1) for n in SWEEP_LENGTHS}
        configs["ragged_b32"] = measure_config("ragged_b32", dev, stream, L, peaks, 0.3)
        configs["bifurcated_mqa"] = measure_config("bif_mqa", dev, stream, L, peaks, 0.15)
        configs["long_b4_peaked"] = measure_config("long_b4", dev, stream, L, peaks, 0.3)
    if rank != 0:
        return 0

    peaks = load_peaks()
    gbs = w.required / (us_per_call * 1e-6) / 1e9 * world
    achieved, peak, per_launch = dominant_roofline(w, dom_us, peaks)
    line = {
        "metric": METRIC, "value": round(us_per_call, 3), "unit": "us/call",
        "n_gpus": world, "steps": args.steps, "warmup": warm,
        "ms_per_step": t["ms_per_step"], "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": getattr(w, "dtype", "bf16"),
        "data": "synthetic",
        "config": line_config(w, ns, world),
        "timing": {"step": t["timing"], "calls_per_step": t["calls_per_step"],
                   "calls_timed": t["calls_per_step"] * args.steps,
                   "window_ms": round(t["ms_per_step"] * args.steps, 3),
                   "value": "device microseconds per call, CUDA events around the steps"},
        "achieved_gbs": round(gbs, 1),
        "frac_of_nominal_8tbs": round(gbs / world / 8000.0, 4),
        "frac_of_measured_hbm": round(gbs / world / peaks["hbm_gbs"], 4),
        "direct_call_us": round(us_direct, 3),
        "kernels": kern,
        "roofline": {"bound": w.bound, "achieved": round(achieved, 1), "peak": peak,
                     "unit": w.unit, "frac": round(achieved / peak, 4),
                     "traffic": measured_traffic(w.dominant, w.short),
                     "kernel": getattr(w, "kernel_name", KERNEL_NAMES[w.dominant]),
                     "peak_kind": peaks["kind"],
                     "per_launch": per_launch, "launch_us": round(dom_us, 3)},
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"],
                   "reasons": clk["reasons"], "samples": clk["samples"]},
        "e2e": {"value": round(e2e_us, 3), "unit": "us/call", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": int(round(launches_per_call * t["calls_per_step"] * args.steps)),
    }
    line.update(extra)
    if configs:
        line["configs"] = configs
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_ref_arm(w, args.workload)
    print(json.dumps(line), flush=True)
    return 0


def run_sweep(args):
    """--sweep-splits: per split count (and split-kernel variant, through
    the library's FD_SPLIT_VARIANT knob), the device time per call of graph
    steps over rotating copies (as the headline is timed) and of direct
    calls, and the split kernel's event-timed launch; one JSON line each,
    marking the library heuristic's own choice.  With --sweep-lengths, the
    batch-1 layer at each of those lengths instead of --workload.  A tuning
    aid, not the benchmark line."""
    import torch
    import decode_attention_20_b300 as fd
    from decode_attention_20_b300 import _lib
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    L = _lib.lib()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    stream = torch.cuda.Stream(device=dev)
    variants = args.sweep_variants.split(",") if args.sweep_variants else [""]
    shorts = ([f"b1_L{int(x)}" for x in args.sweep_lengths.split(",")] if args.sweep_lengths
              else [args.workload])
    for short in shorts:
        w = make_workload(short, dev)
        chosen = (fd.choose_num_splits(w.B, w.Hkv, w.Lcap, sms)
                  if isinstance(w, DecodeWorkload) else 0)
        for var in variants:
            if var:
                os.environ["FD_SPLIT_VARIANT"] = var
            else:
                os.environ.pop("FD_SPLIT_VARIANT", None)
            for ns in [int(x) for x in args.sweep_splits.split(",")]:
                w.prepare(L, stream, ns)
                with torch.cuda.stream(stream):
                    for i in range(max(3, w.nbuf)):
                        w.call(i)
                stream.synchronize()
                t = time_steps(w, stream, 5, 2, args.window_ms / 1e3)
                direct = time_direct(w, stream, max(32, min(400, w.nbuf * 2)))
                kern, _ = kernel_times(w, stream, 64, direct)
                fd.check_device_error(stream)
                row = {"workload": w.name, "variant": var or "default", "splits": ns,
                       "heuristic": ns == chosen, "call_us": round(t["us_per_call"], 3),
                       "direct_us": round(direct, 3), **kern}
                if isinstance(w, DecodeWorkload):
                    row["call_gbs"] = round(w.required / (t["us_per_call"] * 1e-6) / 1e9, 1)
                    row["split_gbs"] = round(w.dominant_units / (kern["split_us"] * 1e-6) / 1e9, 1)
                print(json.dumps(row), flush=True)
        del w
        torch.cuda.empty_cache()
    return 0


def run_bif_sweep(args):
    """--bif-sweep: bifurcated attention against the replicated-context
    decode path over samples n, context length Lc and kv heads (32 query
    heads, head dim 128, bf16, decode lengths uniform in [1, 256]); one JSON
    line each with both times, their ratio, the K/V byte ratio and h/g.  A
    measurement aid, not the benchmark line."""
    import torch
    import decode_attention_20_b300 as fd
    from decode_attention_20_b300 import inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    iters = max(5, min(args.steps, 50))

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        tot = 0.0
        for _ in range(iters):
            flush.fill_(1)                  # every call starts with L2 cleared
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            tot += e0.elapsed_time(e1)
        return tot * 1e3 / iters

    for hkv in [1, 8]:
        for lc in [2048, 8192, 32768]:
            for n in [8, 32, 64, 128]:
                c = inputs.bifurcated_case(n, 32, hkv, 128, lc, 256, seed=n + lc + hkv,
                                           ragged_dec=(1, 256), device="cuda")
                dl = c.dec_lens.cuda()
                bif_us = timed(lambda: fd.bifurcated_attention(c.q, c.k_ctx, c.v_ctx, c.k_dec,
                                                               c.v_dec, dl, c.scale))
                rep = inputs.replicate_context(c)
                sl = rep.seqlens.cuda()
                rep_us = timed(lambda: fd.decode_attention(rep.q, rep.k, rep.v, sl, 0, rep.scale))
                fd.check_device_error()
                kv_bif = c.k_ctx.numel() * 4 + sum(c.lens) * hkv * 128 * 4
                kv_rep = sum(rep.lens) * hkv * 128 * 4
                print(json.dumps({"samples": n, "context_len": lc, "kv_heads": hkv, "q_heads": 32,
                                  "bifurcated_us": round(bif_us, 2),
                                  "replicated_us": round(rep_us, 2),
                                  "speedup": round(rep_us / bif_us, 2),
                                  "kv_byte_ratio": round(kv_rep / kv_bif, 2),
                                  "h_over_g": 32 // hkv}), flush=True)
                del c, rep
                torch.cuda.empty_cache()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--window-ms", type=float, default=400.0,
                    help="device time the timed steps should span (sets the calls per step)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads and the length sweep in the line")
    ap.add_argument("--impl", choices=["fd", "reference"], default="fd")
    ap.add_argument("--workload", default="b1_64k",
                    choices=["b1_64k", "tiny_fp32", "ragged_b32", "long_b4", "bif_mqa",
                             "paged_b1_64k", "int8_b1_64k", "e4m3_b1_64k", "verify4_b1_64k"])
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep-splits", default="",
                    help="comma-separated split counts: print one timing line per count instead")
    ap.add_argument("--sweep-variants", default="",
                    help="with --sweep-splits: comma-separated FD_SPLIT_VARIANT values")
    ap.add_argument("--sweep-lengths", default="",
                    help="with --sweep-splits: comma-separated batch-1 layer lengths instead of --workload")
    ap.add_argument("--bif-sweep", action="store_true",
                    help="bifurcated vs replicated-context over n, Lc and kv heads instead")
    args = ap.parse_args(argv)
    if args.sweep_splits:
        return run_sweep(args)
    if args.bif_sweep:
        return run_bif_sweep(args)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    try:
        return run_fd(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
