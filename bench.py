"""Benchmark of the decode-attention hot path on one B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fd|reference]
                    [--workload b1_64k|ragged_b32|long_b4|bif_mqa|paged_b1_64k|
                                int8_b1_64k|e4m3_b1_64k|verify4_b1_64k]
                    [--num-splits S] [--bif-sweep]

Default workload: split-KV decode attention at batch 1 over a 65536-token
history of a CodeLlama-34B-shaped layer (64 query heads, 8 kv heads, head
dim 128, bf16 K/V, fp32 out + LSE).  One step = one library call (split
kernel + log-sum-exp combine) over the whole history.  Other workloads:
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
  value        device-timed microseconds per call: CUDA events around K calls
               replayed from a CUDA graph, inputs resident in HBM and rotated
               over enough copies that every call reads past L2
  e2e          microseconds per step through the Python API: H2D from pinned
               host memory of the step's new inputs (query, one new K/V row per
               sequence), the call, D2H of out (+ lse), synchronised per step
  roofline     the dominant kernel's algorithmic bytes (or FLOPs) per launch /
               its mean CUDA-event duration (launches queued back to back,
               without programmatic dependent launch), against the peak
  cpu_baseline the fp64 CPU oracle timed on a bounded sample of the same
               workload on the host cores (rank 0, N = 1)
With --gpus N > 1 (torchrun), every rank runs an independent replica (the
method has no cross-GPU exchange); value is the max over ranks.

--impl reference times the fp64 CPU oracle instead (each step a bounded
sample of the same workload, extrapolated to one full call).
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

# Source files each roofline kernel is built from: a DRAM-traffic figure in
# profiles/traffic.json is used only while their code (comments and
# whitespace aside) hashes to the value it was captured with; otherwise the
# kernel has changed and traffic is null.
KERNEL_SOURCES = {
    FD_KERNEL_SPLIT: ["fd_split_mma.cuh", "fd_split.cuh", "fd_device.cuh"],
    FD_KERNEL_BIF_CTX: ["fd_bif_ctx.cuh", "fd_tcgen05.cuh", "fd_split.cuh", "fd_device.cuh"],
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
                 "-lms", "50", "-i", str(self.gpu_id)],
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


def _host_loop_us(stream, steps, step, warmup=5):
    """Wall-clock microseconds per call of step(i) on `stream`, after
    `warmup` untimed calls (first-use costs: lazy kernel loading, pinned
    staging, pool growth)."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(steps):
            step(i)
    return (time.perf_counter() - t0) * 1e6 / steps


class DecodeWorkload(Workload):
    dominant = FD_KERNEL_SPLIT

    def __init__(self, short, builder, device):
        import torch
        from decode_attention_20_b300 import inputs
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
        self.nbuf = max(1, min(8, math.ceil(2 * L2_BYTES / kv_bytes) + (1 if kv_bytes < 4 * L2_BYTES else 0)))
        self.ks = [c.k] + [c.k.clone() for _ in range(self.nbuf - 1)]
        self.vs = [c.v] + [c.v.clone() for _ in range(self.nbuf - 1)]
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

    def api_call(self, q, k, v, stream):
        import decode_attention_20_b300 as fd
        fd.decode_attention(q, k, v, self.seqlens_dev, self.ns, self.case.scale, out=self.out,
                            lse=self.lse, stream=stream)

    def e2e(self, stream, steps):
        """Per step: H2D of the new query and one new K/V row per sequence
        (written at position len_b - 1), the call, D2H of out + lse."""
        import torch
        import decode_attention_20_b300 as fd
        c = self.case
        hq = torch.empty(c.q.shape, dtype=c.q.dtype).pin_memory()
        hq.copy_(c.q.cpu())
        # the Tq newest rows of every sequence (positions len_b - Tq .. len_b - 1)
        pos = [(b, j) for b, n in enumerate(self.lens) for j in range(max(0, n - self.Tq), max(n, 1))]
        nr = len(pos)
        hk = torch.empty((nr, self.Hkv, self.D), dtype=c.k.dtype).pin_memory()
        hv = torch.empty_like(hk).pin_memory()
        for i, (b, j) in enumerate(pos):
            hk[i].copy_(c.k[b, j].cpu())
            hv[i].copy_(c.v[b, j].cpu())
        hout = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()
        hlse = torch.empty(self.lse.shape, dtype=torch.float32).pin_memory()
        rows = torch.tensor([b * self.Lcap + j for b, j in pos], dtype=torch.int64,
                            device=c.q.device)
        dk = torch.empty((nr, self.Hkv * self.D), dtype=c.k.dtype, device=c.q.device)
        dv = torch.empty_like(dk)

        def step(i):
            kb, vb = self.ks[i % self.nbuf], self.vs[i % self.nbuf]
            c.q.copy_(hq, non_blocking=True)
            dk.copy_(hk.view(nr, -1), non_blocking=True)
            dv.copy_(hv.view(nr, -1), non_blocking=True)
            _rows(kb, self.B * self.Lcap).index_copy_(0, rows, _rows(dk, nr))
            _rows(vb, self.B * self.Lcap).index_copy_(0, rows, _rows(dv, nr))
            self.api_call(c.q, kb, vb, stream)
            hout.copy_(self.out, non_blocking=True)
            hlse.copy_(self.lse, non_blocking=True)
            stream.synchronize()

        us = _host_loop_us(stream, steps, step)
        h2d = hq.numel() * hq.element_size() + hk.numel() * hk.element_size() * 2
        d2h = hout.numel() * 4 + hlse.numel() * 4
        return us, h2d, d2h

    def _oracle_inputs(self, n0):
        c = self.case
        return f64(c.q[0:1]), f64(c.k[0:1, :n0]), f64(c.v[0:1, :n0])

    def _oracle_call(self, q, k, v, T):
        import oracle
        oracle.decode_attention_ref(q, k[:, :T], v[:, :T], None, self.case.scale)

    def oracle_sample(self, target_s):
        """Time the oracle on the first T tokens of sequence 0 (all kv
        heads), T sized for about target_s seconds (at least 64 tokens);
        returns (us per full call extrapolated by tokens, sample text,
        seconds of the sample)."""
        if not hasattr(self, "_of"):
            n0 = max(self.lens[0], 1)
            self._of = self._oracle_inputs(n0)
            q, k, v = self._of
            T0 = min(n0, 2048)
            t0 = time.perf_counter()
            self._oracle_call(q, k, v, T0)
            self._per_tok = (time.perf_counter() - t0) / T0
        q, k, v = self._of
        T = int(max(min(64, self.lens[0]), min(self.lens[0], target_s / self._per_tok)))
        t0 = time.perf_counter()
        self._oracle_call(q, k, v, T)
        dt = time.perf_counter() - t0
        full = dt * (sum(self.lens) / T)
        return full * 1e6, (f"sequence 0, first {T} tokens x all {self.Hkv} kv heads per call, "
                            f"extrapolated linearly to {sum(self.lens)} tokens x {self.B} sequences"), dt


class BifWorkload(Workload):
    dominant = FD_KERNEL_BIF_CTX

    def __init__(self, device):
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
        self.nbuf = max(1, math.ceil(2 * L2_BYTES / per_copy))
        self.bufs = [(c.q, c.k_ctx, c.v_ctx, c.k_dec, c.v_dec)] + [
            tuple(x.clone() for x in (c.q, c.k_ctx, c.v_ctx, c.k_dec, c.v_dec))
            for _ in range(self.nbuf - 1)]
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
        """Per step: H2D of the queries and one new decode K/V row per sample,
        the call, D2H of out + lse."""
        import torch
        import decode_attention_20_b300 as fd
        c = self.case
        hq = torch.empty(c.q.shape, dtype=c.q.dtype).pin_memory()
        hq.copy_(c.q.cpu())
        hk = torch.empty((self.n, self.Hkv, self.D), dtype=c.k_dec.dtype).pin_memory()
        hv = torch.empty_like(hk).pin_memory()
        pos = [max(0, x - 1) for x in c.lens]
        for b in range(self.n):
            hk[b].copy_(c.k_dec[b, pos[b]].cpu())
            hv[b].copy_(c.v_dec[b, pos[b]].cpu())
        hout = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()
        hlse = torch.empty(self.lse.shape, dtype=torch.float32).pin_memory()
        rows = torch.tensor([b * self.Ld + pos[b] for b in range(self.n)], dtype=torch.int64,
                            device=c.q.device)
        dk = torch.empty((self.n, self.Hkv * self.D), dtype=c.k_dec.dtype, device=c.q.device)
        dv = torch.empty_like(dk)

        def step(i):
            q, kc, vc, kd, vd = self.bufs[i % self.nbuf]
            q.copy_(hq, non_blocking=True)
            dk.copy_(hk.view(self.n, -1), non_blocking=True)
            dv.copy_(hv.view(self.n, -1), non_blocking=True)
            kd.view(self.n * self.Ld, -1).index_copy_(0, rows, dk)
            vd.view(self.n * self.Ld, -1).index_copy_(0, rows, dv)
            fd.bifurcated_attention(q, kc, vc, kd, vd, self.dec_dev, c.scale, out=self.out,
                                    lse=self.lse, ctx_splits=self.ns, return_lse=True,
                                    stream=stream)
            hout.copy_(self.out, non_blocking=True)
            hlse.copy_(self.lse, non_blocking=True)
            stream.synchronize()

        us = _host_loop_us(stream, steps, step)
        h2d = hq.numel() * 2 + hk.numel() * 2 * 2
        d2h = hout.numel() * 4 + hlse.numel() * 4
        return us, h2d, d2h

    def oracle_sample(self, target_s):
        """Time the oracle on sample 0 with the first T context tokens (and
        its own decode tokens), T sized for about target_s seconds (at least
        64); returns (us per full call extrapolated by tokens and samples,
        sample text, seconds of the sample)."""
        import oracle
        c = self.case
        lens = c.lens
        if not hasattr(self, "_of"):
            self._of = (f64(c.q[:1]), f64(c.k_ctx), f64(c.v_ctx), f64(c.k_dec[:1]), f64(c.v_dec[:1]))
            q, kc, vc, kd, vd = self._of
            T0 = min(self.Lc, 2048)
            t0 = time.perf_counter()
            oracle.bifurcated_attention_ref(q, kc[:T0], vc[:T0], kd, vd, [lens[0]], c.scale)
            self._per_tok = (time.perf_counter() - t0) / (T0 + lens[0])
        q, kc, vc, kd, vd = self._of
        T = int(max(64, min(self.Lc, target_s / self._per_tok - lens[0])))
        t0 = time.perf_counter()
        oracle.bifurcated_attention_ref(q, kc[:T], vc[:T], kd, vd, [lens[0]], c.scale)
        dt = time.perf_counter() - t0
        full_tokens = sum(self.Lc + x for x in lens)
        return dt * full_tokens / (T + lens[0]) * 1e6, (
            f"sample 0 with the first {T} of {self.Lc} context tokens and its {lens[0]} decode "
            f"tokens per call, extrapolated linearly to {self.n} samples"), dt


class PagedWorkload(DecodeWorkload):
    """The batch-1 64K layer with its history in scattered 64-token pages
    (fd_decode_attention_paged)."""

    def __init__(self, device):
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
        self.nbuf = max(1, min(8, math.ceil(2 * L2_BYTES / kv_bytes) + (1 if kv_bytes < 4 * L2_BYTES else 0)))
        self.ks = [c.k_pages] + [c.k_pages.clone() for _ in range(self.nbuf - 1)]
        self.vs = [c.v_pages] + [c.v_pages.clone() for _ in range(self.nbuf - 1)]
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
        """Per step: H2D of the new query and of the newest token's K/V row
        into its page, the paged call, D2H of out + lse."""
        import torch
        import decode_attention_20_b300 as fd
        c = self.pcase
        hq = torch.empty(c.q.shape, dtype=c.q.dtype).pin_memory()
        hq.copy_(c.q.cpu())
        last = self.Lcap - 1
        pid = int(c.block_table[0, last // self.page_size])
        row = pid * self.page_size + last % self.page_size
        hk = torch.empty((1, self.Hkv * self.D), dtype=c.k_pages.dtype).pin_memory()
        hv = torch.empty_like(hk).pin_memory()
        hk.copy_(c.k_pages.view(-1, self.Hkv * self.D)[row:row + 1].cpu())
        hv.copy_(c.v_pages.view(-1, self.Hkv * self.D)[row:row + 1].cpu())
        hout = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()
        hlse = torch.empty(self.lse.shape, dtype=torch.float32).pin_memory()

        def step(i):
            kb, vb = self.ks[i % self.nbuf], self.vs[i % self.nbuf]
            c.q.copy_(hq, non_blocking=True)
            kb.view(-1, self.Hkv * self.D)[row:row + 1].copy_(hk, non_blocking=True)
            vb.view(-1, self.Hkv * self.D)[row:row + 1].copy_(hv, non_blocking=True)
            fd.decode_attention_paged(c.q, kb, vb, self.bt_dev, None, self.ns, c.scale,
                                      out=self.out, lse=self.lse, stream=stream)
            hout.copy_(self.out, non_blocking=True)
            hlse.copy_(self.lse, non_blocking=True)
            stream.synchronize()

        us = _host_loop_us(stream, steps, step)
        return us, hq.numel() * 2 + hk.numel() * 2 * 2, hout.numel() * 4 + hlse.numel() * 4


class MultiWorkload(DecodeWorkload):
    """The batch-1 64K-token layer verifying Tq new tokens at once
    (fd_decode_attention_multi)."""

    def __init__(self, short, tq, device):
        from decode_attention_20_b300 import inputs
        super().__init__(short, lambda d: inputs.speculative_b1(65536, tq=tq, device=d), device)

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

    def api_call(self, q, k, v, stream):
        import decode_attention_20_b300 as fd
        fd.decode_attention_multi(q, k, v, self.seqlens_dev, self.ns, self.case.scale,
                                  out=self.out, lse=self.lse, stream=stream)

    def _oracle_call(self, q, k, v, T):
        import oracle
        oracle.multi_token_decode_ref(q, k[:, :T], v[:, :T], None, self.case.scale)


class QuantWorkload(DecodeWorkload):
    """The batch-1 64K-token layer over an 8-bit cache (int8 or e4m3 codes,
    one scale per kv head): fd_decode_attention_quant."""
    dtype = "f16"
    kernel_name = "split_mma_kernel (mma.sync f16 over 8-bit codes, TMA ring)"

    def __init__(self, short, kind, device):
        from decode_attention_20_b300 import inputs
        super().__init__(short, lambda d: inputs.quant_flash_decoding_b1(65536, kind=kind, device=d),
                         device)
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

    def api_call(self, q, k, v, stream):
        import decode_attention_20_b300 as fd
        c = self.case
        fd.decode_attention_quant(q, k, v, c.k_scale, c.v_scale, self.seqlens_dev, self.ns,
                                  c.scale, out=self.out, lse=self.lse, stream=stream)

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


def make_workload(short, device):
    from decode_attention_20_b300 import inputs
    if short == "b1_64k":
        return DecodeWorkload(short, lambda d: inputs.flash_decoding_b1(65536, seed=0, device=d), device)
    if short == "ragged_b32":
        return DecodeWorkload(short, lambda d: inputs.ragged_batch(device=d), device)
    if short == "long_b4":
        return DecodeWorkload(short, lambda d: inputs.long_context_peaked(device=d), device)
    if short == "bif_mqa":
        return BifWorkload(device)
    if short == "paged_b1_64k":
        return PagedWorkload(device)
    if short == "verify4_b1_64k":
        return MultiWorkload(short, 4, device)
    if short == "int8_b1_64k":
        return QuantWorkload(short, "int8", device)
    if short == "e4m3_b1_64k":
        return QuantWorkload(short, "e4m3", device)
    raise SystemExit(f"unknown workload {short}")


# ------------------------------------------------------------------ reference arm

def run_reference(args, rank):
    """--impl reference: the fp64 oracle on host cores, same workload."""
    if rank != 0:
        return 0
    w = make_workload(args.workload, "cpu")
    budget = 100.0 / max(1, args.steps + args.warmup)
    us = []
    sample = ""
    step_s = []
    for i in range(args.warmup + args.steps):
        u, sample, dt = w.oracle_sample(budget)
        if i >= args.warmup:
            us.append(u)
            step_s.append(dt)
    value = statistics.median(us)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "us/call",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.median(step_s) * 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": w.config(args.num_splits),
        "cpu_baseline": {"value": round(value, 1), "unit": "us/call", "cores": blas_threads(),
                         "kind": "oracle", "sample": sample},
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
        for i in range(warm):
            w.call(i)
    stream.synchronize()
    fd.check_device_error(stream)

    # CUDA graph of nbuf consecutive calls (one per rotating input copy)
    # One graph holds at least 16 back-to-back calls (cycling the rotating
    # input copies), so graph-launch boundaries, which break the
    # programmatic overlap of consecutive calls, are rare.
    glen = w.nbuf * max(1, math.ceil(16 / w.nbuf))
    reps = max(1, math.ceil(args.steps / glen))
    steps = reps * glen
    graph = None
    timing = f"CUDA graph of {glen} calls, replayed"
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(glen):
                w.call(i)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        graph = g
    except Exception as ex:  # capture unsupported: time direct calls instead
        timing = f"direct calls (graph capture failed: {type(ex).__name__})"
        torch.cuda.synchronize()

    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    gpu_id = vis.split(",")[dev.index] if vis else str(dev.index)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        if graph is not None:
            for _ in range(reps):
                graph.replay()
        else:
            for i in range(steps):
                w.call(i)
        e1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    us_per_call = e0.elapsed_time(e1) * 1e3 / steps
    del graph

    # Direct API calls (no graph), same rotation: launch overhead included.
    dsteps = min(steps, 2000)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(dsteps):
            w.call(i)
        e1.record(stream)
    stream.synchronize()
    us_direct = e0.elapsed_time(e1) * 1e3 / dsteps

    # Per-kernel durations (CUDA events around each launch on its stream).
    # The calls are queued behind a device-side delay longer than the host
    # takes to issue them, so the GPU runs them back to back and each event
    # pair brackets its kernel, not the host's time to issue the next call
    # (short calls are host-bound when issued one by one).
    psteps = min(dsteps, 128)
    delay_us = 2.0 * psteps * us_direct + 5000.0
    fd.profile_enable(True)
    sleep = getattr(torch.cuda, "_sleep", None)       # a device-side spin of N clock cycles
    with torch.cuda.stream(stream):
        if sleep is not None:
            sleep(int(delay_us * SLEEP_CYCLES_PER_US))
        for i in range(psteps):
            w.call(i)
    stream.synchronize()
    kern = {}
    launches = 0
    for kind, label in [(FD_KERNEL_SPLIT, "split"), (FD_KERNEL_COMBINE, "combine"),
                        (FD_KERNEL_BIF_CTX, "bif_ctx")]:
        n, ms = fd.profile_read(kind)
        launches += n
        if n:
            kern[label + "_us"] = round(ms * 1e3 / n, 3)
            kern[label + "_launches_per_call"] = n / psteps
    fd.profile_enable(False)
    launches_per_call = launches / psteps
    dom_label = {FD_KERNEL_SPLIT: "split", FD_KERNEL_BIF_CTX: "bif_ctx"}[w.dominant]
    dom_us = kern[dom_label + "_us"]

    extra = {}
    if isinstance(w, BifWorkload):
        rep_us, rep_kv = w.replicated_us(stream, min(steps, 400), 0)
        extra["replicated_context_us"] = round(rep_us, 3)
        extra["speedup_vs_replicated"] = round(rep_us / us_per_call, 3)
        kv_bif = w.case.k_ctx.numel() * 4 + sum(w.case.lens) * w.Hkv * w.D * 4
        extra["kv_byte_ratio_replicated_over_bifurcated"] = round(rep_kv / kv_bif, 3)
        extra["h_over_g"] = w.Hq // w.Hkv

    e2e_us, h2d, d2h = w.e2e(stream, max(1, min(steps, 1000)))
    fd.check_device_error(stream)

    vals = torch.tensor([us_per_call, e2e_us, dom_us], dtype=torch.float64, device=dev)
    vals = max_over_ranks(vals, world)
    us_per_call, e2e_us, dom_us = [float(x) for x in vals.tolist()]
    if rank != 0:
        return 0

    peaks = load_peaks()
    gbs = w.required / (us_per_call * 1e-6) / 1e9 * world
    if w.bound == "hbm":
        achieved = w.dominant_units / (dom_us * 1e-6) / 1e9
        peak = peaks["hbm_gbs"]
        per_launch = int(w.dominant_units)
    else:
        achieved = w.dominant_units / (dom_us * 1e-6) / 1e12
        peak = peaks["bf16_tflops"]
        per_launch = w.dominant_units
    line = {
        "metric": METRIC, "value": round(us_per_call, 3), "unit": "us/call",
        "n_gpus": world, "steps": steps, "warmup": warm,
        "ms_per_step": us_per_call / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": getattr(w, "dtype", "bf16"),
        "data": "synthetic",
        "config": dict(w.config(ns), parallelism="replicas" if world > 1 else "single",
                       l2=f"inputs larger than L2: {w.nbuf} rotating input copies",
                       timing=timing),
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
        "gpu_launches": int(round(launches_per_call * steps)),
    }
    line.update(extra)
    if world == 1 and not args.no_cpu_baseline:
        import torch as _t
        u, sample, dt = w.oracle_sample(args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(u, 1), "unit": "us/call", "cores": blas_threads(),
                                "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)
    return 0


def run_sweep(args):
    """--sweep-splits: per split count (and split-kernel variant, through
    the library's FD_SPLIT_VARIANT knob), the device time per call of back-
    to-back calls and the split kernel's event-timed launch; one JSON line
    each.  A tuning aid, not the benchmark line."""
    import torch
    import decode_attention_20_b300 as fd
    from decode_attention_20_b300 import _lib
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    L = _lib.lib()
    w = make_workload(args.workload, dev)
    stream = torch.cuda.Stream(device=dev)
    variants = args.sweep_variants.split(",") if args.sweep_variants else [""]
    iters = max(10, min(args.steps, 200))
    for var in variants:
        if var:
            os.environ["FD_SPLIT_VARIANT"] = var
        else:
            os.environ.pop("FD_SPLIT_VARIANT", None)
        for ns in [int(x) for x in args.sweep_splits.split(",")]:
            w.prepare(L, stream, ns)
            with torch.cuda.stream(stream):
                for i in range(3):
                    w.call(i)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for i in range(iters):
                    w.call(i)
                e1.record(stream)
            stream.synchronize()
            call_us = e0.elapsed_time(e1) * 1e3 / iters
            fd.profile_enable(True)
            with torch.cuda.stream(stream):
                for i in range(iters):
                    w.call(i)
            stream.synchronize()
            kern = {}
            for kind, label in [(FD_KERNEL_SPLIT, "split"), (FD_KERNEL_COMBINE, "combine"),
                                (FD_KERNEL_BIF_CTX, "bif_ctx")]:
                n, ms = fd.profile_read(kind)
                if n:
                    kern[label + "_us"] = round(ms * 1e3 / n, 3)
            fd.profile_enable(False)
            fd.check_device_error(stream)
            row = {"workload": w.name, "variant": var or "default", "splits": ns,
                   "call_us": round(call_us, 3), **kern}
            if isinstance(w, DecodeWorkload):
                row["split_gbs"] = round(w.dominant_units / (kern["split_us"] * 1e-6) / 1e9, 1)
            print(json.dumps(row), flush=True)
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
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["fd", "reference"], default="fd")
    ap.add_argument("--workload", default="b1_64k",
                    choices=["b1_64k", "ragged_b32", "long_b4", "bif_mqa", "paged_b1_64k",
                             "int8_b1_64k", "e4m3_b1_64k", "verify4_b1_64k"])
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep-splits", default="",
                    help="comma-separated split counts: print one timing line per count instead")
    ap.add_argument("--sweep-variants", default="",
                    help="with --sweep-splits: comma-separated FD_SPLIT_VARIANT values")
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
        return run_reference(args, rank)
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
