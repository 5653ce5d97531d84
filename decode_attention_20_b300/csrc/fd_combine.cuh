// Log-sum-exp combine kernel.
//
// For every output row r (a (sequence, query head) pair) with S partial
// results (O_i, lse_i):
//   LSE = ln sum_i e^(lse_i)   (evaluated as M + ln sum_i e^(lse_i - M))
//   O   = sum_i e^(lse_i - LSE) * O_i
// Rows whose partials are all empty (every lse_i = -inf) give O = 0 and
// LSE = -inf.  Source: Flash-Decoding page ("What is Flash-Decoding and when
// does it speed up LLMs?"), section "Why decoding needs different
// scheduling": a final reduction merges the per-split results exactly.
//
// One warp per row; each lane owns 4 consecutive head-dim elements (16-byte
// loads, coalesced across the warp).  Launched with programmatic stream
// serialisation behind the split kernel: the prologue overlaps its tail, and
// griddepcontrol.wait orders the reads after the partial writes.
#pragma once

#include "fd_device.cuh"

namespace fd {

constexpr int kCombineWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;

__global__ void __launch_bounds__(kCombineWarps * 32)
    lse_combine_kernel(const __grid_constant__ CombineParams p) {
  constexpr float kNegInfC = -__builtin_huge_valf();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kCombineWarps + warp;
  const int rows = p.R1 * p.R2;
  pdl_wait_prerequisites();
  if (row >= rows) return;
  const int r1 = row / p.R2;
  const int r2 = row - r1 * p.R2;
  const float* pl = p.part_lse + r1 * p.pl_r1 + r2 * p.pl_r2;
  const float* po = p.part_o + r1 * p.po_r1 + r2 * p.po_r2;

  // Pass 1 (lanes over splits, all loads in parallel): M and sum e^(lse-M).
  float M = kNegInfC;
  for (int s0 = 0; s0 < p.S; s0 += 32) {
    const int s = s0 + lane;
    M = fmaxf(M, s < p.S ? pl[s * p.pl_s] : kNegInfC);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const bool empty = (M == kNegInfC);
  float tot = 0.f;
  if (!empty) {
    for (int s0 = 0; s0 < p.S; s0 += 32) {
      const int s = s0 + lane;
      if (s < p.S) tot += fast_exp2((pl[s * p.pl_s] - M) * kLog2e);
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const float inv_tot = empty ? 0.f : 1.f / tot;

  // Pass 2: each lane owns 4 consecutive head-dim elements; the weight of
  // split s is broadcast from lane s of the chunk; loads are batched.
  // (Every lane runs every iteration so the full-warp shuffles stay
  // converged; lanes past the head dimension only skip their loads/stores.)
  for (int c0 = 0; c0 * 4 < p.D; c0 += 32) {
    const int c = c0 + lane;
    const bool active = c * 4 < p.D;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!empty) {
      for (int s0 = 0; s0 < p.S; s0 += 32) {
        const int sl = s0 + lane;
        const float w_lane = sl < p.S ? fast_exp2((pl[sl * p.pl_s] - M) * kLog2e) * inv_tot : 0.f;
        const int nchunk = min(32, p.S - s0);
#pragma unroll 8
        for (int j = 0; j < nchunk; ++j) {
          const float w = __shfl_sync(0xffffffffu, w_lane, j);
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (active && w != 0.f)                       // empty split: ignore its O
            v = *reinterpret_cast<const float4*>(po + (s0 + j) * p.po_s + c * 4);
          acc.x = fmaf(w, v.x, acc.x);
          acc.y = fmaf(w, v.y, acc.y);
          acc.z = fmaf(w, v.z, acc.z);
          acc.w = fmaf(w, v.w, acc.w);
        }
      }
    }
    if (active) {
      float* out = p.out + r1 * p.out_r1 + r2 * p.out_r2 + c * 4;
      out[0] = acc.x;
      out[1] = acc.y;
      out[2] = acc.z;
      out[3] = acc.w;
    }
  }
  if (lane == 0 && p.lse != nullptr)
    p.lse[r1 * p.lse_r1 + r2 * p.lse_r2] = empty ? M : M + __logf(tot);
}

}  // namespace fd
