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

  float M = -__int_as_float(0x7f800000);
  for (int s = lane; s < p.S; s += 32) M = fmaxf(M, pl[s * p.pl_s]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const bool empty = (M == -__int_as_float(0x7f800000));
  float tot = 0.f;
  if (!empty)
    for (int s = lane; s < p.S; s += 32) tot += fast_exp2((pl[s * p.pl_s] - M) * kLog2e);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  // LSE in base 2 relative to M: weights are 2^((lse_i - M) log2 e) / tot.
  const float inv_tot = empty ? 0.f : 1.f / tot;

  for (int c = lane; c * 4 < p.D; c += 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!empty) {
      for (int s = 0; s < p.S; ++s) {
        const float w = fast_exp2((pl[s * p.pl_s] - M) * kLog2e) * inv_tot;
        if (w != 0.f) {
          const float4 v = *reinterpret_cast<const float4*>(po + s * p.po_s + c * 4);
          acc.x = fmaf(w, v.x, acc.x);
          acc.y = fmaf(w, v.y, acc.y);
          acc.z = fmaf(w, v.z, acc.z);
          acc.w = fmaf(w, v.w, acc.w);
        }
      }
    }
    float* out = p.out + r1 * p.out_r1 + r2 * p.out_r2 + c * 4;
    out[0] = acc.x;
    out[1] = acc.y;
    out[2] = acc.z;
    out[3] = acc.w;
  }
  if (lane == 0 && p.lse != nullptr)
    p.lse[r1 * p.lse_r1 + r2 * p.lse_r2] = empty ? M : M + __logf(tot);
}

}  // namespace fd
