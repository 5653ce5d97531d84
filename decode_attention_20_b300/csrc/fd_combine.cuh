// Log-sum-exp combine kernel.
//
// For every output row r (a (sequence, query head) pair, or a (sequence,
// query token, query head) triple for multi-token decode) with S partial
// results (O_i, lse_i):
//   LSE = ln sum_i e^(lse_i)   (evaluated as M + ln sum_i e^(lse_i - M))
//   O   = sum_i e^(lse_i - LSE) * O_i
// Rows whose partials are all empty (every lse_i = -inf) give O = 0 and
// LSE = -inf; an empty split's O_i is never used (its weight selects 0, so
// whatever it holds, even NaN, does not reach the result).  Source:
// Flash-Decoding page ("What is Flash-Decoding and when does it speed up
// LLMs?"), section "Why decoding needs different scheduling": a final
// reduction merges the per-split results exactly.
//
// Two layouts, both one CTA per row:
//   - lse_combine_kernel (grids of up to kCombineFewRows rows, where each
//     row's latency is the cost): 128 to 512 threads, more when a row has
//     many splits, laid out so that a row's loads go out in one round.
//     Thread t owns 4 consecutive head-dim elements c = t % (D/4) of the
//     split group g = t / (D/4) (splits s = g, g + SG, g + 2 SG, ...); it
//     first issues the loads of up to kCombineBatch of its splits' partial
//     rows and their lse_i; meanwhile every warp computes M and
//     sum_i e^(lse_i - M) over all splits by itself (lanes stride over the
//     splits, shuffle reductions), so no block barrier stands between the
//     loads and the weights; then each thread weights and sums its rows (a
//     further batch only past kCombineBatch splits per group) and the SG
//     group sums are added through shared memory.
//   - lse_combine_many_kernel (larger grids, where CTAs resident per SM
//     matter): 128 threads and few registers.  Pass 1: threads stride over
//     the splits for M and sum e^(lse - M) (block reductions); pass 2: the
//     same thread layout as above, each thread recomputing its splits'
//     weights from lse directly so its partial-row loads depend on nothing
//     but the addresses.
// Launched with programmatic stream serialisation behind the split kernel:
// the launch overlaps its tail, and griddepcontrol.wait orders the reads
// after the partial writes.  Each lets its own dependents launch at once.
#pragma once

#include "fd_device.cuh"

namespace fd {

constexpr int kCombineMaxThreads = 512;
constexpr int kCombineBatch = 8;        // partial rows in flight per thread
constexpr int kCombineFewRows = 512;    // grids up to this many rows: lse_combine_kernel
constexpr int kCombineManyThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

// Threads per CTA of lse_combine_kernel for rows of S partials of head dim
// D: enough split groups that one batch covers every split, 128 to 512.
inline int combine_threads(int S, int D) {
  const int CD = D / 4;
  const int groups = (S + kCombineBatch - 1) / kCombineBatch;
  int t = 128;
  while (t < kCombineMaxThreads && (t / CD) < groups) t *= 2;
  return t;
}

// MULTI: rows carry a middle (query token) index; compiled separately so
// the single-token path keeps its shorter index arithmetic.
template <bool MULTI>
__global__ void __launch_bounds__(kCombineMaxThreads)
    lse_combine_kernel(const __grid_constant__ CombineParams p) {
  constexpr float kNegInfC = -__builtin_huge_valf();
  __shared__ float4 acc_s[kCombineMaxThreads];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int nthreads = blockDim.x;
  // The next kernel on the stream (the next call's split kernel, launched
  // with PDL) may start now: it waits for this grid before touching memory.
  pdl_launch_dependents();
  pdl_wait_prerequisites();
  // (Row decode and block size written out as here: a variant that read
  // blockDim.x in place and decoded rows through a helper compiled, for
  // multi-token rows, to a schedule measured 1.5 us slower per call.)
  const int row = blockIdx.x;
  int r1, rm = 0, r2;
  if constexpr (MULTI) {                 // (sequence, query token, head) rows
    if (row >= p.R1 * p.Rm * p.R2) return;
    r1 = row / (p.Rm * p.R2);
    const int rr = row - r1 * (p.Rm * p.R2);
    rm = rr / p.R2;
    r2 = rr - rm * p.R2;
  } else {
    if (row >= p.R1 * p.R2) return;
    r1 = row / p.R2;
    r2 = row - r1 * p.R2;
  }
  const float* pl = p.part_lse + r1 * p.pl_r1 + r2 * p.pl_r2 + (MULTI ? rm * p.pl_rm : 0);
  const float* po = p.part_o + r1 * p.po_r1 + r2 * p.po_r2 + (MULTI ? rm * p.po_rm : 0);
  const int S = p.S;
  const int CD = p.D >> 2;                            // float4 chunks per row (<= 128)
  const int SG = nthreads / CD;                       // split groups (>= 1)
  const int c = tid % CD;
  const int sg = tid / CD;
  const bool owner = sg < SG;                         // threads past SG * CD only reduce
  const float* pc = po + c * 4;

  // ---- first batch of this thread's partial rows and their lse_i
  float4 v[kCombineBatch];
  float ls[kCombineBatch];
#pragma unroll
  for (int k = 0; k < kCombineBatch; ++k) {
    const int s = sg + k * SG;
    if (owner && s < S) {
      v[k] = *reinterpret_cast<const float4*>(pc + s * p.po_s);
      ls[k] = pl[s * p.pl_s];
    } else {
      v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      ls[k] = kNegInfC;
    }
  }

  // ---- per warp: M = max_i lse_i, tot = sum_i e^(lse_i - M)
  float M = kNegInfC;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, pl[s * p.pl_s]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const bool empty = (M == kNegInfC);
  float tot = 0.f;
  if (!empty)
    for (int s = lane; s < S; s += 32) tot += fast_exp2((pl[s * p.pl_s] - M) * kLog2e);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const float inv_tot = empty ? 0.f : 1.f / tot;

  // ---- O = sum_i w_i O_i over this thread's splits (w_i = 0 selects nothing,
  // so an empty split's row, whatever it holds, is never used)
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [&](const float4& x, float lse_i) {
    const float w = fast_exp2((lse_i - M) * kLog2e) * inv_tot;   // -inf -> 0
    if (w != 0.f) {
      acc.x = fmaf(w, x.x, acc.x);
      acc.y = fmaf(w, x.y, acc.y);
      acc.z = fmaf(w, x.z, acc.z);
      acc.w = fmaf(w, x.w, acc.w);
    }
  };
  if (!empty) {
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k) add(v[k], ls[k]);
    for (int s0 = sg + kCombineBatch * SG; owner && s0 < S; s0 += kCombineBatch * SG) {
#pragma unroll
      for (int k = 0; k < kCombineBatch; ++k) {
        const int s = s0 + k * SG;
        if (s < S) {
          v[k] = *reinterpret_cast<const float4*>(pc + s * p.po_s);
          ls[k] = pl[s * p.pl_s];
        } else {
          ls[k] = kNegInfC;
        }
      }
#pragma unroll
      for (int k = 0; k < kCombineBatch; ++k)
        if (ls[k] != kNegInfC) add(v[k], ls[k]);
    }
  }
  acc_s[tid] = acc;
  __syncthreads();
  if (tid < CD) {
    float4 o = acc_s[tid];
    for (int gI = 1; gI < SG; ++gI) {
      const float4 a = acc_s[gI * CD + tid];
      o.x += a.x;
      o.y += a.y;
      o.z += a.z;
      o.w += a.w;
    }
    float* out = p.out + r1 * p.out_r1 + r2 * p.out_r2 + (MULTI ? rm * p.out_rm : 0) + tid * 4;
    out[0] = o.x;
    out[1] = o.y;
    out[2] = o.z;
    out[3] = o.w;
  }
  if (tid == 0 && p.lse != nullptr)
    p.lse[r1 * p.lse_r1 + r2 * p.lse_r2 + (MULTI ? rm * p.lse_rm : 0)] = empty ? M : M + __logf(tot);
}

template <bool MULTI>
__global__ void __launch_bounds__(kCombineManyThreads)
    lse_combine_many_kernel(const __grid_constant__ CombineParams p) {
  constexpr float kNegInfC = -__builtin_huge_valf();
  constexpr int T = kCombineManyThreads;
  __shared__ float red_s[T / 32];
  __shared__ float4 acc_s[T];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int row = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait_prerequisites();
  int r1, rm = 0, r2;
  if constexpr (MULTI) {                 // (sequence, query token, head) rows
    if (row >= p.R1 * p.Rm * p.R2) return;
    r1 = row / (p.Rm * p.R2);
    const int rr = row - r1 * (p.Rm * p.R2);
    rm = rr / p.R2;
    r2 = rr - rm * p.R2;
  } else {
    if (row >= p.R1 * p.R2) return;
    r1 = row / p.R2;
    r2 = row - r1 * p.R2;
  }
  const float* pl = p.part_lse + r1 * p.pl_r1 + r2 * p.pl_r2 + (MULTI ? rm * p.pl_rm : 0);
  const float* po = p.part_o + r1 * p.po_r1 + r2 * p.po_r2 + (MULTI ? rm * p.po_rm : 0);

  // ---- pass 1: M = max_i lse_i, tot = sum_i e^(lse_i - M)
  float M = kNegInfC;
  for (int s = tid; s < p.S; s += T) M = fmaxf(M, pl[s * p.pl_s]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) red_s[warp] = M;
  __syncthreads();
  M = red_s[0];
#pragma unroll
  for (int w = 1; w < T / 32; ++w) M = fmaxf(M, red_s[w]);
  const bool empty = (M == kNegInfC);
  float tot = 0.f;
  if (!empty)
    for (int s = tid; s < p.S; s += T) tot += fast_exp2((pl[s * p.pl_s] - M) * kLog2e);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  __syncthreads();                       // everyone has read red_s (max)
  if (lane == 0) red_s[warp] = tot;
  __syncthreads();
  tot = 0.f;
#pragma unroll
  for (int w = 0; w < T / 32; ++w) tot += red_s[w];
  const float inv_tot = empty ? 0.f : 1.f / tot;

  // ---- pass 2: O = sum_i w_i O_i, split groups in parallel
  const int CD = p.D >> 2;
  const int SG = T / CD;
  const int c = tid % CD;
  const int sg = tid / CD;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!empty && sg < SG) {
    const float* pc = po + c * 4;
#pragma unroll 4
    for (int s = sg; s < p.S; s += SG) {
      const float ls = pl[s * p.pl_s];
      const float4 v = *reinterpret_cast<const float4*>(pc + s * p.po_s);
      const float w = fast_exp2((ls - M) * kLog2e) * inv_tot;   // -inf -> 0
      if (w != 0.f) {
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
    }
  }
  acc_s[tid] = acc;
  __syncthreads();
  if (tid < CD) {
    float4 o = acc_s[tid];
    for (int gI = 1; gI < SG; ++gI) {
      const float4 a = acc_s[gI * CD + tid];
      o.x += a.x;
      o.y += a.y;
      o.z += a.z;
      o.w += a.w;
    }
    float* out = p.out + r1 * p.out_r1 + r2 * p.out_r2 + (MULTI ? rm * p.out_rm : 0) + tid * 4;
    out[0] = o.x;
    out[1] = o.y;
    out[2] = o.z;
    out[3] = o.w;
  }
  if (tid == 0 && p.lse != nullptr)
    p.lse[r1 * p.lse_r1 + r2 * p.lse_r2 + (MULTI ? rm * p.lse_rm : 0)] = empty ? M : M + __logf(tot);
}

// Warp-per-row layout for grids of many rows with at most 32 splits and a
// head dim of at most 128 (D / 4 lanes own 4 consecutive elements each):
// lane s loads lse_s, the warp's shuffle reductions give M and
// sum_i e^(lse_i - M) with no block barrier, and the partial-row loads
// (up to kCombineRowBatch splits at a time, issued before the weights are
// known) go out with the lse loads, so a row costs about one round of
// memory latency.  kCombineRowWarps rows per CTA.
constexpr int kCombineRowWarps = 4;
constexpr int kCombineRowBatch = 16;

template <bool MULTI>
__global__ void __launch_bounds__(kCombineRowWarps * 32)
    lse_combine_rows_kernel(const __grid_constant__ CombineParams p) {
  constexpr float kNegInfC = -__builtin_huge_valf();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kCombineRowWarps + (threadIdx.x >> 5);
  pdl_launch_dependents();
  pdl_wait_prerequisites();
  int r1, rm = 0, r2;
  if constexpr (MULTI) {                 // (sequence, query token, head) rows
    if (row >= p.R1 * p.Rm * p.R2) return;
    r1 = row / (p.Rm * p.R2);
    const int rr = row - r1 * (p.Rm * p.R2);
    rm = rr / p.R2;
    r2 = rr - rm * p.R2;
  } else {
    if (row >= p.R1 * p.R2) return;
    r1 = row / p.R2;
    r2 = row - r1 * p.R2;
  }
  const float* pl = p.part_lse + r1 * p.pl_r1 + r2 * p.pl_r2 + (MULTI ? rm * p.pl_rm : 0);
  const float* po = p.part_o + r1 * p.po_r1 + r2 * p.po_r2 + (MULTI ? rm * p.po_rm : 0);
  const int CD = p.D >> 2;
  const bool owner = lane < CD;
  const float* pc = po + lane * 4;
  // First batch of partial rows and every lse, all in flight at once.
  float4 v[kCombineRowBatch];
#pragma unroll
  for (int k = 0; k < kCombineRowBatch; ++k)
    v[k] = (owner && k < p.S) ? *reinterpret_cast<const float4*>(pc + k * p.po_s)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
  const float ls = lane < p.S ? pl[lane * p.pl_s] : kNegInfC;
  float M = ls;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const bool empty = (M == kNegInfC);
  const float e = empty ? 0.f : fast_exp2((ls - M) * kLog2e);   // -inf -> 0
  float tot = e;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const float w_mine = empty ? 0.f : e / tot;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [&](const float4& x, float w) {
    if (w != 0.f) {              // an empty split's row is never used (it may hold anything)
      acc.x = fmaf(w, x.x, acc.x);
      acc.y = fmaf(w, x.y, acc.y);
      acc.z = fmaf(w, x.z, acc.z);
      acc.w = fmaf(w, x.w, acc.w);
    }
  };
#pragma unroll
  for (int k = 0; k < kCombineRowBatch; ++k) add(v[k], __shfl_sync(0xffffffffu, w_mine, k));
  for (int s0 = kCombineRowBatch; s0 < p.S; s0 += kCombineRowBatch) {
#pragma unroll
    for (int k = 0; k < kCombineRowBatch; ++k)
      v[k] = (owner && s0 + k < p.S) ? *reinterpret_cast<const float4*>(pc + (s0 + k) * p.po_s)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kCombineRowBatch; ++k) add(v[k], __shfl_sync(0xffffffffu, w_mine, (s0 + k) & 31));
  }
  if (owner) {
    float* out = p.out + r1 * p.out_r1 + r2 * p.out_r2 + (MULTI ? rm * p.out_rm : 0) + lane * 4;
    out[0] = acc.x;
    out[1] = acc.y;
    out[2] = acc.z;
    out[3] = acc.w;
  }
  if (lane == 0 && p.lse != nullptr)
    p.lse[r1 * p.lse_r1 + r2 * p.lse_r2 + (MULTI ? rm * p.lse_rm : 0)] = empty ? M : M + __logf(tot);
}

}  // namespace fd
