// Bifurcated attention, context part, on the 5th-generation tensor cores.
//
// n samples share one context KV [Lc, Hkv, D].  For kv head g, the rows of
// the problem are all (sample s, query head r of group g) pairs, so the
// context part is a dense attention of M = n * G query rows against Lc keys:
//   S = Q_g K_ctx[g]^T          (GEMM 1, K-dim = D)
//   online softmax over the tokens of a split
//   O = P V_ctx[g]              (GEMM 2, K-dim = tokens)
// and the context KV is read once per M-tile instead of once per sample.
// Each CTA writes, for its 128 rows and one token split of the context, the
// normalised partial output and its natural-log log-sum-exp, in the same
// partial format as the split kernel; the log-sum-exp reduction then merges
// them with the per-sample decode part.  Source: summary of "Bifurcated
// Attention for Single-Context Large-Batch Sampling" (linnk.ai), sections
// "Tiivistelmä" (two GEMMs, prefill KV and decode KV, exact result) and
// "Tilastot" (KV I/O b*g*m*k instead of b*h*m*k); online softmax after
// "How does Flash Attention reduce memory traffic during local inference?",
// section on online softmax.
//
// CTA = one 128-row M-tile x one context split x one kv head; 6 warps:
//   warp 0      TMA producer: the Q tile once, then K and V tiles of 128
//               tokens into separate rings (3 K stages, 2 V stages), all with
//               the 128-byte swizzle (two 64-column boxes per tile).
//   warp 1      allocates 512 TMEM columns; one thread issues every MMA:
//               S_j = Q K_j^T into one of two TMEM score buffers (128 cols
//               each), O += P_j V_j into the TMEM accumulator (128 cols).
//   warps 2..5  softmax: thread = one row (its TMEM lane).  Reads the row of
//               S_j, keeps the running max m / sum l in base 2, writes the
//               probabilities as bf16 into the K-major P tile in shared
//               memory, and rescales the TMEM accumulator on the rare tiles
//               where the running max grows by more than 8 (lazy rescale;
//               p <= 256 always, and numerator and denominator share m).
// Overlap: while the softmax warps work on S_j, the tensor core computes
// S_{j+1} into the other buffer and finishes O += P_{j-1} V_{j-1}.
// Every wait is bounded; on a timeout the CTA drains its copies and MMAs,
// frees its tensor memory and returns with the device error flag set.
#pragma once

#include "fd_split.cuh"
#include "fd_tcgen05.cuh"

namespace fd {

// 3-D tiled tensor load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

struct BifCfg {
  static constexpr int M = 128;                 // rows per CTA (TMEM lanes)
  static constexpr int D = 128;                 // head dim
  static constexpr int TN = kBifTileTokens;     // tokens per tile
  static constexpr int NK = 3;                  // K stages
  static constexpr int NV = 2;                  // V stages
  static constexpr int THREADS = 192;
  static constexpr int CHUNK_BYTES = 128 * 128; // 128 rows x 64 bf16 (one swizzled box)
  static constexpr int Q_BYTES = 2 * CHUNK_BYTES;
  static constexpr int KV_BYTES = 2 * TN * 128; // one K or V tile (two 64-col boxes)
  static constexpr int P_BYTES = 2 * CHUNK_BYTES;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + NK * KV_BYTES;
  static constexpr int OFF_P = OFF_V + NV * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  // barriers: q_full, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV],
  // s_full[2], p_full, o_done, drain
  static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 2 + 3;
  static constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256;
  static_assert(TN == 128, "score buffers and P tile are laid out for 128-token tiles");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

// Context split i of ns over [0, Lc): whole 128-token tiles.
__device__ __forceinline__ void bif_split_range(int Lc, int ns, int i, int& begin, int& end) {
  const int per = (Lc + ns - 1) / ns;
  const long long chunk = (long long)((per + BifCfg::TN - 1) / BifCfg::TN) * BifCfg::TN;
  const long long b0 = (long long)i * chunk;
  begin = (int)(b0 < Lc ? b0 : Lc);
  end = (int)(b0 + chunk < Lc ? b0 + chunk : Lc);
}

__global__ void __launch_bounds__(BifCfg::THREADS, 1)
    bif_ctx_kernel(const __grid_constant__ BifCtxParams p, const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using C = BifCfg;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + C::NK;
  uint64_t* v_full = k_empty + C::NK;
  uint64_t* v_empty = v_full + C::NV;
  uint64_t* s_full = v_empty + C::NV;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* drain = o_done + 1;
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_s = reinterpret_cast<int*>(taddr_s + 1);

  const int mtile = blockIdx.x;
  const int split = blockIdx.y;
  const int g = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int begin, end;
  bif_split_range(p.Lc, p.ns, split, begin, end);
  const int ntiles = (end - begin + C::TN - 1) / C::TN;
  const int rows_per_tile_samples = C::M / p.G;   // samples per M-tile

  if (ntiles == 0) {
    // Empty split: O = 0, lse = -inf for every valid row.
    if (threadIdx.x < C::M) {
      const int m = mtile * C::M + threadIdx.x;
      if (m < p.rows) {
        const int s = m / p.G, h = g * p.G + (m - s * p.G);
        float* o = p.o + s * p.o_sb + h * p.o_sh + split * p.o_ss;
        for (int d = 0; d < C::D; d += 4) *reinterpret_cast<float4*>(o + d) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.lse) p.lse[s * p.l_sb + h * p.l_sh + split * p.l_ss] = kNegInf;
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) mbar_init(&bars[i], &bars[i] == p_full ? 128 : 1);
    *abort_s = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(taddr_s, C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *taddr_s;

  const uint32_t sbase = smem_u32(smem);
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
      const int s0 = mtile * rows_per_tile_samples;
      tma_load_3d(smem + C::OFF_Q, &tmQ, q_full, 0, g * p.G, s0);
      tma_load_3d(smem + C::OFF_Q + C::CHUNK_BYTES, &tmQ, q_full, 64, g * p.G, s0);
      int kt = 0, vt = 0;                           // next K / V tile to issue
      bool ok = true;
      while (ok && (kt < ntiles || vt < ntiles)) {
        // K runs up to NK tiles ahead; V follows.
        if (kt < ntiles && (kt < vt + C::NK)) {
          const int st = kt % C::NK;
          if (kt >= C::NK) ok = mbar_wait_or_abort(&k_empty[st], ((kt / C::NK) - 1) & 1, abort_s);
          if (!ok) break;
          unsigned char* dst = smem + C::OFF_K + st * C::KV_BYTES;
          mbar_arrive_expect_tx(&k_full[st], C::KV_BYTES);
          const int tok = begin + kt * C::TN;
          tma_load_3d(dst, &tmK, &k_full[st], 0, g, tok);
          tma_load_3d(dst + C::KV_BYTES / 2, &tmK, &k_full[st], 64, g, tok);
          ++kt;
        }
        if (vt < ntiles && vt < kt) {
          const int st = vt % C::NV;
          if (vt >= C::NV) ok = mbar_wait_or_abort(&v_empty[st], ((vt / C::NV) - 1) & 1, abort_s);
          if (!ok) break;
          unsigned char* dst = smem + C::OFF_V + st * C::KV_BYTES;
          mbar_arrive_expect_tx(&v_full[st], C::KV_BYTES);
          const int tok = begin + vt * C::TN;
          tma_load_3d(dst, &tmV, &v_full[st], 0, g, tok);
          tma_load_3d(dst + C::KV_BYTES / 2, &tmV, &v_full[st], 64, g, tok);
          ++vt;
        }
      }
      // Never leave with copies in flight: wait for the last load of every
      // stage (earlier loads of a stage completed before it was refilled).
      mbar_wait_bounded(q_full, 0);
      for (int t = (kt > C::NK ? kt - C::NK : 0); t < kt; ++t)
        mbar_wait_bounded(&k_full[t % C::NK], (t / C::NK) & 1);
      for (int t = (vt > C::NV ? vt - C::NV : 0); t < vt; ++t)
        mbar_wait_bounded(&v_full[t % C::NV], (t / C::NV) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = tc::idesc_bf16_f32(C::M, C::TN, false, false);
      constexpr uint32_t IDESC_O = tc::idesc_bf16_f32(C::M, C::D, false, true);
      const uint32_t q_addr = sbase + C::OFF_Q;
      const uint32_t p_addr = sbase + C::OFF_P;
      bool ok = mbar_wait_or_abort(q_full, 0, abort_s);
      // S_j = Q K_j^T into score buffer j & 1 (8 MMAs of K = 16).
      auto issue_s = [&](int j) -> bool {
        const int st = j % C::NK;
        if (!mbar_wait_or_abort(&k_full[st], (j / C::NK) & 1, abort_s)) return false;
        tc::fence_after_sync();
        const uint32_t k_addr = sbase + C::OFF_K + st * C::KV_BYTES;
        const uint32_t d_tmem = tmem + ((j & 1) ? C::COL_S1 : C::COL_S0);
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
          const uint32_t koff = (kk >> 2) * (C::KV_BYTES / 2) + (kk & 3) * 32;
          tc::mma_bf16_ss(d_tmem, tc::smem_desc_sw128(q_addr + off, 16, 1024),
                          tc::smem_desc_sw128(k_addr + koff, 16, 1024), IDESC_S, kk > 0);
        }
        tc::commit(&k_empty[st]);
        tc::commit(&s_full[j & 1]);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && ntiles > 1) ok = issue_s(1);
      for (int j = 0; ok && j < ntiles; ++j) {
        // O += P_j V_j once the softmax warps have written P_j (and
        // rescaled O where needed).
        if (!mbar_wait_or_abort(p_full, j & 1, abort_s)) break;
        tc::fence_after_sync();
        const int st = j % C::NV;
        if (!mbar_wait_or_abort(&v_full[st], (j / C::NV) & 1, abort_s)) break;
        const uint32_t v_addr = sbase + C::OFF_V + st * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::TN / 16; ++kk) {
          // A = P: K-major, tokens 16kk..16kk+15; B = V: MN-major (head dim
          // contiguous), 16 token rows starting at 16kk, two 64-wide blocks
          // KV_BYTES/2 apart.
          const uint32_t poff = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
          tc::mma_bf16_ss(tmem + C::COL_O, tc::smem_desc_sw128(p_addr + poff, 16, 1024),
                          tc::smem_desc_sw128(v_addr + kk * 16 * 128, C::KV_BYTES / 2, 1024),
                          IDESC_O, (j > 0) || (kk > 0));
        }
        tc::commit(&v_empty[st]);
        tc::commit(o_done);
        if (j + 2 < ntiles) ok = issue_s(j + 2);
      }
      // Drain: every MMA issued above completes before the TMEM is freed.
      tc::commit(drain);
      mbar_wait_bounded(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;                    // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;               // row of the M-tile
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    unsigned char* P_s = smem + C::OFF_P;
    float m_run = kNegInf, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      // Waits are made warp-uniform before any .sync.aligned tcgen05 access.
      const bool got = mbar_wait_or_abort(&s_full[j & 1], (j >> 1) & 1, abort_s);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc::fence_after_sync();
      uint32_t sr[4][32];
      const uint32_t s_tmem = tmem + lane_base + ((j & 1) ? C::COL_S1 : C::COL_S0);
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld32(s_tmem + c * 32, sr[c]);
      tc::tmem_wait_ld();
      const int nvalid = min(C::TN, end - (begin + j * C::TN));
      float mx = kNegInf;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float v = __uint_as_float(sr[c][i]) * p.scale_log2;
          if (c * 32 + i >= nvalid) v = kNegInf;
          sr[c][i] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      const float m_new = (mx > m_run + 8.f) ? mx : m_run;
      const float alpha = (m_new == m_run) ? 1.f : fast_exp2(m_run - m_new);
      const float m_use = (m_new == kNegInf) ? 0.f : m_new;   // all -inf: p = 0, not NaN
      float rowsum = 0.f;
      uint32_t pk[4][16];                           // bf16 pairs of the row
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = fast_exp2(__uint_as_float(sr[c][2 * i]) - m_use);
          const float p1 = fast_exp2(__uint_as_float(sr[c][2 * i + 1]) - m_use);
          rowsum += p0 + p1;
          uint32_t w;
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(p1), "f"(p0));
          pk[c][i] = w;
        }
      // P_j may overwrite the P tile and O may be rescaled only once
      // O += P_{j-1} V_{j-1} has completed.
      if (j > 0) {
        const bool got_o = mbar_wait_or_abort(o_done, (j - 1) & 1, abort_s);
        if (!__all_sync(0xffffffffu, got_o)) { ok = false; break; }
        tc::fence_after_sync();
      }
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        const uint32_t o_tmem = tmem + lane_base + C::COL_O;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t orr[32];
          tc::tmem_ld32(o_tmem + c * 32, orr);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
          tc::tmem_st32(o_tmem + c * 32, orr);
        }
        tc::tmem_wait_st();
      }
      // P row r, tokens 64h..64h+63 in swizzled box h: 16-byte chunk c8
      // (tokens 8c8..8c8+7) at (c8 ^ (r & 7)) * 16.
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int chunk = c * 4 + q4;             // 16-byte chunk of the 256-byte row
          const int box = chunk >> 3;
          const int c8 = chunk & 7;
          uint4 val = make_uint4(pk[c][q4 * 4 + 0], pk[c][q4 * 4 + 1], pk[c][q4 * 4 + 2],
                                 pk[c][q4 * 4 + 3]);
          *reinterpret_cast<uint4*>(P_s + box * C::CHUNK_BYTES + r * 128 + ((c8 ^ (r & 7)) << 4)) = val;
        }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      mbar_arrive(p_full);
      l_run = l_run * alpha + rowsum;
      m_run = m_new;
    }
    // ------------------------------------------------------------ epilogue
    const bool got_last = ok && mbar_wait_or_abort(o_done, (ntiles - 1) & 1, abort_s);
    if (__all_sync(0xffffffffu, got_last)) {
      tc::fence_after_sync();
      const int m = mtile * C::M + r;
      const bool valid = m < p.rows;
      const int s = m / p.G;
      const int h = g * p.G + (m - s * p.G);
      const float inv_l = 1.f / l_run;
      float* o = p.o + (valid ? (s * p.o_sb + h * p.o_sh + split * p.o_ss) : 0);
      const uint32_t o_tmem = tmem + lane_base + C::COL_O;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t orr[32];
        tc::tmem_ld32(o_tmem + c * 32, orr);
        tc::tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(o + c * 32 + i) =
                make_float4(__uint_as_float(orr[i]) * inv_l, __uint_as_float(orr[i + 1]) * inv_l,
                            __uint_as_float(orr[i + 2]) * inv_l, __uint_as_float(orr[i + 3]) * inv_l);
        }
      }
      if (valid && p.lse) p.lse[s * p.l_sb + h * p.l_sh + split * p.l_ss] = (m_run + __log2f(l_run)) * kLn2;
    }
  }
  pdl_launch_dependents();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace fd
