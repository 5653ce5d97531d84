// Bifurcated attention, context part, on the 5th-generation tensor cores.
//
// n samples share one context KV [Lc, Hkv, D].  For kv head g, the rows of
// the problem are all (sample s, query head r of group g) pairs, so the
// context part is a dense attention of M = n * G query rows against Lc keys:
//   S = Q_g K_ctx[g]^T          (GEMM 1, K-dim = D)
//   online softmax over the tokens of a split
//   O = P V_ctx[g]              (GEMM 2, K-dim = tokens)
// and the context KV is read once per pair of 128-row query tiles instead of
// once per sample.  Each CTA writes, for its rows and one token split of the
// context, the normalised partial output and its natural-log log-sum-exp, in
// the same partial format as the split kernel; the log-sum-exp reduction then
// merges them with the per-sample decode part.  Source: summary of
// "Bifurcated Attention for Single-Context Large-Batch Sampling" (linnk.ai),
// sections "Tiivistelmä" (two GEMMs, prefill KV and decode KV, exact result)
// and "Tilastot" (KV I/O b*g*m*k instead of b*h*m*k); online softmax after
// "How does Flash Attention reduce memory traffic during local inference?",
// section on online softmax.
//
// CTA = two 128-row query tiles (256 rows) x one context split x one kv head;
// 10 warps:
//   warp 0      TMA producer: K and V tiles of 64 tokens into separate
//               5-stage rings, 128-byte swizzle (two 64-column boxes per
//               tile).  Every K/V tile feeds both query tiles.
//   warp 1      allocates all 512 TMEM columns; one thread issues every MMA.
//               TMEM per query tile t: Q_t (bf16 pairs, 64 columns at 64 t),
//               S_t (64 fp32 columns at 128 + 64 t), O_t (128 fp32 columns
//               at 256 + 128 t).
//                 S_t  = Q_t K_j^T     A = Q_t from TMEM, B = K from shared
//                                      memory (K-major)
//                 O_t += P_t V_j       A = P_t from TMEM, B = V from shared
//                                      memory (MN-major)
//               P_t (bf16 pairs, 32 columns) overwrites the first half of
//               S_t.  With both A operands in tensor memory each MMA reads
//               only its B tile from shared memory.
//   warps 2..5  query tile 0, warps 6..9 query tile 1; thread = one row (its
//               TMEM lane).  First each thread loads its query row from
//               global memory into Q_t; then, per tile, it reads its row of
//               S_t, keeps the running max m / sum l in base 2, writes the
//               bf16 probabilities back into TMEM, and rescales O_t on the
//               rare tiles where the running max grows by more than 8 (lazy
//               rescale; p <= 256 always; numerator and denominator share m).
// The two query tiles ping-pong on the tensor core: while one warpgroup runs
// its softmax, the tensor core runs the other tile's P V and next Q K^T.
// Ordering needs no extra waits: the MMAs of one thread execute in issue
// order, and the barrier that signals "S_t of tile j is ready" is committed
// after O_t += P_t V_{j-1}, so when a softmax warp sees S_t it may also
// rescale O_t and overwrite P_t.
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
  static constexpr int MT = 128;                // rows per query tile (TMEM lanes)
  static constexpr int NQ = kBifQueryTiles;     // query tiles per CTA
  static constexpr int ROWS = MT * NQ;          // rows per CTA
  static constexpr int D = 128;                 // head dim
  static constexpr int TN = kBifTileTokens;     // tokens per K/V tile
  static constexpr int NK = 5;                  // K stages
  static constexpr int NV = 5;                  // V stages
  static constexpr int NSW = 4 * NQ;            // softmax warps
  static constexpr int THREADS = 64 + NSW * 32;
  static constexpr int KV_CHUNK = TN * 128;     // TN rows x 64 bf16 (one swizzled box)
  static constexpr int KV_BYTES = 2 * KV_CHUNK; // one K or V tile (two boxes)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NK * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + NV * KV_BYTES;
  // barriers: k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], q_ready,
  // s_full[NQ], p_full[NQ], o_done, drain
  static constexpr int NBAR = 2 * NK + 2 * NV + 1 + 2 * NQ + 2;
  static constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_Q = 0;          // + 64 t
  static constexpr uint32_t COL_S = 128;        // + 64 t
  static constexpr uint32_t COL_O = 256;        // + 128 t
  static_assert(TN == 64, "score columns are laid out for 64-token tiles");
  static_assert(NQ == 2, "TMEM holds two query tiles");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(NQ * MT * (D + 4) * 4 <= OFF_BAR, "epilogue staging fits the K/V rings");
};

// Context split i of ns over [0, Lc): whole 64-token tiles.
__device__ __forceinline__ void bif_split_range(int Lc, int ns, int i, int& begin, int& end) {
  const int per = (Lc + ns - 1) / ns;
  const long long chunk = (long long)((per + BifCfg::TN - 1) / BifCfg::TN) * BifCfg::TN;
  const long long b0 = (long long)i * chunk;
  begin = (int)(b0 < Lc ? b0 : Lc);
  end = (int)(b0 + chunk < Lc ? b0 + chunk : Lc);
}

__global__ void __launch_bounds__(BifCfg::THREADS, 1)
    bif_ctx_kernel(const __grid_constant__ BifCtxParams p, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV) {
  using C = BifCfg;
  pdl_wait_prerequisites();   // launched with PDL: no memory access before this
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + C::NK;
  uint64_t* v_full = k_empty + C::NK;
  uint64_t* v_empty = v_full + C::NV;
  uint64_t* q_ready = v_empty + C::NV;
  uint64_t* s_full = q_ready + 1;               // [NQ]
  uint64_t* p_full = s_full + C::NQ;            // [NQ]
  uint64_t* o_done = p_full + C::NQ;
  uint64_t* drain = o_done + 1;
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_s = reinterpret_cast<int*>(taddr_s + 1);

  const int mtile = blockIdx.x;                 // pair of 128-row query tiles
  const int split = blockIdx.y;
  const int g = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int begin, end;
  bif_split_range(p.Lc, p.ns, split, begin, end);
  const int ntiles = (end - begin + C::TN - 1) / C::TN;

  if (ntiles == 0) {
    // Empty split: O = 0, lse = -inf for every valid row.
    for (int rr = threadIdx.x; rr < C::ROWS; rr += C::THREADS) {
      const int m = mtile * C::ROWS + rr;
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
    for (int i = 0; i < C::NBAR; ++i) {
      const bool is_q = &bars[i] == q_ready;
      const bool is_p = (&bars[i] >= p_full) && (&bars[i] < p_full + C::NQ);
      mbar_init(&bars[i], is_q ? C::NSW * 32 : (is_p ? 128 : 1));
    }
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
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      int kt = 0, vt = 0;                           // next K / V tile to issue
      bool ok = true;
      while (ok && (kt < ntiles || vt < ntiles)) {
        // K runs up to NK tiles ahead of V; V follows.
        if (kt < ntiles && kt < vt + C::NK) {
          const int st = kt % C::NK;
          if (kt >= C::NK) ok = mbar_wait_or_abort(&k_empty[st], ((kt / C::NK) - 1) & 1, abort_s);
          if (!ok) break;
          unsigned char* dst = smem + C::OFF_K + st * C::KV_BYTES;
          mbar_arrive_expect_tx(&k_full[st], C::KV_BYTES);
          const int tok = begin + kt * C::TN;
          tma_load_3d(dst, &tmK, &k_full[st], 0, g, tok);
          tma_load_3d(dst + C::KV_CHUNK, &tmK, &k_full[st], 64, g, tok);
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
          tma_load_3d(dst + C::KV_CHUNK, &tmV, &v_full[st], 64, g, tok);
          ++vt;
        }
      }
      // Never leave with copies in flight: wait for the last load of every
      // stage (earlier loads of a stage completed before it was refilled).
      for (int t = (kt > C::NK ? kt - C::NK : 0); t < kt; ++t)
        mbar_wait_bounded(&k_full[t % C::NK], (t / C::NK) & 1);
      for (int t = (vt > C::NV ? vt - C::NV : 0); t < vt; ++t)
        mbar_wait_bounded(&v_full[t % C::NV], (t / C::NV) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = tc::idesc_bf16_f32(C::MT, C::TN, false, false);
      constexpr uint32_t IDESC_O = tc::idesc_bf16_f32(C::MT, C::D, false, true);
      // S_t = Q_t K_j^T (8 MMAs of K = 16 head dims; Q_t columns 8 kk).
      auto issue_s = [&](int t, int j) {
        const uint32_t k_addr = sbase + C::OFF_K + (j % C::NK) * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
          tc::mma_bf16_ts(tmem + C::COL_S + t * 64, tmem + C::COL_Q + t * 64 + kk * 8,
                          tc::smem_desc_sw128(k_addr + koff, 16, 1024), IDESC_S, kk > 0);
        }
        tc::commit(&s_full[t]);
      };
      // O_t += P_t V_j (4 MMAs of K = 16 tokens; P_t from the first 32
      // columns of S_t, 8 per MMA; V MN-major: 16 token rows at 16 kk, two
      // 64-wide head-dim blocks KV_CHUNK apart).
      auto issue_pv = [&](int t, int j) {
        const uint32_t v_addr = sbase + C::OFF_V + (j % C::NV) * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::TN / 16; ++kk)
          tc::mma_bf16_ts(tmem + C::COL_O + t * 128, tmem + C::COL_S + t * 64 + kk * 8,
                          tc::smem_desc_sw128(v_addr + kk * 16 * 128, C::KV_CHUNK, 1024),
                          IDESC_O, (j > 0) || (kk > 0));
      };
      bool ok = mbar_wait_or_abort(q_ready, 0, abort_s);
      if (ok) ok = mbar_wait_or_abort(&k_full[0], 0, abort_s);
      if (ok) {
        tc::fence_after_sync();
        issue_s(0, 0);
        issue_s(1, 0);
        tc::commit(&k_empty[0]);
      }
      for (int j = 0; ok && j < ntiles; ++j) {
        const bool more = j + 1 < ntiles;
        if (!mbar_wait_or_abort(&v_full[j % C::NV], (j / C::NV) & 1, abort_s)) break;
        // query tile 0: O_0 += P_0 V_j, then S_0 of tile j+1
        if (!mbar_wait_or_abort(&p_full[0], j & 1, abort_s)) break;
        tc::fence_after_sync();
        issue_pv(0, j);
        if (more) {
          if (!mbar_wait_or_abort(&k_full[(j + 1) % C::NK], ((j + 1) / C::NK) & 1, abort_s)) break;
          issue_s(0, j + 1);
        }
        // query tile 1: O_1 += P_1 V_j, then S_1 of tile j+1
        if (!mbar_wait_or_abort(&p_full[1], j & 1, abort_s)) break;
        tc::fence_after_sync();
        issue_pv(1, j);
        tc::commit(&v_empty[j % C::NV]);
        if (more) {
          issue_s(1, j + 1);
          tc::commit(&k_empty[(j + 1) % C::NK]);
        }
      }
      tc::commit(o_done);
      // Drain: every MMA issued above completes before the TMEM is freed.
      tc::commit(drain);
      mbar_wait_bounded(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 2) >> 2;                // query tile of this warpgroup
    const int quad = warp & 3;                    // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;               // row of the query tile
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t q_tmem = tmem + lane_base + C::COL_Q + t * 64;
    const uint32_t s_tmem = tmem + lane_base + C::COL_S + t * 64;
    const uint32_t o_tmem = tmem + lane_base + C::COL_O + t * 128;
    const int m0 = (mtile * C::NQ + t) * C::MT;   // first row of this tile
    {
      // Query row -> Q_t (bf16 pairs, dim 2c in the low half of column c).
      // Rows past n * G load zeros.  A negative scale is folded in here (the
      // sign bits flip), so the softmax below always scales by |scale|.
      uint32_t qv[2][32];
      const int m = m0 + r;
      if (m < p.rows) {
        const int s = m / p.G;
        const int h = g * p.G + (m - s * p.G);
        const uint4* src = reinterpret_cast<const uint4*>(p.q + s * p.q_sb + h * p.q_sh);
        const uint32_t flip = p.negate_q ? 0x80008000u : 0u;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint4 w = src[i];
          qv[i >> 3][(i & 7) * 4 + 0] = w.x ^ flip;
          qv[i >> 3][(i & 7) * 4 + 1] = w.y ^ flip;
          qv[i >> 3][(i & 7) * 4 + 2] = w.z ^ flip;
          qv[i >> 3][(i & 7) * 4 + 3] = w.w ^ flip;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) qv[0][i] = qv[1][i] = 0u;
      }
      tc::tmem_st32(q_tmem, qv[0]);
      tc::tmem_st32(q_tmem + 32, qv[1]);
      tc::tmem_wait_st();
      tc::fence_before_sync();
      mbar_arrive(q_ready);
    }
    float m_run = kNegInf, l_run = 0.f;
    bool ok = true;
    const float c2 = p.scale_log2;                 // |scale| * log2(e) >= 0
    for (int j = 0; j < ntiles; ++j) {
      // Waits are made warp-uniform before any .sync.aligned tcgen05 access.
      const bool got = mbar_wait_or_abort(&s_full[t], j & 1, abort_s);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc::fence_after_sync();
      uint32_t sr[2][32];
      tc::tmem_ld32(s_tmem, sr[0]);
      tc::tmem_ld32(s_tmem + 32, sr[1]);
      tc::tmem_wait_ld();
      const int nvalid = min(C::TN, end - (begin + j * C::TN));
      if (nvalid < C::TN) {                        // tail tile only (uniform branch)
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c * 32 + i >= nvalid) sr[c][i] = __float_as_uint(kNegInf);
      }
      // Row maximum with 8 independent chains.
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = kNegInf;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sr[c][i]));
#pragma unroll
      for (int k = 1; k < 8; ++k) mx8[0] = fmaxf(mx8[0], mx8[k]);
      const float mx = mx8[0] * c2;                 // -inf stays -inf (c2 > 0)
      const float m_new = (mx > m_run + 8.f) ? mx : m_run;
      const float alpha = (m_new == m_run) ? 1.f : fast_exp2(m_run - m_new);
      const float m_use = (m_new == kNegInf) ? 0.f : m_new;   // all -inf: p = 0, not NaN
      // p = 2^(s * c2 - m); P_t as bf16 pairs (even token in the low half)
      // packed in place and stored into the first 32 columns of S_t.
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(sr[c][2 * i]), c2, -m_use));
          const float p1 = fast_exp2(fmaf(__uint_as_float(sr[c][2 * i + 1]), c2, -m_use));
          sum4[i & 3] += p0 + p1;
          uint32_t w;
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(p1), "f"(p0));
          sr[c][i] = w;
        }
        tc::tmem_st16(s_tmem + c * 16, sr[c]);
      }
      // O_t += P_t V_{j-1} is complete (it was issued before S_t of tile j):
      // rescale O_t where its max moved (rare).
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t orr[32];
          tc::tmem_ld32(o_tmem + c * 32, orr);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
          tc::tmem_st32(o_tmem + c * 32, orr);
          tc::tmem_wait_st();
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      mbar_arrive(&p_full[t]);
      l_run = l_run * alpha + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
      m_run = m_new;
    }
    // ------------------------------------------------------------ epilogue
    // o_done is committed after the last MMA of the CTA: once it fires the
    // K/V rings are dead.  Each row owner normalises its O row into a padded
    // staging tile there, then each warp writes whole rows (512 contiguous
    // bytes per store instruction) instead of 32 rows at once.
    const bool got_last = ok && mbar_wait_or_abort(o_done, 0, abort_s);
    const bool done = __all_sync(0xffffffffu, got_last);
    constexpr int SROW = C::D + 4;                            // padded row (floats)
    float* stage = reinterpret_cast<float*>(smem) + t * (C::MT * SROW);
    if (done) {
      tc::fence_after_sync();
      const int m = m0 + r;
      const float inv_l = 1.f / l_run;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t orr[32];
        tc::tmem_ld32(o_tmem + c * 32, orr);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(stage + r * SROW + c * 32 + i) =
              make_float4(__uint_as_float(orr[i]) * inv_l, __uint_as_float(orr[i + 1]) * inv_l,
                          __uint_as_float(orr[i + 2]) * inv_l, __uint_as_float(orr[i + 3]) * inv_l);
      }
      if (m < p.rows && p.lse) {
        const int s = m / p.G;
        const int h = g * p.G + (m - s * p.G);
        p.lse[s * p.l_sb + h * p.l_sh + split * p.l_ss] = (m_run + __log2f(l_run)) * kLn2;
      }
    }
    // The four warps of this query tile: named barrier 1 + t, 128 threads.
    named_barrier_sync(1 + t, 128);
    if (done) {
      for (int rr = quad; rr < C::MT; rr += 4) {
        const int m = m0 + rr;
        if (m >= p.rows) break;
        const int s = m / p.G;
        const int h = g * p.G + (m - s * p.G);
        float* o = p.o + s * p.o_sb + h * p.o_sh + split * p.o_ss;
        *reinterpret_cast<float4*>(o + lane * 4) =
            *reinterpret_cast<const float4*>(stage + rr * SROW + lane * 4);
      }
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
