// Bifurcated attention, context part, on the 5th-generation tensor cores.
//
// n samples share one context KV [Lc, Hkv, D].  For kv head g, the rows of
// the problem are all (sample s, query head r of group g) pairs, so the
// context part is a dense attention of M = n * G query rows against Lc keys:
//   S = Q_g K_ctx[g]^T          (GEMM 1, K-dim = D)
//   online softmax over the tokens of a split
//   O = P V_ctx[g]              (GEMM 2, K-dim = tokens)
// and the context KV is read once per 128-row query tile instead of once per
// sample.  Each CTA writes, for its rows and one token split of the
// context, the normalised partial output and its natural-log log-sum-exp, in
// the same partial format as the split kernel; the log-sum-exp reduction then
// merges them with the per-sample decode part.  Source: summary of
// "Bifurcated Attention for Single-Context Large-Batch Sampling" (linnk.ai),
// sections "Tiivistelmä" (two GEMMs, prefill KV and decode KV, exact result)
// and "Tilastot" (KV I/O b*g*m*k instead of b*h*m*k); online softmax after
// "How does Flash Attention reduce memory traffic during local inference?",
// section on online softmax.
//
// With 16 or more query heads per kv head, a 128-row query tile spans at
// most 9 samples, and the kernel also takes the decode part ("fold"): each
// decode tile (128 tokens of one sample's own cache, 4-D tensor map over
// [n, Ld, Hkv, D]) joins the tile's list of work with the scores of the
// other samples' rows masked to -inf, and the V rows past the sample's
// length zeroed in shared memory.  The list, context tiles then decode
// tiles, is cut into equal runs, one per split, so every CTA streams about
// the same number of tiles; the log-sum-exp reduction then needs no separate
// decode partial.
//
// CTA = one 128-row query tile x one context split x one kv head; 6 warps:
//   warp 0      TMA producer: K and V tiles of 128 tokens into separate
//               3-stage rings, 128-byte swizzle (two 64-column boxes per
//               tile).
//   warp 1      allocates 512 TMEM columns; one thread issues every MMA.
//               TMEM: Q (bf16 pairs, 64 columns at 0), two score buffers
//               S[0], S[1] (128 fp32 columns each, at 64 and 192) and the
//               output accumulator O (128 fp32 columns at 320).
//                 S[j % 2]  = Q K_j^T     A = Q from TMEM, B = K from shared
//                                         memory (K-major), N = 128 tokens
//                 O        += P_j V_j     A = P_j from TMEM, B = V from shared
//                                         memory (MN-major), N = 128 dims
//               P_j (bf16 pairs, 64 columns) overwrites the first half of the
//               score buffer it was computed from.  Every MMA is 128 x 128 x
//               16 and reads only its B tile from shared memory.
//   warps 2..5  softmax: thread = one row (its TMEM lane).  First each thread
//               loads its query row from global memory into Q; then, per
//               tile, it reads its row of S, keeps the running max m / sum l
//               in base 2, writes the bf16 probabilities back into TMEM, and
//               rescales O on the rare tiles where the running max grows by
//               more than 8 (lazy rescale; p <= 256 always; numerator and
//               denominator share m).
// The score buffers are double-buffered, so the tensor core computes
// S_{j+1} while the softmax warps work on S_j.  The MMAs of one thread
// execute in issue order: S_{j+2} is issued after O += P_j V_j and so never
// overwrites P_j before it is read.  A rescale of O before tile j first
// waits for O += P_{j-1} V_{j-1} (o_done).  The softmax warps may run one
// tile ahead of the MMA issuer, so "S ready" and "P ready" barriers exist
// per score buffer.
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
  static constexpr int MT = 128;                // rows per CTA (TMEM lanes)
  static constexpr int ROWS = MT;
  static constexpr int D = 128;                 // head dim
  static constexpr int TN = kBifTileTokens;     // tokens per K/V tile
  static constexpr int NK = 3;                  // K stages
  static constexpr int NV = 3;                  // V stages
  static constexpr int NSW = 4;                 // softmax warps
  static constexpr int THREADS = 64 + NSW * 32;
  static constexpr int KV_CHUNK = TN * 128;     // TN rows x 64 bf16 (one swizzled box)
  static constexpr int KV_BYTES = 2 * KV_CHUNK; // one K or V tile (two boxes)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NK * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + NV * KV_BYTES;
  // barriers: k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], q_ready,
  // s_full[2], p_full[2], o_done, o_final, drain
  static constexpr int NBAR = 2 * NK + 2 * NV + 1 + 2 + 2 + 3;
  static constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_Q = 0;          // 64 columns
  static constexpr uint32_t COL_S = 64;         // + 128 b
  static constexpr uint32_t COL_O = 320;        // 128 columns
  static_assert(TN == 128, "score buffers are laid out for 128-token tiles");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static constexpr int STAGE_BYTES = MT * (D + 4) * 4;        // padded O rows
  static_assert(STAGE_BYTES + MT * 8 <= OFF_BAR, "epilogue staging fits the K/V rings");
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
    bif_ctx_kernel(const __grid_constant__ BifCtxParams p, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmKd,
                   const __grid_constant__ CUtensorMap tmVd) {
  using C = BifCfg;
  pdl_wait_prerequisites();   // launched with PDL: no memory access before this
  // Every earlier grid has now finished: the decode part (which reads none of
  // this kernel's output) may start on the SMs this grid leaves free.
  pdl_launch_dependents();
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + C::NK;
  uint64_t* v_full = k_empty + C::NK;
  uint64_t* v_empty = v_full + C::NV;
  uint64_t* q_ready = v_empty + C::NV;
  uint64_t* s_full = q_ready + 1;               // [2]
  uint64_t* p_full = s_full + 2;                // [2]
  uint64_t* o_done = p_full + 2;
  uint64_t* o_final = o_done + 1;
  uint64_t* drain = o_final + 1;
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_s = reinterpret_cast<int*>(taddr_s + 1);

  const int mtile = blockIdx.x;                 // 128-row query tile
  const int split = blockIdx.y;
  const int g = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Without the fold: context tiles [begin, end) of this split.  With it:
  // the query tile's work is the list of the nct context tiles followed by
  // the decode tiles of its samples s_first .. s_first + nsamp - 1 (sample
  // after sample, dlen[k] tokens each), and this split takes the run
  // [t0, t0 + ntiles) of that list.
  const bool fold = p.fold != 0;
  const int nct = (p.Lc + C::TN - 1) / C::TN;
  int begin = 0, end = 0, ntiles = 0, t0 = 0, s_first = 0, nsamp = 0;
  int dlen[kBifFoldMaxSamples];
#pragma unroll
  for (int k = 0; k < kBifFoldMaxSamples; ++k) dlen[k] = 0;
  if (!fold) {
    bif_split_range(p.Lc, p.ns, split, begin, end);
    ntiles = (end - begin + C::TN - 1) / C::TN;
  } else {
    const int m0 = mtile * C::MT;
    s_first = m0 / p.G;
    nsamp = (min(m0 + C::MT, p.rows) - 1) / p.G - s_first + 1;
    int total = nct;
#pragma unroll
    for (int k = 0; k < kBifFoldMaxSamples; ++k)
      if (k < nsamp) {
        dlen[k] = resolve_len(p.dec_lens, s_first + k, p.Ld);
        total += (dlen[k] + C::TN - 1) / C::TN;
      }
    const int per = (total + p.ns - 1) / p.ns;
    t0 = min(split * per, total);
    ntiles = min(t0 + per, total) - t0;
  }
  // Tile j (< ntiles) of this CTA -> whether it is a decode tile, its sample
  // index k within the query tile (decode tiles), its first token (in the
  // context, or in sample k's decode cache) and its valid tokens.  Unrolled
  // so dlen stays in registers.
  auto tile_of = [&](int j, bool& is_dec, int& k_out, int& tok, int& nv) {
    if (!fold) {
      is_dec = false;
      k_out = 0;
      tok = begin + j * C::TN;
      nv = min(C::TN, end - tok);
      return;
    }
    int f = t0 + j;
    if (f < nct) {
      is_dec = false;
      k_out = 0;
      tok = f * C::TN;
      nv = min(C::TN, p.Lc - tok);
      return;
    }
    f -= nct;
    int kk = 0, len = 0;
    bool found = false;
#pragma unroll
    for (int k = 0; k < kBifFoldMaxSamples; ++k) {
      const int nt = (dlen[k] + C::TN - 1) / C::TN;
      if (!found && k < nsamp) {
        if (f < nt) {
          kk = k;
          len = dlen[k];
          found = true;
        } else {
          f -= nt;
        }
      }
    }
    is_dec = true;
    k_out = kk;
    tok = f * C::TN;
    nv = min(C::TN, len - tok);
  };

  if (ntiles == 0 && p.cs == 1) {
    // Empty split: O = 0, lse = -inf for every valid row.  (In a cluster an
    // empty split still runs through, stages (m, l) = (-inf, 0) and joins the
    // cluster barriers.)
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
      const bool is_p = (&bars[i] >= p_full) && (&bars[i] < p_full + 2);
      mbar_init(&bars[i], (is_q || is_p) ? C::NSW * 32 : 1);
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
      if (fold) {
        prefetch_tensormap(&tmKd);
        prefetch_tensormap(&tmVd);
      }
      const uint64_t policy = l2_policy_evict_first();
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
          bool is_dec;
          int k, tok, nv;
          tile_of(kt, is_dec, k, tok, nv);
          if (is_dec) {
            tma_load_4d(dst, &tmKd, &k_full[st], 0, g, tok, s_first + k, policy);
            tma_load_4d(dst + C::KV_CHUNK, &tmKd, &k_full[st], 64, g, tok, s_first + k, policy);
          } else {
            tma_load_3d(dst, &tmK, &k_full[st], 0, g, tok);
            tma_load_3d(dst + C::KV_CHUNK, &tmK, &k_full[st], 64, g, tok);
          }
          ++kt;
        }
        if (vt < ntiles && vt < kt) {
          const int st = vt % C::NV;
          if (vt >= C::NV) ok = mbar_wait_or_abort(&v_empty[st], ((vt / C::NV) - 1) & 1, abort_s);
          if (!ok) break;
          unsigned char* dst = smem + C::OFF_V + st * C::KV_BYTES;
          mbar_arrive_expect_tx(&v_full[st], C::KV_BYTES);
          bool is_dec;
          int k, tok, nv;
          tile_of(vt, is_dec, k, tok, nv);
          if (is_dec) {
            tma_load_4d(dst, &tmVd, &v_full[st], 0, g, tok, s_first + k, policy);
            tma_load_4d(dst + C::KV_CHUNK, &tmVd, &v_full[st], 64, g, tok, s_first + k, policy);
          } else {
            tma_load_3d(dst, &tmV, &v_full[st], 0, g, tok);
            tma_load_3d(dst + C::KV_CHUNK, &tmV, &v_full[st], 64, g, tok);
          }
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
      // S[j % 2] = Q K_j^T (8 MMAs of K = 16 head dims; Q columns 8 kk).
      auto issue_s = [&](int j) {
        const uint32_t k_addr = sbase + C::OFF_K + (j % C::NK) * C::KV_BYTES;
        const uint32_t d_tmem = tmem + C::COL_S + (j & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
          tc::mma_bf16_ts(d_tmem, tmem + C::COL_Q + kk * 8,
                          tc::smem_desc_sw128(k_addr + koff, 16, 1024), IDESC_S, kk > 0);
        }
        tc::commit(&s_full[j & 1]);
      };
      // O += P_j V_j (8 MMAs of K = 16 tokens; P_j from the first 64 columns
      // of S[j % 2], 8 per MMA; V MN-major: 16 token rows at 16 kk, two
      // 64-wide head-dim blocks KV_CHUNK apart).
      auto issue_pv = [&](int j) {
        const uint32_t v_addr = sbase + C::OFF_V + (j % C::NV) * C::KV_BYTES;
        const uint32_t a_tmem = tmem + C::COL_S + (j & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < C::TN / 16; ++kk)
          tc::mma_bf16_ts(tmem + C::COL_O, a_tmem + kk * 8,
                          tc::smem_desc_sw128(v_addr + kk * 16 * 128, C::KV_CHUNK, 1024),
                          IDESC_O, (j > 0) || (kk > 0));
        tc::commit(o_done);
      };
      bool ok = mbar_wait_or_abort(q_ready, 0, abort_s);
      // Prologue: scores of tiles 0 and 1.
      for (int j = 0; ok && j < 2 && j < ntiles; ++j) {
        if (!mbar_wait_or_abort(&k_full[j % C::NK], (j / C::NK) & 1, abort_s)) { ok = false; break; }
        tc::fence_after_sync();
        issue_s(j);
        tc::commit(&k_empty[j % C::NK]);
      }
      for (int j = 0; ok && j < ntiles; ++j) {
        if (!mbar_wait_or_abort(&v_full[j % C::NV], (j / C::NV) & 1, abort_s)) break;
        if (!mbar_wait_or_abort(&p_full[j & 1], (j >> 1) & 1, abort_s)) break;
        tc::fence_after_sync();
        issue_pv(j);
        tc::commit(&v_empty[j % C::NV]);
        if (j + 2 < ntiles) {
          if (!mbar_wait_or_abort(&k_full[(j + 2) % C::NK], ((j + 2) / C::NK) & 1, abort_s)) break;
          issue_s(j + 2);
          tc::commit(&k_empty[(j + 2) % C::NK]);
        }
      }
      tc::commit(o_final);
      // Drain: every MMA issued above completes before the TMEM is freed.
      tc::commit(drain);
      mbar_wait_bounded(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;                    // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;               // row of the query tile
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t q_tmem = tmem + lane_base + C::COL_Q;
    const uint32_t o_tmem = tmem + lane_base + C::COL_O;
    const int m0 = mtile * C::MT;                 // first row of this tile
    const int row_s = (m0 + r) / p.G;             // sample of this row
    {
      // Query row -> Q (bf16 pairs, dim 2c in the low half of column c).
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
      const uint32_t s_tmem = tmem + lane_base + C::COL_S + (j & 1) * 128;
      // Waits are made warp-uniform before any .sync.aligned tcgen05 access.
      const bool got = mbar_wait_or_abort(&s_full[j & 1], (j >> 1) & 1, abort_s);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc::fence_after_sync();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld32(s_tmem + c * 32, sr[c]);
      tc::tmem_wait_ld();
      // Context tile: the context's tail; decode tile: its sample's tail,
      // and nothing at all for rows of the tile's other samples.
      bool is_dec;
      int ks, tok, tile_valid;
      tile_of(j, is_dec, ks, tok, tile_valid);
      const int nvalid = (!is_dec || row_s == s_first + ks) ? tile_valid : 0;
      if (nvalid < C::TN) {                        // tail tiles (and other samples' decode tiles)
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c * 32 + i >= nvalid) sr[c][i] = __float_as_uint(kNegInf);
      }
      // Row maximum with 8 independent chains.
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = kNegInf;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sr[c][i]));
#pragma unroll
      for (int k = 1; k < 8; ++k) mx8[0] = fmaxf(mx8[0], mx8[k]);
      const float mx = mx8[0] * c2;                 // -inf stays -inf (c2 > 0)
      const float m_new = (mx > m_run + 8.f) ? mx : m_run;
      const float alpha = (m_new == m_run) ? 1.f : fast_exp2(m_run - m_new);
      const float m_use = (m_new == kNegInf) ? 0.f : m_new;   // all -inf: p = 0, not NaN
      // p = 2^(s * c2 - m); P_j as bf16 pairs (even token in the low half)
      // packed in place and stored into the first 64 columns of the buffer.
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
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
      // Rescale O where its max moved (rare), once O += P_{j-1} V_{j-1} is
      // done: o_done has then completed phases 0..j-1 (phase j needs P_j).
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        const bool got_o = mbar_wait_or_abort(o_done, (j - 1) & 1, abort_s);
        if (!__all_sync(0xffffffffu, got_o)) { ok = false; break; }
        tc::fence_after_sync();
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
      if (is_dec && tile_valid < C::TN) {
        // V rows past the sample's length hold whatever the cache holds
        // there: zero them before O += P V reads the tile (P is 0 on those
        // rows, but 0 times a non-finite value is not 0).
        const bool got_v = mbar_wait_or_abort(&v_full[j % C::NV], (j / C::NV) & 1, abort_s);
        if (!__all_sync(0xffffffffu, got_v)) { ok = false; break; }
        if (r >= tile_valid) {
          unsigned char* vrow = smem + C::OFF_V + (j % C::NV) * C::KV_BYTES + r * 128;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            reinterpret_cast<uint4*>(vrow)[i] = make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4*>(vrow + C::KV_CHUNK)[i] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        tc::fence_proxy_async_smem();
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      mbar_arrive(&p_full[j & 1]);
      l_run = l_run * alpha + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
      m_run = m_new;
    }
    // ------------------------------------------------------------ epilogue
    // o_final is committed after the last MMA of the CTA: once it fires the
    // K/V rings are dead.  Each row owner normalises its O row into a padded
    // staging tile there, then each warp writes whole rows (512 contiguous
    // bytes per store instruction) instead of 32 rows at once.
    const bool got_last = ok && mbar_wait_or_abort(o_final, 0, abort_s);
    const bool done = __all_sync(0xffffffffu, got_last);
    constexpr int SROW = C::D + 4;                            // padded row (floats)
    float* stage = reinterpret_cast<float*>(smem);
    float2* ml_stage = reinterpret_cast<float2*>(smem + C::STAGE_BYTES);
    if (done) {
      tc::fence_after_sync();
      const int m = m0 + r;
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;   // a decode row may see no token
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
      if (p.cs > 1) {
        // Clustered: keep (m, l) of the row for the cluster reduction below.
        ml_stage[r] = make_float2(m_run, l_run);
      } else if (m < p.rows && p.lse) {
        const int s = m / p.G;
        const int h = g * p.G + (m - s * p.G);
        p.lse[s * p.l_sb + h * p.l_sh + split * p.l_ss] = (m_run + __log2f(l_run)) * kLn2;
      }
    } else if (p.cs > 1) {
      ml_stage[r] = make_float2(kNegInf, 0.f);    // aborted: contributes nothing
    }
    if (done && p.cs == 1) {
      // Each thread hands its own staged row to the bulk-copy engine (one
      // 512-byte copy), after making its shared-memory writes visible to
      // the async proxy, and waits for the copy before the CTA can exit.
      const int m = m0 + r;
      tc::fence_proxy_async_smem();
      if (m < p.rows) {
        const int s = m / p.G;
        const int h = g * p.G + (m - s * p.G);
        bulk_store(p.o + s * p.o_sb + h * p.o_sh + split * p.o_ss, stage + r * SROW, C::D * 4);
        bulk_store_commit_and_wait();
      }
    }
  }
  pdl_launch_dependents();
  tc::fence_before_sync();
  __syncthreads();
  if (p.cs > 1) {
    // Cluster reduction over the cs splits of this query tile (the cluster
    // spans consecutive splits of one tile and kv head): every CTA has its
    // normalised O rows and (m, l) staged in shared memory; CTA `rank`
    // merges rows [rank * 128 / cs, (rank + 1) * 128 / cs) of all of them
    // through distributed shared memory and writes one partial per row,
    // partial slot split / cs:
    //   M = max_k m_k,  w_k = l_k 2^(m_k - M),  O = sum_k w_k O_k / sum_k w_k
    //   lse = (M + log2 sum_k w_k) ln 2.
    // One warp per row; lane = 4 head-dim elements.
    cluster_sync_all();
    const uint32_t rank = cluster_ctarank();
    const int rows_per = C::MT / p.cs;
    const uint32_t stage_addr = smem_u32(smem);
    const uint32_t ml_addr = smem_u32(smem + C::STAGE_BYTES);
    for (int rr = warp; rr < rows_per; rr += C::THREADS / 32) {
      const int row = (int)rank * rows_per + rr;
      const int m = mtile * C::MT + row;
      if (m >= p.rows) break;
      float mk[8], lk[8];
      float M = kNegInf;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k < p.cs) {
          const float2 v = dsmem_ld_f2(dsmem_map(ml_addr + row * 8, (uint32_t)k));
          mk[k] = v.x;
          lk[k] = v.y;
          M = fmaxf(M, v.x);
        } else {
          mk[k] = kNegInf;
          lk[k] = 0.f;
        }
      }
      float L = 0.f;
      float wk[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        wk[k] = (mk[k] == kNegInf) ? 0.f : lk[k] * fast_exp2(mk[k] - M);
        L += wk[k];
      }
      const float invL = L > 0.f ? 1.f / L : 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k < p.cs && wk[k] != 0.f) {
          const float4 v =
              dsmem_ld_f4(dsmem_map(stage_addr + (row * (C::D + 4) + lane * 4) * 4, (uint32_t)k));
          const float w = wk[k] * invL;
          acc.x = fmaf(w, v.x, acc.x);
          acc.y = fmaf(w, v.y, acc.y);
          acc.z = fmaf(w, v.z, acc.z);
          acc.w = fmaf(w, v.w, acc.w);
        }
      }
      const int s = m / p.G;
      const int h = g * p.G + (m - s * p.G);
      const int slot = split / p.cs;
      *reinterpret_cast<float4*>(p.o + s * p.o_sb + h * p.o_sh + slot * p.o_ss + lane * 4) = acc;
      if (lane == 0 && p.lse)
        p.lse[s * p.l_sb + h * p.l_sh + slot * p.l_ss] = L > 0.f ? (M + __log2f(L)) * kLn2 : kNegInf;
    }
    // No CTA leaves (and frees its shared memory) while a peer still reads it.
    cluster_sync_all();
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace fd
