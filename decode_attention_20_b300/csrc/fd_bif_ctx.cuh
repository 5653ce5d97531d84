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
// CTA = one 128-row query tile x one context split x one kv head; 10 warps:
//   warp 0      TMA producer (the whole warp runs the loop, one elected lane
//               issues): the query tile (where its tensor map applies), then
//               K and V tiles of 128 tokens into separate 3-stage rings,
//               128-byte swizzle (two 64-column boxes per tile).
//   warp 1      allocates 512 TMEM columns and issues every MMA (whole warp,
//               one elected lane per MMA: warp-uniform operands keep the
//               issue well ahead of the tensor core).  TMEM: Q (bf16 pairs,
//               64 columns at 0), two score buffers S[0], S[1] (128 fp32
//               columns each, at 64 and 192) and the output accumulator O
//               (128 fp32 columns at 320).
//                 S[j % 2]  = Q K_j^T     A = Q from TMEM, B = K from shared
//                                         memory (K-major), N = 128 tokens
//                 O        += P_j V_j     A = P_j from TMEM, B = V from shared
//                                         memory (MN-major), N = 128 dims
//               P_j (bf16 pairs, 64 columns) overwrites the first half of the
//               score buffer it was computed from.  Every MMA is 128 x 128 x
//               16 and reads only its B tile from shared memory.
//   warps 2..9  softmax: two warps per TMEM lane quadrant; a thread owns one
//               row (its TMEM lane) and one half of the 128 columns.  Per
//               tile it reads its 64 scores, the two halves of a row trade
//               their maxima through shared memory, each keeps the running
//               max m / its part of the sum l in base 2, writes its 64 bf16
//               probabilities back into TMEM, and rescales its half of O on
//               the rare tiles where the running max grows by more than 8
//               (lazy rescale; p <= 256 always; numerator and denominator
//               share m).  Two warps per scheduler hide each other's TMEM
//               and exp latencies.
// The score buffers are double-buffered, so the tensor core computes
// S_{j+1} while the softmax warps work on S_j.  The MMAs of one thread
// execute in issue order: S_{j+2} is issued after O += P_j V_j and so never
// overwrites P_j before it is read.  A rescale of O before tile j first
// waits for O += P_{j-1} V_{j-1} (o_done).  The softmax warps may run one
// tile ahead of the MMA issuer, so "S ready" and "P ready" barriers exist
// per score buffer.
// Epilogue: each thread normalises its half row of O into a 128-byte
// swizzled staging tile (four boxes of 32 fp32 columns, bank-conflict free
// writes), and four TMA tensor stores write the 128 partial rows.
// Every wait is bounded; on a timeout the CTA drains its copies and MMAs,
// frees its tensor memory and returns with the device error flag set.  The
// softmax warps of a quadrant meet at a named barrier once per tile whatever
// happened, so a wait that gave up never leaves its partner warp blocked.
#pragma once

#include "fd_split.cuh"
#include "fd_tcgen05.cuh"

namespace fd {

// 5-D tiled tensor store shared -> global, tracked in this thread's bulk
// group; rows outside the tensor are not written.
__device__ __forceinline__ void tma_store_5d(const CUtensorMap* map, const void* smem_src, int c0,
                                             int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

struct BifCfg {
  static constexpr int MT = 128;                // rows per CTA (TMEM lanes)
  static constexpr int ROWS = MT;
  static constexpr int D = 128;                 // head dim
  static constexpr int TN = kBifTileTokens;     // tokens per K/V tile
  static constexpr int NK = 3;                  // K stages
  static constexpr int NV = 3;                  // V stages
  static constexpr int NSW = 8;                 // softmax warps (two per TMEM quadrant)
  static constexpr int HALF = TN / 2;           // score columns per softmax thread
  static constexpr int THREADS = 64 + NSW * 32;
  static constexpr int KV_CHUNK = TN * 128;     // TN rows x 64 bf16 (one swizzled box)
  static constexpr int KV_BYTES = 2 * KV_CHUNK; // one K or V tile (two boxes)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NK * KV_BYTES;
  static constexpr int OFF_Q = OFF_V + NV * KV_BYTES;  // query tile (two swizzled boxes)
  static constexpr int Q_BYTES = MT * D * 2;
  static constexpr int OFF_BAR = OFF_Q + Q_BYTES;
  // barriers: k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], q_ready,
  // s_full[2], p_full[2], o_done, o_final, drain, q_full
  static constexpr int NBAR = 2 * NK + 2 * NV + 1 + 2 + 2 + 3 + 1;
  static constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_Q = 0;          // 64 columns
  static constexpr uint32_t COL_S = 64;         // + 128 b
  static constexpr uint32_t COL_O = 320;        // 128 columns
  // Output staging (epilogue, over the dead K/V rings): four boxes of 32
  // fp32 columns x 128 rows, 128-byte swizzle.
  static constexpr int OBOX_BYTES = MT * 128;
  // Row-pair exchange (in the query staging, dead once the first scores
  // are in): maxima [2 tiles][2 halves][MT], then sums [2 halves][MT].
  static constexpr int XCH_MAX = 0;
  static constexpr int XCH_SUM = 4 * MT * 4;
  static_assert(TN == 128, "score buffers are laid out for 128-token tiles");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(4 * OBOX_BYTES <= OFF_Q, "epilogue staging fits the K/V rings");
  static_assert(XCH_SUM + 2 * MT * 4 <= Q_BYTES, "row-pair exchange fits the query staging");
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
                   const __grid_constant__ CUtensorMap tmVd,
                   const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmO) {
  using C = BifCfg;
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
  uint64_t* q_full = drain + 1;                 // the query tile's TMA load
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(q_full + 1);
  int* abort_s = reinterpret_cast<int*>(taddr_s + 1);

  const int mtile = blockIdx.x;                 // 128-row query tile
  const int split = blockIdx.y;
  const int g = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Set-up that reads no global memory (barriers, tensor memory, the
  // tensor maps in parameter space) runs before the launch wait, so it
  // overlaps the tail of the previous kernel on the stream.
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
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    if (p.fold) {
      prefetch_tensormap(&tmKd);
      prefetch_tensormap(&tmVd);
    }
    if (p.q_tma) prefetch_tensormap(&tmQ);
    if (p.o_tma) prefetch_tensormap(&tmO);
  }
  pdl_wait_prerequisites();   // launched with PDL: no global memory access before this
  // Every earlier grid has now finished: the decode part (which reads none of
  // this kernel's output) may start on the SMs this grid leaves free.
  pdl_launch_dependents();

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

  // Softmax thread coordinates: TMEM lane quadrant, row, column half.
  const int quad = warp & 3;
  const int half = (warp - 2) >> 2;             // softmax warps 2..5: 0, 6..9: 1
  const int r = quad * 32 + lane;               // row of the query tile (softmax warps)

  // Without the query TMA, the softmax threads issue their query loads now
  // (half a row each: 64 head dims as bf16 pairs, dim 2c in the low half of
  // word c), so they are in flight while the CTA finishes its set-up.  Rows
  // past n * G load zeros.  A negative scale is folded in here (the sign
  // bits flip), so the softmax always scales by |scale|.
  uint32_t qv[32];
  if (warp >= 2 && !p.q_tma && ntiles > 0) {
    const int m = mtile * C::MT + r;
    if (m < p.rows) {
      const int s = m / p.G;
      const int h = g * p.G + (m - s * p.G);
      const uint4* src = reinterpret_cast<const uint4*>(p.q + s * p.q_sb + h * p.q_sh + half * 64);
      const uint32_t flip = p.negate_q ? 0x80008000u : 0u;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 w = src[i];
        qv[i * 4 + 0] = w.x ^ flip;
        qv[i * 4 + 1] = w.y ^ flip;
        qv[i * 4 + 2] = w.z ^ flip;
        qv[i * 4 + 3] = w.w ^ flip;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) qv[i] = 0u;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *taddr_s;

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
    if (warp == 1) tc::tmem_dealloc(tmem, C::TMEM_COLS);
    return;
  }

  const uint32_t sbase = smem_u32(smem);
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop (warp-uniform waits and operands); one
    // elected lane issues each copy.
    const uint64_t policy = l2_policy_evict_first();
    if (p.q_tma) {
      // The query tile first: rows m0 .. m0 + 127 of kv head g are heads
      // r0 .. of samples s0 .. (rows past n * G fill with zeros); the
      // query rows of a tile are reused by every split, so they are kept in
      // L2 with priority.
      const int m0 = mtile * C::MT;
      const int s0 = m0 / p.G, r0 = m0 - s0 * p.G;
      const uint64_t qpol = l2_policy_evict_last();
      mbar_arrive_expect_tx_w(q_full, C::Q_BYTES);
      tma_load_4d_w(smem + C::OFF_Q, &tmQ, q_full, 0, r0, g, s0, qpol);
      tma_load_4d_w(smem + C::OFF_Q + C::Q_BYTES / 2, &tmQ, q_full, 64, r0, g, s0, qpol);
    }
    int kt = 0, vt = 0;                             // next K / V tile to issue
    bool ok = true;
    while (ok && (kt < ntiles || vt < ntiles)) {
      // K runs up to NK tiles ahead of V; V follows.
      if (kt < ntiles && kt < vt + C::NK) {
        const int st = kt % C::NK;
        if (kt >= C::NK)
          ok = __all_sync(0xffffffffu,
                          mbar_wait_or_abort(&k_empty[st], ((kt / C::NK) - 1) & 1, abort_s));
        if (!ok) break;
        unsigned char* dst = smem + C::OFF_K + st * C::KV_BYTES;
        mbar_arrive_expect_tx_w(&k_full[st], C::KV_BYTES);
        bool is_dec;
        int k, tok, nv;
        tile_of(kt, is_dec, k, tok, nv);
        if (is_dec) {
          tma_load_4d_w(dst, &tmKd, &k_full[st], 0, g, tok, s_first + k, policy);
          tma_load_4d_w(dst + C::KV_CHUNK, &tmKd, &k_full[st], 64, g, tok, s_first + k, policy);
        } else {
          tma_load_3d_w(dst, &tmK, &k_full[st], 0, g, tok);
          tma_load_3d_w(dst + C::KV_CHUNK, &tmK, &k_full[st], 64, g, tok);
        }
        ++kt;
      }
      if (vt < ntiles && vt < kt) {
        const int st = vt % C::NV;
        if (vt >= C::NV)
          ok = __all_sync(0xffffffffu,
                          mbar_wait_or_abort(&v_empty[st], ((vt / C::NV) - 1) & 1, abort_s));
        if (!ok) break;
        unsigned char* dst = smem + C::OFF_V + st * C::KV_BYTES;
        mbar_arrive_expect_tx_w(&v_full[st], C::KV_BYTES);
        bool is_dec;
        int k, tok, nv;
        tile_of(vt, is_dec, k, tok, nv);
        if (is_dec) {
          tma_load_4d_w(dst, &tmVd, &v_full[st], 0, g, tok, s_first + k, policy);
          tma_load_4d_w(dst + C::KV_CHUNK, &tmVd, &v_full[st], 64, g, tok, s_first + k, policy);
        } else {
          tma_load_3d_w(dst, &tmV, &v_full[st], 0, g, tok);
          tma_load_3d_w(dst + C::KV_CHUNK, &tmV, &v_full[st], 64, g, tok);
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
    if (p.q_tma) mbar_wait_bounded(q_full, 0);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop; one elected lane issues each MMA and
    // commit (warp-uniform descriptors stay in uniform registers, so the
    // issue keeps ahead of the tensor core).
    constexpr uint32_t IDESC_S = tc::idesc_bf16_f32(C::MT, C::TN, false, false);
    constexpr uint32_t IDESC_O = tc::idesc_bf16_f32(C::MT, C::D, false, true);
    // Descriptors of stage 0's K and V boxes.  A stage, a 16-column step
    // of K or a 16-token step of V adds a constant to the start-address
    // field (16-byte units, low bits; shared addresses stay below 2^18, so
    // the field never carries).
    const uint64_t kd0 = tc::smem_desc_sw128(sbase + C::OFF_K, 16, 1024);
    const uint64_t vd0 = tc::smem_desc_sw128(sbase + C::OFF_V, C::KV_CHUNK, 1024);
    const uint32_t q_t = tmem + C::COL_Q;
    // S[j % 2] = Q K_j^T from K stage kst (8 MMAs of K = 16 head dims; Q
    // columns 8 kk; K box kk / 4, 32 bytes per 16 dims within it).
    auto issue_s = [&](int j, int kst) {
      const uint64_t kd = kd0 + (uint64_t)(kst * (C::KV_BYTES >> 4));
      const uint32_t d_tmem = tmem + C::COL_S + (uint32_t)(j & 1) * 128u;
      tc::mma_bf16_ts_w<false>(d_tmem, q_t, kd, IDESC_S);
#pragma unroll
      for (int kk = 1; kk < C::D / 16; ++kk)
        tc::mma_bf16_ts_w<true>(d_tmem, q_t + kk * 8,
                                kd + (uint64_t)(((kk >> 2) * C::KV_CHUNK + (kk & 3) * 32) >> 4),
                                IDESC_S);
      tc::commit_w(&s_full[j & 1]);
    };
    // O += P_j V_j from V stage vst (8 MMAs of K = 16 tokens; P_j from the
    // first 64 columns of S[j % 2], 8 per MMA; V MN-major: 16 token rows
    // of 128 bytes per step, two 64-wide head-dim blocks KV_CHUNK apart).
    auto issue_pv = [&](int j, int vst) {
      const uint64_t vd = vd0 + (uint64_t)(vst * (C::KV_BYTES >> 4));
      const uint32_t a_tmem = tmem + C::COL_S + (uint32_t)(j & 1) * 128u;
      if (j == 0)
        tc::mma_bf16_ts_w<false>(tmem + C::COL_O, a_tmem, vd, IDESC_O);
      else
        tc::mma_bf16_ts_w<true>(tmem + C::COL_O, a_tmem, vd, IDESC_O);
#pragma unroll
      for (int kk = 1; kk < C::TN / 16; ++kk)
        tc::mma_bf16_ts_w<true>(tmem + C::COL_O, a_tmem + kk * 8,
                                vd + (uint64_t)((kk * 16 * 128) >> 4), IDESC_O);
      tc::commit_w(o_done);
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait_or_abort(bar, parity, abort_s));
    };
    bool ok = wait(q_ready, 0);
    if (ok && p.q_tma) {
      // Query tile (shared memory, K-major, 128-byte swizzle) -> Q in
      // tensor memory: 8 copies of 16 head dims, ordered before the MMAs.
      ok = wait(q_full, 0);
      if (ok) {
        tc::fence_after_sync();
        const uint64_t qd0 = tc::smem_desc_sw128(sbase + C::OFF_Q, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk)
          tc::cp_128x256b_w(q_t + kk * 8,
                            qd0 + (uint64_t)(((kk >> 2) * (C::Q_BYTES / 2) + (kk & 3) * 32) >> 4));
      }
    }
    // Prologue: scores of tiles 0 and 1.
    for (int j = 0; ok && j < 2 && j < ntiles; ++j) {
      if (!wait(&k_full[j % C::NK], (j / C::NK) & 1)) { ok = false; break; }
      tc::fence_after_sync();
      issue_s(j, j % C::NK);
      tc::commit_w(&k_empty[j % C::NK]);
    }
    int vst = 0, vph = 0;                          // V stage and phase of tile j
    int kst = 2 % C::NK, kph = (2 / C::NK) & 1;    // K stage and phase of tile j + 2
    for (int j = 0; ok && j < ntiles; ++j) {
      if (!wait(&v_full[vst], (uint32_t)vph)) break;
      if (!wait(&p_full[j & 1], (j >> 1) & 1)) break;
      tc::fence_after_sync();
      issue_pv(j, vst);
      tc::commit_w(&v_empty[vst]);
      if (j + 2 < ntiles) {
        if (!wait(&k_full[kst], (uint32_t)kph)) break;
        issue_s(j + 2, kst);
        tc::commit_w(&k_empty[kst]);
      }
      if (++vst == C::NV) { vst = 0; vph ^= 1; }
      if (++kst == C::NK) { kst = 0; kph ^= 1; }
    }
    tc::commit_w(o_final);
    // Drain: every MMA issued above completes before the TMEM is freed.
    tc::commit_w(drain);
    mbar_wait_bounded(drain, 0);
  } else {
    // ------------------------------------------------------------ softmax
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t q_tmem = tmem + lane_base + C::COL_Q;
    const uint32_t o_tmem = tmem + lane_base + C::COL_O + (uint32_t)(half * 64);
    const int c0 = half * C::HALF;                // first score column of this thread
    const int m0 = mtile * C::MT;                 // first row of this tile
    const int row_s = (m0 + r) / p.G;             // sample of this row
    const int pair_bar = 1 + quad;                // named barrier of the quadrant's two warps
    float* xch = reinterpret_cast<float*>(smem + C::OFF_Q);   // row-pair exchange
    bool ok = true;
    if (!p.q_tma) {
      // Half query row (loaded above) -> Q in tensor memory (32 columns).
      tc::tmem_st32(q_tmem + half * 32, qv);
      tc::tmem_wait_st();
      tc::fence_before_sync();
    } else if (p.negate_q) {
      // A negative scale: flip the sign bits of the staged query tile before
      // the MMA warp copies it (consecutive threads on consecutive 16 bytes).
      ok = __all_sync(0xffffffffu, mbar_wait_or_abort(q_full, 0, abort_s));
      if (ok) {
        uint4* qs = reinterpret_cast<uint4*>(smem + C::OFF_Q);
        for (int i = threadIdx.x - 64; i < C::Q_BYTES / 16; i += C::NSW * 32) {
          uint4 w = qs[i];
          w.x ^= 0x80008000u;
          w.y ^= 0x80008000u;
          w.z ^= 0x80008000u;
          w.w ^= 0x80008000u;
          qs[i] = w;
        }
        tc::fence_proxy_async_smem();
      }
    }
    mbar_arrive(q_ready);

    float m_run = kNegInf, l_run = 0.f;
    const float c2 = p.scale_log2;                 // |scale| * log2(e) >= 0
    const uint64_t c2x2 = f2_pack(c2, c2);
    // Every softmax warp runs all ntiles iterations and meets its partner
    // at the pair barrier in each (also after a wait gave up: ok then only
    // skips the tensor-memory work).
    for (int j = 0; j < ntiles; ++j) {
      const uint32_t s_tmem = tmem + lane_base + C::COL_S + (j & 1) * 128;
      // Waits are made warp-uniform before any .sync.aligned tcgen05 access.
      ok = __all_sync(0xffffffffu, ok && mbar_wait_or_abort(&s_full[j & 1], (j >> 1) & 1, abort_s));
      // Context tile: the context's tail; decode tile: its sample's tail,
      // and nothing at all for rows of the tile's other samples.
      bool is_dec;
      int ks, tok, tile_valid;
      tile_of(j, is_dec, ks, tok, tile_valid);
      const int nvalid = (!is_dec || row_s == s_first + ks) ? tile_valid : 0;
      float m_new = m_run, alpha = 1.f, tile_sum = 0.f;
      // The same for both warps of a quadrant (same rows).
      const bool none = __all_sync(0xffffffffu, nvalid == 0);
      if (none) {
        // A decode tile of a sample none of these rows belongs to: P = 0.
        if (ok) {
          uint32_t z[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] = 0u;
          tc::tmem_st32(s_tmem + half * 32, z);
        }
      } else {
        uint32_t sr[2][32];
        float mx = kNegInf;
        if (ok) {
          tc::fence_after_sync();
          tc::tmem_ld32(s_tmem + c0, sr[0]);
          tc::tmem_ld32(s_tmem + c0 + 32, sr[1]);
          tc::tmem_wait_ld();
          if (nvalid < c0 + C::HALF) {             // tails (and other samples' decode tiles)
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (c0 + c * 32 + i >= nvalid) sr[c][i] = __float_as_uint(kNegInf);
          }
          // Half-row maximum: three-input maxima in 4 independent chains.
          float mx4[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int i = 0; i < 16; ++i)
              mx4[i & 3] = fmax3(mx4[i & 3], __uint_as_float(sr[c][2 * i]),
                                 __uint_as_float(sr[c][2 * i + 1]));
          mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        }
        // Trade half-row maxima with the partner thread (same row, other
        // half).  Past the barrier both halves have read their scores, so
        // P may overwrite them.
        xch[C::XCH_MAX / 4 + ((j & 1) * 2 + half) * C::MT + r] = mx;
        named_barrier_sync(pair_bar, 64);
        mx = fmaxf(mx, xch[C::XCH_MAX / 4 + ((j & 1) * 2 + (half ^ 1)) * C::MT + r]);
        if (ok) {
          mx *= c2;                                  // -inf stays -inf (c2 > 0)
          m_new = (mx > m_run + 8.f) ? mx : m_run;
          alpha = (m_new == m_run) ? 1.f : fast_exp2(m_run - m_new);
          const float m_use = (m_new == kNegInf) ? 0.f : m_new;   // all -inf: p = 0, not NaN
          const uint64_t negm2 = f2_pack(-m_use, -m_use);
          // p = 2^(s * c2 - m): one packed FMA per pair of columns, one ex2
          // per column, the pair packed as bf16 (even token in the low half)
          // and summed with one packed add; this half's 32 P columns go to
          // the first 64 columns of the score buffer.
          uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c][2 * i]),
                                       __uint_as_float(sr[c][2 * i + 1])),
                               c2x2, negm2),
                        x0, x1);
              const float p0 = fast_exp2(x0);
              const float p1 = fast_exp2(x1);
              sum2[i & 3] = f2_add(sum2[i & 3], f2_pack(p0, p1));
              uint32_t w;
              asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(p1), "f"(p0));
              sr[c][i] = w;
            }
            tc::tmem_st16(s_tmem + half * 32 + c * 16, sr[c]);
          }
          float a0, a1, b0, b1;
          f2_unpack(f2_add(sum2[0], sum2[1]), a0, a1);
          f2_unpack(f2_add(sum2[2], sum2[3]), b0, b1);
          tile_sum = (a0 + a1) + (b0 + b1);
        }
      }
      // Rescale this half of O where the max moved (rare), once O +=
      // P_{j-1} V_{j-1} is done: o_done has then completed phases 0..j-1
      // (phase j needs P_j).
      if (ok && j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        ok = __all_sync(0xffffffffu, mbar_wait_or_abort(o_done, (j - 1) & 1, abort_s));
        if (ok) {
          tc::fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t orr[32];
            tc::tmem_ld32(o_tmem + c * 32, orr);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            tc::tmem_st32(o_tmem + c * 32, orr);
            tc::tmem_wait_st();
          }
        }
      }
      if (ok && is_dec && tile_valid < C::TN) {
        // V rows past the sample's length hold whatever the cache holds
        // there: zero them before O += P V reads the tile (P is 0 on those
        // rows, but 0 times a non-finite value is not 0).  This thread
        // clears its row's half (one 64-column box).
        ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&v_full[j % C::NV], (j / C::NV) & 1, abort_s));
        if (ok && r >= tile_valid) {
          uint4* vrow = reinterpret_cast<uint4*>(smem + C::OFF_V + (j % C::NV) * C::KV_BYTES +
                                                 half * C::KV_CHUNK + r * 128);
#pragma unroll
          for (int i = 0; i < 8; ++i) vrow[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        tc::fence_proxy_async_smem();
      }
      if (ok) {
        tc::tmem_wait_st();
        tc::fence_before_sync();
      }
      mbar_arrive(&p_full[j & 1]);
      l_run = l_run * alpha + tile_sum;
      m_run = m_new;
    }
    // ------------------------------------------------------------ epilogue
    // o_final is committed after the last MMA of the CTA: once it fires the
    // K/V rings are dead.  The two halves of a row add their sums; each
    // thread normalises its 64 columns of O into the staging tile, then one
    // thread stores the tile with four TMA tensor stores (or, where no
    // output map applies, each thread writes its half row).
    const bool done = __all_sync(0xffffffffu, ok && mbar_wait_or_abort(o_final, 0, abort_s));
    xch[C::XCH_SUM / 4 + half * C::MT + r] = l_run;
    named_barrier_sync(pair_bar, 64);
    const float l_tot = l_run + xch[C::XCH_SUM / 4 + (half ^ 1) * C::MT + r];
    const int m = m0 + r;
    if (done) {
      tc::fence_after_sync();
      const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;   // a decode row may see no token
      float* orow = nullptr;
      if (!p.o_tma && m < p.rows) {
        const int s = m / p.G;
        const int h = g * p.G + (m - s * p.G);
        orow = p.o + s * p.o_sb + h * p.o_sh + split * p.o_ss + half * 64;
      }
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t orr[32];
        tc::tmem_ld32(o_tmem + c * 32, orr);
        tc::tmem_wait_ld();
        if (p.o_tma) {
          // Box 2 * half + c, row r: chunk k of the row at (k ^ (r % 8)) * 16
          // bytes (the 128-byte swizzle pattern), so the 8 lanes of a phase
          // write 8 distinct 16-byte slots.
          unsigned char* rowp = smem + (2 * half + c) * C::OBOX_BYTES + r * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4*>(rowp + ((k ^ (r & 7)) << 4)) =
                make_float4(__uint_as_float(orr[4 * k]) * inv_l,
                            __uint_as_float(orr[4 * k + 1]) * inv_l,
                            __uint_as_float(orr[4 * k + 2]) * inv_l,
                            __uint_as_float(orr[4 * k + 3]) * inv_l);
        } else if (orow != nullptr) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4*>(orow + c * 32 + 4 * k) =
                make_float4(__uint_as_float(orr[4 * k]) * inv_l,
                            __uint_as_float(orr[4 * k + 1]) * inv_l,
                            __uint_as_float(orr[4 * k + 2]) * inv_l,
                            __uint_as_float(orr[4 * k + 3]) * inv_l);
        }
      }
      if (half == 0 && m < p.rows && p.lse) {
        const int s = m / p.G;
        const int h = g * p.G + (m - s * p.G);
        p.lse[s * p.l_sb + h * p.l_sh + split * p.l_ss] = (m_run + __log2f(l_tot)) * kLn2;
      }
    }
    if (p.o_tma) {
      // Every softmax thread's staging writes, made visible to the async
      // proxy, before one thread stores the tile: rows m0 .. m0 + 127 of kv
      // head g are heads r0 .. of samples s0 .. of partial slot `split`
      // (rows past n * G are outside the tensor and not written).
      tc::fence_proxy_async_smem();
      named_barrier_sync(5, C::NSW * 32);
      if (threadIdx.x == 64 && done) {
        const int s0 = m0 / p.G, r0 = m0 - s0 * p.G;
#pragma unroll
        for (int b = 0; b < 4; ++b)
          tma_store_5d(&tmO, smem + b * C::OBOX_BYTES, 32 * b, r0, g, s0, split);
        bulk_store_commit_and_wait_read();
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
