// Split-KV partial kernels.
//
// One CTA owns one (split i, kv head g, sequence b): the tokens
// [begin_i, end_i) of sequence b (fd_split_bounds), and every query head of
// kv head g's GQA group.  It computes, in one pass over its K/V tokens,
//   scores  s_j = scale * <q_h, k_j>          (kept in base 2: q is pre-scaled
//                                              by scale * log2 e)
//   online softmax  m, l  per head           (running max / running sum)
//   PV      acc_h = sum_j 2^(s_j - m) v_j
// and writes the normalised partial output acc_h / l_h and its natural-log
// log-sum-exp (m + log2 l) * ln 2.  Source: Flash-Decoding page ("What is
// Flash-Decoding and when does it speed up LLMs?"), section "Why decoding
// needs different scheduling": split the history across GPU blocks, each
// block emits a partial result plus a log-sum-exp value; the online softmax
// follows "How does Flash Attention reduce memory traffic during local
// inference?", section on online softmax (running normalisation statistics,
// no materialised score row).
//
// split_tma_kernel (bf16 K/V, head dim 128), 8 warps, one CTA per SM:
//   - thread 0 streams 64-token K and V tiles into a 5-stage shared-memory
//     ring with TMA tensor loads (no multicast), completion tracked by
//     mbarriers (full[s] / empty[s]); a stage is refilled once all 8 warps
//     have released it.  (No separate producer warp: a 9th warp would cap
//     every thread at 168 registers, as the 4 SM sub-partitions each hold
//     a quarter of the register file.)
//   - every warp consumes: 16 lanes per token, 8 head-dim elements
//     (one 16-byte shared load) per lane; every converted K/V element feeds
//     GH query heads held in registers.  The 16 per-lane partial dot products
//     of a batch of 4 tokens x GH heads are reduce-scattered with shuffles;
//     each lane then owns whole scores of one head, runs the online-softmax
//     update for it, and publishes probabilities through shared memory for
//     the PV step.  Query-register order is permuted per lane so the
//     reduce-scatter needs no selects (see `phys_mask`).
//   - epilogue: the 16 (or fewer) token slots of the CTA merge their
//     (m, l, acc) states through shared memory and write the partial.
//
// split_generic_kernel: any supported (dtype, head dim, group size); one CTA
// per (split, query head, sequence); plain global loads.  Used for fp32
// caches, head dim 64 and layouts TMA cannot describe.
#pragma once

#include "fd_device.cuh"

namespace fd {

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kLn2 = 0.6931471805599453f;

// Device copy of the split partition; must equal fd_split_bounds().
// Computed in 64 bits: len may come within a few tokens of INT32_MAX (a
// paged cache's capacity needs no memory behind it), where len + ns - 1
// would overflow an int.
__device__ __forceinline__ void split_range(int len, int ns, int i, int& begin, int& end) {
  const long long per = ((long long)len + ns - 1) / ns;
  const long long chunk = ((per + kSplitAlign - 1) / kSplitAlign) * kSplitAlign;
  const long long b0 = (long long)i * chunk;
  begin = (int)(b0 < len ? b0 : len);
  end = (int)(b0 + chunk < len ? b0 + chunk : len);
}

// Length of sequence b, clamped to [0, cap]; out-of-range values raise the
// device bounds flag.
__device__ __forceinline__ int resolve_len(const int32_t* seqlens, int b, int cap) {
  if (seqlens == nullptr) return cap;
  int len = seqlens[b];
  if (len < 0 || len > cap) {
    raise_device_error(FD_DEVERR_BOUNDS);
    len = len < 0 ? 0 : cap;
  }
  return len;
}

// Page of token j of sequence b in a paged cache; an id outside
// [0, num_pages) raises the device bounds flag and is replaced by `bad`.
__device__ __forceinline__ int page_of(const SplitParams& p, int b, int j, int bad) {
  int pid = p.block_table[(int64_t)b * p.bt_stride + j / p.page_size];
  if (pid < 0 || pid >= p.num_pages) {
    raise_device_error(FD_DEVERR_BOUNDS);
    pid = bad;
  }
  return pid;
}

template <int N>
struct Log2 {
  static constexpr int value = 1 + Log2<N / 2>::value;
};
template <>
struct Log2<1> {
  static constexpr int value = 0;
};

// ------------------------------------------------------------------ TMA kernel

template <int GH_, int HC_>
struct TmaCfg {
  static constexpr int GH = GH_;             // query heads per head chunk (registers)
  static constexpr int HC = HC_;             // head chunks (warp groups) per CTA
  static constexpr int G = GH * HC;          // query heads per kv head
  static constexpr int D = 128;
  static constexpr int T = kSplitTileTokens; // tokens per tile
  static constexpr int NSTAGE = 5;
  static constexpr int NCW = 8;              // warps (all consume; thread 0 also issues TMA)
  static constexpr int THREADS = NCW * 32;
  static constexpr int LPT = 16;             // lanes per token
  static constexpr int EPL = 8;              // bf16 elements per lane
  static constexpr int TS = (NCW / HC) * 2;  // token slots per head chunk
  static constexpr int NSLOT = HC * TS;      // = 2 * NCW
  static constexpr int TOK_PER_SLOT = T / TS;
  static constexpr int NB = 4;               // tokens per softmax batch
  static constexpr int LOG_NB = 2;
  static constexpr int NBATCH = TOK_PER_SLOT / NB;
  static constexpr int V = GH * NB;          // partial scores per lane per batch
  static constexpr int NBITS = Log2<V>::value;
  static constexpr int C = V >= 16 ? V / 16 : 1;          // scores owned after reduction
  static constexpr int SH = NBITS >= 4 ? 0 : 4 - NBITS;   // butterfly-duplicated lane bits
  static constexpr int NTB = NBITS >= 4 ? 4 - Log2<GH>::value : LOG_NB;  // token lane bits
  static constexpr int TILE_BYTES = T * D * 2;             // one K or V tile
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int RING_BYTES = NSTAGE * STAGE_BYTES;
  static constexpr int P_PAIRS = NSLOT * NB * GH;           // probabilities as (p, p)
  static constexpr int A_FLOATS = NSLOT * GH;
  static constexpr int SMEM_BYTES =
      1024 /*align slack*/ + RING_BYTES + P_PAIRS * 8 + A_FLOATS * 4 + 2 * NSTAGE * 8 + 16;
  static_assert(TS * TOK_PER_SLOT == T, "tile must split evenly over slots");
  static_assert(NBATCH >= 1 && NBATCH * NB == TOK_PER_SLOT, "whole batches per slot");
  static_assert(GH <= 8 && (GH & (GH - 1)) == 0, "GH must be 1, 2, 4 or 8");
  static_assert(NSLOT * GH * 2 * 4 + NSLOT * GH * D * 4 <= RING_BYTES, "epilogue fits the ring");
};

template <int GH, int HC>
__global__ void __launch_bounds__(TmaCfg<GH, HC>::THREADS, 1)
    split_tma_kernel(const __grid_constant__ SplitParams p,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV) {
  using C = TmaCfg<GH, HC>;
  if (!p.late_wait) pdl_wait_prerequisites();   // launched with PDL: no memory access before this
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float2* P_s = reinterpret_cast<float2*>(smem + C::RING_BYTES);   // (p, p) pairs
  float* A_s = reinterpret_cast<float*>(P_s + C::P_PAIRS);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(A_s + C::A_FLOATS);
  uint64_t* empty_bar = full_bar + C::NSTAGE;
  int* abort_s = reinterpret_cast<int*>(empty_bar + C::NSTAGE);

  const int split = blockIdx.x;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int len = resolve_len(p.seqlens, b, p.Lcap);
  int begin, end;
  split_range(len, p.ns, split, begin, end);
  const int ntiles = (end - begin + C::T - 1) / C::T;
  const int kvb = p.kv_batch_broadcast ? 0 : b;   // kv batch row of the tensor map

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], C::NCW);
    }
    *abort_s = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const int hc = warp % C::HC;
  const int slot = (warp / C::HC) * 2 + (lane >> 4);
  const int L = lane & 15;
  // Physical/logical index map of the reduce-scatter: logical score index
  // j = head * NB + token sits at register position j ^ phys_mask.
  const int phys_mask = C::NBITS >= 4 ? (L << (C::NBITS - 4)) : (L >> (4 - C::NBITS));
  const int mh = phys_mask >> C::LOG_NB;        // head xor (also: the head this lane owns)
  const int mt = phys_mask & (C::NB - 1);       // token xor
  const bool head_writer = (L & ((1 << (C::SH + C::NTB)) - 1)) == 0;
  const bool p_writer = (L & ((1 << C::SH) - 1)) == 0;

  // Accumulators as (even, odd) head-dim pairs for the paired fp32 FMA.
  float2 acc[GH][C::EPL / 2];
  float m_run = kNegInf, l_run = 0.f;

  // Tile issue (thread 0 only): tiles 0..NSTAGE-1 up front, then tile
  // t-1+NSTAGE once every warp has released tile t-1's stage.
  uint64_t policy = 0;
  int issued = 0;
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    policy = l2_policy_evict_first();
    for (int t = 0; t < C::NSTAGE && t < ntiles; ++t) {
      unsigned char* stage = smem + t * C::STAGE_BYTES;
      mbar_arrive_expect_tx(&full_bar[t], C::STAGE_BYTES);
      const int tok = begin + t * C::T;
      tma_load_4d(stage, &tmK, &full_bar[t], 0, g, tok, kvb, policy);
      tma_load_4d(stage + C::TILE_BYTES, &tmV, &full_bar[t], 0, g, tok, kvb, policy);
      ++issued;
    }
  }
  {
    // Query registers, pre-scaled into base 2, as (even, odd) pairs, in the
    // lane's physical head order.
    float2 qr[GH][C::EPL / 2];
#pragma unroll
    for (int ph = 0; ph < GH; ++ph) {
      const int h = g * C::G + hc * GH + (ph ^ mh);
      float qv[C::EPL];
      if (p.q_bf16) {
        const uint16_t* qp =
            reinterpret_cast<const uint16_t*>(p.q) + b * p.q_sb + h * p.q_sh + L * C::EPL;
#pragma unroll
        for (int e = 0; e < C::EPL; ++e) qv[e] = __uint_as_float(uint32_t(qp[e]) << 16);
      } else {
        const float* qp = reinterpret_cast<const float*>(p.q) + b * p.q_sb + h * p.q_sh + L * C::EPL;
#pragma unroll
        for (int e = 0; e < C::EPL; ++e) qv[e] = qp[e];
      }
#pragma unroll
      for (int e = 0; e < C::EPL / 2; ++e) {
        qr[ph][e] = make_float2(qv[2 * e] * p.scale_log2, qv[2 * e + 1] * p.scale_log2);
        acc[ph][e] = make_float2(0.f, 0.f);
      }
    }
    float2* P_slot = P_s + (hc * C::TS + slot) * C::NB * GH;
    float* A_slot = A_s + (hc * C::TS + slot) * GH;

    for (int t = 0; t < ntiles; ++t) {
      const int s = t % C::NSTAGE;
      if (!mbar_wait_or_abort(&full_bar[s], (t / C::NSTAGE) & 1, abort_s)) break;
      const uint16_t* Ks = reinterpret_cast<const uint16_t*>(smem + s * C::STAGE_BYTES);
      const uint16_t* Vs = Ks + C::T * C::D;
      const int nvalid = min(C::T, end - (begin + t * C::T));
      const bool full_tile = nvalid == C::T;

#pragma unroll 1
      for (int bi = 0; bi < C::NBATCH; ++bi) {
        // ---- QK^T: partial dot products over this lane's 8 elements
        float sp[C::V];
#pragma unroll
        for (int pt = 0; pt < C::NB; ++pt) {
          const int row = (bi * C::NB + (pt ^ mt)) * C::TS + slot;
          const uint4 kr = lds128(Ks + row * C::D + L * C::EPL);
          const float2 k2[4] = {make_float2(bf16lo_to_f32(kr.x), bf16hi_to_f32(kr.x)),
                                make_float2(bf16lo_to_f32(kr.y), bf16hi_to_f32(kr.y)),
                                make_float2(bf16lo_to_f32(kr.z), bf16hi_to_f32(kr.z)),
                                make_float2(bf16lo_to_f32(kr.w), bf16hi_to_f32(kr.w))};
#pragma unroll
          for (int ph = 0; ph < GH; ++ph) {
            float2 a = __fmul2_rn(qr[ph][0], k2[0]);
            a = __ffma2_rn(qr[ph][1], k2[1], a);
            a = __ffma2_rn(qr[ph][2], k2[2], a);
            a = __ffma2_rn(qr[ph][3], k2[3], a);
            sp[ph * C::NB + pt] = a.x + a.y;
          }
        }
        // ---- reduce-scatter over the 16 lanes of the token group
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int o = 8 >> k;
          const int n = C::V >> k;
          if (n >= 2) {
#pragma unroll
            for (int i = 0; i < n / 2; ++i) sp[i] += __shfl_xor_sync(0xffffffffu, sp[i + n / 2], o);
          } else {
            sp[0] += __shfl_xor_sync(0xffffffffu, sp[0], o);
          }
        }
        // sp[c], c < C, is the full score of head mh, token (c ^ mt).
        float mx = kNegInf;
#pragma unroll
        for (int c = 0; c < C::C; ++c) {
          if (!full_tile) {
            const int row = (bi * C::NB + (c ^ mt)) * C::TS + slot;
            if (row >= nvalid) sp[c] = kNegInf;
          }
          mx = fmaxf(mx, sp[c]);
        }
#pragma unroll
        for (int i = 0; i < C::NTB; ++i) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1 << (C::SH + i)));
        // Lazy rescaling: keep the running max unless the batch max exceeds
        // it by more than 8 (base 2), so probabilities stay <= 256 and the
        // accumulators are rescaled rarely.  Exact: the final normalisation
        // uses the same m for numerator and denominator.
        const float m_new = (mx > m_run + 8.f) ? mx : m_run;
        const float alpha = (m_new == m_run) ? 1.f : fast_exp2(m_run - m_new);
        float psum = 0.f;
#pragma unroll
        for (int c = 0; c < C::C; ++c) {
          const float pv = (m_new == kNegInf) ? 0.f : fast_exp2(sp[c] - m_new);
          sp[c] = pv;
          psum += pv;
        }
#pragma unroll
        for (int i = 0; i < C::NTB; ++i) psum += __shfl_xor_sync(0xffffffffu, psum, 1 << (C::SH + i));
        l_run = l_run * alpha + psum;
        m_run = m_new;
        if (p_writer) {
#pragma unroll
          for (int c = 0; c < C::C; ++c) P_slot[(c ^ mt) * GH + mh] = make_float2(sp[c], sp[c]);
        }
        if (head_writer) A_slot[mh] = alpha;
        __syncwarp();
        // ---- rescale accumulators when some head's max moved
        float al[GH];
        if constexpr (GH >= 4) {
#pragma unroll
          for (int h4 = 0; h4 < GH / 4; ++h4) {
            const float4 a4 = lds128f(A_slot + h4 * 4);
            al[h4 * 4 + 0] = a4.x;
            al[h4 * 4 + 1] = a4.y;
            al[h4 * 4 + 2] = a4.z;
            al[h4 * 4 + 3] = a4.w;
          }
        } else {
#pragma unroll
          for (int h = 0; h < GH; ++h) al[h] = A_slot[h];
        }
        bool moved = false;
#pragma unroll
        for (int h = 0; h < GH; ++h) moved |= (al[h] != 1.f);
        if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
          for (int h = 0; h < GH; ++h) {
            const float2 a2 = make_float2(al[h], al[h]);
#pragma unroll
            for (int e = 0; e < C::EPL / 2; ++e) acc[h][e] = __fmul2_rn(acc[h][e], a2);
          }
        }
        // ---- PV
#pragma unroll
        for (int tk = 0; tk < C::NB; ++tk) {
          float2 pr[GH];
          if constexpr (GH >= 2) {
#pragma unroll
            for (int h2 = 0; h2 < GH / 2; ++h2) {
              const float4 p4 = lds128f(P_slot + tk * GH + h2 * 2);
              pr[h2 * 2 + 0] = make_float2(p4.x, p4.y);
              pr[h2 * 2 + 1] = make_float2(p4.z, p4.w);
            }
          } else {
            pr[0] = P_slot[tk * GH];
          }
          const int row = (bi * C::NB + tk) * C::TS + slot;
          uint4 vr = lds128(Vs + row * C::D + L * C::EPL);
          if (!full_tile && row >= nvalid) vr = make_uint4(0u, 0u, 0u, 0u);
          const float2 v2[4] = {make_float2(bf16lo_to_f32(vr.x), bf16hi_to_f32(vr.x)),
                                make_float2(bf16lo_to_f32(vr.y), bf16hi_to_f32(vr.y)),
                                make_float2(bf16lo_to_f32(vr.z), bf16hi_to_f32(vr.z)),
                                make_float2(bf16lo_to_f32(vr.w), bf16hi_to_f32(vr.w))};
#pragma unroll
          for (int h = 0; h < GH; ++h)
#pragma unroll
            for (int e = 0; e < C::EPL / 2; ++e) acc[h][e] = __ffma2_rn(pr[h], v2[e], acc[h][e]);
        }
        __syncwarp();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
      if (threadIdx.x == 0 && t >= 1 && issued < ntiles) {
        const int tp = t - 1;                      // stage released one tile ago
        const int sp_ = tp % C::NSTAGE;
        if (mbar_wait_or_abort(&empty_bar[sp_], (tp / C::NSTAGE) & 1, abort_s)) {
          unsigned char* stage = smem + sp_ * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full_bar[sp_], C::STAGE_BYTES);
          const int tok = begin + issued * C::T;
          tma_load_4d(stage, &tmK, &full_bar[sp_], 0, g, tok, kvb, policy);
          tma_load_4d(stage + C::TILE_BYTES, &tmV, &full_bar[sp_], 0, g, tok, kvb, policy);
          ++issued;
        }
      }
    }
    // Never leave the CTA with copies in flight (matters only after an
    // abort; otherwise every issued phase has already been consumed).
    if (threadIdx.x == 0) {
      const int first = issued > C::NSTAGE ? issued - C::NSTAGE : 0;
      for (int t = first; t < issued; ++t)
        mbar_wait_bounded(&full_bar[t % C::NSTAGE], (t / C::NSTAGE) & 1);
    }
  }

  pdl_launch_dependents();
  __syncthreads();

  // ------------------------------------------------------------ epilogue
  // Merge the token slots' (m, l, acc) states: reuse the ring.
  float* ML_s = reinterpret_cast<float*>(smem);                 // [NSLOT][GH][2]
  float* ACC_s = ML_s + C::NSLOT * GH * 2;                       // [NSLOT][GH][D]
  {
    const int sidx = hc * C::TS + slot;
    if (head_writer) {
      ML_s[(sidx * GH + mh) * 2 + 0] = m_run;
      ML_s[(sidx * GH + mh) * 2 + 1] = l_run;
    }
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      float* dst = ACC_s + (sidx * GH + h) * C::D + L * C::EPL;
      *reinterpret_cast<float4*>(dst) = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < C::G * C::D; idx += C::THREADS) {
    const int hg = idx / C::D;
    const int d = idx - hg * C::D;
    const int hcc = hg / GH;
    const int h = hg - hcc * GH;
    float M = kNegInf;
#pragma unroll 4
    for (int s = 0; s < C::TS; ++s) M = fmaxf(M, ML_s[((hcc * C::TS + s) * GH + h) * 2]);
    float lt = 0.f, o = 0.f;
    if (M != kNegInf) {
#pragma unroll 4
      for (int s = 0; s < C::TS; ++s) {
        const int sidx = hcc * C::TS + s;
        const float ms = ML_s[(sidx * GH + h) * 2];
        const float f = (ms == kNegInf) ? 0.f : fast_exp2(ms - M);
        lt += f * ML_s[(sidx * GH + h) * 2 + 1];
        o += f * ACC_s[(sidx * GH + h) * C::D + d];
      }
    }
    const int hq = g * C::G + hg;
    const float out = lt > 0.f ? o / lt : 0.f;
    p.o[b * p.o_sb + hq * p.o_sh + split * p.o_ss + d] = out;
    if (d == 0 && p.lse != nullptr)
      p.lse[b * p.l_sb + hq * p.l_sh + split * p.l_ss] = lt > 0.f ? (M + __log2f(lt)) * kLn2 : kNegInf;
  }
  if (p.late_wait) pdl_wait_prerequisites();   // complete only after the preceding grid
}

// ------------------------------------------------------------------ generic

// One cache element as fp32 (8-bit kinds: the code, before its scale).
template <int KVK>
__device__ __forceinline__ float kv_elem(const void* base, int64_t i) {
  if constexpr (KVK == kKvBf16) {
    return __uint_as_float(uint32_t(reinterpret_cast<const uint16_t*>(base)[i]) << 16);
  } else if constexpr (KVK == kKvI8) {
    return float(reinterpret_cast<const int8_t*>(base)[i]);
  } else if constexpr (KVK == kKvE4m3) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(reinterpret_cast<const __nv_fp8_storage_t*>(base)[i], __NV_E4M3);
    return __half2float(__half(h));
  } else {
    return reinterpret_cast<const float*>(base)[i];
  }
}

template <int D, int KVK>
__global__ void __launch_bounds__(128) split_generic_kernel(const __grid_constant__ SplitParams p) {
  if (!p.late_wait) pdl_wait_prerequisites();   // launched with PDL: no memory access before this
  constexpr int NW = 4;
  constexpr int EPL = D / 32;
  __shared__ float ml_s[NW][2];
  __shared__ float acc_s[NW][D];
  const int split = blockIdx.x;
  const int TQ = p.tq > 1 ? p.tq : 1;
  const int tqi = blockIdx.y / p.Hq;          // query token (grid.y = tq * Hq)
  const int h = blockIdx.y - tqi * p.Hq;
  const int b = blockIdx.z;
  const int g = h / p.G;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int len = resolve_len(p.seqlens, b, p.Lcap);
  int begin, end;
  split_range(len, p.ns, split, begin, end);
  end = min(end, max(begin, len - TQ + tqi + 1));   // causal limit of query token tqi

  // 8-bit caches: the K scale joins the score scale, the V scale multiplies
  // the normalised output.
  constexpr bool kQuant = (KVK == kKvI8 || KVK == kKvE4m3);
  const float qs = kQuant ? p.scale_log2 * p.k_scale[g] : p.scale_log2;
  const float vs = kQuant ? p.v_scale[g] : 1.f;
  float q[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const int d = lane * EPL + e;
    float x;
    if (p.q_bf16)
      x = __uint_as_float(uint32_t(reinterpret_cast<const uint16_t*>(p.q)[b * p.q_sb + tqi * p.q_st + h * p.q_sh + d]) << 16);
    else
      x = reinterpret_cast<const float*>(p.q)[b * p.q_sb + tqi * p.q_st + h * p.q_sh + d];
    q[e] = x * qs;
  }
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float m = kNegInf, l = 0.f;
  for (int j = begin + warp; j < end; j += NW) {
    float kf[EPL], vf[EPL];
    int64_t kbase, vbase;
    if (p.block_table) {                       // paged: clamp bad ids to page 0
      const int pid = page_of(p, b, j, 0);
      const int off = j % p.page_size;
      kbase = (int64_t)pid * p.k_sb + (int64_t)off * p.k_sl;
      vbase = (int64_t)pid * p.v_sb + (int64_t)off * p.v_sl;
    } else {
      kbase = b * p.k_sb + (int64_t)j * p.k_sl;
      vbase = b * p.v_sb + (int64_t)j * p.v_sl;
    }
    const int64_t ko = kbase + g * p.k_sh + lane * EPL;
    const int64_t vo = vbase + g * p.v_sh + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      kf[e] = kv_elem<KVK>(p.k, ko + e);
      vf[e] = kv_elem<KVK>(p.v, vo + e);
    }
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) s = fmaf(q[e], kf[e], s);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float m_new = fmaxf(m, s);
    const float alpha = fast_exp2(m - m_new);     // m = -inf -> 0
    const float pj = fast_exp2(s - m_new);
    l = l * alpha + pj;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = fmaf(pj, vf[e], acc[e] * alpha);
    m = m_new;
  }
  pdl_launch_dependents();
  if (lane == 0) {
    ml_s[warp][0] = m;
    ml_s[warp][1] = l;
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc_s[warp][lane * EPL + e] = acc[e];
  __syncthreads();
  float M = kNegInf;
#pragma unroll
  for (int w = 0; w < NW; ++w) M = fmaxf(M, ml_s[w][0]);
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float lt = 0.f, o = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = ml_s[w][0] == kNegInf ? 0.f : fast_exp2(ml_s[w][0] - M);
        lt += f * ml_s[w][1];
        o += f * acc_s[w][d];
      }
    }
    p.o[b * p.o_sb + tqi * p.o_st + h * p.o_sh + split * p.o_ss + d] = lt > 0.f ? vs * (o / lt) : 0.f;
    if (d == 0 && p.lse != nullptr)
      p.lse[b * p.l_sb + tqi * p.l_st + h * p.l_sh + split * p.l_ss] =
          lt > 0.f ? (M + __log2f(lt)) * kLn2 : kNegInf;
  }
  if (p.late_wait) pdl_wait_prerequisites();   // complete only after the preceding grid
}

}  // namespace fd
