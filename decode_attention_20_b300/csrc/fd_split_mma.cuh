// Split-KV partial kernel for grouped-query attention on the tensor cores.
//
// Same contract as split_tma_kernel (fd_split.cuh): one CTA per (split i,
// kv head g, sequence b) writes the normalised partial output and the
// natural-log log-sum-exp of its token range for every query head of the
// group.  Source: Flash-Decoding page ("What is Flash-Decoding and when does
// it speed up LLMs?"), section "Why decoding needs different scheduling";
// online softmax after "How does Flash Attention reduce memory traffic during
// local inference?", section on online softmax.
//
// Why tensor cores here: with G query heads sharing every K/V element, the
// per-token work is a real contraction (G x D scores, G x D accumulations).
// On CUDA cores at G = 8 the FMA pipe alone needs about as long as HBM takes
// to deliver the cache (profiled: ~45% FMA-pipe activity over an 83 us
// launch at 64K tokens), so the kernel cannot reach the memory roofline.
// Warp-level mma.sync m16n8k16 (bf16 in, fp32 accumulate) does the same
// arithmetic in ~1/16 of the instructions, leaving the kernel HBM-bound.
//
// Layout of the work (per warp, per 16-token block, per 8-head n-tile):
//   S^T[16 tok x 8 heads]  = K[16 x 128] . Q^T[128 x 8]    8 mma (k = 16 dims)
//   online softmax on the accumulator fragment (each lane: 2 tokens x 2
//   heads; per-head block max over the 8 lanes sharing lane % 4)
//   P^T -> bf16, transposed in registers (movmatrix) into B operands
//   O^T[128 dims x 8 heads] += V^T[128 x 16 tok] . P^T[16 tok x 8 heads]
//                                                   8 mma (k = 16 tokens)
// K and V tiles arrive by TMA with the 128-byte swizzle (two 64-column boxes
// per tile), so every ldmatrix is bank-conflict free.
//
// With a bf16 cache the probabilities enter the PV product as bf16 (8
// significant bits, one MMA); the running sum l stays in fp32, so the
// log-sum-exp carries no rounding of P.
//
// 8-bit caches (int8 or e4m3 codes with one scale per kv head for K and for
// V): one 128-byte box per row, codes turned into exact f16 values in
// registers, f16 mma.sync with the queries in f16 (per-head power-of-two
// rescale); the K scale joins the score scale and the V scale the final
// normalisation.  Half the bytes per token of the bf16 cache.  P enters the
// PV product as one f16 value (11 significant bits), one MMA.
#pragma once

#include <type_traits>

#include "fd_split.cuh"

namespace fd {

// --------------------------------------------------------- warp MMA helpers

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + C (fp32)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// (lo, hi) floats -> bf16x2 with round-to-nearest-even; lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + C (fp32)
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (lo, hi) floats -> f16x2 with round-to-nearest-even; lo in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t u4_word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Four 8-bit cache codes in a word -> two f16x2 values, exactly: bytes 0, 1
// into `lo` (byte 0 in the low half), bytes 2, 3 into `hi`.
//  - int8 (KVQ 1): the word arrives with every byte's sign bit flipped (code
//    + 128 as an unsigned byte u); the f16 with bit pattern 0x6400 | u is
//    1024 + u = code + kI8Bias (integers below 2048 are exact in f16).  The
//    bias is left in: in QK^T it adds kI8Bias * sum_d q_d to every score of
//    a head, which the score computation subtracts again, and in PV it adds
//    kI8Bias * sum_j p_j, which the epilogue removes with the normaliser.
//  - e4m3 (KVQ 2): every e4m3 value is exactly representable in f16 (3 of
//    f16's 10 mantissa bits, exponents 2^-9 .. 2^8 inside f16's range); the
//    hardware converts two at a time.
constexpr float kI8Bias = 1152.f;

template <int KVQ>
__device__ __forceinline__ void q8_to_f16x2x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
  if constexpr (KVQ == 1) {
    lo = __byte_perm(x, 0x64646464u, 0x5140);
    hi = __byte_perm(x, 0x64646464u, 0x7362);
  } else {
    // Each half of the word is one e4m3 pair; the conversion writes the
    // f16 pair straight into a 32-bit register (element order kept).
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(x));
  }
}

// A 16-byte shared-memory load of 8-bit codes, prepared for q8_to_f16x2x2.
template <int KVQ>
__device__ __forceinline__ uint4 lds128_q8(uint32_t addr) {
  uint4 v = lds128(addr);
  if constexpr (KVQ == 1) {
    v.x ^= 0x80808080u;
    v.y ^= 0x80808080u;
    v.z ^= 0x80808080u;
    v.w ^= 0x80808080u;
  }
  return v;
}

// Byte offset of (row, 16-byte chunk) inside a 128-byte-swizzled box whose
// rows are 128 bytes (the TMA SWIZZLE_128B pattern on a 1024-byte aligned
// base: chunk index XOR row % 8).
__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
  return uint32_t(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// ------------------------------------------------------------------ config

template <int KVQ_, int NT_, int WN_, int W_, int T_, int NSTAGE_>
struct MmaCfg {
  static constexpr int KVQ = KVQ_;             // cache: 0 bf16, 1 int8, 2 e4m3
  static constexpr bool Q8 = KVQ_ != 0;
  static constexpr int NT = NT_;               // 8-head n-tiles per kv head (ceil(G/8))
  static constexpr int WN = WN_;               // warps sharing a token block (split n-tiles)
  static constexpr int NPW = NT / WN;          // n-tiles per warp
  static constexpr int W = W_;                 // warps per CTA
  static constexpr int WT = W / WN;            // token groups
  static constexpr int T = T_;                 // tokens per tile
  static constexpr int NSTAGE = NSTAGE_;
  static constexpr int D = 128;
  static constexpr int THREADS = W * 32;
  static constexpr int BLK = T / 16;           // 16-token blocks per tile
  static constexpr int BPW = BLK / WT;         // blocks per warp per tile
  // One swizzled box: [T][64] bf16, or [T][128] 8-bit codes; a stage holds
  // K lo, K hi, V lo, V hi (bf16) or K, V (8-bit).
  static constexpr int HALF_BYTES = T * 128;
  static constexpr int STAGE_BYTES = (Q8 ? 2 : 4) * HALF_BYTES;
  static constexpr int RING_BYTES = NSTAGE * STAGE_BYTES;
  static constexpr int GP = NT * 8;            // padded heads
  // Query staging (bf16 queries, up to 32 rows): rows of D bf16 padded by 16
  // bytes so that the fragment reads of 8 rows hit distinct banks.
  static constexpr bool STAGE_Q = GP <= 32;
  static constexpr int QROW_BYTES = D * 2 + 16;
  static constexpr int OFF_Q = ((RING_BYTES + 2 * NSTAGE * 8 + 16) + 127) / 128 * 128;
  static constexpr int Q_BYTES = STAGE_Q ? GP * QROW_BYTES : 0;
  static constexpr int SMEM_BYTES = 1024 + OFF_Q + Q_BYTES;
  static_assert(NT % WN == 0, "n-tiles split evenly over warps");
  static_assert(W % WN == 0 && BLK % WT == 0 && BPW >= 1, "blocks split evenly over warps");
  // Epilogue accumulator rows: D + 4 floats apart (bank-conflict free
  // stores for the bf16 fragment layout, 2-way with the 8-bit one's swizzle).
  static constexpr int AS = D + 4;
  static_assert(WT * GP * 2 * 4 + WT * GP * AS * 4 + (WT + 1) * GP * 4 <= RING_BYTES,
                "epilogue fits the ring");
  static_assert(Q_BYTES == 0 || OFF_Q % 16 == 0, "staged query rows are 16-byte aligned");
  static_assert(HALF_BYTES % 1024 == 0, "swizzled boxes need 1024-byte alignment");
};

template <int KVQ, int NT, int WN, int W, int T, int NSTAGE>
__global__ void __launch_bounds__(W * 32, (KVQ != 0 && W == 8) ? 2 : 1)
    split_mma_kernel(const __grid_constant__ SplitParams p,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV) {
  using C = MmaCfg<KVQ, NT, WN, W, T, NSTAGE>;
  constexpr int NPW = C::NPW;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::RING_BYTES);
  uint64_t* empty_bar = full_bar + C::NSTAGE;
  int* abort_s = reinterpret_cast<int*>(empty_bar + C::NSTAGE);

  const int split = blockIdx.x;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wn = warp % WN;                    // n-tile group
  const int wt = warp / WN;                    // token group

  // Set-up that reads no global memory (the ring's barriers, the tensor maps
  // in parameter space) runs before the launch wait, so it overlaps the tail
  // of the preceding kernel on the stream.
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], W);
    }
    *abort_s = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (!p.late_wait) pdl_wait_prerequisites();   // launched with PDL: no global memory access before this

  const int len = resolve_len(p.seqlens, b, p.Lcap);
  int begin, end;
  split_range(len, p.ns, split, begin, end);
  const int ntiles = (end - begin + C::T - 1) / C::T;
  const int kvb = p.kv_batch_broadcast ? 0 : b;
  // 8-bit caches: the kv head's scales, loaded now so that their latency
  // hides behind the ring fill (the query set-up and the epilogue use them).
  float ks_g = 1.f, vs_g = 1.f;
  if constexpr (C::Q8) {
    ks_g = p.k_scale[g];
    vs_g = p.v_scale[g];
  }

  // Rows of the kv head: (query token t, head in group hl), row = t * G + hl
  // (plain decode: tq = 1, rows = heads).
  const int G = p.G;
  const int TQ = p.tq > 1 ? p.tq : 1;
  const int R = TQ * G;
  // ---- bf16 query block: one coalesced 16-byte load per chunk per thread,
  // issued before the ring's first copies (scalar fragment loads issued
  // after them queued behind every CTA's ring fill for several
  // microseconds while the full ring waited); stored to shared memory
  // after the copies are issued.
  constexpr int QCH = C::GP * (C::D / 8);                    // 16-byte chunks
  constexpr int QPT = C::STAGE_Q ? (QCH + C::THREADS - 1) / C::THREADS : 1;
  const bool stage_q = C::STAGE_Q && p.q_bf16 && p.q_vec16;
  uint4 qv16[QPT];
  if (stage_q) {
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
      const int c = threadIdx.x + k * C::THREADS;
      const int r = c / (C::D / 8);
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (c < QCH && r < R) {
        const int tqi = r / G;
        const int64_t o = b * p.q_sb + tqi * p.q_st + (g * G + r - tqi * G) * p.q_sh +
                          (c - r * (C::D / 8)) * 8;
        x = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.q) + o);
      }
      qv16[k] = x;
    }
  }

  __syncthreads();

  uint64_t policy = 0;
  int issued = 0;
  // Warp 0 as a whole issues the copies (warp-uniform operands; one elected
  // lane issues each instruction): measured on B300, a copy issued by one
  // lane of a divergent branch costs its warp far more issue time.
  auto issue = [&](int t) {
    const int s = t % C::NSTAGE;
    unsigned char* stage = smem + s * C::STAGE_BYTES;
    mbar_arrive_expect_tx_w(&full_bar[s], C::STAGE_BYTES);
    const int tok = begin + t * C::T;
    if (p.block_table == nullptr) {
      if constexpr (C::Q8) {
        tma_load_4d_w(stage, &tmK, &full_bar[s], 0, g, tok, kvb, policy);
        tma_load_4d_w(stage + C::HALF_BYTES, &tmV, &full_bar[s], 0, g, tok, kvb, policy);
      } else {
        tma_load_4d_w(stage, &tmK, &full_bar[s], 0, g, tok, kvb, policy);
        tma_load_4d_w(stage + C::HALF_BYTES, &tmK, &full_bar[s], 64, g, tok, kvb, policy);
        tma_load_4d_w(stage + 2 * C::HALF_BYTES, &tmV, &full_bar[s], 0, g, tok, kvb, policy);
        tma_load_4d_w(stage + 3 * C::HALF_BYTES, &tmV, &full_bar[s], 64, g, tok, kvb, policy);
      }
    } else {
      // Paged cache: the tile is page_rows-row segments, each inside one page
      // (tiles start on multiples of 64 tokens; page_rows = min(64, page
      // size) divides both).  Segments past the split's end load page -1:
      // out of range, so the copy fills zeros (and still counts its bytes).
      const int nseg = C::T / p.page_rows;
      for (int sg = 0; sg < nseg; ++sg) {
        const int tk = tok + sg * p.page_rows;
        const int pid = tk < end ? page_of(p, b, tk, -1) : -1;
        const int off = tk % p.page_size;
        const int so = sg * p.page_rows * 128;
        if constexpr (C::Q8) {
          tma_load_4d_w(stage + so, &tmK, &full_bar[s], 0, g, off, pid, policy);
          tma_load_4d_w(stage + C::HALF_BYTES + so, &tmV, &full_bar[s], 0, g, off, pid, policy);
        } else {
          tma_load_4d_w(stage + so, &tmK, &full_bar[s], 0, g, off, pid, policy);
          tma_load_4d_w(stage + C::HALF_BYTES + so, &tmK, &full_bar[s], 64, g, off, pid, policy);
          tma_load_4d_w(stage + 2 * C::HALF_BYTES + so, &tmV, &full_bar[s], 0, g, off, pid, policy);
          tma_load_4d_w(stage + 3 * C::HALF_BYTES + so, &tmV, &full_bar[s], 64, g, off, pid, policy);
        }
      }
    }
  };
  // Warp 0 fills the ring.  (A test delay moves the fill after the query
  // staging and spins first, so that the other warps' first waits run out.)
  auto fill_ring = [&]() {
    policy = l2_policy_evict_first();
    for (int t = 0; t < C::NSTAGE && t < ntiles; ++t) {
      issue(t);
      ++issued;
    }
  };
  if (warp == 0 && p.producer_delay_ns == 0) fill_ring();

  // ---- raw query values (fp32 bit patterns), turned into MMA fragments below.
  uint32_t qraw[NPW][8][4];
  unsigned char* q_s = smem + C::OFF_Q;
  if (stage_q) {
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
      const int c = threadIdx.x + k * C::THREADS;
      if (c < QCH) {
        const int r = c / (C::D / 8);
        *reinterpret_cast<uint4*>(q_s + r * C::QROW_BYTES + (c - r * (C::D / 8)) * 16) = qv16[k];
      }
    }
    __syncthreads();
    // Word pairs: bf16 cache dims (d0, d0+1) and (d0+8, d0+9); 8-bit cache
    // dims (d0, d0+1) and (d0+2, d0+3) (the fragment orders below).
#pragma unroll
    for (int j = 0; j < NPW; ++j) {
      const int r = (wn * NPW + j) * 8 + (lane >> 2);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int d0 = C::Q8 ? 16 * (2 * (lane & 3) + (ks >> 2)) + 4 * (ks & 3)
                             : ks * 16 + 2 * (lane & 3);
        const uint32_t* rowp = reinterpret_cast<const uint32_t*>(q_s + r * C::QROW_BYTES);
        const uint32_t w0 = rowp[d0 >> 1];
        const uint32_t w1 = rowp[(d0 + (C::Q8 ? 2 : 8)) >> 1];
        qraw[j][ks][0] = w0 << 16;
        qraw[j][ks][1] = w0 & 0xffff0000u;
        qraw[j][ks][2] = w1 << 16;
        qraw[j][ks][3] = w1 & 0xffff0000u;
      }
    }
  }
  // One uniform branch on the query type outside the unrolled loads (a
  // per-element select here measured 2-4 us slower per launch).
  auto load_q = [&](auto as_bits) {
#pragma unroll
    for (int j = 0; j < NPW; ++j) {
      const int r = (wn * NPW + j) * 8 + (lane >> 2);         // row of this lane's query
      const bool real = r < R;
      const int tqi = real ? r / G : 0;
      const int h = g * G + (real ? r - tqi * G : 0);
      const int64_t base = b * p.q_sb + tqi * p.q_st + h * p.q_sh;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        // bf16 cache: dims ks*16 + 2(lane%4) + {0, 1, 8, 9}; 8-bit cache: dims
        // 16(2(lane%4) + ks/4) + 4(ks%4) + {0, 1, 2, 3} (see the fragments below)
        const int d0 = C::Q8 ? 16 * (2 * (lane & 3) + (ks >> 2)) + 4 * (ks & 3)
                             : ks * 16 + 2 * (lane & 3);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int d = C::Q8 ? d0 + i : d0 + (i & 1) + (i >> 1) * 8;
          qraw[j][ks][i] = real ? as_bits(base + d) : 0u;     // fp32 bit pattern
        }
      }
    }
  };
  if (stage_q) {
  } else if (C::Q8 && !p.q_bf16) {
    load_q([&](int64_t o) { return __float_as_uint(reinterpret_cast<const float*>(p.q)[o]); });
  } else {
    load_q([&](int64_t o) { return uint32_t(reinterpret_cast<const uint16_t*>(p.q)[o]) << 16; });
  }

  // ---- query fragments (B operand of S^T = K . Q^T): B[k = dim][n = head]
  // lane holds dims 2(lane%4)+{0,1} and +8 of head (lane/4) of each n-tile.
  uint32_t qf[NPW][8][2];
  // 8-bit caches: per-lane score multipliers of heads hA = 2(lane%4) and
  // hB = hA + 1 of each n-tile (score scale x K scale x 2^-e of the head's
  // query rescale, below).
  float sl2h[NPW][2];
  float shift[NPW][2];   // int8: sl2h * kI8Bias * sum_d q_d (f16 values) per head
  if constexpr (!C::Q8) {
    // bf16 queries: the top halves of the fp32 patterns are the bf16 values.
#pragma unroll
    for (int j = 0; j < NPW; ++j) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qf[j][ks][0] = (qraw[j][ks][0] >> 16) | (qraw[j][ks][1] & 0xffff0000u);
        qf[j][ks][1] = (qraw[j][ks][2] >> 16) | (qraw[j][ks][3] & 0xffff0000u);
      }
      sl2h[j][0] = sl2h[j][1] = p.scale_log2;
      shift[j][0] = shift[j][1] = 0.f;
    }
  } else {
    // The contraction over head dims may take the dims in any order, as long
    // as the K and Q fragments agree.  Lane (n = lane/4, t = lane%4) reads
    // whole words of a K row, so in k-step ks its k positions 2t, 2t+1 are
    // dims 16c + 4w + {0, 1} and positions 2t+8, 2t+9 dims 16c + 4w + {2, 3},
    // with c = 2t + ks/4 (the row's 16-byte chunk) and w = ks % 4 (its word).
    // The queries of each head are scaled by 2^e (e from the head's largest
    // |q|, so that it lands in [2^14, 2^15)) and rounded to f16; the score
    // multiplier takes 2^-e back.
#pragma unroll
    for (int j = 0; j < NPW; ++j) {
      float qv[8][4];
      float amax = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          qv[ks][i] = __uint_as_float(qraw[j][ks][i]);
          amax = fmaxf(amax, fabsf(qv[ks][i]));
        }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const int E = int((__float_as_uint(amax) >> 23) & 0xffu);
      const int e = (E == 0) ? 0 : min(100, max(-100, 141 - E));
      const float up = __uint_as_float(uint32_t(127 + e) << 23);       // 2^e
      const float down = __uint_as_float(uint32_t(127 - e) << 23);     // 2^-e
      float qsum = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qf[j][ks][0] = pack_f16x2(qv[ks][0] * up, qv[ks][1] * up);
        qf[j][ks][1] = pack_f16x2(qv[ks][2] * up, qv[ks][3] * up);
        if constexpr (KVQ == 1) {
          const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&qf[j][ks][0]));
          const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&qf[j][ks][1]));
          qsum += (a.x + a.y) + (c.x + c.y);
        }
      }
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
      const float mine = p.scale_log2 * ks_g * down;                  // head lane/4
      const float mshift = (KVQ == 1) ? mine * (kI8Bias * qsum) : 0.f;
      sl2h[j][0] = __shfl_sync(0xffffffffu, mine, 8 * (lane & 3));     // head 2(lane%4)
      sl2h[j][1] = __shfl_sync(0xffffffffu, mine, 8 * (lane & 3) + 4); // head 2(lane%4)+1
      shift[j][0] = __shfl_sync(0xffffffffu, mshift, 8 * (lane & 3));
      shift[j][1] = __shfl_sync(0xffffffffu, mshift, 8 * (lane & 3) + 4);
    }
  }

  float acc[NPW][8][4];
  float m_run[NPW][2], l_run[NPW][2];
#pragma unroll
  for (int j = 0; j < NPW; ++j) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][mt][e] = 0.f;
    m_run[j][0] = m_run[j][1] = kNegInf;
    l_run[j][0] = l_run[j][1] = 0.f;
  }
  const float sl2 = p.scale_log2;
  const int r8 = lane & 7;
  // Causal limit of this lane's two score columns (rows hA, hB of each
  // n-tile): query token t sees tokens j < len - tq + t + 1.  For tq = 1 the
  // limit is len, which the split range already enforces.
  int limA[NPW], limB[NPW];
#pragma unroll
  for (int j = 0; j < NPW; ++j) {
    const int rA = (wn * NPW + j) * 8 + 2 * (lane & 3);
    limA[j] = len - TQ + min(rA, R - 1) / G + 1;
    limB[j] = len - TQ + min(rA + 1, R - 1) / G + 1;
  }

  if (warp == 0 && p.producer_delay_ns != 0) {
    const uint64_t t0 = globaltimer_ns();
    while (__any_sync(0xffffffffu, globaltimer_ns() - t0 < p.producer_delay_ns)) {
    }
    fill_ring();
  }

  for (int t = 0; t < ntiles; ++t) {
    const int s = t % C::NSTAGE;
    // Warp-uniform: a lane must not run on into the warp-wide MMAs and
    // shuffles of a tile that another lane of its warp has given up on.
    const bool got = mbar_wait_or_abort(&full_bar[s], (t / C::NSTAGE) & 1, abort_s, p.wait_limit_ns);
    if (!__all_sync(0xffffffffu, got)) break;
    const uint32_t kbase = smem_u32(smem + s * C::STAGE_BYTES);
    const uint32_t vbase = kbase + (C::Q8 ? 1 : 2) * C::HALF_BYTES;   // V box(es) after K
    const int nvalid = min(C::T, end - (begin + t * C::T));
#pragma unroll 1
    for (int bb = 0; bb < C::BPW; ++bb) {
      const int row0 = (bb * C::WT + wt) * 16;       // first token row of this block
      // ---- S^T = K . Q^T
      // Two accumulators per n-tile (even and odd head-dim steps) halve the
      // chain of dependent MMAs; they are summed once below.
      float sacc2[NPW][2][4];
#pragma unroll
      for (int j = 0; j < NPW; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc2[j][0][e] = sacc2[j][1][e] = 0.f;
      if constexpr (!C::Q8) {
        const int arow = row0 + r8 + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const int col = ks * 16 + (lane >> 4) * 8;           // 0..127
          const uint32_t addr =
              kbase + (col >> 6) * C::HALF_BYTES + swz128(arow, (col & 63) >> 3);
          uint32_t a0, a1, a2, a3;
          ldsm_x4(addr, a0, a1, a2, a3);
#pragma unroll
          for (int j = 0; j < NPW; ++j)
            mma_bf16_16816(sacc2[j][ks & 1], a0, a1, a2, a3, qf[j][ks][0], qf[j][ks][1]);
        }
      } else {
        // A = K rows row0 + lane/4 (a0, a2) and + 8 (a1, a3); chunks 2t and
        // 2t + 1 of each (the dims order of the query fragments).  Rows of
        // one parity read even chunks, the others odd ones after the
        // swizzle, so the 16-byte loads are bank-conflict free.
        const int ra = row0 + (lane >> 2);
        const int c0 = 2 * (lane & 3);
        const uint4 kA0 = lds128_q8<KVQ>(kbase + swz128(ra, c0));
        const uint4 kA1 = lds128_q8<KVQ>(kbase + swz128(ra, c0 + 1));
        const uint4 kB0 = lds128_q8<KVQ>(kbase + swz128(ra + 8, c0));
        const uint4 kB1 = lds128_q8<KVQ>(kbase + swz128(ra + 8, c0 + 1));
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t a0, a1, a2, a3;
          q8_to_f16x2x2<KVQ>(u4_word(ks < 4 ? kA0 : kA1, ks & 3), a0, a2);
          q8_to_f16x2x2<KVQ>(u4_word(ks < 4 ? kB0 : kB1, ks & 3), a1, a3);
#pragma unroll
          for (int j = 0; j < NPW; ++j)
            mma_f16_16816(sacc2[j][ks & 1], a0, a1, a2, a3, qf[j][ks][0], qf[j][ks][1]);
        }
      }
      float sacc[NPW][4];
#pragma unroll
      for (int j = 0; j < NPW; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[j][e] = sacc2[j][0][e] + sacc2[j][1][e];
      // ---- online softmax; lane holds tokens tA = lane/4, tB = tA + 8 and
      // heads hA = 2(lane%4), hB = hA + 1 of each n-tile
      const int tokA = row0 + (lane >> 2);
      const bool vA = tokA < nvalid;
      const bool vB = tokA + 8 < nvalid;
      const int absA = begin + t * C::T + tokA;                  // absolute token index
      uint32_t pb[NPW][2];
      bool moved = false;
      float alpha[NPW][2];
#pragma unroll
      for (int j = 0; j < NPW; ++j) {
        const float f0 = C::Q8 ? sl2h[j][0] : sl2;
        const float f1 = C::Q8 ? sl2h[j][1] : sl2;
        // (int8: one fused multiply-add also removes the code bias's share
        // of the score, exactly rounded once.)
        float sA0 = (vA && absA < limA[j]) ? fmaf(sacc[j][0], f0, -shift[j][0]) : kNegInf;      // (tA, hA)
        float sA1 = (vA && absA < limB[j]) ? fmaf(sacc[j][1], f1, -shift[j][1]) : kNegInf;      // (tA, hB)
        float sB0 = (vB && absA + 8 < limA[j]) ? fmaf(sacc[j][2], f0, -shift[j][0]) : kNegInf;  // (tB, hA)
        float sB1 = (vB && absA + 8 < limB[j]) ? fmaf(sacc[j][3], f1, -shift[j][1]) : kNegInf;  // (tB, hB)
        float mx0 = fmaxf(sA0, sB0), mx1 = fmaxf(sA1, sB1);
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        // Lazy rescaling (threshold 8 in base 2): probabilities stay <= 256.
        const float mn0 = (mx0 > m_run[j][0] + 8.f) ? mx0 : m_run[j][0];
        const float mn1 = (mx1 > m_run[j][1] + 8.f) ? mx1 : m_run[j][1];
        alpha[j][0] = (mn0 == m_run[j][0]) ? 1.f : fast_exp2(m_run[j][0] - mn0);
        alpha[j][1] = (mn1 == m_run[j][1]) ? 1.f : fast_exp2(m_run[j][1] - mn1);
        moved |= (alpha[j][0] != 1.f) | (alpha[j][1] != 1.f);
        m_run[j][0] = mn0;
        m_run[j][1] = mn1;
        const float pA0 = (mn0 == kNegInf) ? 0.f : fast_exp2(sA0 - mn0);
        const float pB0 = (mn0 == kNegInf) ? 0.f : fast_exp2(sB0 - mn0);
        const float pA1 = (mn1 == kNegInf) ? 0.f : fast_exp2(sA1 - mn1);
        const float pB1 = (mn1 == kNegInf) ? 0.f : fast_exp2(sB1 - mn1);
        // Probabilities enter the PV product as bf16 (round to nearest even,
        // at most 2^-9 relative per p) and the running sum keeps the fp32
        // values, so the log-sum-exp carries no rounding of P.
        if constexpr (KVQ == 1) {
          // The normaliser sums the f16 probabilities the PV product uses,
          // so that the epilogue's bias removal is exact.
          const uint32_t XA = pack_f16x2(pA0, pA1);
          const uint32_t XB = pack_f16x2(pB0, pB1);
          const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&XA));
          const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&XB));
          l_run[j][0] = l_run[j][0] * alpha[j][0] + (a.x + c.x);
          l_run[j][1] = l_run[j][1] * alpha[j][1] + (a.y + c.y);
          pb[j][0] = movmatrix_trans(XA);
          pb[j][1] = movmatrix_trans(XB);
        } else {
          l_run[j][0] = l_run[j][0] * alpha[j][0] + (pA0 + pB0);
          l_run[j][1] = l_run[j][1] * alpha[j][1] + (pA1 + pB1);
        }
        if constexpr (!C::Q8) {
          const uint32_t XA = pack_bf16x2(pA0, pA1);      // token tA, heads hA hB
          const uint32_t XB = pack_bf16x2(pB0, pB1);      // token tB
          pb[j][0] = movmatrix_trans(XA);                 // B[k = tokens 0-7][n = head]
          pb[j][1] = movmatrix_trans(XB);                 // B[k = tokens 8-15][n = head]
        } else if constexpr (KVQ == 2) {
          // f16 keeps 11 significant bits of p (<= 256 under the lazy
          // rescale): one PV product suffices.
          pb[j][0] = movmatrix_trans(pack_f16x2(pA0, pA1));
          pb[j][1] = movmatrix_trans(pack_f16x2(pB0, pB1));
        }
      }
      if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
        for (int j = 0; j < NPW; ++j)
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            acc[j][mt][0] *= alpha[j][0];
            acc[j][mt][1] *= alpha[j][1];
            acc[j][mt][2] *= alpha[j][0];
            acc[j][mt][3] *= alpha[j][1];
          }
      }
      // ---- O^T += V^T . P^T   (A = V^T via transposing ldmatrix)
      {
        // In the last, partial tile, rows past the split may hold anything
        // (even NaN padding): clear this lane's V elements of those tokens
        // (low half = token 2(lane%4), high half = the next token), so
        // zero-probability rows contribute exactly zero.
        uint32_t keep01 = 0xffffffffu, keep23 = 0xffffffffu;
        if (nvalid < C::T) {
          const int tk = row0 + 2 * (lane & 3);
          keep01 = (tk < nvalid ? 0x0000ffffu : 0u) | (tk + 1 < nvalid ? 0xffff0000u : 0u);
          keep23 = (tk + 8 < nvalid ? 0x0000ffffu : 0u) | (tk + 9 < nvalid ? 0xffff0000u : 0u);
        }
        if constexpr (!C::Q8) {
          const int vrow = row0 + r8 + (lane >> 4) * 8;
          // Only the last, partial tile of a range clears its V elements (a
          // tile-uniform branch; full tiles spend nothing on it).
          auto pv = [&](auto clear) {
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              const int col = mt * 16 + ((lane >> 3) & 1) * 8;
              const uint32_t addr =
                  vbase + (col >> 6) * C::HALF_BYTES + swz128(vrow, (col & 63) >> 3);
              uint32_t a0, a1, a2, a3;
              ldsm_x4_trans(addr, a0, a1, a2, a3);
              if constexpr (decltype(clear)::value) {
                a0 &= keep01;
                a1 &= keep01;
                a2 &= keep23;
                a3 &= keep23;
              }
#pragma unroll
              for (int j = 0; j < NPW; ++j) mma_bf16_16816(acc[j][mt], a0, a1, a2, a3, pb[j][0], pb[j][1]);
            }
          };
          if (nvalid < C::T)
            pv(std::integral_constant<bool, true>{});
          else
            pv(std::integral_constant<bool, false>{});
        } else {
          // A = V^T with the dims reordered so that a lane reads whole
          // 16-byte chunks: lane (r = lane/4, t = lane%4) reads chunk r of
          // token rows 2t, 2t+1, 2t+8, 2t+9; row r of m-tile mt is dim
          // 16r + 2mt and row r + 8 is dim 16r + 2mt + 1.  A byte permute
          // pairs the two tokens of each f16x2 operand.  Row parities split
          // the even and odd chunks, so the loads are conflict free.
          const int vr = row0 + 2 * (lane & 3);
          const int ch = lane >> 2;
          const uint4 vA = lds128_q8<KVQ>(vbase + swz128(vr, ch));
          const uint4 vB = lds128_q8<KVQ>(vbase + swz128(vr + 1, ch));
          const uint4 vC = lds128_q8<KVQ>(vbase + swz128(vr + 8, ch));
          const uint4 vD = lds128_q8<KVQ>(vbase + swz128(vr + 9, ch));
          // e4m3 codes past the split may be NaN: the last, partial tile of
          // a range clears them after the conversion (a tile-uniform
          // branch, so full tiles spend nothing on it).
          auto pv = [&](auto clear) {
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
              const uint32_t iAB = __byte_perm(u4_word(vA, mt >> 1), u4_word(vB, mt >> 1), sel);
              const uint32_t iCD = __byte_perm(u4_word(vC, mt >> 1), u4_word(vD, mt >> 1), sel);
              uint32_t a0, a1, a2, a3;
              q8_to_f16x2x2<KVQ>(iAB, a0, a1);
              q8_to_f16x2x2<KVQ>(iCD, a2, a3);
              if constexpr (decltype(clear)::value) {
                a0 &= keep01;
                a1 &= keep01;
                a2 &= keep23;
                a3 &= keep23;
              }
#pragma unroll
              for (int j = 0; j < NPW; ++j) mma_f16_16816(acc[j][mt], a0, a1, a2, a3, pb[j][0], pb[j][1]);
            }
          };
          if (KVQ == 2 && nvalid < C::T)
            pv(std::integral_constant<bool, KVQ == 2>{});
          else
            pv(std::integral_constant<bool, false>{});
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[s]);
    if (warp == 0 && t >= 1 && issued < ntiles) {
      const int tp = t - 1;
      if (__all_sync(0xffffffffu, mbar_wait_or_abort(&empty_bar[tp % C::NSTAGE], (tp / C::NSTAGE) & 1,
                                                     abort_s, p.wait_limit_ns))) {
        issue(issued);
        ++issued;
      }
    }
  }
  if (threadIdx.x == 0) {
    const int first = issued > C::NSTAGE ? issued - C::NSTAGE : 0;
    for (int t = first; t < issued; ++t)
      mbar_wait_bounded(&full_bar[t % C::NSTAGE], (t / C::NSTAGE) & 1);
  }

  pdl_launch_dependents();
  __syncthreads();

  // ------------------------------------------------------------ epilogue
  // Sum l over the 8 lanes that share each head, then merge the token
  // groups' (m, l, acc) through shared memory (the ring is free now).
  float* ML_s = reinterpret_cast<float*>(smem);              // [WT][GP][2]
  float* ACC_s = ML_s + C::WT * C::GP * 2;                   // [WT][GP][AS]
  // Position of dim d in an accumulator row: the 8-bit fragments put the
  // lanes' dims 16 apart, so bits 2..4 are swizzled with d / 16 (float4
  // groups and even/odd pairs stay together).
  auto acc_col = [](int d) { return C::Q8 ? (d ^ (((d >> 4) & 7) << 2)) : d; };
#pragma unroll
  for (int j = 0; j < NPW; ++j) {
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      l_run[j][0] += __shfl_xor_sync(0xffffffffu, l_run[j][0], o);
      l_run[j][1] += __shfl_xor_sync(0xffffffffu, l_run[j][1], o);
    }
    const int hbase = (wn * NPW + j) * 8;
    if (lane < 4) {
      const int h0 = hbase + 2 * lane;
      ML_s[(wt * C::GP + h0) * 2 + 0] = m_run[j][0];
      ML_s[(wt * C::GP + h0) * 2 + 1] = l_run[j][0];
      ML_s[(wt * C::GP + h0 + 1) * 2 + 0] = m_run[j][1];
      ML_s[(wt * C::GP + h0 + 1) * 2 + 1] = l_run[j][1];
    }
    const int hA = hbase + 2 * (lane & 3);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      // Accumulator rows r = lane/4 and r + 8 of m-tile mt are dims
      // mt*16 + r and + 8 (bf16), or 16r + 2mt and 16r + 2mt + 1 (8-bit:
      // one 8-byte store per row).
      float* rowA = ACC_s + (wt * C::GP + hA) * C::AS;
      float* rowB = rowA + C::AS;
      if constexpr (C::Q8) {
        const int d = acc_col(16 * (lane >> 2) + 2 * mt);
        *reinterpret_cast<float2*>(rowA + d) = make_float2(acc[j][mt][0], acc[j][mt][2]);
        *reinterpret_cast<float2*>(rowB + d) = make_float2(acc[j][mt][1], acc[j][mt][3]);
      } else {
        const int d = mt * 16 + (lane >> 2);
        rowA[d] = acc[j][mt][0];
        rowB[d] = acc[j][mt][1];
        rowA[d + 8] = acc[j][mt][2];
        rowB[d + 8] = acc[j][mt][3];
      }
    }
  }
  __syncthreads();
  // Per head: the common max, each token group's weight 2^(m_w - M) / l_tot
  // (into SF_s) and the log-sum-exp; then every output element is a short
  // weighted sum over the token groups, four elements per thread at a time.
  float* SF_s = ACC_s + C::WT * C::GP * C::AS;               // [WT][GP]
  float* SB_s = SF_s + C::WT * C::GP;                         // [GP]
  for (int h = threadIdx.x; h < R; h += C::THREADS) {         // h: row (t * G + head)
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < C::WT; ++w) M = fmaxf(M, ML_s[(w * C::GP + h) * 2]);
    float lt = 0.f;
    float f[C::WT];
#pragma unroll
    for (int w = 0; w < C::WT; ++w) {
      const float ms = ML_s[(w * C::GP + h) * 2];
      f[w] = (ms == kNegInf) ? 0.f : fast_exp2(ms - M);
      lt += f[w] * ML_s[(w * C::GP + h) * 2 + 1];
    }
    // 8-bit caches: the kv head's V scale joins the normalisation; int8
    // subtracts the code bias (times the V scale) from the normalised sum.
    const float vsc = vs_g;
    const float inv = lt > 0.f ? vsc / lt : 0.f;
#pragma unroll
    for (int w = 0; w < C::WT; ++w) SF_s[w * C::GP + h] = f[w] * inv;
    SB_s[h] = (KVQ == 1 && lt > 0.f) ? vsc * kI8Bias : 0.f;
    const int tqi = TQ == 1 ? 0 : h / G;       // (a runtime division costs here)
    const int hq = g * G + (h - tqi * G);
    if (p.lse != nullptr)
      p.lse[b * p.l_sb + tqi * p.l_st + hq * p.l_sh + split * p.l_ss] =
          lt > 0.f ? (M + __log2f(lt)) * kLn2 : kNegInf;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < R * (C::D / 4); idx += C::THREADS) {
    const int h = idx / (C::D / 4);
    const int d = (idx - h * (C::D / 4)) * 4;
    const float bias = SB_s[h];
    float4 o = make_float4(-bias, -bias, -bias, -bias);
#pragma unroll
    for (int w = 0; w < C::WT; ++w) {
      const float sf = SF_s[w * C::GP + h];
      const float4 a = *reinterpret_cast<const float4*>(ACC_s + (w * C::GP + h) * C::AS + acc_col(d));
      o.x = fmaf(sf, a.x, o.x);
      o.y = fmaf(sf, a.y, o.y);
      o.z = fmaf(sf, a.z, o.z);
      o.w = fmaf(sf, a.w, o.w);
    }
    const int tqi = TQ == 1 ? 0 : h / G;
    const int hq = g * G + (h - tqi * G);
    float* dst = p.o + b * p.o_sb + tqi * p.o_st + hq * p.o_sh + split * p.o_ss + d;
    if (p.o_vec4) {
      *reinterpret_cast<float4*>(dst) = o;
    } else {
      dst[0] = o.x;
      dst[1] = o.y;
      dst[2] = o.z;
      dst[3] = o.w;
    }
  }
  if (p.late_wait) pdl_wait_prerequisites();   // complete only after the preceding grid
}

}  // namespace fd
