// Internal host/device declarations of the decode-attention library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fd {

// Device error word bits.
constexpr unsigned int FD_DEVERR_BOUNDS = 1u;   // a length outside [0, capacity]
constexpr unsigned int FD_DEVERR_TIMEOUT = 2u;  // a bounded wait gave up

// Longest any on-device wait may spin before giving up (1 s).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

constexpr int kSplitAlign = 64;   // FD_SPLIT_ALIGN
constexpr int kMaxSplits = 256;   // FD_MAX_SPLITS

// Arguments of the split-partial kernels (one CTA per (split, kv head, b)).
// Cache element kinds of the split kernels.
constexpr int kKvF32 = 0;
constexpr int kKvBf16 = 1;
constexpr int kKvI8 = 2;
constexpr int kKvE4m3 = 3;

struct SplitParams {
  const void* q;              // [B, Hq, D], or [B, tq, Hq, D] with tq > 1
  int64_t q_sb, q_sh;         // element strides
  int64_t q_st;               // stride over the query tokens (tq > 1)
  int tq;                     // new query positions per sequence (1: plain decode);
                              // query t sees keys j < len - tq + t + 1
  int q_bf16;                 // 1: bf16, 0: fp32
  const void* k;              // [B, Lcap, Hkv, D] (generic kernel only; the TMA
  const void* v;              //  kernel reads through tensor maps)
  int64_t k_sb, k_sl, k_sh;
  int64_t v_sb, v_sl, v_sh;
  const int32_t* seqlens;     // [B] or nullptr (= Lcap)
  int B, Hq, Hkv, G, Lcap, ns;
  float scale_log2;           // scale * log2(e): scores are kept in base 2
  float* o;                   // partial (or final, ns == 1) output, fp32
  int64_t o_sb, o_sh, o_ss;   // strides over (b, q head, split)
  int64_t o_st, l_st;         // strides over the query tokens (tq > 1)
  int o_vec4;                 // 1: o and its strides allow 16-byte stores
  float* lse;                 // natural-log lse, or nullptr
  int64_t l_sb, l_sh, l_ss;
  int kv_batch_broadcast;     // 1: every sequence reads kv batch row 0
  // 1: do not wait for the preceding grid before reading the inputs, only
  // before exiting.  Set only when the preceding kernel is one of this
  // library's, which triggers its dependents after its own launch wait (so
  // every earlier grid has finished) and writes nothing this kernel reads:
  // the split kernel then overlaps it, and still completes after it.
  int late_wait;
  // 1: q rows are 16-byte aligned (base and strides), so the tensor-core
  // kernel stages its query block through shared memory with vector loads.
  int q_vec16;
  // Element type of the cache (kKvF32, kKvBf16, kKvI8, kKvE4m3); the 8-bit
  // kinds carry one dequantisation scale per kv head for K and for V.
  int kv_kind;
  const float* k_scale;       // [Hkv] device, 8-bit kinds only
  const float* v_scale;
  // Paged cache (block_table != nullptr): k / v are [num_pages, page_size,
  // Hkv, D]; token j of sequence b is row j % page_size of page
  // block_table[b * bt_stride + j / page_size].  The TMA kernels load
  // page_rows = min(64, page_size) rows per box.
  const int32_t* block_table;
  int64_t bt_stride;
  int page_size, num_pages, page_rows;
  // Limit of the tensor-core split kernel's pipeline waits (its final drain
  // of copies in flight always allows kWaitLimitNs), and a delay its
  // producer thread spins before issuing its first copies: kWaitLimitNs and
  // 0 except under the test knobs that make a wait run out on purpose
  // (FD_TEST_WAIT_LIMIT_NS, FD_TEST_PRODUCER_DELAY_NS).
  unsigned long long wait_limit_ns;
  unsigned int producer_delay_ns;
};

// Longest producer delay the test knob may ask for (10 ms).
constexpr unsigned int kMaxProducerDelayNs = 10000000u;

// Arguments of the log-sum-exp combine kernel.
struct CombineParams {
  const float* part_o;        // rows x splits x D
  int64_t po_r1, po_r2, po_s; // row index r = (r1 * Rm + rm) * R2 + r2 ; split stride
  const float* part_lse;
  int64_t pl_r1, pl_r2, pl_s;
  float* out;
  int64_t out_r1, out_r2;
  float* lse;                 // may be nullptr
  int64_t lse_r1, lse_r2;
  int R1, R2, S, D;
  int Rm;                     // middle row dimension (query tokens), 1 if none
  int64_t po_rm, pl_rm, out_rm, lse_rm;
};

// Arguments of the bifurcated context kernel (one CTA per (128-row M-tile,
// context split, kv head)); rows of kv head g are (sample, head-in-group)
// pairs, row m = sample * G + r.
struct BifCtxParams {
  const uint16_t* q;          // [n, Hq, D] bf16, rows 16-byte aligned
  int64_t q_sb, q_sh;         // element strides over (sample, q head)
  int n, Hq, Hkv, G, Lc, ns;
  int rows;                   // n * G
  float scale_log2;           // |scale| * log2(e)
  int negate_q;               // 1: scale < 0, the kernel negates Q as it loads it
  float* o;                   // partial outputs, fp32
  int64_t o_sb, o_sh, o_ss;   // strides over (sample, q head, split)
  float* lse;                 // natural-log partial lse
  int64_t l_sb, l_sh, l_ss;
  // Decode part folded into this kernel (fold = 1; needs G >= 16, so a
  // 128-row query tile spans at most 9 samples).  A query tile's work is
  // then one list of 128-token tiles, the context's followed by the decode
  // tiles of the tile's samples (dec_lens[s] tokens each, nullptr: all Ld;
  // each masked to the rows of its own sample), cut into ns equal runs, one
  // per split.
  int fold;
  const int32_t* dec_lens;
  int Ld;
  // 1: the query tile arrives by one TMA load (tensor map over q as
  // [n][Hkv][G][D], a box of min(G, 128) heads x max(1, 128 / G) samples;
  // G divides 128 or 128 divides G) into shared memory and is copied into
  // tensor memory by the MMA warp (tcgen05.cp); 0: each softmax thread
  // loads its query row from global memory into tensor memory.
  int q_tma;
  // 1: the 128 partial rows of a CTA leave by TMA tensor stores (tensor map
  // over the partial outputs as [S][n][Hkv][G][D], same box rule as the
  // query map); 0: each softmax thread writes its half row.
  int o_tma;
};

// Most samples a 128-row query tile can span when the decode part is folded.
constexpr int kBifFoldMaxSamples = 9;

// Tokens per tile, and 128-row query tiles per CTA, of the bifurcated
// context kernel.
constexpr int kBifTileTokens = 128;
constexpr int kBifQueryTiles = 1;

// Host launchers (return a cudaError_t from the launch).  `pdl` launches
// with programmatic stream serialisation (the kernel may start while the
// previous kernel on the stream drains; it waits before touching memory).
cudaError_t launch_split_tma(const SplitParams& p, const CUtensorMap& tmK,
                             const CUtensorMap& tmV, int D, int G, cudaStream_t st,
                             bool* launched, bool pdl);
cudaError_t launch_split_mma(const SplitParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             int G, int variant, cudaStream_t st, bool* launched, bool pdl);
int mma_tile_tokens(int variant, int kv_kind);
cudaError_t launch_split_generic(const SplitParams& p, int D, cudaStream_t st, bool pdl);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_bif_ctx(const BifCtxParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const CUtensorMap& tmKd, const CUtensorMap& tmVd,
                           const CUtensorMap& tmQ, const CUtensorMap& tmO, int mtiles,
                           cudaStream_t st, bool pdl);

// Tile height (tokens) of the TMA split kernel; the tensor-map box uses it.
constexpr int kSplitTileTokens = 64;


}  // namespace fd
