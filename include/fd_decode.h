/*
 * fd_decode.h — C ABI of the B300 (sm_103a) decode-attention library
 * (libfd_decode.so).
 *
 * Exact single-query decode attention over a long KV cache, computed two ways:
 *
 *  1. Split-KV ("Flash-Decoding"): the cached history of every (sequence,
 *     kv head) is cut into splits; independent CTAs each produce a partial
 *     output and its log-sum-exp; a separate log-sum-exp reduction merges the
 *     partials into the exact full-history result.
 *     Source: "What is Flash-Decoding and when does it speed up LLMs?"
 *     (slavadubrov.com), section "Why decoding needs different scheduling".
 *
 *  2. Bifurcated attention for single-context batch sampling: one context KV
 *     shared by n samples is read once for all of them as a GEMM, a second
 *     part covers each sample's own decode KV, and the two are merged exactly.
 *     Source: summary of "Bifurcated Attention for Single-Context Large-Batch
 *     Sampling" (linnk.ai), sections "Tiivistelmä" and "Tilastot".
 *
 * Definition computed (both entry points), for batch row b and query head h,
 * with G = Hq / Hkv and kv head g = h / G (contiguous GQA groups):
 *     s_j = scale * <q[b,h,:], K[b,j,g,:]>      for j < len_b
 *     O[b,h,:] = sum_j softmax(s)_j * V[b,j,g,:]
 *     LSE[b,h] = ln sum_j exp(s_j)              (natural log, scaled scores)
 * len_b == 0 gives O = 0 and LSE = -inf.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors travel as fd_tensor descriptors: a data pointer, a dtype, a rank
 *    and per-dimension shape and stride.  Strides are in ELEMENTS; the
 *    innermost stride must be 1.  All data pointers given to compute entry
 *    points are DEVICE pointers on the current CUDA device.
 *  - Ownership: the caller owns every tensor and the stream.  The library
 *    keeps no pointer after the call returns beyond the work it enqueued.
 *  - Asynchrony: compute calls only enqueue work on `stream` (a cudaStream_t,
 *    NULL = the legacy default stream) and return; outputs are valid once the
 *    stream reaches that point.
 *  - Errors: every call returns an fd_status.  Argument errors are detected on
 *    the host before anything is enqueued (nothing is launched, outputs are
 *    untouched).  fd_last_error() returns a thread-local message for the most
 *    recent failure on the calling thread.  Data errors that only the device
 *    can see (a seqlens entry outside [0, Lcap]) are clamped on the device and
 *    recorded in a device error word that fd_check_device_error() reports.
 *  - Workspace: calls that need scratch memory for partial results allocate
 *    it stream-ordered (cudaMallocAsync / cudaFreeAsync on `stream`), so
 *    calls on different streams or threads never share scratch.
 *  - Arithmetic: no step of the method is approximated; sums and the online
 *    softmax are fp32 and the partial results fp32.  With bf16 caches the
 *    tensor-core kernels round each softmax probability to bf16 (relative
 *    error at most 2^-9) before the P.V product, while the normaliser and
 *    the LSE use the fp32 probabilities; with 8-bit caches the probability
 *    is rounded to f16 (2^-11) and the codes become exact f16 values; fp32
 *    caches run in fp32 throughout.  Exponentials use the hardware ex2
 *    approximation.
 */
#ifndef FD_DECODE_H
#define FD_DECODE_H

#include <stdint.h>

#if defined(__GNUC__)
#define FD_API __attribute__((visibility("default")))
#else
#define FD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define FD_MAX_DIMS 4
/* Largest accepted num_splits. */
#define FD_MAX_SPLITS 256
/* Split partition granule in tokens (see fd_split_bounds). */
#define FD_SPLIT_ALIGN 64

typedef int32_t fd_status;
enum {
  FD_OK = 0,
  FD_ERR_NULL = 1,          /* a required pointer or descriptor is NULL            */
  FD_ERR_SHAPE = 2,         /* ranks or extents disagree                           */
  FD_ERR_DTYPE = 3,         /* unsupported dtype combination                       */
  FD_ERR_LAYOUT = 4,        /* inner stride != 1, or 16-byte alignment violated    */
  FD_ERR_ARG = 5,           /* num_splits out of range, non-finite scale, ...      */
  FD_ERR_UNSUPPORTED = 6,   /* head dim not in {64,128}, Hq % Hkv != 0, ...        */
  FD_ERR_ARCH = 7,          /* current device is not sm_103 / sm_100 family       */
  FD_ERR_CUDA = 8,          /* a CUDA runtime call failed                          */
  FD_ERR_DEVICE_BOUNDS = 9, /* device saw a length outside [0, capacity]           */
  FD_ERR_DEVICE_TIMEOUT = 10/* a bounded on-device wait gave up                    */
};

/* Element types.  FD_I8 is a signed 8-bit integer code, FD_E4M3 the 8-bit
 * float with 1 sign, 4 exponent (bias 7) and 3 mantissa bits (no infinity;
 * codes 0x7F / 0xFF are NaN; largest finite 448).  Both appear only as the
 * cache of fd_decode_attention_quant. */
enum { FD_F32 = 0, FD_BF16 = 1, FD_I32 = 2, FD_I8 = 3, FD_E4M3 = 4 };

typedef struct fd_tensor {
  void* data;                    /* device pointer (host pointer only where stated) */
  int32_t dtype;                 /* FD_F32, FD_BF16, FD_I32, FD_I8 or FD_E4M3      */
  int32_t ndim;                  /* 1..4                                           */
  int64_t shape[FD_MAX_DIMS];    /* extents, outermost first                        */
  int64_t stride[FD_MAX_DIMS];   /* strides in elements, outermost first            */
} fd_tensor;

/* A cudaStream_t passed as an opaque pointer. */
typedef void* fd_stream;

/*
 * fd_decode_attention — split-KV decode attention.
 *   q        [B, Hq, D]            FD_BF16 or FD_F32
 *   k_cache  [B, Lcap, Hkv, D]     FD_BF16 or FD_F32 (same dtype as v_cache)
 *   v_cache  [B, Lcap, Hkv, D]
 *   seqlens  [B] FD_I32 device tensor, or NULL meaning every len_b = Lcap.
 *            Entries outside [0, Lcap] are clamped on the device and flagged
 *            (FD_ERR_DEVICE_BOUNDS from fd_check_device_error).
 *   num_splits  0 = choose with fd_choose_num_splits(B, Hkv, Lcap, #SMs);
 *               1..FD_MAX_SPLITS = use that many splits per (b, kv head).
 *   scale    finite multiplier of the dot product (typically 1/sqrt(D)).
 *   out      [B, Hq, D] FD_F32 (written).
 *   lse      [B, Hq] FD_F32 (written), or NULL.
 * D must be 64 or 128 and Hq a multiple of Hkv.  Base pointers and the
 * strides of k_cache / v_cache must be 16-byte aligned.
 * Source: Flash-Decoding page, section "Why decoding needs different
 * scheduling" (split the history, per-split partial + log-sum-exp, reduce).
 */
FD_API fd_status fd_decode_attention(const fd_tensor* q, const fd_tensor* k_cache,
                              const fd_tensor* v_cache, const fd_tensor* seqlens,
                              int32_t num_splits, float scale, fd_tensor* out,
                              fd_tensor* lse, fd_stream stream);

/*
 * fd_decode_attention_quant — split-KV decode attention over an 8-bit KV
 * cache with one dequantisation scale per kv head (the bandwidth lever of
 * quantisation: 8-bit codes instead of 16-bit floats halve the bytes that
 * cross the memory bus; memory-bound decoding explainer, section on fighting
 * the memory wall).
 *   q        [B, Hq, D]            FD_BF16 or FD_F32
 *   k_cache  [B, Lcap, Hkv, D]     FD_I8 or FD_E4M3 (same dtype as v_cache)
 *   v_cache  [B, Lcap, Hkv, D]
 *   k_scale  [Hkv] FD_F32 device tensor: K[b,j,g,:] = k_scale[g] * k_cache[b,j,g,:]
 *   v_scale  [Hkv] FD_F32 device tensor: V[b,j,g,:] = v_scale[g] * v_cache[b,j,g,:]
 *   seqlens, num_splits, scale, out, lse: as fd_decode_attention.
 * The result is the definition above evaluated on the dequantised K and V
 * (codes times scales, exact).  Non-finite scales, or NaN codes of an E4M3
 * cache inside len_b, give non-finite outputs; codes past len_b are never
 * used.  D must be 64 or 128 and Hq a multiple of Hkv; base pointers and the
 * strides of the caches must be 16-byte aligned.  Queries are taken to f16
 * inside the kernel after a per-head power-of-two rescale, so |q| up to
 * 2^100 is represented without overflow.
 */
FD_API fd_status fd_decode_attention_quant(const fd_tensor* q, const fd_tensor* k_cache,
                                           const fd_tensor* v_cache, const fd_tensor* k_scale,
                                           const fd_tensor* v_scale, const fd_tensor* seqlens,
                                           int32_t num_splits, float scale, fd_tensor* out,
                                           fd_tensor* lse, fd_stream stream);

/*
 * fd_decode_attention_multi — split-KV decode attention with several new
 * query positions per sequence (the verification step of speculative
 * decoding: between prefill, which processes many query positions at once,
 * and usual decoding, one new position per sequence; Flash-Decoding page,
 * section "Why decoding needs different scheduling").
 *   q        [B, Tq, Hq, D]        FD_BF16 or FD_F32; Tq >= 1 new positions
 *   k_cache  [B, Lcap, Hkv, D]     FD_BF16 or FD_F32 (same dtype as v_cache),
 *   v_cache  [B, Lcap, Hkv, D]     holding the history INCLUDING the Tq new
 *                                  tokens at its end
 *   seqlens  [B] FD_I32 or NULL: len_b cached tokens, new ones included.
 *            Query t of sequence b sits at position len_b - Tq + t and sees
 *            the keys j < len_b - Tq + t + 1 (causal among the new tokens);
 *            a query with no visible key gets O = 0, LSE = -inf.
 *   out      [B, Tq, Hq, D] FD_F32; lse [B, Tq, Hq] FD_F32 or NULL.
 *   num_splits, scale: as fd_decode_attention.
 * Tq = 1 is fd_decode_attention with q viewed as [B, 1, Hq, D].
 * Tq * Hq <= 65535.  The tensor-core kernel takes Tq * G <= 64 rows per kv
 * head (bf16 queries and cache, head dim 128); other shapes use the
 * CUDA-core kernel.
 */
FD_API fd_status fd_decode_attention_multi(const fd_tensor* q, const fd_tensor* k_cache,
                                           const fd_tensor* v_cache, const fd_tensor* seqlens,
                                           int32_t num_splits, float scale, fd_tensor* out,
                                           fd_tensor* lse, fd_stream stream);

/*
 * fd_decode_attention_paged — split-KV decode attention over a paged KV
 * cache: fixed-size pages of tokens, each sequence's pages listed in a block
 * table (the indirection-table storage named among the memory-wall
 * techniques of the memory-bound decoding explainer).
 *   q           [B, Hq, D]                FD_BF16 or FD_F32
 *   k_pages     [num_pages, page_size, Hkv, D]   FD_BF16 or FD_F32 (same
 *   v_pages     [num_pages, page_size, Hkv, D]    dtype for both)
 *   block_table [B, max_pages] FD_I32 device tensor, rows contiguous: token j
 *               of sequence b is row j % page_size of page
 *               block_table[b, j / page_size].  Entries past a sequence's
 *               last page are never read.
 *   seqlens     [B] FD_I32 device tensor, or NULL meaning every sequence
 *               holds max_pages * page_size tokens (its capacity).
 *   num_splits, scale, out, lse, stream: as fd_decode_attention, with the
 *               capacity max_pages * page_size in place of Lcap.
 * Lengths outside [0, capacity] and page ids outside [0, num_pages) are
 * caught on the device: the length is clamped, a bad page reads as zeros,
 * and fd_check_device_error reports FD_ERR_DEVICE_BOUNDS.  The tensor-core
 * split kernel streams pages whose size is 16, 32 or a multiple of 64
 * tokens (bf16, head dim 128, group size 4..64); other shapes run on the
 * generic kernel.  Workspace and asynchrony as fd_decode_attention.
 */
FD_API fd_status fd_decode_attention_paged(const fd_tensor* q, const fd_tensor* k_pages,
                                           const fd_tensor* v_pages,
                                           const fd_tensor* block_table,
                                           const fd_tensor* seqlens, int32_t num_splits,
                                           float scale, fd_tensor* out, fd_tensor* lse,
                                           fd_stream stream);

/*
 * fd_decode_attention_noalloc — fd_decode_attention without any device
 * allocation.  (The pages have no counterpart: this is a library service.)
 *
 * For callers that cannot allocate GPU memory while they run: code inside a
 * region where a memory pool must not grow, a runtime that owns all device
 * memory itself, or a deadline-bound loop that cannot risk an allocation
 * stall.  Same arguments, results and errors as fd_decode_attention, but the
 * partial results of the split stage go to a fixed, library-owned device
 * array of FD_NOALLOC_SCRATCH_BYTES bytes instead of stream-ordered
 * workspace.  That array exists on every GPU that loads the library, for the
 * life of the process.
 *   - num_splits = 0: the heuristic's split count, lowered where needed to
 *     the largest count whose partial results fit the array, so the
 *     library's own choice is never refused.
 *   - An explicit num_splits whose partial results would not fit
 *     (fd_workspace_bytes(B, Hq, D, num_splits) > FD_NOALLOC_SCRATCH_BYTES)
 *     returns FD_ERR_UNSUPPORTED and enqueues nothing; pass a smaller
 *     num_splits or use fd_decode_attention.
 *   - All calls on a device share the one array: two calls whose work
 *     overlaps on the GPU (different streams, no ordering between them) race
 *     and may return wrong results.  Order them on one stream or with events.
 *   - The first call on each device looks up the array's device address
 *     (once, with that device current); make that first call before any
 *     stream capture.
 *   - Nothing in the array has to start at zero; each call writes every
 *     partial result before reading it.
 */
FD_API fd_status fd_decode_attention_noalloc(const fd_tensor* q, const fd_tensor* k_cache,
                                             const fd_tensor* v_cache, const fd_tensor* seqlens,
                                             int32_t num_splits, float scale, fd_tensor* out,
                                             fd_tensor* lse, fd_stream stream);

/* Size of the fixed scratch used by fd_decode_attention_noalloc (8 MiB). */
#define FD_NOALLOC_SCRATCH_BYTES (8 * 1024 * 1024)

/*
 * fd_decode_attention_partials — the split stage alone (diagnostics and
 * partial-level tests).  Same inputs as fd_decode_attention with an explicit
 * num_splits (1..FD_MAX_SPLITS); writes, instead of the merged result,
 *   part_o   [B, Hq, num_splits, D] FD_F32: the NORMALISED partial output of
 *            split i (attention restricted to fd_split_bounds(len_b, ns, i));
 *   part_lse [B, Hq, num_splits] FD_F32: that split's log-sum-exp (natural
 *            log); an empty split writes part_o = 0 and part_lse = -inf.
 * Allocates nothing.
 */
FD_API fd_status fd_decode_attention_partials(const fd_tensor* q, const fd_tensor* k_cache,
                                       const fd_tensor* v_cache, const fd_tensor* seqlens,
                                       int32_t num_splits, float scale, fd_tensor* part_o,
                                       fd_tensor* part_lse, fd_stream stream);

/*
 * fd_lse_combine — the log-sum-exp reduction alone.
 *   part_o [R, S, D] FD_F32, part_lse [R, S] FD_F32 (S splits per row)
 *   out    [R, D] FD_F32, lse [R] FD_F32 or NULL.
 *   LSE = ln sum_i exp(lse_i);  O = sum_i exp(lse_i - LSE) * O_i;
 *   rows whose lse_i are all -inf give O = 0, LSE = -inf.
 * D must be a multiple of 4 and at most 512; S at most 4096.
 * Source: Flash-Decoding page, section "Why decoding needs different
 * scheduling" (the final reduction over partial results).
 */
FD_API fd_status fd_lse_combine(const fd_tensor* part_o, const fd_tensor* part_lse,
                         fd_tensor* out, fd_tensor* lse, fd_stream stream);

/*
 * fd_bifurcated_attention — attention of n samples that share one context.
 *   q        [n, Hq, D]            FD_BF16
 *   k_ctx    [Lc, Hkv, D]          FD_BF16 (shared by every sample; Lc >= 1)
 *   v_ctx    [Lc, Hkv, D]
 *   k_dec    [n, Ld, Hkv, D]       FD_BF16 (sample i's own decode tokens)
 *   v_dec    [n, Ld, Hkv, D]
 *   dec_lens [n] FD_I32 device tensor, or NULL meaning all Ld.
 *   out      [n, Hq, D] FD_F32.
 * Sample i attends over concat(context, its first dec_lens[i] decode tokens).
 * The context part runs as a tensor-core contraction whose rows are all
 * (sample, query head) pairs of a kv-head group, so the context KV is read
 * once for all samples; partials are merged by the log-sum-exp reduction.
 * The decode part runs inside the same tensor-core kernel when a group holds
 * 16 or more query heads (each sample's decode tiles as extra tiles of the
 * query tile that holds its rows), else on the split kernel.  Decode tokens
 * past dec_lens[i] are never used, whatever they hold.  With the decode part
 * inside the tensor-core kernel, a NaN or infinity inside sample i's first
 * dec_lens[i] values of v_dec also reaches the other samples whose rows share
 * its 128-row query tile (their zero weights times the value); finite caches
 * are unaffected.  Environment FD_BIF_FOLD=0 keeps the decode part on the
 * split kernel, which isolates samples also for non-finite caches.
 * Source: bifurcated-attention summary, section "Tiivistelmä" (two GEMMs,
 * one over the prefill KV and one over the decode KV; exact result).
 */
FD_API fd_status fd_bifurcated_attention(const fd_tensor* q, const fd_tensor* k_ctx,
                                  const fd_tensor* v_ctx, const fd_tensor* k_dec,
                                  const fd_tensor* v_dec, const fd_tensor* dec_lens,
                                  float scale, fd_tensor* out, fd_stream stream);

/*
 * fd_bifurcated_attention_lse — fd_bifurcated_attention that also writes
 * lse [n, Hq] FD_F32 (may be NULL) and takes an explicit context split count
 * (0 = library choice; 1..FD_MAX_SPLITS, else FD_ERR_ARG).  With the decode
 * part inside the tensor-core kernel, the count is the number of equal runs
 * a query tile's context and decode tiles are cut into.
 */
FD_API fd_status fd_bifurcated_attention_lse(const fd_tensor* q, const fd_tensor* k_ctx,
                                      const fd_tensor* v_ctx, const fd_tensor* k_dec,
                                      const fd_tensor* v_dec, const fd_tensor* dec_lens,
                                      float scale, int32_t ctx_splits, fd_tensor* out,
                                      fd_tensor* lse, fd_stream stream);

/*
 * fd_choose_num_splits — split-count heuristic (pure host function).
 * Returns the smallest ns in [1, min(FD_MAX_SPLITS, ceil(max_len / 256))]
 * that minimises the modelled makespan
 *     waves(ns) * (chunk(ns) + 256)
 * where chunk(ns) is the fd_split_bounds chunk of a max_len history and
 * waves(ns) = ceil(batch * kv_heads * nonempty_splits / (2 * num_sms))
 * rounds of two CTAs per SM (the split kernel's occupancy); the 256 tokens
 * charge each wave its fixed start-up and epilogue time.  Returns 1 for any non-positive argument.  The
 * Flash-Decoding page ("Why decoding needs different scheduling") fixes only
 * the direction: split when the batch leaves SMs idle, not when the history
 * is short or the batch already fills the GPU.
 */
FD_API int32_t fd_choose_num_splits(int64_t batch, int64_t kv_heads, int64_t max_len,
                             int32_t num_sms);

/*
 * fd_split_bounds — token range [*begin, *end) of split i (pure host function).
 *   chunk = ceil(ceil(len / ns) / FD_SPLIT_ALIGN) * FD_SPLIT_ALIGN
 *   begin = min(i * chunk, len), end = min((i + 1) * chunk, len).
 * Returns FD_ERR_ARG (outputs untouched) unless 1 <= ns, 0 <= i < ns,
 * len >= 0; FD_ERR_NULL if begin or end is NULL.
 */
FD_API fd_status fd_split_bounds(int64_t len, int32_t ns, int32_t i, int64_t* begin,
                          int64_t* end);

/* Bytes of scratch fd_decode_attention allocates for (B, Hq, D, ns). */
FD_API int64_t fd_workspace_bytes(int64_t batch, int64_t q_heads, int64_t head_dim,
                           int32_t num_splits);

/*
 * fd_check_device_error — SYNCHRONISES `stream`, then reads and clears the
 * device error word of the current device.  Returns FD_OK, FD_ERR_DEVICE_BOUNDS
 * (a length was clamped), FD_ERR_DEVICE_TIMEOUT (a bounded wait gave up; the
 * affected outputs are undefined) or FD_ERR_CUDA.
 */
FD_API fd_status fd_check_device_error(fd_stream stream);

/* Static English text for a status code. */
FD_API const char* fd_status_string(fd_status status);

/* Message of the last failing call on this thread ("" if none). */
FD_API const char* fd_last_error(void);

/*
 * Kernel timing hooks.  While enabled, every kernel the library launches is
 * bracketed by CUDA events recorded on its launch stream; fd_profile_read
 * synchronises those events and returns, for one kernel kind, the number of
 * launches and their summed duration in milliseconds since the last enable.
 * Kernel kinds: 0 split partial, 1 log-sum-exp combine, 2 bifurcated context.
 * Not thread-safe; meant for benchmarks.
 */
enum { FD_KERNEL_SPLIT = 0, FD_KERNEL_COMBINE = 1, FD_KERNEL_BIF_CTX = 2, FD_KERNEL_KINDS = 3 };
FD_API fd_status fd_profile_enable(int32_t on);
FD_API fd_status fd_profile_read(int32_t kernel_kind, int64_t* launches, double* total_ms);

/* Library version string. */
FD_API const char* fd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FD_DECODE_H */
