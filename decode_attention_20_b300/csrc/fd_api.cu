// C ABI of the decode-attention library: argument validation, kernel
// selection, stream-ordered workspace, TMA descriptors, error state and
// kernel timing hooks.  Host code only; kernels live in fd_kernels.cu.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/fd_decode.h"
#include "fd_internal.h"

namespace fd {
cudaError_t read_and_clear_device_error(unsigned int* bits, cudaStream_t st);

}

using namespace fd;

namespace {

// ------------------------------------------------------------------ errors

thread_local std::string g_last_error;

fd_status fail(fd_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

fd_status cuda_fail(cudaError_t e, const char* what) {
  return fail(FD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ------------------------------------------------------------------ device info

struct DeviceInfo {
  bool ok = false;
  int sms = 0;
  int major = 0, minor = 0;
  cudaMemPool_t pool = nullptr;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[64];

fd_status current_device(int* dev_out, DeviceInfo** info_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(FD_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ok) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(cc major)");
    e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(cc minor)");
    if (!(d.major == 10 && d.minor == 3))
      return fail(FD_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                  d.major, d.minor);
    // A library-private stream-ordered pool that keeps freed workspace cached.
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    e = cudaMemPoolCreate(&d.pool, &props);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
    uint64_t thresh = ~0ull;
    e = cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &thresh);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolSetAttribute");
    d.ok = true;
  }
  *dev_out = dev;
  *info_out = &d;
  return FD_OK;
}

// ------------------------------------------------------------------ profiling

struct ProfRecord {
  cudaEvent_t start, stop;
};
struct ProfState {
  std::atomic<bool> on{false};   // read without the lock on every launch
  std::vector<ProfRecord> rec[FD_KERNEL_KINDS];
  std::vector<ProfRecord> pool;
} g_prof;
std::mutex g_prof_mu;

bool prof_begin(int kind, cudaStream_t st, ProfRecord* r) {
  if (!g_prof.on.load(std::memory_order_relaxed)) return false;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (!g_prof.pool.empty()) {
    *r = g_prof.pool.back();
    g_prof.pool.pop_back();
  } else {
    if (cudaEventCreate(&r->start) != cudaSuccess) return false;
    if (cudaEventCreate(&r->stop) != cudaSuccess) return false;
  }
  cudaEventRecord(r->start, st);
  (void)kind;
  return true;
}

void prof_end(int kind, cudaStream_t st, bool active, const ProfRecord& r) {
  if (!active) return;
  cudaEventRecord(r.stop, st);
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof.rec[kind].push_back(r);
}

// ------------------------------------------------------------------ TMA maps

// The driver's tensor-map encoder, looked up once (atomic: calls may come
// from several host threads; two lookups store the same pointer).
std::atomic<PFN_cuTensorMapEncodeTiled_v12000> g_encode_fn{nullptr};

fd_status get_encoder() {
  if (g_encode_fn.load(std::memory_order_acquire)) return FD_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
    return fail(FD_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  g_encode_fn.store(reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn),
                    std::memory_order_release);
  return FD_OK;
}

// Callers run get_encoder() first.
inline PFN_cuTensorMapEncodeTiled_v12000 g_encode() {
  return g_encode_fn.load(std::memory_order_acquire);
}

// 4-D map over a [B, L, Hkv, D] cache of bf16 (esz 2) or 8-bit codes (esz
// 1) with box {box_d, 1, tile, 1}; a 128-byte box row uses the 128-byte
// swizzle (one swizzle row per token), other widths leave the tile
// unswizzled.
bool make_kv_map(CUtensorMap* map, const void* base, int64_t B, int64_t L, int64_t Hkv,
                 int64_t D, int64_t sb, int64_t sl, int64_t sh, int tile, int box_d = 0,
                 int64_t esz = 2) {
  if (box_d == 0) box_d = (int)D;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)L, (cuuint64_t)B};
  // A unit batch extent never steps along its stride; give it a legal one.
  const int64_t sb_eff = (B == 1) ? sl * L : sb;
  cuuint64_t strides[3] = {(cuuint64_t)(sh * esz), (cuuint64_t)(sl * esz),
                           (cuuint64_t)(sb_eff * esz)};
  cuuint32_t box[4] = {(cuuint32_t)box_d, 1u, (cuuint32_t)tile, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUtensorMapSwizzle swz =
      (box_d * esz == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  const CUtensorMapDataType dt =
      esz == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = g_encode()(map, dt, 4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D bf16 map {D, dim1, dim2} with byte strides {s1, s2} and box
// {64, box1, box2}, 128-byte swizzle (one swizzle row per 64-element box row).
bool make_3d_map(CUtensorMap* map, const void* base, int64_t D, int64_t n1, int64_t n2,
                 int64_t s1_elems, int64_t s2_elems, int box1, int box2) {
  const int64_t esz = 2;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)n1, (cuuint64_t)n2};
  // A unit outer extent never steps along its stride; give it a legal one.
  const int64_t s2_eff = (n2 == 1) ? s1_elems * n1 : s2_elems;
  cuuint64_t strides[2] = {(cuuint64_t)(s1_elems * esz), (cuuint64_t)(s2_eff * esz)};
  cuuint32_t box[3] = {64u, (cuuint32_t)box1, (cuuint32_t)box2};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = g_encode()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D bf16 map over the queries of a bifurcated call, q [n, Hq, D] seen as
// [n][Hkv][G][D] (element strides q_sb, q_sh), with a box of 64 head dims x
// rb heads x 1 kv head x sb samples (rb = min(G, 128), sb = 128 / rb) and
// the 128-byte swizzle: one box is half a 128-row query tile of kv head g in
// row order (sample, head).  Needs G to divide 128 or 128 to divide G.
bool make_q_map(CUtensorMap* map, const void* base, int64_t n, int64_t Hkv, int64_t G,
                int64_t D, int64_t q_sb, int64_t q_sh) {
  if (!(128 % G == 0 || G % 128 == 0)) return false;
  const int64_t rb = G < 128 ? G : 128, sb = 128 / rb;
  const int64_t esz = 2;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)G, (cuuint64_t)Hkv, (cuuint64_t)n};
  // Unit extents never step along their strides; give them legal ones.
  const int64_t sg = G * q_sh;
  const int64_t ss = (n == 1) ? sg * Hkv : q_sb;
  cuuint64_t strides[3] = {(cuuint64_t)(q_sh * esz), (cuuint64_t)(sg * esz),
                           (cuuint64_t)(ss * esz)};
  cuuint32_t box[4] = {64u, (cuuint32_t)rb, 1u, (cuuint32_t)sb};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = g_encode()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 5-D fp32 map over the bifurcated partial outputs [S][n][Hq][D] (element
// strides o_ss, o_sb, o_sh) seen as [S][n][Hkv][G][D], with a box of 32
// head dims x rb heads x 1 kv head x sb samples x 1 slot (rb = min(G, 128),
// sb = 128 / rb) and the 128-byte swizzle: four boxes are the 128 partial
// rows of one context CTA.  Needs G to divide 128 or 128 to divide G.
bool make_o_map(CUtensorMap* map, void* base, int64_t S, int64_t n, int64_t Hkv, int64_t G,
                int64_t D, int64_t o_ss, int64_t o_sb, int64_t o_sh) {
  if (!(128 % G == 0 || G % 128 == 0)) return false;
  const int64_t rb = G < 128 ? G : 128, sb = 128 / rb;
  const int64_t esz = 4;
  cuuint64_t dims[5] = {(cuuint64_t)D, (cuuint64_t)G, (cuuint64_t)Hkv, (cuuint64_t)n,
                        (cuuint64_t)S};
  const int64_t sg = G * o_sh;
  cuuint64_t strides[4] = {(cuuint64_t)(o_sh * esz), (cuuint64_t)(sg * esz),
                           (cuuint64_t)(o_sb * esz), (cuuint64_t)(o_ss * esz)};
  cuuint32_t box[5] = {32u, (cuuint32_t)rb, 1u, (cuuint32_t)sb, 1u};
  cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  CUresult r = g_encode()(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ validation

int64_t esize(int32_t dt) {
  return dt == FD_BF16 ? 2 : (dt == FD_I8 || dt == FD_E4M3) ? 1 : 4;
}

bool is_q8(int32_t dt) { return dt == FD_I8 || dt == FD_E4M3; }

int kv_kind_of(int32_t dt) {
  switch (dt) {
    case FD_BF16: return kKvBf16;
    case FD_I8: return kKvI8;
    case FD_E4M3: return kKvE4m3;
    default: return kKvF32;
  }
}

fd_status check_tensor(const fd_tensor* t, const char* name, int ndim) {
  if (t == nullptr) return fail(FD_ERR_NULL, "%s descriptor is NULL", name);
  if (t->ndim != ndim) return fail(FD_ERR_SHAPE, "%s must have %d dims, got %d", name, ndim, t->ndim);
  int64_t numel = 1;
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0) return fail(FD_ERR_SHAPE, "%s has a negative extent", name);
    numel *= t->shape[i];
  }
  if (numel > 0 && t->data == nullptr) return fail(FD_ERR_NULL, "%s data pointer is NULL", name);
  if (t->dtype != FD_F32 && t->dtype != FD_BF16 && t->dtype != FD_I32 && !is_q8(t->dtype))
    return fail(FD_ERR_DTYPE, "%s has unknown dtype %d", name, t->dtype);
  if (t->stride[ndim - 1] != 1 && t->shape[ndim - 1] > 1)
    return fail(FD_ERR_LAYOUT, "%s innermost stride must be 1", name);
  for (int i = 0; i < ndim; ++i)
    if (t->stride[i] < 0) return fail(FD_ERR_LAYOUT, "%s has a negative stride", name);
  if (reinterpret_cast<uintptr_t>(t->data) % esize(t->dtype) != 0)
    return fail(FD_ERR_LAYOUT, "%s data pointer is not element-aligned", name);
  return FD_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DecodeDesc {
  int64_t B, Hq, Hkv, D, Lcap, G;
  int32_t q_dt, kv_dt;
  int64_t tq = 1;                   // query positions per sequence (q is [B, tq, Hq, D] if > 1)
  const float* k_scale = nullptr;   // 8-bit caches: [Hkv] device
  const float* v_scale = nullptr;
};

// Validates q / k / v / seqlens / out / lse of a decode call.  `out_dims`
// 3: out [B,Hq,D], lse [B,Hq];  4: partials out [B,Hq,ns,D], lse [B,Hq,ns].
// `quant_kv`: the caches hold 8-bit codes (FD_I8 / FD_E4M3) instead of
// bf16 / f32 values.
fd_status validate_decode(const fd_tensor* q, const fd_tensor* k, const fd_tensor* v,
                          const fd_tensor* seqlens, const fd_tensor* out, const fd_tensor* lse,
                          int out_dims, int ns, DecodeDesc* d, bool quant_kv = false) {
  fd_status st;
  if ((st = check_tensor(q, "q", 3))) return st;
  if ((st = check_tensor(k, "k_cache", 4))) return st;
  if ((st = check_tensor(v, "v_cache", 4))) return st;
  if ((st = check_tensor(out, "out", out_dims))) return st;
  if (lse && (st = check_tensor(lse, "lse", out_dims - 1))) return st;
  if (seqlens && (st = check_tensor(seqlens, "seqlens", 1))) return st;
  d->B = q->shape[0];
  d->Hq = q->shape[1];
  d->D = q->shape[2];
  d->Lcap = k->shape[1];
  d->Hkv = k->shape[2];
  for (int i = 0; i < 4; ++i)
    if (k->shape[i] != v->shape[i]) return fail(FD_ERR_SHAPE, "k_cache and v_cache shapes differ");
  if (k->shape[0] != d->B) return fail(FD_ERR_SHAPE, "k_cache batch %lld != q batch %lld",
                                       (long long)k->shape[0], (long long)d->B);
  if (k->shape[3] != d->D) return fail(FD_ERR_SHAPE, "k_cache head dim != q head dim");
  if (q->dtype != FD_BF16 && q->dtype != FD_F32) return fail(FD_ERR_DTYPE, "q must be bf16 or f32");
  if (k->dtype != v->dtype) return fail(FD_ERR_DTYPE, "k_cache and v_cache dtypes differ");
  if (quant_kv && !is_q8(k->dtype))
    return fail(FD_ERR_DTYPE, "k_cache/v_cache must be int8 or e4m3 codes");
  if (!quant_kv && k->dtype != FD_BF16 && k->dtype != FD_F32)
    return fail(FD_ERR_DTYPE, "k_cache/v_cache must be bf16 or f32");
  if (out->dtype != FD_F32) return fail(FD_ERR_DTYPE, "out must be f32");
  if (lse && lse->dtype != FD_F32) return fail(FD_ERR_DTYPE, "lse must be f32");
  if (seqlens) {
    if (seqlens->dtype != FD_I32) return fail(FD_ERR_DTYPE, "seqlens must be int32");
    if (seqlens->shape[0] != d->B) return fail(FD_ERR_SHAPE, "seqlens must have B entries");
    if (seqlens->stride[0] != 1 && d->B > 1) return fail(FD_ERR_LAYOUT, "seqlens must be contiguous");
  }
  if (out_dims == 3) {
    if (out->shape[0] != d->B || out->shape[1] != d->Hq || out->shape[2] != d->D)
      return fail(FD_ERR_SHAPE, "out must be [B, Hq, D]");
    if (lse && (lse->shape[0] != d->B || lse->shape[1] != d->Hq))
      return fail(FD_ERR_SHAPE, "lse must be [B, Hq]");
  } else {
    if (out->shape[0] != d->B || out->shape[1] != d->Hq || out->shape[2] != ns || out->shape[3] != d->D)
      return fail(FD_ERR_SHAPE, "part_o must be [B, Hq, num_splits, D]");
    if (lse && (lse->shape[0] != d->B || lse->shape[1] != d->Hq || lse->shape[2] != ns))
      return fail(FD_ERR_SHAPE, "part_lse must be [B, Hq, num_splits]");
  }
  if (d->Hkv < 1 || d->Hq < 1 || d->Hq % d->Hkv != 0)
    return fail(FD_ERR_UNSUPPORTED, "Hq (%lld) must be a positive multiple of Hkv (%lld)",
                (long long)d->Hq, (long long)d->Hkv);
  if (d->D != 64 && d->D != 128) return fail(FD_ERR_UNSUPPORTED, "head dim %lld not in {64, 128}", (long long)d->D);
  if (d->B > 65535 || d->Hq > 65535) return fail(FD_ERR_UNSUPPORTED, "batch and query heads must be <= 65535");
  if (d->Lcap > (int64_t)INT32_MAX - 2 * kSplitAlign) return fail(FD_ERR_UNSUPPORTED, "cache length too large");
  d->G = d->Hq / d->Hkv;
  d->q_dt = q->dtype;
  d->kv_dt = k->dtype;
  return FD_OK;
}

// Whether the TMA kernel can stream this cache: bf16, head dim 128, 16-byte
// aligned base and strides (token, kv head, batch), a group size it is
// instantiated for.
// (8-bit caches: the same with 1-byte codes.)
bool tma_ok(const DecodeDesc& d, const void* kd, const void* vd, const int64_t (&strides)[6],
            int64_t batch_extent) {
  if ((d.kv_dt != FD_BF16 && !is_q8(d.kv_dt)) || d.D != 128 || d.Lcap < kSplitTileTokens)
    return false;
  if (!(d.G == 1 || d.G == 2 || d.G == 4 || d.G == 8 || d.G == 16 || d.G == 32 || d.G == 64)) return false;
  if (!aligned16(kd) || !aligned16(vd)) return false;
  const int64_t esz = esize(d.kv_dt);
  for (int i = 0; i < 6; ++i) {
    if (i >= 4 && batch_extent == 1) continue;   // batch strides unused
    if (strides[i] <= 0 || (strides[i] * esz) % 16 != 0 || strides[i] * esz >= (1ll << 40)) return false;
  }
  return true;
}

// Which split kernel variant to use.  Tuning and test knob, read on every
// call: FD_SPLIT_VARIANT = "cuda" forces the CUDA-core kernel, "mma0" /
// "mma1" / "mma2" pick a tensor-core tiling.  Unset, from the variant sweeps
// on B300 (batch-1 64K layer, 32 and 37 splits):
//  - bf16 caches: "mma2" (3-stage ring of 64-token tiles, two CTAs per SM):
//    it matched the 6-stage one-CTA-per-SM tiling at batch 1 and beat it by
//    5% on the ragged batch, the second resident CTA covering the first
//    one's start and tail; paged caches 46.2 us against 53.2 and 71.3.
//  - 8-bit caches: "mma1" (8 warps, 128-token tiles, 3 stages): e4m3 33.2 us
//    against 36.2 (4 warps) and 38.8 (64-token tiles), the extra warps
//    hiding the latency of the code conversions; int8 28.9 us, level with
//    4 warps and 2 us ahead of 64-token tiles.
int split_variant(int kv_kind) {
  const char* e = getenv("FD_SPLIT_VARIANT");
  if (e == nullptr || e[0] == 0) return (kv_kind == kKvI8 || kv_kind == kKvE4m3) ? 1 : 2;
  if (!strcmp(e, "cuda")) return -1;
  if (!strcmp(e, "mma1")) return 1;
  if (!strcmp(e, "mma2")) return 2;
  return 0;
}

// Test knobs of the bounded-wait error path, read on every call:
// FD_TEST_WAIT_LIMIT_NS shortens the tensor-core split kernel's pipeline
// waits (1 ns .. 1 s) and FD_TEST_PRODUCER_DELAY_NS makes its producer spin
// that long (at most kMaxProducerDelayNs) before its first copies, so a test
// can make a wait run out on a small, complete problem.  Unset: the 1 s limit
// and no delay.
void test_wait_knobs(unsigned long long* limit_ns, unsigned int* delay_ns) {
  *limit_ns = kWaitLimitNs;
  *delay_ns = 0u;
  if (const char* e = getenv("FD_TEST_WAIT_LIMIT_NS")) {
    const long long v = atoll(e);
    if (v > 0) *limit_ns = (unsigned long long)std::min<long long>(v, (long long)kWaitLimitNs);
  }
  if (const char* e = getenv("FD_TEST_PRODUCER_DELAY_NS")) {
    const long long v = atoll(e);
    if (v > 0) *delay_ns = (unsigned int)std::min<long long>(v, (long long)kMaxProducerDelayNs);
  }
}

bool mma_group_ok(int64_t G) { return G == 4 || G == 8 || G == 16 || G == 32 || G == 64; }

// Split-count heuristic: the smallest ns with the lowest makespan
// waves(ns) * (chunk(ns) + kSplitOverheadTokens), where chunk is the
// fd_split_bounds chunk of a max_len history and waves counts rounds of two
// CTAs per SM (the default split kernel's occupancy) over batch * kv_heads *
// (non-empty splits) CTAs; ns is capped at ceil(max_len / 64) (chunks of
// at least one 64-token tile: the split-count sweeps find the fastest call
// there for histories of 512 to 2048 tokens) and FD_MAX_SPLITS.
int32_t choose_splits_host(int64_t batch, int64_t kv_heads, int64_t max_len, int32_t num_sms) {
  constexpr int64_t kMinChunk = 64;
  constexpr int64_t kSplitOverheadTokens = 256;
  if (batch <= 0 || kv_heads <= 0 || max_len <= 0 || num_sms <= 0) return 1;
  const int64_t units = batch * kv_heads;
  int64_t cap = (max_len + kMinChunk - 1) / kMinChunk;
  if (cap > kMaxSplits) cap = kMaxSplits;
  if (cap < 1) cap = 1;
  int64_t best_ns = 1, best_cost = -1;
  for (int64_t ns = 1; ns <= cap; ++ns) {
    const int64_t per = (max_len + ns - 1) / ns;
    const int64_t chunk = ((per + kSplitAlign - 1) / kSplitAlign) * kSplitAlign;
    const int64_t used = (max_len + chunk - 1) / chunk;
    const int64_t waves = (units * used + 2 * (int64_t)num_sms - 1) / (2 * (int64_t)num_sms);
    const int64_t cost = waves * (chunk + kSplitOverheadTokens);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_ns = ns;
    }
  }
  return (int32_t)best_ns;
}

// Enqueue the split stage for one cache.
// A paged cache: k / v tensors are [num_pages, page_size, Hkv, D].
struct PageDesc {
  const int32_t* table;       // [B, max_pages] device
  int64_t stride;             // elements between rows of the table
  int page_size, num_pages;
};

// Page sizes the TMA split kernel streams (every box stays inside a page).
bool page_size_tma_ok(int ps) { return ps == 16 || ps == 32 || (ps >= 64 && ps % 64 == 0); }

fd_status enqueue_split(const DecodeDesc& d, const fd_tensor* q, const fd_tensor* k,
                        const fd_tensor* v, const int32_t* seqlens, int ns, float scale,
                        float* o, int64_t o_sb, int64_t o_sh, int64_t o_ss, float* lse,
                        int64_t l_sb, int64_t l_sh, int64_t l_ss, bool kv_broadcast,
                        cudaStream_t st, const PageDesc* pg = nullptr, int64_t o_st = 0,
                        int64_t l_st = 0, bool late_wait = false) {
  SplitParams p = {};
  p.late_wait = late_wait ? 1 : 0;
  test_wait_knobs(&p.wait_limit_ns, &p.producer_delay_ns);
  if (pg) {
    p.block_table = pg->table;
    p.bt_stride = pg->stride;
    p.page_size = pg->page_size;
    p.num_pages = pg->num_pages;
    p.page_rows = pg->page_size < 64 ? pg->page_size : 64;
  }
  p.q = q->data;
  p.tq = (int)d.tq;
  p.q_sb = q->stride[0];
  p.q_st = q->ndim == 4 ? q->stride[1] : 0;          // [B, tq, Hq, D] or [B, Hq, D]
  p.q_sh = q->ndim == 4 ? q->stride[2] : q->stride[1];
  p.o_st = o_st;
  p.l_st = l_st;
  p.q_vec16 = d.q_dt == FD_BF16 && aligned16(q->data) && p.q_sb % 8 == 0 && p.q_sh % 8 == 0 &&
              p.q_st % 8 == 0;
  p.q_bf16 = d.q_dt == FD_BF16;
  p.k = k->data;
  p.v = v->data;
  // kv tensors are [B, L, Hkv, D] or, when broadcast, [L, Hkv, D]
  const int dim0 = kv_broadcast ? 1 : 0;
  p.k_sb = kv_broadcast ? 0 : k->stride[0];
  p.k_sl = k->stride[1 - dim0];
  p.k_sh = k->stride[2 - dim0];
  p.v_sb = kv_broadcast ? 0 : v->stride[0];
  p.v_sl = v->stride[1 - dim0];
  p.v_sh = v->stride[2 - dim0];
  p.seqlens = seqlens;
  p.B = (int)d.B;
  p.Hq = (int)d.Hq;
  p.Hkv = (int)d.Hkv;
  p.G = (int)d.G;
  p.Lcap = (int)d.Lcap;
  p.ns = ns;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o = o;
  p.o_sb = o_sb;
  p.o_sh = o_sh;
  p.o_ss = o_ss;
  p.o_vec4 = aligned16(o) && o_sb % 4 == 0 && o_sh % 4 == 0 && o_ss % 4 == 0 && o_st % 4 == 0;
  p.lse = lse;
  p.l_sb = l_sb;
  p.l_sh = l_sh;
  p.l_ss = l_ss;
  p.kv_batch_broadcast = kv_broadcast ? 1 : 0;
  p.kv_kind = kv_kind_of(d.kv_dt);
  p.k_scale = d.k_scale;
  p.v_scale = d.v_scale;
  const bool q8 = is_q8(d.kv_dt);

  ProfRecord rec;
  bool launched = false;
  cudaError_t e = cudaSuccess;
  // The tensor maps span the kv batch, or for a paged cache the pages (a
  // page is a "sequence" of page_size tokens, boxes page_rows tall).
  const int64_t kv_batch = pg ? pg->num_pages : (kv_broadcast ? 1 : d.B);
  const int64_t map_len = pg ? pg->page_size : d.Lcap;
  const int64_t strides[6] = {p.k_sl, p.k_sh, p.v_sl, p.v_sh, p.k_sb, p.v_sb};
  const int variant = split_variant(p.kv_kind);
  // The tensor-core kernel takes bf16 queries over a bf16 cache, or bf16 /
  // f32 queries over an 8-bit cache (converted to f16 in the kernel).
  const int mtile = mma_tile_tokens(variant, p.kv_kind);
  // Multi-token decode puts tq * G rows on the n-tiles (up to 64).
  const bool rows_ok = d.tq > 1 ? d.tq * d.G <= 64 : mma_group_ok(d.G);
  if (variant >= 0 && (d.q_dt == FD_BF16 || q8) && rows_ok && d.Lcap >= mtile &&
      tma_ok(d, k->data, v->data, strides, kv_batch) &&
      (!pg || page_size_tma_ok(pg->page_size))) {
    fd_status gs = get_encoder();
    if (gs) return gs;
    CUtensorMap tmK, tmV;
    const int tile = pg ? p.page_rows : mtile;
    const int box_d = q8 ? 128 : 64;            // 128-byte box rows either way
    const int64_t esz = esize(d.kv_dt);
    const bool okk = make_kv_map(&tmK, k->data, kv_batch, map_len, d.Hkv, d.D, p.k_sb, p.k_sl,
                                 p.k_sh, tile, box_d, esz);
    const bool okv = make_kv_map(&tmV, v->data, kv_batch, map_len, d.Hkv, d.D, p.v_sb, p.v_sl,
                                 p.v_sh, tile, box_d, esz);
    if (okk && okv) {
      const bool prof = prof_begin(FD_KERNEL_SPLIT, st, &rec);
      e = launch_split_mma(p, tmK, tmV, (int)d.G, variant, st, &launched, !prof);
      prof_end(FD_KERNEL_SPLIT, st, prof && launched, rec);
      if (prof && !launched) {
        std::lock_guard<std::mutex> lock(g_prof_mu);
        g_prof.pool.push_back(rec);
      }
      if (e != cudaSuccess) return cuda_fail(e, "split kernel launch");
    }
  }
  if (!launched && !pg && !q8 && d.tq == 1 && tma_ok(d, k->data, v->data, strides, kv_batch)) {
    fd_status gs = get_encoder();
    if (gs) return gs;
    CUtensorMap tmK, tmV;
    const bool okk = make_kv_map(&tmK, k->data, kv_batch, d.Lcap, d.Hkv, d.D, p.k_sb, p.k_sl,
                                 p.k_sh, kSplitTileTokens);
    const bool okv = make_kv_map(&tmV, v->data, kv_batch, d.Lcap, d.Hkv, d.D, p.v_sb, p.v_sl,
                                 p.v_sh, kSplitTileTokens);
    if (okk && okv) {
      const bool prof = prof_begin(FD_KERNEL_SPLIT, st, &rec);
      e = launch_split_tma(p, tmK, tmV, (int)d.D, (int)d.G, st, &launched, !prof);
      prof_end(FD_KERNEL_SPLIT, st, prof && launched, rec);
      if (prof && !launched) {
        std::lock_guard<std::mutex> lock(g_prof_mu);
        g_prof.pool.push_back(rec);
      }
      if (e != cudaSuccess) return cuda_fail(e, "split kernel launch");
    }
  }
  if (!launched) {
    const bool prof = prof_begin(FD_KERNEL_SPLIT, st, &rec);
    e = launch_split_generic(p, (int)d.D, st, !prof);
    prof_end(FD_KERNEL_SPLIT, st, prof, rec);
    if (e != cudaSuccess) return cuda_fail(e, "split kernel launch");
  }
  return FD_OK;
}

fd_status enqueue_combine(const CombineParams& cp, cudaStream_t st, bool pdl) {
  ProfRecord rec;
  const bool prof = prof_begin(FD_KERNEL_COMBINE, st, &rec);
  // Event records between the kernels would defeat the programmatic
  // overlap, so timing runs launch the combine without it.
  cudaError_t e = launch_combine(cp, st, pdl && !prof);
  prof_end(FD_KERNEL_COMBINE, st, prof, rec);
  if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
  return FD_OK;
}

// Context split count of the bifurcated tensor-core kernel: the fewest
// splits that reach the smallest makespan waves x (tiles per split + 2) when
// `units` CTAs (query tiles x kv heads) run per split on `num_sms` SMs, one
// CTA per SM; the 2 tiles (256 tokens) charge each CTA its start-up (query
// load, pipeline fill) and epilogue.
int choose_ctx_splits(int64_t Lc, int64_t units, int num_sms) {
  constexpr int64_t kCtaOverheadTiles = 2;
  const int64_t tiles = (Lc + kBifTileTokens - 1) / kBifTileTokens;
  int best_ns = 1;
  int64_t best_cost = -1;
  for (int ns = 1; ns <= kMaxSplits && ns <= tiles; ++ns) {
    const int64_t per = (tiles + ns - 1) / ns;          // tiles per split
    const int64_t used = (tiles + per - 1) / per;        // non-empty splits
    const int64_t ctas = used * units;
    const int64_t waves = (ctas + num_sms - 1) / num_sms;
    const int64_t cost = waves * (per + kCtaOverheadTiles);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_ns = (int)used;
    }
  }
  return best_ns;
}

// Which context path the bifurcated call takes.  Tuning and test knob, read
// on every call: FD_BIF_CTX = "split" forces the split kernel over a
// batch-broadcast view of the context; unset = the tensor-core kernel where
// it applies.
bool bif_ctx_tensor_core_allowed() {
  const char* e = getenv("FD_BIF_CTX");
  return !(e && !strcmp(e, "split"));
}

int64_t workspace_bytes(int64_t B, int64_t Hq, int64_t D, int64_t ns) {
  const int64_t o_bytes = B * Hq * ns * D * 4;
  const int64_t l_bytes = B * Hq * ns * 4;
  return ((o_bytes + 255) / 256) * 256 + ((l_bytes + 255) / 256) * 256;
}

}  // namespace

// ------------------------------------------------------- allocation-free scratch
//
// For callers that must not allocate device memory while they run (see
// fd_decode_attention_noalloc in fd_decode.h): the partial-result workspace
// of the split stage lives in this fixed array instead of the stream-ordered
// pool.  Every GPU that loads the library holds it until the process exits.
// Host code must never pass the array's name to a kernel (on the host it is
// only a stand-in for the symbol); the device address comes from
// cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FD_NOALLOC_SCRATCH_BYTES];

namespace {

struct NoAllocDevice {
  bool ok = false;
  int sms = 0;
  void* scratch = nullptr;   // device address of g_noalloc_scratch on this device
};
std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[64];

// One-time set-up for the current device: architecture check, SM count and
// the scratch array's device address.  Allocates nothing.
fd_status noalloc_setup(NoAllocDevice** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(FD_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!d.ok) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(cc major)");
    e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(cc minor)");
    if (!(major == 10 && minor == 3))
      return fail(FD_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                  major, minor);
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    d.scratch = ptr;
    d.ok = true;
  }
  *out = &d;
  return FD_OK;
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

const char* fd_version(void) { return "fd_decode 0.1 (sm_103a)"; }

const char* fd_last_error(void) { return g_last_error.c_str(); }

const char* fd_status_string(fd_status s) {
  switch (s) {
    case FD_OK: return "ok";
    case FD_ERR_NULL: return "null pointer or descriptor";
    case FD_ERR_SHAPE: return "shape mismatch";
    case FD_ERR_DTYPE: return "unsupported dtype";
    case FD_ERR_LAYOUT: return "unsupported layout or alignment";
    case FD_ERR_ARG: return "invalid argument";
    case FD_ERR_UNSUPPORTED: return "unsupported problem";
    case FD_ERR_ARCH: return "unsupported GPU architecture";
    case FD_ERR_CUDA: return "CUDA error";
    case FD_ERR_DEVICE_BOUNDS: return "device saw a length outside [0, capacity]";
    case FD_ERR_DEVICE_TIMEOUT: return "a bounded device wait timed out";
    default: return "unknown status";
  }
}

int32_t fd_choose_num_splits(int64_t batch, int64_t kv_heads, int64_t max_len, int32_t num_sms) {
  return choose_splits_host(batch, kv_heads, max_len, num_sms);
}

fd_status fd_split_bounds(int64_t len, int32_t ns, int32_t i, int64_t* begin, int64_t* end) {
  if (begin == nullptr || end == nullptr) return fail(FD_ERR_NULL, "begin/end is NULL");
  if (ns < 1 || i < 0 || i >= ns || len < 0) return fail(FD_ERR_ARG, "bad split arguments");
  const int64_t per = (len + ns - 1) / ns;
  const int64_t chunk = ((per + kSplitAlign - 1) / kSplitAlign) * kSplitAlign;
  const int64_t b0 = (int64_t)i * chunk;
  *begin = b0 < len ? b0 : len;
  *end = b0 + chunk < len ? b0 + chunk : len;
  return FD_OK;
}

int64_t fd_workspace_bytes(int64_t batch, int64_t q_heads, int64_t head_dim, int32_t num_splits) {
  if (batch < 0 || q_heads < 0 || head_dim < 0 || num_splits <= 1) return 0;
  return workspace_bytes(batch, q_heads, head_dim, num_splits);
}

}  // extern "C"

namespace {

// Split stage + log-sum-exp combine into out / lse, workspace from the
// library pool (shared by the contiguous and the paged entry points).
fd_status run_decode(const DecodeDesc& d, const fd_tensor* q, const fd_tensor* k_cache,
                     const fd_tensor* v_cache, const fd_tensor* seqlens, int32_t num_splits,
                     float scale, fd_tensor* out, fd_tensor* lse, fd_stream stream,
                     const PageDesc* pg) {
  fd_status st;
  int dev;
  DeviceInfo* info;
  if ((st = current_device(&dev, &info))) return st;
  if (d.B == 0 || d.Hq == 0) return FD_OK;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int ns = num_splits > 0 ? num_splits : choose_splits_host(d.B, d.Hkv, d.Lcap, info->sms);
  const int32_t* sl = seqlens ? reinterpret_cast<const int32_t*>(seqlens->data) : nullptr;
  float* o = reinterpret_cast<float*>(out->data);
  float* l = lse ? reinterpret_cast<float*>(lse->data) : nullptr;
  if (ns == 1) {
    return enqueue_split(d, q, k_cache, v_cache, sl, 1, scale, o, out->stride[0], out->stride[1],
                         0, l, lse ? lse->stride[0] : 0, lse ? lse->stride[1] : 0, 0, false, cs,
                         pg);
  }
  const int64_t bytes = workspace_bytes(d.B, d.Hq, d.D, ns);
  void* ws = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&ws, (size_t)bytes, info->pool, cs);
  if (e != cudaSuccess) return cuda_fail(e, "workspace allocation");
  float* po = reinterpret_cast<float*>(ws);
  float* pl = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) +
                                       ((d.B * d.Hq * ns * d.D * 4 + 255) / 256) * 256);
  st = enqueue_split(d, q, k_cache, v_cache, sl, ns, scale, po, d.Hq * ns * d.D, ns * d.D, d.D,
                     pl, d.Hq * ns, ns, 1, false, cs, pg);
  if (st == FD_OK) {
    CombineParams cp = {};
    cp.part_o = po;
    cp.po_r1 = d.Hq * ns * d.D;
    cp.po_r2 = ns * d.D;
    cp.po_s = d.D;
    cp.part_lse = pl;
    cp.pl_r1 = d.Hq * ns;
    cp.pl_r2 = ns;
    cp.pl_s = 1;
    cp.out = o;
    cp.out_r1 = out->stride[0];
    cp.out_r2 = out->stride[1];
    cp.lse = l;
    cp.lse_r1 = lse ? lse->stride[0] : 0;
    cp.lse_r2 = lse ? lse->stride[1] : 0;
    cp.R1 = (int)d.B;
    cp.R2 = (int)d.Hq;
    cp.S = ns;
    cp.D = (int)d.D;
    st = enqueue_combine(cp, cs, true);
  }
  e = cudaFreeAsync(ws, cs);
  if (st) return st;
  if (e != cudaSuccess) return cuda_fail(e, "workspace release");
  return FD_OK;
}

}  // namespace

extern "C" {

fd_status fd_decode_attention(const fd_tensor* q, const fd_tensor* k_cache,
                              const fd_tensor* v_cache, const fd_tensor* seqlens,
                              int32_t num_splits, float scale, fd_tensor* out, fd_tensor* lse,
                              fd_stream stream) {
  DecodeDesc d;
  fd_status st = validate_decode(q, k_cache, v_cache, seqlens, out, lse, 3, 0, &d);
  if (st) return st;
  if (num_splits < 0 || num_splits > kMaxSplits)
    return fail(FD_ERR_ARG, "num_splits %d outside [0, %d]", num_splits, kMaxSplits);
  if (!std::isfinite(scale)) return fail(FD_ERR_ARG, "scale must be finite");
  return run_decode(d, q, k_cache, v_cache, seqlens, num_splits, scale, out, lse, stream, nullptr);
}

fd_status fd_decode_attention_quant(const fd_tensor* q, const fd_tensor* k_cache,
                                    const fd_tensor* v_cache, const fd_tensor* k_scale,
                                    const fd_tensor* v_scale, const fd_tensor* seqlens,
                                    int32_t num_splits, float scale, fd_tensor* out,
                                    fd_tensor* lse, fd_stream stream) {
  DecodeDesc d;
  fd_status st = validate_decode(q, k_cache, v_cache, seqlens, out, lse, 3, 0, &d, true);
  if (st) return st;
  if ((st = check_tensor(k_scale, "k_scale", 1))) return st;
  if ((st = check_tensor(v_scale, "v_scale", 1))) return st;
  if (k_scale->dtype != FD_F32 || v_scale->dtype != FD_F32)
    return fail(FD_ERR_DTYPE, "k_scale / v_scale must be f32");
  if (k_scale->shape[0] != d.Hkv || v_scale->shape[0] != d.Hkv)
    return fail(FD_ERR_SHAPE, "k_scale / v_scale must have Hkv (%lld) entries", (long long)d.Hkv);
  if (num_splits < 0 || num_splits > kMaxSplits)
    return fail(FD_ERR_ARG, "num_splits %d outside [0, %d]", num_splits, kMaxSplits);
  if (!std::isfinite(scale)) return fail(FD_ERR_ARG, "scale must be finite");
  d.k_scale = reinterpret_cast<const float*>(k_scale->data);
  d.v_scale = reinterpret_cast<const float*>(v_scale->data);
  return run_decode(d, q, k_cache, v_cache, seqlens, num_splits, scale, out, lse, stream, nullptr);
}

fd_status fd_decode_attention_multi(const fd_tensor* q, const fd_tensor* k_cache,
                                    const fd_tensor* v_cache, const fd_tensor* seqlens,
                                    int32_t num_splits, float scale, fd_tensor* out,
                                    fd_tensor* lse, fd_stream stream) {
  fd_status st;
  if ((st = check_tensor(q, "q", 4))) return st;
  if ((st = check_tensor(k_cache, "k_cache", 4))) return st;
  if ((st = check_tensor(v_cache, "v_cache", 4))) return st;
  if ((st = check_tensor(out, "out", 4))) return st;
  if (lse && (st = check_tensor(lse, "lse", 3))) return st;
  if (seqlens && (st = check_tensor(seqlens, "seqlens", 1))) return st;
  DecodeDesc d;
  d.B = q->shape[0];
  d.tq = q->shape[1];
  d.Hq = q->shape[2];
  d.D = q->shape[3];
  d.Lcap = k_cache->shape[1];
  d.Hkv = k_cache->shape[2];
  for (int i = 0; i < 4; ++i)
    if (k_cache->shape[i] != v_cache->shape[i])
      return fail(FD_ERR_SHAPE, "k_cache and v_cache shapes differ");
  if (k_cache->shape[0] != d.B) return fail(FD_ERR_SHAPE, "k_cache batch != q batch");
  if (k_cache->shape[3] != d.D) return fail(FD_ERR_SHAPE, "k_cache head dim != q head dim");
  if (d.tq < 1) return fail(FD_ERR_SHAPE, "q must hold at least one query token per sequence");
  if (q->dtype != FD_BF16 && q->dtype != FD_F32) return fail(FD_ERR_DTYPE, "q must be bf16 or f32");
  if (k_cache->dtype != v_cache->dtype) return fail(FD_ERR_DTYPE, "k_cache and v_cache dtypes differ");
  if (k_cache->dtype != FD_BF16 && k_cache->dtype != FD_F32)
    return fail(FD_ERR_DTYPE, "k_cache/v_cache must be bf16 or f32");
  if (out->dtype != FD_F32 || (lse && lse->dtype != FD_F32))
    return fail(FD_ERR_DTYPE, "out / lse must be f32");
  for (int i = 0; i < 4; ++i)
    if (out->shape[i] != q->shape[i]) return fail(FD_ERR_SHAPE, "out must be [B, Tq, Hq, D]");
  if (lse && (lse->shape[0] != d.B || lse->shape[1] != d.tq || lse->shape[2] != d.Hq))
    return fail(FD_ERR_SHAPE, "lse must be [B, Tq, Hq]");
  if (seqlens) {
    if (seqlens->dtype != FD_I32) return fail(FD_ERR_DTYPE, "seqlens must be int32");
    if (seqlens->shape[0] != d.B) return fail(FD_ERR_SHAPE, "seqlens must have B entries");
    if (seqlens->stride[0] != 1 && d.B > 1) return fail(FD_ERR_LAYOUT, "seqlens must be contiguous");
  }
  if (d.Hkv < 1 || d.Hq < 1 || d.Hq % d.Hkv != 0)
    return fail(FD_ERR_UNSUPPORTED, "Hq must be a positive multiple of Hkv");
  if (d.D != 64 && d.D != 128) return fail(FD_ERR_UNSUPPORTED, "head dim not in {64, 128}");
  if (d.B > 65535 || d.tq * d.Hq > 65535)
    return fail(FD_ERR_UNSUPPORTED, "batch and query tokens x heads must be <= 65535");
  if (d.Lcap > (int64_t)INT32_MAX - 2 * kSplitAlign) return fail(FD_ERR_UNSUPPORTED, "cache length too large");
  if (num_splits < 0 || num_splits > kMaxSplits)
    return fail(FD_ERR_ARG, "num_splits %d outside [0, %d]", num_splits, kMaxSplits);
  if (!std::isfinite(scale)) return fail(FD_ERR_ARG, "scale must be finite");
  d.G = d.Hq / d.Hkv;
  d.q_dt = q->dtype;
  d.kv_dt = k_cache->dtype;

  int dev;
  DeviceInfo* info;
  if ((st = current_device(&dev, &info))) return st;
  if (d.B == 0) return FD_OK;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int ns = num_splits > 0 ? num_splits : choose_splits_host(d.B, d.Hkv, d.Lcap, info->sms);
  const int32_t* sl = seqlens ? reinterpret_cast<const int32_t*>(seqlens->data) : nullptr;
  float* o = reinterpret_cast<float*>(out->data);
  float* l = lse ? reinterpret_cast<float*>(lse->data) : nullptr;
  const int64_t l0 = lse ? lse->stride[0] : 0, l1 = lse ? lse->stride[1] : 0,
                l2 = lse ? lse->stride[2] : 0;
  if (ns == 1)
    return enqueue_split(d, q, k_cache, v_cache, sl, 1, scale, o, out->stride[0], out->stride[2],
                         0, l, l0, l2, 0, false, cs, nullptr, out->stride[1], l1);
  // Partials [B, Tq, Hq, ns, D] and [B, Tq, Hq, ns], merged per (b, t, h).
  const int64_t rows = d.B * d.tq;
  const int64_t bytes = workspace_bytes(rows, d.Hq, d.D, ns);
  void* ws = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&ws, (size_t)bytes, info->pool, cs);
  if (e != cudaSuccess) return cuda_fail(e, "workspace allocation");
  float* po = reinterpret_cast<float*>(ws);
  float* pl = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) +
                                       ((rows * d.Hq * ns * d.D * 4 + 255) / 256) * 256);
  const int64_t po_h = ns * d.D, po_t = d.Hq * po_h, po_b = d.tq * po_t;
  const int64_t pl_h = ns, pl_t = d.Hq * pl_h, pl_b = d.tq * pl_t;
  st = enqueue_split(d, q, k_cache, v_cache, sl, ns, scale, po, po_b, po_h, d.D, pl, pl_b, pl_h, 1,
                     false, cs, nullptr, po_t, pl_t);
  if (st == FD_OK) {
    CombineParams cp = {};
    cp.part_o = po;
    cp.po_r1 = po_b;
    cp.po_rm = po_t;
    cp.po_r2 = po_h;
    cp.po_s = d.D;
    cp.part_lse = pl;
    cp.pl_r1 = pl_b;
    cp.pl_rm = pl_t;
    cp.pl_r2 = pl_h;
    cp.pl_s = 1;
    cp.out = o;
    cp.out_r1 = out->stride[0];
    cp.out_rm = out->stride[1];
    cp.out_r2 = out->stride[2];
    cp.lse = l;
    cp.lse_r1 = l0;
    cp.lse_rm = l1;
    cp.lse_r2 = l2;
    cp.R1 = (int)d.B;
    cp.Rm = (int)d.tq;
    cp.R2 = (int)d.Hq;
    cp.S = ns;
    cp.D = (int)d.D;
    st = enqueue_combine(cp, cs, true);
  }
  e = cudaFreeAsync(ws, cs);
  if (st) return st;
  if (e != cudaSuccess) return cuda_fail(e, "workspace release");
  return FD_OK;
}

fd_status fd_decode_attention_paged(const fd_tensor* q, const fd_tensor* k_pages,
                                    const fd_tensor* v_pages, const fd_tensor* block_table,
                                    const fd_tensor* seqlens, int32_t num_splits, float scale,
                                    fd_tensor* out, fd_tensor* lse, fd_stream stream) {
  fd_status st;
  if ((st = check_tensor(q, "q", 3))) return st;
  if ((st = check_tensor(k_pages, "k_pages", 4))) return st;
  if ((st = check_tensor(v_pages, "v_pages", 4))) return st;
  if ((st = check_tensor(block_table, "block_table", 2))) return st;
  if ((st = check_tensor(out, "out", 3))) return st;
  if (lse && (st = check_tensor(lse, "lse", 2))) return st;
  if (seqlens && (st = check_tensor(seqlens, "seqlens", 1))) return st;
  DecodeDesc d;
  d.B = q->shape[0];
  d.Hq = q->shape[1];
  d.D = q->shape[2];
  const int64_t P = k_pages->shape[0], ps = k_pages->shape[1];
  d.Hkv = k_pages->shape[2];
  for (int i = 0; i < 4; ++i)
    if (k_pages->shape[i] != v_pages->shape[i])
      return fail(FD_ERR_SHAPE, "k_pages and v_pages shapes differ");
  if (k_pages->shape[3] != d.D) return fail(FD_ERR_SHAPE, "k_pages head dim != q head dim");
  if (block_table->dtype != FD_I32) return fail(FD_ERR_DTYPE, "block_table must be int32");
  if (block_table->shape[0] != d.B) return fail(FD_ERR_SHAPE, "block_table must have B rows");
  if (block_table->stride[1] != 1 && block_table->shape[1] > 1)
    return fail(FD_ERR_LAYOUT, "block_table rows must be contiguous");
  if (ps < 1 || P < 1) return fail(FD_ERR_SHAPE, "k_pages must hold at least one page of one token");
  d.Lcap = block_table->shape[1] * ps;
  if (q->dtype != FD_BF16 && q->dtype != FD_F32) return fail(FD_ERR_DTYPE, "q must be bf16 or f32");
  if (k_pages->dtype != v_pages->dtype) return fail(FD_ERR_DTYPE, "k_pages and v_pages dtypes differ");
  if (k_pages->dtype != FD_BF16 && k_pages->dtype != FD_F32)
    return fail(FD_ERR_DTYPE, "k_pages / v_pages must be bf16 or f32");
  if (out->dtype != FD_F32 || (lse && lse->dtype != FD_F32)) return fail(FD_ERR_DTYPE, "out / lse must be f32");
  if (out->shape[0] != d.B || out->shape[1] != d.Hq || out->shape[2] != d.D)
    return fail(FD_ERR_SHAPE, "out must be [B, Hq, D]");
  if (lse && (lse->shape[0] != d.B || lse->shape[1] != d.Hq)) return fail(FD_ERR_SHAPE, "lse must be [B, Hq]");
  if (seqlens) {
    if (seqlens->dtype != FD_I32) return fail(FD_ERR_DTYPE, "seqlens must be int32");
    if (seqlens->shape[0] != d.B) return fail(FD_ERR_SHAPE, "seqlens must have B entries");
    if (seqlens->stride[0] != 1 && d.B > 1) return fail(FD_ERR_LAYOUT, "seqlens must be contiguous");
  }
  if (d.Hkv < 1 || d.Hq < 1 || d.Hq % d.Hkv != 0)
    return fail(FD_ERR_UNSUPPORTED, "Hq must be a positive multiple of Hkv");
  if (d.D != 64 && d.D != 128) return fail(FD_ERR_UNSUPPORTED, "head dim not in {64, 128}");
  if (d.B > 65535 || d.Hq > 65535) return fail(FD_ERR_UNSUPPORTED, "batch and query heads must be <= 65535");
  if (d.Lcap > (int64_t)INT32_MAX - 2 * kSplitAlign || P > INT32_MAX)
    return fail(FD_ERR_UNSUPPORTED, "paged cache too large");
  if (num_splits < 0 || num_splits > kMaxSplits)
    return fail(FD_ERR_ARG, "num_splits %d outside [0, %d]", num_splits, kMaxSplits);
  if (!std::isfinite(scale)) return fail(FD_ERR_ARG, "scale must be finite");
  d.G = d.Hq / d.Hkv;
  d.q_dt = q->dtype;
  d.kv_dt = k_pages->dtype;
  PageDesc pg = {reinterpret_cast<const int32_t*>(block_table->data), block_table->stride[0],
                 (int)ps, (int)P};
  return run_decode(d, q, k_pages, v_pages, seqlens, num_splits, scale, out, lse, stream, &pg);
}

fd_status fd_decode_attention_noalloc(const fd_tensor* q, const fd_tensor* k_cache,
                                      const fd_tensor* v_cache, const fd_tensor* seqlens,
                                      int32_t num_splits, float scale, fd_tensor* out,
                                      fd_tensor* lse, fd_stream stream) {
  DecodeDesc d;
  fd_status st = validate_decode(q, k_cache, v_cache, seqlens, out, lse, 3, 0, &d);
  if (st) return st;
  if (num_splits < 0 || num_splits > kMaxSplits)
    return fail(FD_ERR_ARG, "num_splits %d outside [0, %d]", num_splits, kMaxSplits);
  if (!std::isfinite(scale)) return fail(FD_ERR_ARG, "scale must be finite");
  NoAllocDevice* dev = nullptr;
  if ((st = noalloc_setup(&dev))) return st;
  if (d.B == 0 || d.Hq == 0) return FD_OK;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int ns = num_splits;
  if (ns == 0) {
    // The library's own choice never exceeds the scratch: the heuristic's
    // count, lowered to the largest that fits (one split needs no scratch).
    ns = choose_splits_host(d.B, d.Hkv, d.Lcap, dev->sms);
    while (ns > 1 && workspace_bytes(d.B, d.Hq, d.D, ns) > (int64_t)FD_NOALLOC_SCRATCH_BYTES) --ns;
  }
  const int32_t* sl = seqlens ? reinterpret_cast<const int32_t*>(seqlens->data) : nullptr;
  float* o = reinterpret_cast<float*>(out->data);
  float* l = lse ? reinterpret_cast<float*>(lse->data) : nullptr;
  if (ns == 1) {
    return enqueue_split(d, q, k_cache, v_cache, sl, 1, scale, o, out->stride[0], out->stride[1],
                         0, l, lse ? lse->stride[0] : 0, lse ? lse->stride[1] : 0, 0, false, cs);
  }
  const int64_t bytes = workspace_bytes(d.B, d.Hq, d.D, ns);
  if (bytes > (int64_t)FD_NOALLOC_SCRATCH_BYTES)
    return fail(FD_ERR_UNSUPPORTED,
                "partial results need %lld bytes (B=%lld, Hq=%lld, D=%lld, %d splits) but the "
                "static scratch holds %lld; use fewer splits or fd_decode_attention",
                (long long)bytes, (long long)d.B, (long long)d.Hq, (long long)d.D, ns,
                (long long)FD_NOALLOC_SCRATCH_BYTES);
  // Nothing in the scratch has to start at zero: the split kernel writes
  // every partial (O_i, lse_i) that the combine kernel then reads.
  float* po = reinterpret_cast<float*>(dev->scratch);
  float* pl = reinterpret_cast<float*>(reinterpret_cast<char*>(dev->scratch) +
                                       ((d.B * d.Hq * ns * d.D * 4 + 255) / 256) * 256);
  st = enqueue_split(d, q, k_cache, v_cache, sl, ns, scale, po, d.Hq * ns * d.D, ns * d.D, d.D,
                     pl, d.Hq * ns, ns, 1, false, cs);
  if (st) return st;
  CombineParams cp = {};
  cp.part_o = po;
  cp.po_r1 = d.Hq * ns * d.D;
  cp.po_r2 = ns * d.D;
  cp.po_s = d.D;
  cp.part_lse = pl;
  cp.pl_r1 = d.Hq * ns;
  cp.pl_r2 = ns;
  cp.pl_s = 1;
  cp.out = o;
  cp.out_r1 = out->stride[0];
  cp.out_r2 = out->stride[1];
  cp.lse = l;
  cp.lse_r1 = lse ? lse->stride[0] : 0;
  cp.lse_r2 = lse ? lse->stride[1] : 0;
  cp.R1 = (int)d.B;
  cp.R2 = (int)d.Hq;
  cp.S = ns;
  cp.D = (int)d.D;
  return enqueue_combine(cp, cs, true);
}

fd_status fd_decode_attention_partials(const fd_tensor* q, const fd_tensor* k_cache,
                                       const fd_tensor* v_cache, const fd_tensor* seqlens,
                                       int32_t num_splits, float scale, fd_tensor* part_o,
                                       fd_tensor* part_lse, fd_stream stream) {
  if (num_splits < 1 || num_splits > kMaxSplits)
    return fail(FD_ERR_ARG, "num_splits %d outside [1, %d]", num_splits, kMaxSplits);
  DecodeDesc d;
  fd_status st =
      validate_decode(q, k_cache, v_cache, seqlens, part_o, part_lse, 4, num_splits, &d);
  if (st) return st;
  if (!part_lse) return fail(FD_ERR_NULL, "part_lse is required");
  if (!std::isfinite(scale)) return fail(FD_ERR_ARG, "scale must be finite");
  int dev;
  DeviceInfo* info;
  if ((st = current_device(&dev, &info))) return st;
  if (d.B == 0 || d.Hq == 0) return FD_OK;
  const int32_t* sl = seqlens ? reinterpret_cast<const int32_t*>(seqlens->data) : nullptr;
  return enqueue_split(d, q, k_cache, v_cache, sl, num_splits, scale,
                       reinterpret_cast<float*>(part_o->data), part_o->stride[0],
                       part_o->stride[1], part_o->stride[2],
                       reinterpret_cast<float*>(part_lse->data), part_lse->stride[0],
                       part_lse->stride[1], part_lse->stride[2], false,
                       reinterpret_cast<cudaStream_t>(stream));
}

fd_status fd_lse_combine(const fd_tensor* part_o, const fd_tensor* part_lse, fd_tensor* out,
                         fd_tensor* lse, fd_stream stream) {
  fd_status st;
  if ((st = check_tensor(part_o, "part_o", 3))) return st;
  if ((st = check_tensor(part_lse, "part_lse", 2))) return st;
  if ((st = check_tensor(out, "out", 2))) return st;
  if (lse && (st = check_tensor(lse, "lse", 1))) return st;
  const int64_t R = part_o->shape[0], S = part_o->shape[1], D = part_o->shape[2];
  if (part_o->dtype != FD_F32 || part_lse->dtype != FD_F32 || out->dtype != FD_F32)
    return fail(FD_ERR_DTYPE, "combine tensors must be f32");
  if (lse && lse->dtype != FD_F32) return fail(FD_ERR_DTYPE, "lse must be f32");
  if (part_lse->shape[0] != R || part_lse->shape[1] != S)
    return fail(FD_ERR_SHAPE, "part_lse must be [R, S]");
  if (out->shape[0] != R || out->shape[1] != D) return fail(FD_ERR_SHAPE, "out must be [R, D]");
  if (lse && lse->shape[0] != R) return fail(FD_ERR_SHAPE, "lse must be [R]");
  if (D % 4 != 0 || D > 512 || D < 4) return fail(FD_ERR_UNSUPPORTED, "D must be a multiple of 4 in [4, 512]");
  if (S < 1 || S > 4096) return fail(FD_ERR_UNSUPPORTED, "S must be in [1, 4096]");
  if (R > INT32_MAX) return fail(FD_ERR_UNSUPPORTED, "too many rows");
  if (!aligned16(part_o->data) || part_o->stride[0] % 4 != 0 || part_o->stride[1] % 4 != 0)
    return fail(FD_ERR_LAYOUT, "part_o must be 16-byte aligned with strides multiple of 4");
  int dev;
  DeviceInfo* info;
  if ((st = current_device(&dev, &info))) return st;
  if (R == 0) return FD_OK;
  CombineParams cp = {};
  cp.part_o = reinterpret_cast<const float*>(part_o->data);
  cp.po_r1 = 0;
  cp.po_r2 = part_o->stride[0];
  cp.po_s = part_o->stride[1];
  cp.part_lse = reinterpret_cast<const float*>(part_lse->data);
  cp.pl_r1 = 0;
  cp.pl_r2 = part_lse->stride[0];
  cp.pl_s = part_lse->stride[1];
  cp.out = reinterpret_cast<float*>(out->data);
  cp.out_r1 = 0;
  cp.out_r2 = out->stride[0];
  cp.lse = lse ? reinterpret_cast<float*>(lse->data) : nullptr;
  cp.lse_r1 = 0;
  cp.lse_r2 = lse ? lse->stride[0] : 0;
  cp.R1 = 1;
  cp.R2 = (int)R;
  cp.S = (int)S;
  cp.D = (int)D;
  return enqueue_combine(cp, reinterpret_cast<cudaStream_t>(stream), false);
}

fd_status fd_bifurcated_attention_lse(const fd_tensor* q, const fd_tensor* k_ctx,
                                      const fd_tensor* v_ctx, const fd_tensor* k_dec,
                                      const fd_tensor* v_dec, const fd_tensor* dec_lens,
                                      float scale, int32_t ctx_splits, fd_tensor* out,
                                      fd_tensor* lse, fd_stream stream) {
  fd_status st;
  if ((st = check_tensor(q, "q", 3))) return st;
  if ((st = check_tensor(k_ctx, "k_ctx", 3))) return st;
  if ((st = check_tensor(v_ctx, "v_ctx", 3))) return st;
  if ((st = check_tensor(k_dec, "k_dec", 4))) return st;
  if ((st = check_tensor(v_dec, "v_dec", 4))) return st;
  if ((st = check_tensor(out, "out", 3))) return st;
  if (lse && (st = check_tensor(lse, "lse", 2))) return st;
  if (dec_lens && (st = check_tensor(dec_lens, "dec_lens", 1))) return st;
  const int64_t n = q->shape[0], Hq = q->shape[1], D = q->shape[2];
  const int64_t Lc = k_ctx->shape[0], Hkv = k_ctx->shape[1], Ld = k_dec->shape[1];
  for (int i = 0; i < 3; ++i)
    if (k_ctx->shape[i] != v_ctx->shape[i]) return fail(FD_ERR_SHAPE, "k_ctx and v_ctx shapes differ");
  for (int i = 0; i < 4; ++i)
    if (k_dec->shape[i] != v_dec->shape[i]) return fail(FD_ERR_SHAPE, "k_dec and v_dec shapes differ");
  if (k_ctx->shape[2] != D || k_dec->shape[3] != D) return fail(FD_ERR_SHAPE, "head dims differ");
  if (k_dec->shape[0] != n) return fail(FD_ERR_SHAPE, "k_dec must have n samples");
  if (k_dec->shape[2] != Hkv) return fail(FD_ERR_SHAPE, "k_dec and k_ctx kv heads differ");
  if (out->shape[0] != n || out->shape[1] != Hq || out->shape[2] != D)
    return fail(FD_ERR_SHAPE, "out must be [n, Hq, D]");
  if (lse && (lse->shape[0] != n || lse->shape[1] != Hq)) return fail(FD_ERR_SHAPE, "lse must be [n, Hq]");
  if (dec_lens) {
    if (dec_lens->dtype != FD_I32) return fail(FD_ERR_DTYPE, "dec_lens must be int32");
    if (dec_lens->shape[0] != n) return fail(FD_ERR_SHAPE, "dec_lens must have n entries");
    if (dec_lens->stride[0] != 1 && n > 1) return fail(FD_ERR_LAYOUT, "dec_lens must be contiguous");
  }
  for (const fd_tensor* t : {q, k_ctx, v_ctx, k_dec, v_dec})
    if (t->dtype != FD_BF16) return fail(FD_ERR_DTYPE, "bifurcated q/k/v must be bf16");
  if (out->dtype != FD_F32 || (lse && lse->dtype != FD_F32)) return fail(FD_ERR_DTYPE, "out/lse must be f32");
  if (Lc < 1) return fail(FD_ERR_SHAPE, "the shared context must hold at least one token");
  if (Hkv < 1 || Hq % Hkv != 0) return fail(FD_ERR_UNSUPPORTED, "Hq must be a multiple of Hkv");
  if (D != 64 && D != 128) return fail(FD_ERR_UNSUPPORTED, "head dim not in {64, 128}");
  if (n > 65535 || Hq > 65535) return fail(FD_ERR_UNSUPPORTED, "n and Hq must be <= 65535");
  if (Lc > (int64_t)INT32_MAX - 2 * kSplitAlign || Ld > (int64_t)INT32_MAX - 2 * kSplitAlign)
    return fail(FD_ERR_UNSUPPORTED, "lengths too large");
  if (ctx_splits < 0 || ctx_splits > kMaxSplits) return fail(FD_ERR_ARG, "ctx_splits out of range");
  if (!std::isfinite(scale)) return fail(FD_ERR_ARG, "scale must be finite");
  int dev;
  DeviceInfo* info;
  if ((st = current_device(&dev, &info))) return st;
  if (n == 0 || Hq == 0) return FD_OK;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

  // Tensor-core context path: head dim 128, 16-byte aligned bases and
  // strides (query rows are read as 16-byte vectors, K/V through TMA).
  const int64_t G = Hq / Hkv;
  bool tc_ok = bif_ctx_tensor_core_allowed() && D == 128 &&
                     aligned16(q->data) && aligned16(k_ctx->data) && aligned16(v_ctx->data) &&
                     (q->stride[1] * 2) % 16 == 0 && (q->stride[0] * 2) % 16 == 0 &&
                     q->stride[1] > 0 && (q->stride[0] > 0 || n == 1) &&
                     (k_ctx->stride[1] * 2) % 16 == 0 && (k_ctx->stride[0] * 2) % 16 == 0 &&
                     (v_ctx->stride[1] * 2) % 16 == 0 && (v_ctx->stride[0] * 2) % 16 == 0 &&
                     k_ctx->stride[1] > 0 && v_ctx->stride[1] > 0 && k_ctx->stride[0] > 0 &&
                     v_ctx->stride[0] > 0;
  // Tensor maps of the context K / V (the tensor-core path needs both).
  CUtensorMap tmK, tmV;
  if (tc_ok) {
    if ((st = get_encoder())) return st;
    tc_ok = make_3d_map(&tmK, k_ctx->data, D, Hkv, Lc, k_ctx->stride[1], k_ctx->stride[0], 1,
                        kBifTileTokens) &&
            make_3d_map(&tmV, v_ctx->data, D, Hkv, Lc, v_ctx->stride[1], v_ctx->stride[0], 1,
                        kBifTileTokens);
  }
  const int64_t mtiles = (n * G + 128 * kBifQueryTiles - 1) / (128 * kBifQueryTiles);
  // Decode part folded into the context kernel: each query tile's decode
  // tiles join its list of context tiles, masked per sample, and the list is
  // shared out evenly over the splits.  Used when a 128-row tile spans few
  // samples (G >= 16) and the decode caches can
  // be streamed by TMA; FD_BIF_FOLD = 0 turns it off (tuning and test knob,
  // read on every call).
  CUtensorMap tmKd, tmVd;
  bool fold = false;
  if (tc_ok && G >= 16 && Ld > 0) {
    const char* fe = getenv("FD_BIF_FOLD");
    fold = !(fe && fe[0] == '0') && aligned16(k_dec->data) && aligned16(v_dec->data);
    for (int i = 0; fold && i < 3; ++i)
      fold = (k_dec->stride[i] * 2) % 16 == 0 && (v_dec->stride[i] * 2) % 16 == 0 &&
             k_dec->stride[i] > 0 && v_dec->stride[i] > 0;
    fold = fold && make_kv_map(&tmKd, k_dec->data, n, Ld, Hkv, D, k_dec->stride[0],
                               k_dec->stride[1], k_dec->stride[2], kBifTileTokens, 64) &&
           make_kv_map(&tmVd, v_dec->data, n, Ld, Hkv, D, v_dec->stride[0], v_dec->stride[1],
                       v_dec->stride[2], kBifTileTokens, 64);
  }
  // Split count.  Folded: over the longest list a query tile can have (its
  // context tiles plus full decode caches of the most samples a tile spans).
  int64_t work_tokens = Lc;
  if (fold) {
    int64_t most = 1;
    for (int64_t t = 0; t < mtiles; ++t) {
      const int64_t m0 = t * 128, last = std::min<int64_t>(m0 + 128, n * G) - 1;
      most = std::max<int64_t>(most, last / G - m0 / G + 1);
    }
    work_tokens = ((Lc + kBifTileTokens - 1) / kBifTileTokens +
                   most * ((Ld + kBifTileTokens - 1) / kBifTileTokens)) * kBifTileTokens;
  }
  const int ns_ctx = ctx_splits > 0 ? ctx_splits
                     : tc_ok ? choose_ctx_splits(work_tokens, mtiles * Hkv, info->sms)
                             : choose_splits_host(n, Hkv, Lc, info->sms);
  // Decode part on the split kernel (not folded): about two CTAs per SM over
  // (sample, kv head) units, at most one 64-token tile per split.
  int ns_dec = 0;
  if (Ld > 0 && !fold) {
    int64_t want = (2 * (int64_t)info->sms) / (n * Hkv);
    // Tuning knob, read on every call: FD_BIF_DEC_SPLITS fixes the count.
    if (const char* e = getenv("FD_BIF_DEC_SPLITS")) {
      if (atoi(e) > 0) want = atoi(e);
    }
    const int64_t cap = (Ld + 63) / 64;
    if (want > cap) want = cap;
    if (want > kMaxSplits) want = kMaxSplits;
    ns_dec = want < 1 ? 1 : (int)want;
  }
  const int S = ns_ctx + ns_dec;
  const int64_t bytes = workspace_bytes(n, Hq, D, S);
  void* ws = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&ws, (size_t)bytes, info->pool, cs);
  if (e != cudaSuccess) return cuda_fail(e, "workspace allocation");
  // Partials slot-major, [S][n][Hq][D] and [S][n][Hq]: a context CTA's 128
  // rows are then one contiguous block (for one kv head).
  float* po = reinterpret_cast<float*>(ws);
  float* pl = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + ((n * Hq * S * D * 4 + 255) / 256) * 256);

  st = FD_OK;
  bool ctx_done = false;
  if (tc_ok) {
    // Context part on the tensor cores: rows (sample, head of the group).
    {
      {
        BifCtxParams bp = {};
        bp.q = reinterpret_cast<const uint16_t*>(q->data);
        bp.q_sb = q->stride[0];
        bp.q_sh = q->stride[1];
        bp.n = (int)n;
        bp.Hq = (int)Hq;
        bp.Hkv = (int)Hkv;
        bp.G = (int)G;
        bp.Lc = (int)Lc;
        bp.ns = ns_ctx;
        bp.rows = (int)(n * G);
        // A zero scale becomes 1e-30: every scaled score then rounds to an
        // exponent of 0 in fp32 (uniform weights, as scale 0 means), while
        // masked tail scores stay at -inf instead of 0 * inf = NaN.
        bp.scale_log2 = scale == 0.f ? 1e-30f : std::fabs(scale) * 1.4426950408889634f;
        bp.negate_q = scale < 0.f ? 1 : 0;
        bp.o = po;
        bp.o_sb = Hq * D;
        bp.o_sh = D;
        bp.o_ss = n * Hq * D;
        bp.lse = pl;
        bp.l_sb = Hq;
        bp.l_sh = 1;
        bp.l_ss = n * Hq;
        ProfRecord rec;
        const bool prof = prof_begin(FD_KERNEL_BIF_CTX, cs, &rec);
        bp.fold = fold ? 1 : 0;
        bp.dec_lens = dec_lens ? reinterpret_cast<const int32_t*>(dec_lens->data) : nullptr;
        bp.Ld = (int)Ld;
        // The query tile by one TMA load where the map can describe it
        // (tuning and test knob, read on every call: FD_BIF_Q_TMA = 0 keeps
        // the per-thread query loads).
        CUtensorMap tmQ = tmK;
        const char* qe = getenv("FD_BIF_Q_TMA");
        bp.q_tma = (!(qe && qe[0] == '0') &&
                    make_q_map(&tmQ, q->data, n, Hkv, G, D, q->stride[0], q->stride[1]))
                       ? 1 : 0;
        // The partial rows leave by TMA tensor stores where the same box
        // rule describes them (FD_BIF_O_TMA = 0: per-thread stores).
        CUtensorMap tmO = tmK;
        const char* oe = getenv("FD_BIF_O_TMA");
        bp.o_tma = (!(oe && oe[0] == '0') &&
                    make_o_map(&tmO, po, S, n, Hkv, G, D, bp.o_ss, bp.o_sb, bp.o_sh))
                       ? 1 : 0;
        e = launch_bif_ctx(bp, tmK, tmV, fold ? tmKd : tmK, fold ? tmVd : tmV, tmQ, tmO,
                           (int)mtiles, cs, !prof);
        prof_end(FD_KERNEL_BIF_CTX, cs, prof, rec);
        if (e != cudaSuccess) st = cuda_fail(e, "bifurcated context kernel launch");
        ctx_done = true;
      }
    }
  }
  if (st == FD_OK && !ctx_done) {
    // Context part on the split kernel: every sample reads the one shared
    // context through a batch-broadcast view (batch stride 0).
    DecodeDesc dc = {n, Hq, Hkv, D, Lc, Hq / Hkv, FD_BF16, FD_BF16};
    st = enqueue_split(dc, q, k_ctx, v_ctx, nullptr, ns_ctx, scale, po, Hq * D, D, n * Hq * D, pl,
                       Hq, 1, n * Hq, true, cs);
  }
  // Decode part: each sample's own tokens, ns_dec splits, written after
  // the context splits.
  if (st == FD_OK && ns_dec) {
    DecodeDesc dd = {n, Hq, Hkv, D, Ld, Hq / Hkv, FD_BF16, FD_BF16};
    st = enqueue_split(dd, q, k_dec, v_dec,
                       dec_lens ? reinterpret_cast<const int32_t*>(dec_lens->data) : nullptr,
                       ns_dec, scale, po + (int64_t)ns_ctx * n * Hq * D, Hq * D, D,
                       n * Hq * D, pl + (int64_t)ns_ctx * n * Hq, Hq, 1, n * Hq, false,
                       cs, nullptr, 0, 0, /*late_wait=*/ctx_done);
  }
  if (st == FD_OK) {
    CombineParams cp = {};
    cp.part_o = po;
    cp.po_r1 = Hq * D;
    cp.po_r2 = D;
    cp.po_s = n * Hq * D;
    cp.part_lse = pl;
    cp.pl_r1 = Hq;
    cp.pl_r2 = 1;
    cp.pl_s = n * Hq;
    cp.out = reinterpret_cast<float*>(out->data);
    cp.out_r1 = out->stride[0];
    cp.out_r2 = out->stride[1];
    cp.lse = lse ? reinterpret_cast<float*>(lse->data) : nullptr;
    cp.lse_r1 = lse ? lse->stride[0] : 0;
    cp.lse_r2 = lse ? lse->stride[1] : 0;
    cp.R1 = (int)n;
    cp.R2 = (int)Hq;
    cp.S = S;
    cp.D = (int)D;
    st = enqueue_combine(cp, cs, true);
  }
  e = cudaFreeAsync(ws, cs);
  if (st) return st;
  if (e != cudaSuccess) return cuda_fail(e, "workspace release");
  return FD_OK;
}

fd_status fd_bifurcated_attention(const fd_tensor* q, const fd_tensor* k_ctx,
                                  const fd_tensor* v_ctx, const fd_tensor* k_dec,
                                  const fd_tensor* v_dec, const fd_tensor* dec_lens, float scale,
                                  fd_tensor* out, fd_stream stream) {
  return fd_bifurcated_attention_lse(q, k_ctx, v_ctx, k_dec, v_dec, dec_lens, scale, 0, out,
                                     nullptr, stream);
}

fd_status fd_check_device_error(fd_stream stream) {
  unsigned int bits = 0;
  cudaError_t e = read_and_clear_device_error(&bits, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (bits & FD_DEVERR_TIMEOUT) return fail(FD_ERR_DEVICE_TIMEOUT, "a bounded device wait timed out");
  if (bits & FD_DEVERR_BOUNDS) return fail(FD_ERR_DEVICE_BOUNDS, "a length outside [0, capacity] was clamped");
  return FD_OK;
}

fd_status fd_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  for (int k = 0; k < FD_KERNEL_KINDS; ++k) {
    for (auto& r : g_prof.rec[k]) g_prof.pool.push_back(r);
    g_prof.rec[k].clear();
  }
  g_prof.on.store(on != 0, std::memory_order_relaxed);
  return FD_OK;
}

fd_status fd_profile_read(int32_t kind, int64_t* launches, double* total_ms) {
  if (kind < 0 || kind >= FD_KERNEL_KINDS) return fail(FD_ERR_ARG, "unknown kernel kind");
  if (!launches || !total_ms) return fail(FD_ERR_NULL, "output pointer is NULL");
  std::lock_guard<std::mutex> lock(g_prof_mu);
  double tot = 0.0;
  for (auto& r : g_prof.rec[kind]) {
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, r.start, r.stop);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
    tot += ms;
  }
  *launches = (int64_t)g_prof.rec[kind].size();
  *total_ms = tot;
  return FD_OK;
}

}  // extern "C"
