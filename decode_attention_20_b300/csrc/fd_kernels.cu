// Device code of the decode-attention library and its host launchers.
// (All device code lives in this translation unit, so the device error word
// needs no relocatable device code.)
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <utility>

#include "fd_combine.cuh"
#include "fd_internal.h"
#include "fd_split.cuh"
#include "fd_split_mma.cuh"
#include "fd_bif_ctx.cuh"

namespace fd {

// Launch with cudaLaunchKernelEx; `pdl` adds programmatic stream
// serialisation, so the grid may start while the previous kernel on the
// stream finishes (every kernel here executes griddepcontrol.wait before its
// first global-memory access).
template <typename... KArgs, typename... Args>
static cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// The dynamic shared-memory opt-in of a kernel is per (function, device).
// `done` keeps one bit per device index below 64 (higher indices set the
// attribute on every call).  Atomic, since calls may come from several host
// threads; two threads that both set the attribute do no harm.
template <typename K>
static cudaError_t smem_optin(K kern, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

cudaError_t read_and_clear_device_error(unsigned int* bits, cudaStream_t st) {
  unsigned int zero = 0u;
  cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_device_error, sizeof(unsigned int), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(unsigned int), 0,
                              cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(st);
}

template <int GH, int HC>
static cudaError_t launch_tma_variant(const SplitParams& p, const CUtensorMap& tmK,
                                      const CUtensorMap& tmV, cudaStream_t st, bool pdl) {
  using C = TmaCfg<GH, HC>;
  auto kern = split_tma_kernel<GH, HC>;
  static std::atomic<unsigned long long> optin{0ull};
  const cudaError_t e = smem_optin(kern, C::SMEM_BYTES, optin);
  if (e != cudaSuccess) return e;
  return launch_ex(kern, dim3(p.ns, p.Hkv, p.B), dim3(C::THREADS), C::SMEM_BYTES, st, pdl, p,
                   tmK, tmV);
}

cudaError_t launch_split_tma(const SplitParams& p, const CUtensorMap& tmK,
                             const CUtensorMap& tmV, int D, int G, cudaStream_t st,
                             bool* launched, bool pdl) {
  *launched = false;
  if (D != 128) return cudaSuccess;
  *launched = true;
  switch (G) {
    case 1: return launch_tma_variant<1, 1>(p, tmK, tmV, st, pdl);
    case 2: return launch_tma_variant<2, 1>(p, tmK, tmV, st, pdl);
    case 4: return launch_tma_variant<4, 1>(p, tmK, tmV, st, pdl);
    case 8: return launch_tma_variant<8, 1>(p, tmK, tmV, st, pdl);
    case 16: return launch_tma_variant<8, 2>(p, tmK, tmV, st, pdl);
    case 32: return launch_tma_variant<8, 4>(p, tmK, tmV, st, pdl);
    case 64: return launch_tma_variant<8, 8>(p, tmK, tmV, st, pdl);
    default: *launched = false; return cudaSuccess;
  }
}

template <int KVQ, int NT, int WN, int W, int T, int NSTAGE>
static cudaError_t launch_mma_variant(const SplitParams& p, const CUtensorMap& tmK,
                                      const CUtensorMap& tmV, cudaStream_t st, bool pdl) {
  using C = MmaCfg<KVQ, NT, WN, W, T, NSTAGE>;
  auto kern = split_mma_kernel<KVQ, NT, WN, W, T, NSTAGE>;
  static std::atomic<unsigned long long> optin{0ull};
  const cudaError_t e = smem_optin(kern, C::SMEM_BYTES, optin);
  if (e != cudaSuccess) return e;
  return launch_ex(kern, dim3(p.ns, p.Hkv, p.B), dim3(C::THREADS), C::SMEM_BYTES, st, pdl, p,
                   tmK, tmV);
}

int mma_tile_tokens(int variant, int kv_kind) {
  if (kv_kind == kKvI8 || kv_kind == kKvE4m3) return variant == 2 ? 64 : 128;
  return variant == 1 ? 128 : 64;
}

template <int KVQ>
static cudaError_t launch_split_mma_kind(const SplitParams& p, const CUtensorMap& tmK,
                                         const CUtensorMap& tmV, int G, int variant,
                                         cudaStream_t st, bool* launched, bool pdl) {
  *launched = true;
  if (KVQ != 0 && variant == 2) {   // 8-bit: 4 warps, 64-token tiles (8 KB + 8 KB), 6 stages
    switch (G) {
      case 4: case 8: return launch_mma_variant<KVQ, 1, 1, 4, 64, 6>(p, tmK, tmV, st, pdl);
      case 16: return launch_mma_variant<KVQ, 2, 1, 4, 64, 6>(p, tmK, tmV, st, pdl);
      case 32: return launch_mma_variant<KVQ, 4, 2, 4, 64, 6>(p, tmK, tmV, st, pdl);
      case 64: return launch_mma_variant<KVQ, 8, 4, 4, 64, 6>(p, tmK, tmV, st, pdl);
      default: break;
    }
  } else if (KVQ != 0) {         // 8-bit: 128-token tiles (16 KB + 16 KB), 3 stages;
    switch (G) {                 // 8 warps (variant 1, one n-tile) or 4
      case 4: case 8:
        if (variant == 1) return launch_mma_variant<KVQ, 1, 1, 8, 128, 3>(p, tmK, tmV, st, pdl);
        return launch_mma_variant<KVQ, 1, 1, 4, 128, 3>(p, tmK, tmV, st, pdl);
      case 16: return launch_mma_variant<KVQ, 2, 1, 4, 128, 3>(p, tmK, tmV, st, pdl);
      case 32: return launch_mma_variant<KVQ, 4, 2, 4, 128, 3>(p, tmK, tmV, st, pdl);
      case 64: return launch_mma_variant<KVQ, 8, 4, 4, 128, 3>(p, tmK, tmV, st, pdl);
      default: break;
    }
  } else if (variant == 1) {     // 8 warps, 128-token tiles, 3 stages
    switch (G) {
      case 4: case 8: return launch_mma_variant<0, 1, 1, 8, 128, 3>(p, tmK, tmV, st, pdl);
      case 16: return launch_mma_variant<0, 2, 1, 8, 128, 3>(p, tmK, tmV, st, pdl);
      case 32: return launch_mma_variant<0, 4, 2, 8, 128, 3>(p, tmK, tmV, st, pdl);
      case 64: return launch_mma_variant<0, 8, 4, 8, 128, 3>(p, tmK, tmV, st, pdl);
      default: break;
    }
  } else if (variant == 2) {     // 4 warps, 64-token tiles, 3 stages (two CTAs per SM)
    switch (G) {
      case 4: case 8: return launch_mma_variant<0, 1, 1, 4, 64, 3>(p, tmK, tmV, st, pdl);
      case 16: return launch_mma_variant<0, 2, 1, 4, 64, 3>(p, tmK, tmV, st, pdl);
      case 32: return launch_mma_variant<0, 4, 2, 4, 64, 3>(p, tmK, tmV, st, pdl);
      case 64: return launch_mma_variant<0, 8, 4, 4, 64, 3>(p, tmK, tmV, st, pdl);
      default: break;
    }
  } else {                       // 4 warps, 64-token tiles, 6 stages
    switch (G) {
      case 4: case 8: return launch_mma_variant<0, 1, 1, 4, 64, 6>(p, tmK, tmV, st, pdl);
      case 16: return launch_mma_variant<0, 2, 1, 4, 64, 6>(p, tmK, tmV, st, pdl);
      case 32: return launch_mma_variant<0, 4, 2, 4, 64, 6>(p, tmK, tmV, st, pdl);
      case 64: return launch_mma_variant<0, 8, 4, 4, 64, 6>(p, tmK, tmV, st, pdl);
      default: break;
    }
  }
  *launched = false;
  return cudaSuccess;
}

cudaError_t launch_split_mma(const SplitParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             int G, int variant, cudaStream_t st, bool* launched, bool pdl) {
  // The n-tiles hold the kv head's rows: its G query heads, times the query
  // tokens for multi-token decode; round up to an instantiated row count.
  const int rows = G * (p.tq > 1 ? p.tq : 1);
  if (p.tq > 1) G = rows <= 8 ? 8 : rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : 0;
  switch (p.kv_kind) {
    case kKvBf16: return launch_split_mma_kind<0>(p, tmK, tmV, G, variant, st, launched, pdl);
    case kKvI8: return launch_split_mma_kind<1>(p, tmK, tmV, G, variant, st, launched, pdl);
    case kKvE4m3: return launch_split_mma_kind<2>(p, tmK, tmV, G, variant, st, launched, pdl);
    default: *launched = false; return cudaSuccess;
  }
}

template <int D>
static cudaError_t launch_generic_d(const SplitParams& p, cudaStream_t st, bool pdl) {
  const dim3 grid(p.ns, p.Hq * (p.tq > 1 ? p.tq : 1), p.B);
  switch (p.kv_kind) {
    case kKvF32: return launch_ex(split_generic_kernel<D, kKvF32>, grid, dim3(128), 0, st, pdl, p);
    case kKvBf16: return launch_ex(split_generic_kernel<D, kKvBf16>, grid, dim3(128), 0, st, pdl, p);
    case kKvI8: return launch_ex(split_generic_kernel<D, kKvI8>, grid, dim3(128), 0, st, pdl, p);
    case kKvE4m3: return launch_ex(split_generic_kernel<D, kKvE4m3>, grid, dim3(128), 0, st, pdl, p);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_split_generic(const SplitParams& p, int D, cudaStream_t st, bool pdl) {
  if (D == 128) return launch_generic_d<128>(p, st, pdl);
  if (D == 64) return launch_generic_d<64>(p, st, pdl);
  return cudaErrorInvalidValue;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t st, bool pdl) {
  const int rows = p.R1 * (p.Rm > 1 ? p.Rm : 1) * p.R2;   // Rm is 0 or 1 without query tokens
  if (rows > kCombineFewRows && p.S <= 32 && p.D <= 128) {
    const dim3 grid((rows + kCombineRowWarps - 1) / kCombineRowWarps);
    return p.Rm > 1 ? launch_ex(lse_combine_rows_kernel<true>, grid, dim3(kCombineRowWarps * 32),
                                0, st, pdl, p)
                    : launch_ex(lse_combine_rows_kernel<false>, grid, dim3(kCombineRowWarps * 32),
                                0, st, pdl, p);
  }
  if (rows > kCombineFewRows)
    return p.Rm > 1 ? launch_ex(lse_combine_many_kernel<true>, dim3(rows),
                                dim3(kCombineManyThreads), 0, st, pdl, p)
                    : launch_ex(lse_combine_many_kernel<false>, dim3(rows),
                                dim3(kCombineManyThreads), 0, st, pdl, p);
  const int threads = combine_threads(p.S, p.D);
  return p.Rm > 1 ? launch_ex(lse_combine_kernel<true>, dim3(rows), dim3(threads), 0, st, pdl, p)
                  : launch_ex(lse_combine_kernel<false>, dim3(rows), dim3(threads), 0, st, pdl, p);
}

cudaError_t launch_bif_ctx(const BifCtxParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const CUtensorMap& tmKd, const CUtensorMap& tmVd,
                           const CUtensorMap& tmQ, const CUtensorMap& tmO, int mtiles,
                           cudaStream_t st, bool pdl) {
  static std::atomic<unsigned long long> optin{0ull};
  const cudaError_t e = smem_optin(bif_ctx_kernel, BifCfg::SMEM_BYTES, optin);
  if (e != cudaSuccess) return e;
  return launch_ex(bif_ctx_kernel, dim3(mtiles, p.ns, p.Hkv), dim3(BifCfg::THREADS),
                   BifCfg::SMEM_BYTES, st, pdl, p, tmK, tmV, tmKd, tmVd, tmQ, tmO);
}

}  // namespace fd
