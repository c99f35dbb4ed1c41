// Shared device-side definitions of the eviction-step kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/bkv.h"
#include "ptx.cuh"

namespace bkv {

// Workspace header (bytes 0..255): status word and the site that set it.
struct WsHeader {
  int32_t status;
  int32_t site;
  int32_t pad[62];
};
constexpr size_t kWsHeaderBytes = 256;

// Sites that can record an error (reported through WsHeader::site).
enum ErrSite : int32_t {
  kSiteFpsState = 1,
  kSiteFpsWait = 2,
  kSiteScoreWait = 3,
  kSiteScoreState = 4,
  kSiteSelectState = 5,
  kSiteSelectWait = 6,
};

__device__ __forceinline__ void record_error(WsHeader* ws, int32_t code, int32_t site) {
  if (atomicCAS(&ws->status, 0, code) == 0) atomicExch(&ws->site, site);
}

// Bounded mbarrier wait measured in wall time (%globaltimer, ns).
constexpr uint64_t kWaitBudgetNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity,
                                         uint64_t budget_ns = kWaitBudgetNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && globaltimer() - t0 > budget_ns) return false;
  }
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Offset (bytes) of element e of row r inside a K-major operand stored as
// 128-byte-swizzled atoms of 64 bf16 columns: atoms of `rows` rows each are
// placed one after another along K.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t e, uint32_t rows) {
  const uint32_t atom = e >> 6, ce = e & 63u;
  const uint32_t chunk = (ce >> 3) ^ (r & 7u);
  return atom * rows * 128u + r * 128u + (chunk << 4) + ((ce & 7u) << 1);
}

// Host: raise a kernel's dynamic shared-memory limit to `bytes` once per
// (kernel, device) instead of on every call (the attribute is sticky).
inline cudaError_t set_smem_once(const void* fn, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(fn, dev);
  const auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes));
  if (e == cudaSuccess) done[key] = bytes;
  return e;
}

}  // namespace bkv
