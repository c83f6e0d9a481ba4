// Launch helper for one instantiation of the tcgen05 GEMM engine.
#pragma once
#include <atomic>
#include "gemm_tc.cuh"
#include "internal.h"

namespace tpl {

template <bool SWAP, int KIND, int BN, int NA>
cudaError_t launch_one(const CUtensorMap& map_act, const CUtensorMap& map_w, const GemmParams& p,
                       int grid, cudaStream_t st) {
  using S = GemmShape<SWAP, KIND, BN, NA>;
  auto kernel = tc_gemm_kernel<SWAP, KIND, BN, NA>;
  static std::atomic<uint64_t> attr_done{0};  // one bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  kernel<<<grid, 192, S::kSmemBytes, st>>>(map_act, map_w, p);
  return cudaGetLastError();
}

}  // namespace tpl
