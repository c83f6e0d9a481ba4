// Launch helper for one instantiation of the tcgen05 GEMM engine.
#pragma once
#include <atomic>
#include "gemm_tc.cuh"
#include "internal.h"

namespace tpl {

template <bool SWAP, int KIND, int BN, int KIND2 = -1>
cudaError_t launch_one(const CUtensorMap& map_act, const GemmParams& p, int grid, cudaStream_t st,
                       const CUtensorMap* map_act2 = nullptr, const GemmParams* p2 = nullptr) {
  using S = GemmShape<SWAP, KIND, BN>;
  auto kernel = tc_gemm_kernel<SWAP, KIND, BN, KIND2>;
  const CUtensorMap& m2 = map_act2 != nullptr ? *map_act2 : map_act;
  GemmParams q2{};
  if (p2 != nullptr) q2 = *p2;
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
  if (p.splits == 1) {
    kernel<<<grid, 192, S::kSmemBytes, st>>>(map_act, m2, p, q2);
    return cudaGetLastError();
  }
  // split-K ends in a grid-wide barrier: launch cooperatively so every CTA is resident
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = S::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, map_act, m2, p, q2);
}

}  // namespace tpl
