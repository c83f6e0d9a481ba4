// Mixture-of-experts routing around the grouped GEMMs ("Tensor Parallelism",
// MoE Expert Parallelism, Within-Expert Parallel: each expert's FFN is split
// with the dense column/row pattern; the routing is the caller's).
//
//   moe_route_kernel    one CTA: a stable counting sort of the T*k (token,
//                       slot) entries by expert. Each expert's rows start on
//                       a 128-row boundary, so no token tile mixes experts:
//                       tile m belongs to tile_expert[m], m < *m_valid.
//                       perm_row[entry] = its row; row_src[row] = its token
//                       (-1 for padding rows). For the CTA-pair engine it
//                       also lists each expert's tiles two by two
//                       (pair_tiles, -1 when an expert's last tile is alone)
//   moe_gather_kernel   x_perm[row] = x[row_src[row]] (zero for padding)
//   (grouped gate_up and down GEMMs on x_perm, per-tile expert weights)
//   moe_combine_kernel  y[i] = sum_j gate[i][j] * y_perm[perm_row[i*k + j]],
//                       fp32 in slot order, rounded once to bf16
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"

namespace tpl {

namespace {
constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;
}  // namespace

// Shared memory: cnt[E] running counts, off[E + 1] padded offsets, wcnt[32][E]
// per-warp counts of the current chunk (turned into per-warp bases in place).
__global__ void __launch_bounds__(kRouteThreads, 1)
    moe_route_kernel(const int* __restrict__ ids, int n_entries, int k, int E, int max_rows,
                     int* __restrict__ rank, int* __restrict__ perm_row, int* __restrict__ row_src,
                     int* __restrict__ tile_expert, int* __restrict__ m_valid, int* __restrict__ pair_tiles,
                     int* __restrict__ pair_count, int* __restrict__ status) {
  extern __shared__ int sm[];
  int* cnt = sm;
  int* off = cnt + E;
  int* wcnt = off + E + 1;
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int e = tid; e < E; e += kRouteThreads) cnt[e] = 0;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  // pass 1: rank of every entry among the entries of its expert, in entry order
  for (int c0 = 0; c0 < n_entries; c0 += kRouteThreads) {
    for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) wcnt[i] = 0;
    __syncthreads();
    const int i = c0 + tid;
    int e = -1;
    if (i < n_entries) {
      e = ids[i];
      if (e < 0 || e >= E) {
        atomicExch(&s_bad, 1);
        e = -1;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int in_warp = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && in_warp == 0) wcnt[w * E + e] = __popc(peers);
    __syncthreads();
    // per expert: exclusive scan over the warps of this chunk, added to the running count
    for (int x = tid; x < E; x += kRouteThreads) {
      int run = cnt[x];
      for (int ww = 0; ww < kRouteWarps; ++ww) {
        const int v = wcnt[ww * E + x];
        wcnt[ww * E + x] = run;
        run += v;
      }
      cnt[x] = run;
    }
    __syncthreads();
    if (e >= 0) rank[i] = wcnt[w * E + e] + in_warp;
    __syncthreads();
  }
  if (s_bad) {
    // ids out of range: no rows, every entry contributes nothing
    for (int i = tid; i < n_entries; i += kRouteThreads) perm_row[i] = -1;
    if (tid == 0) {
      *m_valid = 0;
      *pair_count = 0;
      atomicExch(status, -2);  // TP_ERR_SHAPE
    }
    return;
  }
  if (tid == 0) {
    int acc = 0;
    for (int x = 0; x < E; ++x) {
      off[x] = acc;
      acc += (cnt[x] + 127) & ~127;
    }
    off[E] = acc;
    *m_valid = acc / 128;
  }
  __syncthreads();
  const int rows = off[E];   // <= max_rows by construction of the workspace
  for (int r = tid; r < rows && r < max_rows; r += kRouteThreads) row_src[r] = -1;
  for (int m = tid; m < rows / 128; m += kRouteThreads) {
    int x = 0;
    while (off[x + 1] <= m * 128) ++x;
    tile_expert[m] = x;
  }
  if (tid == 0) {
    // pairs of tiles of one expert, experts in order (the CTA-pair engine)
    int np = 0;
    for (int x = 0; x < E; ++x) {
      const int t0 = off[x] / 128, nt = (off[x + 1] - off[x]) / 128;
      for (int i = 0; i < nt; i += 2) {
        pair_tiles[2 * np] = t0 + i;
        pair_tiles[2 * np + 1] = i + 1 < nt ? t0 + i + 1 : -1;
        ++np;
      }
    }
    *pair_count = np;
  }
  __syncthreads();
  for (int i = tid; i < n_entries; i += kRouteThreads) {
    const int row = off[ids[i]] + rank[i];
    perm_row[i] = row;
    row_src[row] = i / k;
  }
}

__global__ void moe_gather_kernel(const __nv_bfloat16* __restrict__ x, int H, const int* __restrict__ row_src,
                                  const int* __restrict__ m_valid, __nv_bfloat16* __restrict__ x_perm) {
  const int rows = *m_valid * 128;
  const int vec = H / 8;
  const long long total = (long long)rows * vec;
  for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(it / vec), c = (int)(it - (long long)r * vec);
    const int src = row_src[r];
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (src >= 0) v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)src * H) + c);
    reinterpret_cast<uint4*>(x_perm + (size_t)r * H)[c] = v;
  }
}

__global__ void moe_combine_kernel(const __nv_bfloat16* __restrict__ y_perm, int H, int T, int k,
                                   const int* __restrict__ perm_row, const float* __restrict__ gates,
                                   __nv_bfloat16* __restrict__ y) {
  const int vec = H / 8;
  const long long total = (long long)T * vec;
  for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const int i = (int)(it / vec), c = (int)(it - (long long)i * vec);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      const int row = perm_row[i * k + j];
      if (row < 0) continue;
      const float gw = gates[i * k + j];
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(y_perm + (size_t)row * H) + c);
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(b[q]);
        acc[2 * q] += gw * f.x;
        acc[2 * q + 1] += gw * f.y;
      }
    }
    uint4 o;
    __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int q = 0; q < 4; ++q) ob[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
    reinterpret_cast<uint4*>(y + (size_t)i * H)[c] = o;
  }
}

cudaError_t launch_moe_route(const int* ids, int n_entries, int k, int E, int max_rows, int* rank, int* perm_row,
                             int* row_src, int* tile_expert, int* m_valid, int* pair_tiles, int* pair_count,
                             int* status, cudaStream_t st) {
  const size_t smem = sizeof(int) * ((size_t)E + E + 1 + (size_t)kRouteWarps * E);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(moe_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  moe_route_kernel<<<1, kRouteThreads, smem, st>>>(ids, n_entries, k, E, max_rows, rank, perm_row, row_src,
                                                   tile_expert, m_valid, pair_tiles, pair_count, status);
  return cudaGetLastError();
}

cudaError_t launch_moe_gather(const void* x, int H, const int* row_src, const int* m_valid, int max_rows,
                              void* x_perm, int nsm, cudaStream_t st) {
  const long long work = (long long)max_rows * (H / 8);
  const int grid = (int)std::min<long long>((work + 255) / 256, 4LL * nsm);
  moe_gather_kernel<<<grid > 0 ? grid : 1, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), H, row_src, m_valid,
                                                          static_cast<__nv_bfloat16*>(x_perm));
  return cudaGetLastError();
}

cudaError_t launch_moe_combine(const void* y_perm, int H, int T, int k, const int* perm_row, const float* gates,
                               void* y, int nsm, cudaStream_t st) {
  const long long work = (long long)T * (H / 8);
  const int grid = (int)std::min<long long>((work + 255) / 256, 4LL * nsm);
  moe_combine_kernel<<<grid > 0 ? grid : 1, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(y_perm), H, T, k,
                                                           perm_row, gates, static_cast<__nv_bfloat16*>(y));
  return cudaGetLastError();
}

}  // namespace tpl
