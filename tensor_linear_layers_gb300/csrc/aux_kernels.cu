// Memory-bound kernels of the block: fused residual add + RMSNorm, the
// activation-capture gather, and create-time weight packing into the shard
// layout.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>

#include "internal.h"

namespace tpl {

// ======================================================================= RMSNorm
// Per token row: r = a + residual (fp32, rounded to bf16 and stored as the
// updated residual); x = r_bf16 * rsqrt(mean(r_bf16^2) + eps) * gamma.
// "Tensor & pipeline parallelism", residual_stream: post_attention_layernorm
// folds the residual add and the norm together and returns both tensors.

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(b[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 f32_to_bf16x8(const float* f) {
  uint4 v;
  __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) b[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return v;
}

// One warp per row, kNormRows rows per CTA, so that an SM keeps dozens of rows' loads
// in flight (one CTA per row kept a few). Pass 1 loads a and the residual, kNormChunk
// vectors per lane at a time, all issued before any is used; it stores r and sums r^2.
// Pass 2 re-reads r (this thread's own stores, in L2) for x, so nothing of the row stays
// in registers and any H is handled.
constexpr int kNormRows = 8;
constexpr int kNormChunk = 8;

__global__ void __launch_bounds__(32 * kNormRows)
    add_rms_norm_kernel(const __nv_bfloat16* __restrict__ a, const __nv_bfloat16* __restrict__ res,
                        const __nv_bfloat16* __restrict__ gamma, float eps, int T, int H,
                        __nv_bfloat16* __restrict__ res_out, __nv_bfloat16* __restrict__ x_out) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kNormRows + (threadIdx.x >> 5);
  if (row >= T) return;
  const int nvec = H >> 3;
  const size_t roff = (size_t)row * H;
  const uint4* av = reinterpret_cast<const uint4*>(a + roff);
  const uint4* rv = res != nullptr ? reinterpret_cast<const uint4*>(res + roff) : nullptr;
  uint4* ro = reinterpret_cast<uint4*>(res_out + roff);
  float ss = 0.f;
  for (int v0 = 0; v0 < nvec; v0 += kNormChunk * 32) {
    uint4 la[kNormChunk], lr[kNormChunk];
#pragma unroll
    for (int k = 0; k < kNormChunk; ++k) {
      const int v = v0 + k * 32 + lane;
      if (v < nvec) {
        la[k] = __ldg(av + v);
        if (rv != nullptr) lr[k] = __ldg(rv + v);
      }
    }
#pragma unroll
    for (int k = 0; k < kNormChunk; ++k) {
      const int v = v0 + k * 32 + lane;
      if (v < nvec) {
        float fa[8], fr[8];
        bf16x8_to_f32(la[k], fa);
        if (rv != nullptr) {  // no residual (a model's first layer): r = a
          bf16x8_to_f32(lr[k], fr);
#pragma unroll
          for (int i = 0; i < 8; ++i) fa[i] += fr[i];
        }
        const uint4 packed = f32_to_bf16x8(fa);
        ro[v] = packed;
        bf16x8_to_f32(packed, fa);  // the stored (bf16) residual is what gets normalised
#pragma unroll
        for (int i = 0; i < 8; ++i) ss += fa[i] * fa[i];
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = rsqrtf(ss / (float)H + eps);
  const uint4* gv = reinterpret_cast<const uint4*>(gamma);
  uint4* xo = reinterpret_cast<uint4*>(x_out + roff);
  for (int v0 = 0; v0 < nvec; v0 += kNormChunk * 32) {
    uint4 lq[kNormChunk], lg[kNormChunk];
#pragma unroll
    for (int k = 0; k < kNormChunk; ++k) {
      const int v = v0 + k * 32 + lane;
      if (v < nvec) {
        lq[k] = ro[v];   // written by this thread above
        lg[k] = __ldg(gv + v);
      }
    }
#pragma unroll
    for (int k = 0; k < kNormChunk; ++k) {
      const int v = v0 + k * 32 + lane;
      if (v < nvec) {
        float q[8], g[8], o[8];
        bf16x8_to_f32(lq[k], q);
        bf16x8_to_f32(lg[k], g);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = q[i] * inv * g[i];
        xo[v] = f32_to_bf16x8(o);
      }
    }
  }
}

cudaError_t launch_add_rms_norm(int T, int H, const void* a, const void* res, const void* gamma,
                                float eps, void* res_out, void* x_out, cudaStream_t st) {
  add_rms_norm_kernel<<<(T + kNormRows - 1) / kNormRows, 32 * kNormRows, 0, st>>>(
      static_cast<const __nv_bfloat16*>(a), static_cast<const __nv_bfloat16*>(res),
      static_cast<const __nv_bfloat16*>(gamma), eps, T, H, static_cast<__nv_bfloat16*>(res_out),
      static_cast<__nv_bfloat16*>(x_out));
  return cudaGetLastError();
}
// Hidden sizes accepted with the norm (both norm kernels loop over any H; this is the
// range the library supports and tests for).
int max_norm_hidden() { return 16384; }

// ======================================================================= capture
// "Tensor & pipeline parallelism", What the adapter hooks / Duplicate records:
// select rows whose (request_id, token_pos) key was registered, record them
// per tensor in batch-row order; a key selected twice still yields one record.
constexpr int kCapThreads = 1024;
constexpr uint64_t kEmpty = 0xFFFFFFFFFFFFFFFFull;

__device__ __forceinline__ uint64_t mix64(uint64_t k) {
  // MurmurHash3 64-bit finaliser
  k ^= k >> 33;
  k *= 0xff51afd7ed558ccdull;
  k ^= k >> 33;
  k *= 0xc4ceb9fe1a85ec53ull;
  k ^= k >> 33;
  return k;
}

__device__ __forceinline__ uint64_t row_key(int req, int pos) {
  return (static_cast<uint64_t>(static_cast<uint32_t>(req)) << 32) | static_cast<uint32_t>(pos);
}

__global__ void __launch_bounds__(kCapThreads)
    capture_match_kernel(int T, const int32_t* __restrict__ row_req, const int32_t* __restrict__ row_pos,
                         const int64_t* __restrict__ sel, int n_sel, uint64_t* gtable, int cap_log2,
                         CaptureMeta meta, int64_t capacity, int64_t* n_out_dev,
                         int32_t* match_rows, int32_t* n_match_ws, int* status) {
  extern __shared__ uint64_t stable[];
  uint64_t* table = gtable != nullptr ? gtable : stable;
  const uint32_t cap = 1u << cap_log2;
  const uint32_t mask = cap - 1u;
  __shared__ int s_has_empty;
  __shared__ int warp_cnt[kCapThreads / 32];
  __shared__ int warp_off[kCapThreads / 32];
  __shared__ int s_chunk;
  __shared__ int s_running;
  if (threadIdx.x == 0) {
    s_has_empty = 0;
    s_running = 0;
  }
  for (uint32_t i = threadIdx.x; i < cap; i += kCapThreads) table[i] = kEmpty;
  __syncthreads();
  for (int i = threadIdx.x; i < n_sel; i += kCapThreads) {
    const uint64_t key = static_cast<uint64_t>(sel[i]);
    if (key == kEmpty) {
      s_has_empty = 1;
      continue;
    }
    uint32_t h = static_cast<uint32_t>(mix64(key)) & mask;
    for (uint32_t probe = 0; probe < cap; ++probe) {
      const unsigned long long prev =
          atomicCAS(reinterpret_cast<unsigned long long*>(table + h), kEmpty, key);
      if (prev == kEmpty || prev == key) break;
      h = (h + 1u) & mask;
    }
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  // rows in chunks of one CTA: flag, block-wide exclusive scan, order-preserving compaction
  for (int base = 0; base < T; base += kCapThreads) {
    const int i = base + threadIdx.x;
    int hit = 0;
    if (i < T) {
      const uint64_t key = row_key(row_req[i], row_pos[i]);
      if (key == kEmpty) {
        hit = s_has_empty;
      } else {
        // volatile: the table was filled with atomics at L2 and must not be read from a stale L1 line
        const volatile uint64_t* vt = table;
        uint32_t h = static_cast<uint32_t>(mix64(key)) & mask;
        for (uint32_t probe = 0; probe < cap; ++probe) {
          const uint64_t v = vt[h];
          if (v == key) {
            hit = 1;
            break;
          }
          if (v == kEmpty) break;
          h = (h + 1u) & mask;
        }
      }
    }
    const unsigned ball = __ballot_sync(0xffffffffu, hit);
    const int before = __popc(ball & ((1u << lane) - 1u));
    if (lane == 0) warp_cnt[wid] = __popc(ball);
    __syncthreads();
    if (wid == 0) {
      const int v = warp_cnt[lane];
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      warp_off[lane] = incl - v;
      if (lane == 31) s_chunk = incl;
    }
    __syncthreads();
    if (hit) match_rows[s_running + warp_off[wid] + before] = i;
    __syncthreads();
    if (threadIdx.x == 0) s_running += s_chunk;
    __syncthreads();
  }
  const int n_match = s_running;
  const int64_t n_rec = static_cast<int64_t>(meta.n_tensors) * n_match;
  if (threadIdx.x == 0) {
    *n_match_ws = n_match;
    *n_out_dev = n_rec;
    if (n_rec > capacity) atomicCAS(status, 0, kStatusCapacity);
  }
  const int64_t n_write = n_rec < capacity ? n_rec : capacity;
  for (int64_t j = threadIdx.x; j < n_write; j += kCapThreads) {
    const int k = static_cast<int>(j / n_match);
    const int m = static_cast<int>(j - static_cast<int64_t>(k) * n_match);
    const int row = match_rows[m];
    int32_t* h = meta.hdr + j * 6;
    h[0] = row_req[row];
    h[1] = row_pos[row];
    h[2] = meta.types[k];
    h[3] = meta.layer;
    h[4] = row;
    h[5] = 0;
  }
}

__global__ void __launch_bounds__(256)
    capture_copy_kernel(int H, CaptureMeta meta, int64_t capacity, const int32_t* __restrict__ match_rows,
                        const int32_t* __restrict__ n_match_ws, __nv_bfloat16* __restrict__ rows_out) {
  const int n_match = *n_match_ws;
  int64_t n_rec = static_cast<int64_t>(meta.n_tensors) * n_match;
  if (n_rec > capacity) n_rec = capacity;
  const int nvec = H >> 3;
  for (int64_t j = blockIdx.x; j < n_rec; j += gridDim.x) {
    const int k = static_cast<int>(j / n_match);
    const int m = static_cast<int>(j - static_cast<int64_t>(k) * n_match);
    const uint4* src = reinterpret_cast<const uint4*>(meta.tensors[k] + (size_t)match_rows[m] * H);
    uint4* dst = reinterpret_cast<uint4*>(rows_out + (size_t)j * H);
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) dst[v] = __ldg(src + v);
  }
}

// One launch for small selector sets (the table in shared memory) and T <= 64 * 256:
// every CTA builds the selector table and matches all T rows itself (a few KB, from
// L2), so no CTA waits for another and no list of matched rows goes through global
// memory; then each CTA copies records j = blockIdx.x, blockIdx.x + gridDim.x, ... and
// writes their headers. Thread t owns rows [t R, (t + 1) R), so a block-wide scan of
// the per-thread hit counts gives every match its place in batch-row order.
constexpr int kCapFusedThreads = 256;
constexpr int kCapFusedMaxRowsPerThread = 64;   // one 64-bit hit mask per thread

__global__ void __launch_bounds__(kCapFusedThreads)
    capture_fused_kernel(int T, int H, const int32_t* __restrict__ row_req, const int32_t* __restrict__ row_pos,
                         const int64_t* __restrict__ sel, int n_sel, int cap_log2, CaptureMeta meta,
                         int64_t capacity, int64_t* n_out_dev, int* status) {
  extern __shared__ uint64_t cap_smem[];
  uint64_t* table = cap_smem;                                               // 1 << cap_log2 slots
  int32_t* s_match = reinterpret_cast<int32_t*>(cap_smem + (1u << cap_log2));  // T entries
  __shared__ int s_has_empty;
  __shared__ int s_warp[kCapFusedThreads / 32];
  const uint32_t cap = 1u << cap_log2;
  const uint32_t mask = cap - 1u;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int R = (T + kCapFusedThreads - 1) / kCapFusedThreads;
  const int r0 = min(T, tid * R), r1 = min(T, r0 + R);
  if (tid == 0) s_has_empty = 0;
  for (uint32_t i = tid; i < cap; i += kCapFusedThreads) table[i] = kEmpty;
  __syncthreads();
  for (int i = tid; i < n_sel; i += kCapFusedThreads) {
    const uint64_t key = static_cast<uint64_t>(sel[i]);
    if (key == kEmpty) {
      s_has_empty = 1;
      continue;
    }
    uint32_t h = static_cast<uint32_t>(mix64(key)) & mask;
    for (uint32_t probe = 0; probe < cap; ++probe) {
      const unsigned long long prev = atomicCAS(reinterpret_cast<unsigned long long*>(table + h), kEmpty, key);
      if (prev == kEmpty || prev == key) break;
      h = (h + 1u) & mask;
    }
  }
  __syncthreads();
  // this thread's rows: hit bits, eight rows' keys loaded at a time
  uint64_t hits = 0;
  for (int c = r0; c < r1; c += 8) {
    int rq[8], ps[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (c + u < r1) {
        rq[u] = row_req[c + u];
        ps[u] = row_pos[c + u];
      }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (c + u < r1) {
        const uint64_t key = row_key(rq[u], ps[u]);
        bool hit = false;
        if (key == kEmpty) {
          hit = s_has_empty != 0;
        } else {
          uint32_t h = static_cast<uint32_t>(mix64(key)) & mask;
          for (uint32_t probe = 0; probe < cap; ++probe) {
            const uint64_t v = table[h];
            if (v == key) {
              hit = true;
              break;
            }
            if (v == kEmpty) break;
            h = (h + 1u) & mask;
          }
        }
        if (hit) hits |= 1ull << (c + u - r0);
      }
  }
  // exclusive scan of the hit counts over the block (thread order = row order)
  const int cnt = __popcll(hits);
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_warp[wid] = incl;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kCapFusedThreads / 32; ++w) {
    const int v = s_warp[w];
    if (w < wid) before += v;
    total += v;
  }
  int o = before + incl - cnt;
  for (uint64_t b = hits; b != 0ull; b &= b - 1ull) s_match[o++] = r0 + __ffsll(static_cast<long long>(b)) - 1;
  __syncthreads();
  const int n_match = total;
  const int64_t n_rec = static_cast<int64_t>(meta.n_tensors) * n_match;
  if (blockIdx.x == 0 && tid == 0) {
    *n_out_dev = n_rec;
    if (n_rec > capacity) atomicCAS(status, 0, kStatusCapacity);
  }
  const int64_t n_write = n_rec < capacity ? n_rec : capacity;
  const int nvec = H >> 3;
  __nv_bfloat16* rows_out = static_cast<__nv_bfloat16*>(meta.rows_out);
  for (int64_t j = blockIdx.x; j < n_write; j += gridDim.x) {
    const int k = static_cast<int>(j / n_match);
    const int m = static_cast<int>(j - static_cast<int64_t>(k) * n_match);
    const int row = s_match[m];
    if (tid == 0) {
      int32_t* hd = meta.hdr + j * 6;
      hd[0] = row_req[row];
      hd[1] = row_pos[row];
      hd[2] = meta.types[k];
      hd[3] = meta.layer;
      hd[4] = row;
      hd[5] = 0;
    }
    const uint4* src = reinterpret_cast<const uint4*>(meta.tensors[k] + (size_t)row * H);
    uint4* dst = reinterpret_cast<uint4*>(rows_out + (size_t)j * H);
    for (int v = tid; v < nvec; v += kCapFusedThreads) dst[v] = __ldg(src + v);
  }
}

cudaError_t launch_capture(int T, int H, const int32_t* row_req, const int32_t* row_pos,
                           const int64_t* sel, int n_sel, uint64_t* gtable, int cap_log2,
                           size_t table_smem, const CaptureMeta& meta, int64_t capacity,
                           int64_t* n_out_dev, int32_t* match_rows, int32_t* n_match_ws, int* status,
                           int copy_grid, cudaStream_t st) {
  // small selector sets: one launch (table and match list in each CTA's shared memory)
  const size_t fused_smem = table_smem + 4 * (size_t)T;
  if (gtable == nullptr && T <= kCapFusedThreads * kCapFusedMaxRowsPerThread && fused_smem <= 160 * 1024) {
    if (fused_smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(capture_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(fused_smem));
      if (e != cudaSuccess) return e;
    }
    capture_fused_kernel<<<copy_grid, kCapFusedThreads, fused_smem, st>>>(T, H, row_req, row_pos, sel, n_sel,
                                                                          cap_log2, meta, capacity, n_out_dev, status);
    return cudaGetLastError();
  }
  if (table_smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(capture_match_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(table_smem));
    if (e != cudaSuccess) return e;
  }
  capture_match_kernel<<<1, kCapThreads, table_smem, st>>>(T, row_req, row_pos, sel, n_sel, gtable,
                                                           cap_log2, meta, capacity, n_out_dev,
                                                           match_rows, n_match_ws, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  capture_copy_kernel<<<copy_grid, 256, 0, st>>>(H, meta, capacity, match_rows, n_match_ws,
                                                 static_cast<__nv_bfloat16*>(meta.rows_out));
  return cudaGetLastError();
}

// ======================================================================= packing
// Build the shard layout of a weight ("weight_loader": each rank narrows the
// full checkpoint tensor to its shard), tiled into 32 KB blocks of 256 rows x
// 64 K elements, each 16-byte chunk stored at its 128-byte-swizzled position:
// within a row rr of a block, logical chunk c sits at physical chunk
// c ^ (rr % 8). One thread writes one 16-byte chunk.
__global__ void __launch_bounds__(256) pack_tiles_kernel(PackSpec s, int64_t n_chunks, uint4* __restrict__ dst) {
  for (int64_t id = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; id < n_chunks;
       id += (int64_t)gridDim.x * blockDim.x) {
    const int64_t blk = id >> 11;          // 2048 chunks per block
    const int rr = (int)((id >> 3) & 255);
    const int c = (int)(id & 7) ^ (rr & 7);
    const int64_t wt = blk / s.nkb, kb = blk - wt * s.nkb;
    const __nv_bfloat16* src = nullptr;
    if (s.mode == PACK_GATE_UP) {
      // block = [128 gate rows | 128 up rows] of shard r, feature block b
      const int64_t r = wt / s.nb, b = wt - r * s.nb;
      const int64_t i = b * 128 + (rr & 127), k = kb * 64 + c * 8;
      if (i < s.Is && k < s.H) src = s.src[rr >> 7] + (r * s.Is + i) * s.H + k;
    } else if (s.mode == PACK_QKV) {
      // packed row n = [shard r: q heads | k heads | v heads]
      const int64_t n = wt * 256 + rr, k = kb * 64 + c * 8;
      if (n < s.n_col && k < s.H) {
        const int64_t r = n / s.ws, cc = n - r * s.ws;
        const int64_t qpart = (int64_t)s.q_per * s.hd, kvpart = (int64_t)s.kv_per * s.hd;
        if (cc < qpart) {
          src = s.src[0] + (r * qpart + cc) * s.H + k;
        } else {
          const int64_t e = cc - qpart;
          const int which = e < kvpart ? 1 : 2;
          const int64_t ek = e < kvpart ? e : e - kvpart;
          const int64_t head = (s.rep > 1) ? (r / s.rep) : (r * s.kv_per + ek / s.hd);
          src = s.src[which] + (head * s.hd + ek % s.hd) * s.H + k;
        }
      }
    } else {
      // PACK_ROW: output row n, global k-block kb = shard r, local k-block kk
      const int64_t n = wt * 256 + rr;
      const int64_t r = kb / s.kbs, kk = kb - r * s.kbs;
      const int64_t k = kk * 64 + c * 8;
      if (n < s.H && k < s.Is) src = s.src[0] + n * (s.t * s.Is) + r * s.Is + k;
    }
    dst[id] = src != nullptr ? *reinterpret_cast<const uint4*>(src) : make_uint4(0u, 0u, 0u, 0u);
  }
}

cudaError_t launch_pack(const PackSpec& s, int64_t n_blocks, void* dst, cudaStream_t st) {
  if (n_blocks <= 0) return cudaSuccess;
  const int64_t n_chunks = n_blocks * 2048;
  const int64_t grid = std::min<int64_t>((n_chunks + 255) / 256, 1 << 16);
  pack_tiles_kernel<<<(unsigned)grid, 256, 0, st>>>(s, n_chunks, static_cast<uint4*>(dst));
  return cudaGetLastError();
}

}  // namespace tpl
