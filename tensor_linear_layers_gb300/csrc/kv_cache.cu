// Paged KV cache of the attention core ("vLLM Code Reading (Section 5)", §13:
// each rank's attention kernel writes the KV cache of the heads it holds; the
// model runner derives every new token's slot from the block table).
//
// Cache layout, per shard r: cache[r][block][offset][kv_per][hd] bf16, slot s =
// block * block_size + offset. Attention of new tokens over their requests'
// cached keys is HBM-bound at decode (every cached key and value is read once
// per step for a handful of queries), so it runs on the CUDA cores, split
// along the sequence (flash-decoding):
//
//   kv_write_kernel     each token's k and v heads of every shard to its slot
//   paged_attn_kernel   one CTA per (request, shard, kv head, sequence split):
//                       the queries of every q head that reads this kv head and
//                       every new token of the request, over the split's keys
//                       in chunks of 128: thread = key for q.k (key row read
//                       from its block), a warp per query for the running max
//                       and sum, thread = head dimension for p.v. Writes the
//                       split's (max, sum, unnormalised o) per query.
//   paged_combine_kernel the splits of every query merged (log-sum-exp), o / l
//                       rounded to bf16 into the attention output layout
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "gemm_tc.cuh"
#include "internal.h"

namespace tpl {

namespace {
constexpr int kHd = 128;
constexpr int kChunk = 128;     // keys per pass; one per thread
constexpr int kAttnThreads = 256;
constexpr int kStatusShape = -2;  // TP_ERR_SHAPE
}  // namespace

__global__ void kv_write_kernel(const __nv_bfloat16* __restrict__ qkv, int T, int t, long long sstride, int rstride,
                                int q_per, int kv_per,
                                const int* __restrict__ slots, long long n_slots, __nv_bfloat16* __restrict__ ck,
                                __nv_bfloat16* __restrict__ cv, int* __restrict__ status) {
  const int vec = kv_per * kHd / 8;                 // 16-byte vectors of one token's k (or v) heads
  const long long total = (long long)T * t * 2 * vec;
  for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    long long rest = it;
    const int c = (int)(rest % vec);
    rest /= vec;
    const int which = (int)(rest % 2);              // 0: k, 1: v
    rest /= 2;
    const int r = (int)(rest % t);
    const int i = (int)(rest / t);
    const int s = slots[i];
    if (s < 0) continue;                            // padding token
    if (s >= n_slots) {
      atomicExch(status, kStatusShape);
      continue;
    }
    const __nv_bfloat16* src = qkv + (size_t)r * sstride + (size_t)i * rstride + (q_per + which * kv_per) * kHd;
    __nv_bfloat16* dst = (which ? cv : ck) + ((size_t)r * n_slots + s) * kv_per * kHd;
    reinterpret_cast<uint4*>(dst)[c] = __ldg(reinterpret_cast<const uint4*>(src) + c);
  }
}

// 16-byte global -> shared copy without a register round trip; src_bytes 0 fills zeros
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most one committed group of this thread is still in flight
__device__ __forceinline__ void cp_async_wait_but_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Warp-level tensor-core product m16n8k16 (bf16 x bf16 -> fp32) and its operand loads.
__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ void ldsm_x4(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}

namespace {
constexpr int kRow = kHd + 8;                      // bf16 row stride in shared memory: ldmatrix rows hit distinct banks
constexpr int kMRows = 16;                         // query rows of one pass (the m16 tile)
constexpr int kPagedSmem = 2 * kChunk * kRow * 2 + 2 * kMRows * kRow * 2 + kMRows * kChunk * 4;
}  // namespace

// One CTA (8 warps) per (request, shard, kv head, split). The split's keys go in
// chunks of 128, staged in shared memory with 16-byte copies: the next chunk's
// keys load during this chunk's softmax and p . v, this chunk's values during its
// q . k (cp.async groups complete oldest first; a thread copies the same positions
// of every chunk). Up to 16 queries per pass (the q heads of the kv group times
// the request's new tokens) form the rows of m16n8k16 tensor-core products:
// S = Q K^T with warp w taking keys [16 w, 16 w + 16), O += P V with warp w
// taking head dimensions [16 w, 16 w + 16); the running max and sum are kept per
// query in fp32, P is rounded to bf16.
__global__ void __launch_bounds__(kAttnThreads)
    paged_attn_kernel(const PagedAttnParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __nv_bfloat16* ks = reinterpret_cast<__nv_bfloat16*>(smem);                     // [128 keys][kRow]
  __nv_bfloat16* vs = ks + kChunk * kRow;                                          // [128 keys][kRow]
  __nv_bfloat16* qsb = vs + kChunk * kRow;                                         // [16 queries][kRow]
  __nv_bfloat16* psb = qsb + kMRows * kRow;                                        // [16 queries][kRow] (keys)
  float (*sc)[kChunk] = reinterpret_cast<float (*)[kChunk]>(psb + kMRows * kRow);   // [16][128]
  __shared__ long long rowoff[2][kChunk];   // element offset of each key's row in the cache (-1: none), per chunk parity
  __shared__ float s_m[kMRows], s_l[kMRows], s_f[kMRows];
  __shared__ int s_pos[kMRows];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gr = lane >> 2, tq = lane & 3;   // fragment row group and column pair of this lane
  // item -> (request, shard, local kv head, split)
  int item = blockIdx.x;
  const int sp = item % p.n_splits;
  item /= p.n_splits;
  const int g = item % p.kv_per;
  item /= p.kv_per;
  const int r = item % p.t;
  const int b = item / p.t;
  const int q0 = p.qsl[b], n_new = p.qsl[b + 1] - q0;
  const int L = p.seq_lens[b];
  const int k0 = sp * p.split_len, k1 = min(L, k0 + p.split_len);
  if (n_new < 0 || n_new > p.max_query_len || L < n_new || L > p.max_seq_len) {
    if (tid == 0 && sp == 0 && r == 0 && g == 0) atomicExch(p.status, kStatusShape);
    return;
  }
  // the q heads of shard r that read local kv head g: [h0, h0 + gq)
  const int gq = p.q_per / (p.rep > 1 ? 1 : p.kv_per);
  const int h0 = g * gq;
  const int nq = n_new * gq;                       // queries of this item
  float* part = p.partials + (size_t)blockIdx.x * p.q_stride * (kHd + 2);
  auto lookup = [&](int c0, int par) {             // its row through the block table, one key per thread
    if (tid < kChunk) {
      const int key = c0 + tid;
      long long off = -1;
      if (key < k1) {
        const int blk = p.block_tables[(size_t)b * p.max_blocks + key / p.block_size];
        if (blk >= 0 && blk < p.num_blocks)
          off = (((long long)r * p.num_blocks + blk) * p.block_size + key % p.block_size) * p.kv_per * kHd + g * kHd;
        else
          atomicExch(p.status, kStatusShape);
      }
      rowoff[par][tid] = off;
    }
  };
  // 16-byte copies, 16 per row; missing rows read as zero (a committed group per call)
  auto load_rows = [&](__nv_bfloat16* dst, const __nv_bfloat16* cache, int par) {
#pragma unroll 4
    for (int e = tid; e < kChunk * 16; e += kAttnThreads) {
      const int row = e >> 4, c = e & 15;
      const long long ro = rowoff[par][row];
      const bool have = ro >= 0;
      cp_async16(dst + row * kRow + c * 8, cache + (have ? ro : 0) + c * 8, have ? 16 : 0);
    }
    cp_async_commit();
  };
  int ci = 0;   // chunks of this CTA so far: chunk ci uses rowoff[ci & 1]
  for (int qa = 0; qa < nq; qa += kMRows) {
    const int qc = min(kMRows, nq - qa);
    // the pass's queries as bf16 rows (rows past qc zero); query j: token q0 + (qa + j) / gq,
    // head h0 + (qa + j) % gq
    for (int e = tid; e < kMRows * kHd; e += kAttnThreads) {
      const int j = e / kHd, d = e - j * kHd;
      __nv_bfloat16 v = __float2bfloat16_rn(0.f);
      if (j < qc) {
        const int tok = q0 + (qa + j) / gq, h = h0 + (qa + j) % gq;
        v = p.qkv[(size_t)r * p.sstride_in + (size_t)tok * p.rstride_in + h * kHd + d];
      }
      qsb[j * kRow + d] = v;
      psb[j * kRow + d] = __float2bfloat16_rn(0.f);
    }
    if (tid < kMRows) {
      s_m[tid] = -INFINITY;
      s_l[tid] = 0.f;
      s_f[tid] = 0.f;
      s_pos[tid] = tid < qc ? L - n_new + (qa + tid) / gq : -1;
    }
    float oacc[2][4];                                // O rows gr, gr + 8; head dims 16 warp + 8 nt + 2 tq, +1
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) oacc[nt][i] = 0.f;
    if (k0 < k1) {
      lookup(k0, ci & 1);
      __syncthreads();
      load_rows(ks, p.cache_k, ci & 1);
      load_rows(vs, p.cache_v, ci & 1);
    }
    for (int c0 = k0; c0 < k1; c0 += kChunk, ++ci) {
      const int par = ci & 1;
      const bool more = c0 + kChunk < k1;
      if (more) lookup(c0 + kChunk, par ^ 1);
      cp_async_wait_but_one();             // this chunk's K (its V may still be in flight)
      __syncthreads();
      {
        // S = Q K^T for keys [16 warp, +16): 8 k-steps of 16 head dimensions, 2 n-tiles of 8 keys
        float cs[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < kHd / 16; ++kk) {
          uint32_t a[4], bk[4];
          ldsm_x4(a, qsb + ((lane & 7) + 8 * ((lane >> 3) & 1)) * kRow + 16 * kk + 8 * (lane >> 4));
          ldsm_x4(bk, ks + (16 * warp + (lane & 7) + 8 * (lane >> 4)) * kRow + 16 * kk + 8 * ((lane >> 3) & 1));
          mma_bf16_16816(cs[0], a, bk);
          mma_bf16_16816(cs[1], a, bk + 2);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = gr + 8 * (i >> 1), kl = 16 * warp + 8 * nt + 2 * tq + (i & 1);
            const int key = c0 + kl;
            if (row < qc)
              sc[row][kl] = (rowoff[par][kl] >= 0 && key <= s_pos[row]) ? cs[nt][i] * p.scale_log2 : -INFINITY;
          }
      }
      __syncthreads();
      // the keys are read: the next chunk's keys start loading
      if (more) load_rows(ks, p.cache_k, par ^ 1);
      else cp_async_commit();              // an empty group keeps the count uniform
      // running max and sum, a warp per query; P as bf16 rows for the product with V
      for (int j = warp; j < qc; j += kAttnThreads / 32) {
        float mx = -INFINITY;
        for (int e = lane; e < kChunk; e += 32) mx = fmaxf(mx, sc[j][e]);
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        const float m_old = s_m[j];
        const float m_new = fmaxf(m_old, mx);
        float sum = 0.f;
        for (int e = lane; e < kChunk; e += 32) {
          const float pe = m_new == -INFINITY ? 0.f : exp2f(sc[j][e] - m_new);
          psb[j * kRow + e] = __float2bfloat16_rn(pe);
          sum += pe;
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o2);
        if (lane == 0) {
          const float f = (m_old == -INFINITY) ? 0.f : exp2f(m_old - m_new);
          s_f[j] = f;
          s_l[j] = s_l[j] * f + sum;
          s_m[j] = m_new;
        }
      }
      cp_async_wait_but_one();             // this chunk's V (the next chunk's K may still be in flight)
      __syncthreads();
      {
        // O = O * f + P V for head dimensions [16 warp, +16): 8 k-steps of 16 keys, 2 n-tiles of 8
        const float f0 = s_f[gr], f1 = s_f[gr + 8];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          oacc[nt][0] *= f0;
          oacc[nt][1] *= f0;
          oacc[nt][2] *= f1;
          oacc[nt][3] *= f1;
        }
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk) {
          uint32_t a[4], bv[4];
          ldsm_x4(a, psb + ((lane & 7) + 8 * ((lane >> 3) & 1)) * kRow + 16 * kk + 8 * (lane >> 4));
          ldsm_x4_t(bv, vs + (16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1)) * kRow + 16 * warp + 8 * (lane >> 4));
          mma_bf16_16816(oacc[0], a, bv);
          mma_bf16_16816(oacc[1], a, bv + 2);
        }
      }
      __syncthreads();
      // the values are read: the next chunk's values start loading
      if (more) load_rows(vs, p.cache_v, par ^ 1);
    }
    // this split's partial result of every query of the pass
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = gr + 8 * (i >> 1);
        if (row < qc) part[(size_t)(qa + row) * (kHd + 2) + 16 * warp + 8 * nt + 2 * tq + (i & 1)] = oacc[nt][i];
      }
    if (tid < qc) {
      part[(size_t)(qa + tid) * (kHd + 2) + kHd] = s_m[tid];
      part[(size_t)(qa + tid) * (kHd + 2) + kHd + 1] = s_l[tid];
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kHd)
    paged_combine_kernel(const PagedAttnParams p) {
  // block -> (request, shard, (token, local q head) of the request)
  int idx = blockIdx.x;
  const int qi = idx % p.c_stride;
  idx /= p.c_stride;
  const int r = idx % p.t;
  const int b = idx / p.t;
  const int q0 = p.qsl[b], n_new = p.qsl[b + 1] - q0;
  const int gq = p.q_per / (p.rep > 1 ? 1 : p.kv_per);
  if (n_new < 0 || n_new > p.max_query_len) return;
  const int n_items_q = n_new * p.q_per;          // (token, local q head) pairs of the request and shard
  if (qi >= n_items_q) return;
  const int tok = qi / p.q_per, h = qi % p.q_per;  // local q head h reads local kv head h / gq
  const int g = h / gq;
  const int jq = tok * gq + (h - g * gq);          // its query index within item (b, r, g)
  const int L = p.seq_lens[b];
  const int ns = L > 0 ? min(p.n_splits, (L + p.split_len - 1) / p.split_len) : 0;
  const size_t item0 = (((size_t)b * p.t + r) * p.kv_per + g) * p.n_splits;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, p.partials[((item0 + s) * p.q_stride + jq) * (kHd + 2) + kHd]);
  float o = 0.f, l = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float* pj = p.partials + ((item0 + s) * p.q_stride + jq) * (kHd + 2);
    const float ms = pj[kHd];
    if (ms == -INFINITY) continue;
    const float f = exp2f(ms - M);
    o += pj[threadIdx.x] * f;
    l += pj[kHd + 1] * f;
  }
  const float val = l > 0.f ? o / l : 0.f;
  p.out[(size_t)r * p.sstride_out + (size_t)(q0 + tok) * p.rstride_out + h * kHd + threadIdx.x] = __float2bfloat16_rn(val);
}

cudaError_t launch_kv_write(const void* qkv, int T, int t, long long sstride, int rstride, int q_per, int kv_per,
                            const int* slots, long long n_slots, void* ck, void* cv, int* status, int nsm,
                            cudaStream_t st) {
  const long long work = (long long)T * t * 2 * (kv_per * kHd / 8);
  const int grid = (int)std::max<long long>(1, std::min<long long>((work + 255) / 256, 8LL * nsm));
  kv_write_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(qkv), T, t, sstride, rstride, q_per, kv_per,
                                        slots, n_slots,
                                        static_cast<__nv_bfloat16*>(ck), static_cast<__nv_bfloat16*>(cv), status);
  return cudaGetLastError();
}

cudaError_t launch_paged_attention(const PagedAttnParams& p, int n_reqs, cudaStream_t st) {
  const long long items = (long long)n_reqs * p.t * p.kv_per * p.n_splits;
  static bool attr_done = false;   // the same attribute on every device
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(paged_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPagedSmem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  paged_attn_kernel<<<(unsigned)items, kAttnThreads, kPagedSmem, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  paged_combine_kernel<<<(unsigned)((long long)n_reqs * p.t * p.c_stride), kHd, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace tpl
