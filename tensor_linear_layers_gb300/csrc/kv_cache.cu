// Paged KV cache of the attention core ("vLLM Code Reading (Section 5)", §13:
// each rank's attention kernel writes the KV cache of the heads it holds; the
// model runner derives every new token's slot from the block table).
//
// Cache layout, per shard r: cache[r][block][offset][kv_per][hd] bf16, slot s =
// block * block_size + offset. Attention of new tokens over their requests'
// cached keys is HBM-bound at decode (every cached key and value is read once
// per step for a handful of queries), so it is split along the sequence
// (flash-decoding) to fill the GPU, and its two small products per chunk of
// keys run as warp-level m16n8k16 tensor-core tiles:
//
//   kv_write_kernel     each token's k and v heads of every shard to its slot
//   paged_attn_kernel   one CTA per (request, shard, kv head, sequence split):
//                       the queries of every q head that reads this kv head and
//                       every new token of the request (16 per pass), over the
//                       split's keys in chunks of 128 staged in shared memory.
//                       Writes the split's (max, sum, unnormalised o) per query.
//   paged_merge_kernel  one CTA per (request, shard, kv head, query): the splits
//                       merged (log-sum-exp), o / l as bf16 in the attention
//                       output layout
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

// 16-byte global -> shared copy without a register round trip; src_bytes 0 fills zeros;
// pol: L2 eviction policy of the line read
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes, uint64_t pol) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(s), "l"(gmem), "r"(src_bytes),
               "l"(pol)
               : "memory");
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
constexpr int kMRows = 16;                               // query rows of one pass (the m16 tile)
constexpr int kWarps = kAttnThreads / 32;
constexpr int kPagedSmem = (2 * kChunk + 2 * kMRows) * kHd * 2;   // K, V, Q, P tiles (bf16, 256-byte rows)
}  // namespace

// Byte offset of element (row, col) of a bf16 tile with 256-byte rows: the 16-byte
// pieces of a row are permuted by the row's low three bits, so eight consecutive
// rows read at the same column (an ldmatrix) fall in eight distinct bank groups.
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return row * 256 + ((((col >> 3) ^ row) & 7) | ((col >> 3) & 8)) * 16 + (col & 7) * 2;
}

// One CTA (8 warps) per (request, shard, kv head, split). The split's keys go in
// chunks of 128, staged in shared memory with 16-byte copies: the next chunk's
// keys load during this chunk's softmax and p . v, this chunk's values during its
// q . k (cp.async groups complete oldest first; a thread copies the same positions
// of every chunk). Up to 16 queries per pass (the q heads of the kv group times
// the request's new tokens) form the rows of m16n8k16 tensor-core products:
// S = Q K^T with warp w taking keys [16 w, 16 w + 16), O += P V with warp w
// taking head dimensions [16 w, 16 w + 16). The softmax stays in the S
// fragments: the chunk's row maxima are exchanged through a small table, every
// lane keeps the running max of its two rows, each warp its partial row sums
// (merged at the end of the pass); P is rounded to bf16 for the second product.
__global__ void __launch_bounds__(kAttnThreads)
    paged_attn_kernel(const PagedAttnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ks = smem;                                      // [128 keys][128] bf16, swizzled
  uint8_t* vs = ks + kChunk * 256;                         // [128 keys][128]
  uint8_t* qsb = vs + kChunk * 256;                        // [16 queries][128]
  uint8_t* psb = qsb + kMRows * 256;                       // [16 queries][128 keys]
  __shared__ long long rowoff[2][kChunk];   // element offset of each key's k (or v) head in a cache (-1: none), per parity
  __shared__ float xch[kWarps][kMRows];                    // per-warp row maxima, then row sums
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gr = lane >> 2, tq = lane & 3;   // fragment row group and column pair of this lane
  griddep_launch_dependents();               // the merge grid may be scheduled once every split has started
  // item -> (request, shard, local kv head, split)
  int item = blockIdx.x;
  const int sp = item % p.n_splits;
  item /= p.n_splits;
  const int g = item % p.kv_per;
  item /= p.kv_per;
  const int r = item % p.t;
  const int b = item / p.t;
  const int k0 = sp * p.split_len;
  // the block-table entries of the first chunk's keys load together with the request's
  // offsets and length (they do not depend on them)
  int blk_first = -1;
  if (tid < kChunk && (k0 + tid) / p.block_size < p.max_blocks)
    blk_first = p.block_tables[(size_t)b * p.max_blocks + (k0 + tid) / p.block_size];
  const int q0 = p.qsl[b], n_new = p.qsl[b + 1] - q0;
  const int L = p.seq_lens[b];
  const int k1 = min(L, k0 + p.split_len);
  if (n_new < 0 || n_new > p.max_query_len || L < n_new || L > p.max_seq_len) {
    if (tid == 0 && sp == 0 && r == 0 && g == 0) atomicExch(p.status, kStatusShape);
    return;
  }
  // the q heads of shard r that read local kv head g: [h0, h0 + gq)
  const int gq = p.q_per / (p.rep > 1 ? 1 : p.kv_per);
  const int h0 = g * gq;
  const int nq = n_new * gq;                       // queries of this item
  const long long row_elems = (long long)p.kv_per * kHd;
  // The new tokens whose positions fall in this split: their k and v heads of (shard r,
  // kv head g) go to their slots first. No other CTA reads those positions, and this one
  // reads them back only after the barrier.
  if (p.slots != nullptr) {
    const int first = max(0, k0 - (L - n_new)), last = min(n_new, k1 - (L - n_new));   // new tokens [first, last)
    for (int e = tid; e < (last - first) * 32; e += kAttnThreads) {
      const int i = first + (e >> 5), which = (e >> 4) & 1, c = e & 15;   // which: 0 k, 1 v
      const int s = p.slots[q0 + i];
      if (s < 0) continue;                         // padding token
      if (s >= p.n_slots) {
        atomicExch(p.status, kStatusShape);
        continue;
      }
      const __nv_bfloat16* src = p.qkv + (size_t)r * p.sstride_in + (size_t)(q0 + i) * p.rstride_in +
                                 (p.q_per + which * p.kv_per + g) * kHd + c * 8;
      __nv_bfloat16* dst = (which ? p.cache_v : p.cache_k) + ((size_t)r * p.n_slots + s) * row_elems + g * kHd + c * 8;
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    }
    __syncthreads();
  }
  float* part = p.partials + (size_t)blockIdx.x * p.q_stride * (kHd + 2);
  // each key's cache row through the block table, one key per thread (blk: its entry, if loaded)
  auto lookup = [&](int c0, int par, bool have_blk, int blk) {
    if (tid < kChunk) {
      const int key = c0 + tid;
      long long off = -1;
      if (key < k1) {
        if (!have_blk) blk = p.block_tables[(size_t)b * p.max_blocks + key / p.block_size];
        if (blk >= 0 && blk < p.num_blocks)
          off = (long long)((r * p.num_blocks + blk) * p.block_size + key % p.block_size) * row_elems + g * kHd;
        else
          atomicExch(p.status, kStatusShape);
      }
      rowoff[par][tid] = off;
    }
  };
  // 16-byte copies, 16 per row; missing rows read as zero (a committed group per call). The
  // cache is read once per step: its lines go first from L2, the splits' partials stay.
  const uint64_t pol = policy_evict_first();
  // thread = 16-byte piece lc of rows lr, lr + 16, ..., lr + 112: its shared-memory
  // offsets differ by 16 rows, the same swizzle
  const int lr = tid >> 4, lc = tid & 15;
  const uint32_t ldst = swz(lr, lc * 8);
  auto load_rows = [&](uint8_t* dst, const __nv_bfloat16* cache, int par) {
#pragma unroll
    for (int k0 = 0; k0 < kChunk / 16; k0 += 4) {
      long long o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) o[k] = rowoff[par][lr + 16 * (k0 + k)];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        cp_async16(dst + ldst + (k0 + k) * 16 * 256, cache + (o[k] >= 0 ? o[k] : 0) + lc * 8, o[k] >= 0 ? 16 : 0, pol);
    }
    cp_async_commit();
  };
  // ldmatrix lane addresses: A tiles (rows 16, k 16) and the two B n-tiles of one k-step
  const int a_row = (lane & 7) + 8 * ((lane >> 3) & 1), a_col = 8 * (lane >> 4);
  const int bk_row = (lane & 7) + 8 * (lane >> 4), bk_col = 8 * ((lane >> 3) & 1);
  const int bv_row = (lane & 7) + 8 * ((lane >> 3) & 1), bv_col = 8 * (lane >> 4);
  int ci = 0;   // chunks of this CTA so far: chunk ci uses rowoff[ci & 1]
  for (int qa = 0; qa < nq; qa += kMRows) {
    const int qc = min(kMRows, nq - qa);
    // the first chunk's keys and values start loading
    if (k0 < k1) {
      lookup(k0, ci & 1, qa == 0, blk_first);
      __syncthreads();
      load_rows(ks, p.cache_k, ci & 1);
      load_rows(vs, p.cache_v, ci & 1);
    }
    // the pass's queries as bf16 rows (rows past qc zero); query j: token q0 + (qa + j) / gq,
    // head h0 + (qa + j) % gq
    for (int e = tid; e < kMRows * kHd / 8; e += kAttnThreads) {
      const int j = e >> 4, c = e & 15;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (j < qc) {
        const int tok = q0 + (qa + j) / gq, h = h0 + (qa + j) % gq;
        v = *reinterpret_cast<const uint4*>(p.qkv + (size_t)r * p.sstride_in + (size_t)tok * p.rstride_in + h * kHd +
                                            c * 8);
      }
      *reinterpret_cast<uint4*>(qsb + swz(j, c * 8)) = v;
    }
    // causal limit of this lane's rows gr and gr + 8 (-1: no query), and of the pass's first query
    const int pos_min = L - n_new + qa / gq;
    int pos[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int row = gr + 8 * h2;
      pos[h2] = row < qc ? L - n_new + (qa + row) / gq : -1;
    }
    float m_run[2] = {-INFINITY, -INFINITY}, l_w[2] = {0.f, 0.f};
    float oacc[2][4];                                // O rows gr, gr + 8; head dims 16 warp + 8 nt + 2 tq, +1
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) oacc[nt][i] = 0.f;
    for (int c0 = k0; c0 < k1; c0 += kChunk, ++ci) {
      const int par = ci & 1;
      const bool more = c0 + kChunk < k1;
      if (more) lookup(c0 + kChunk, par ^ 1, false, 0);
      cp_async_wait_but_one();             // this chunk's K (its V may still be in flight)
      __syncthreads();
      // S = Q K^T for keys [16 warp, +16): 8 k-steps of 16 head dimensions, 2 n-tiles of 8 keys
      float cs[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < kHd / 16; ++kk) {
        uint32_t a[4], bk[4];
        ldsm_x4(a, qsb + swz(a_row, 16 * kk + a_col));
        ldsm_x4(bk, ks + swz(16 * warp + bk_row, 16 * kk + bk_col));
        mma_bf16_16816(cs[0], a, bk);
        mma_bf16_16816(cs[1], a, bk + 2);
      }
      // scaled scores with the mask (missing key or after the query), and this warp's row maxima;
      // a chunk whose keys all exist and precede every query of the pass needs no mask (rows
      // without a query then score 0 and are never stored; a key of a block id out of range
      // reads zeros and has raised the status)
      float mloc[2] = {-INFINITY, -INFINITY};
      if (c0 + kChunk <= k1 && c0 + kChunk - 1 <= pos_min) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            cs[nt][i] *= p.scale_log2;
            mloc[i >> 1] = fmaxf(mloc[i >> 1], cs[nt][i]);
          }
      } else {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int kl = 16 * warp + 8 * nt + 2 * tq + (i & 1);
            const bool ok = rowoff[par][kl] >= 0 && c0 + kl <= pos[i >> 1];
            cs[nt][i] = ok ? cs[nt][i] * p.scale_log2 : -INFINITY;
            mloc[i >> 1] = fmaxf(mloc[i >> 1], cs[nt][i]);
          }
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        mloc[h2] = fmaxf(mloc[h2], __shfl_xor_sync(0xffffffffu, mloc[h2], 1));
        mloc[h2] = fmaxf(mloc[h2], __shfl_xor_sync(0xffffffffu, mloc[h2], 2));
        if (tq == 0) xch[warp][gr + 8 * h2] = mloc[h2];
      }
      __syncthreads();
      // the keys are read: the next chunk's keys start loading
      if (more) load_rows(ks, p.cache_k, par ^ 1);
      else cp_async_commit();              // an empty group keeps the count uniform
      // new running max of this lane's rows, P = 2^(s - m) as bf16, rescale factors
      float f[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float mx = m_run[h2];
#pragma unroll
        for (int w2 = 0; w2 < kWarps; ++w2) mx = fmaxf(mx, xch[w2][gr + 8 * h2]);
        f[h2] = m_run[h2] == -INFINITY ? 0.f : exp2f(m_run[h2] - mx);
        l_w[h2] *= f[h2];
        m_run[h2] = mx;
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const float mx = m_run[h2];
          const float p0 = mx == -INFINITY ? 0.f : exp2f(cs[nt][2 * h2] - mx);
          const float p1 = mx == -INFINITY ? 0.f : exp2f(cs[nt][2 * h2 + 1] - mx);
          l_w[h2] += p0 + p1;
          *reinterpret_cast<__nv_bfloat162*>(psb + swz(gr + 8 * h2, 16 * warp + 8 * nt + 2 * tq)) =
              __floats2bfloat162_rn(p0, p1);
        }
      cp_async_wait_but_one();             // this chunk's V (the next chunk's K may still be in flight)
      __syncthreads();
      // O = O * f + P V for head dimensions [16 warp, +16): 8 k-steps of 16 keys, 2 n-tiles of 8
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        oacc[nt][0] *= f[0];
        oacc[nt][1] *= f[0];
        oacc[nt][2] *= f[1];
        oacc[nt][3] *= f[1];
      }
#pragma unroll
      for (int kk = 0; kk < kChunk / 16; ++kk) {
        uint32_t a[4], bv[4];
        ldsm_x4(a, psb + swz(a_row, 16 * kk + a_col));
        ldsm_x4_t(bv, vs + swz(16 * kk + bv_row, 16 * warp + bv_col));
        mma_bf16_16816(oacc[0], a, bv);
        mma_bf16_16816(oacc[1], a, bv + 2);
      }
      __syncthreads();
      // the values are read: the next chunk's values start loading
      if (more) load_rows(vs, p.cache_v, par ^ 1);
    }
    // this split's partial result of every query of the pass: o per warp's head dimensions,
    // the running max (the same in every lane of a row), the row sums merged over lanes and warps
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = gr + 8 * (i >> 1);
        if (row < qc) part[(size_t)(qa + row) * (kHd + 2) + 16 * warp + 8 * nt + 2 * tq + (i & 1)] = oacc[nt][i];
      }
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      float l = l_w[h2];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      const int row = gr + 8 * h2;
      if (tq == 0) xch[warp][row] = l;
      if (warp == 0 && tq == 0 && row < qc) part[(size_t)(qa + row) * (kHd + 2) + kHd] = m_run[h2];
    }
    __syncthreads();
    if (tid < qc) {
      float l = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) l += xch[w2][tid];
      part[(size_t)(qa + tid) * (kHd + 2) + kHd + 1] = l;
    }
    __syncthreads();
  }
}

// One CTA per (request, shard, kv head, query slot), a thread per head dimension: the
// splits' partial results of the query merged (log-sum-exp, running over batches of
// eight splits whose max, sum and o are loaded together) and o / l written as bf16
// in the attention output layout. Launched behind the attention grid with
// programmatic serialisation: it is scheduled while the attention grid's last CTAs
// run and waits for its completion (griddepcontrol.wait) before reading a partial.
__global__ void __launch_bounds__(kHd)
    paged_merge_kernel(const PagedAttnParams p) {
  int idx = blockIdx.x;
  const int j = idx % p.q_stride;                          // query of the group
  idx /= p.q_stride;
  const int g = idx % p.kv_per;
  idx /= p.kv_per;
  const int r = idx % p.t;
  const int b = idx / p.t;
  const int q0 = p.qsl[b], n_new = p.qsl[b + 1] - q0;
  const int L = p.seq_lens[b];
  griddep_wait();
  if (n_new < 0 || n_new > p.max_query_len || L < n_new || L > p.max_seq_len) return;   // reported by the splits
  const int gq = p.q_per / (p.rep > 1 ? 1 : p.kv_per);
  if (j >= n_new * gq) return;
  const int d = threadIdx.x;
  const int ns = min(p.n_splits, (L + p.split_len - 1) / p.split_len);   // splits that hold keys
  const size_t split_stride = (size_t)p.q_stride * (kHd + 2);
  const float* pj = p.partials + (size_t)(blockIdx.x / p.q_stride) * p.n_splits * split_stride + (size_t)j * (kHd + 2);
  float M = -INFINITY, o = 0.f, l = 0.f;
  for (int s0 = 0; s0 < ns; s0 += 8) {
    float mb[8], lb[8], ob[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const bool have = s0 + i < ns;
      const float* ps = pj + (size_t)(s0 + i) * split_stride;
      mb[i] = have ? __ldcg(ps + kHd) : -INFINITY;
      lb[i] = have ? __ldcg(ps + kHd + 1) : 0.f;
      ob[i] = have ? __ldcg(ps + d) : 0.f;
    }
    float mn = M;
#pragma unroll
    for (int i = 0; i < 8; ++i) mn = fmaxf(mn, mb[i]);
    if (mn == -INFINITY) continue;
    const float f = M == -INFINITY ? 0.f : exp2f(M - mn);
    o *= f;
    l *= f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float w = mb[i] == -INFINITY ? 0.f : exp2f(mb[i] - mn);
      o += w * ob[i];
      l += w * lb[i];
    }
    M = mn;
  }
  const int tok = q0 + j / gq, h = g * gq + j % gq;
  p.out[(size_t)r * p.sstride_out + (size_t)tok * p.rstride_out + h * kHd + d] = __float2bfloat16_rn(l > 0.f ? o / l : 0.f);
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
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(paged_attn_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  paged_attn_kernel<<<(unsigned)items, kAttnThreads, kPagedSmem, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)((long long)n_reqs * p.t * p.kv_per * p.q_stride));
  cfg.blockDim = dim3(kHd);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, paged_merge_kernel, p);
}

}  // namespace tpl
