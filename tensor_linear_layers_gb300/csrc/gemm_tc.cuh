// Persistent, warp-specialised tcgen05 GEMM engine for the tensor-parallel
// linear block.
//
//   warp 0      : producer (one elected thread): the weight block of a stage
//                 is one contiguous 32 KB bulk copy, the activation tile a
//                 TMA tensor copy; a ring of shared-memory stages guarded by
//                 full/empty mbarrier pairs
//   warp 1      : tensor-memory allocator + MMA issuer (one elected thread)
//   warps 2..5  : epilogue: tcgen05.ld from the fp32 accumulator, fused
//                 SiLU*mul / residual add, bf16 stores; split-K fix-up
//
// Weights are packed once, at create time, as blocks of 256 rows x 64 K
// elements (32 KB), already in the 128-byte-swizzled K-major image that the
// MMA reads from shared memory; block (w_tile, kb) lives at
// w_packed + (w_tile * nkb + kb) * 32 KB, so a unit of work streams one
// contiguous stretch of memory.
//
// Operand A feeds the UMMA M side (128 rows per accumulator, NA
// accumulators), operand B the N side (BN rows):
//   SWAP = false (prefill): A = 128 tokens, B = 256 weight rows (BN = 256).
//   SWAP = true  (decode) : A = 256 weight rows (two M=128 accumulators),
//                           B = the step's tokens (BN = 16 .. 128).
//
// Kinds:
//   KIND_GATE_UP : column-parallel merged gate/up. A weight block holds 128
//                  gate rows and the matching 128 up rows of one shard, so
//                  one thread holds g and u of the same intermediate feature
//                  and applies silu(g) * u in registers. Output h [t][T][I/t].
//   KIND_COL     : column-parallel plain store, output split per shard
//                  [t][T][w_s] (QKV by head).
//   KIND_ROW     : row-parallel: the K loop runs over all t shards in turn,
//                  so the shards' partial sums add up in the accumulator (the
//                  on-chip replacement of the all-reduce). Output y [T][N],
//                  optional y + residual.
//
// Split-K (splits > 1, few tiles): every unit writes its fp32 partial tile;
// after a grid-wide barrier (cooperative launch, so all CTAs are resident;
// the wait is bounded) all CTAs together add the partials of each tile in
// ascending split order (deterministic) and apply the epilogue.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <type_traits>
#include "ptx.cuh"

namespace tpl {

enum GemmKind : int { KIND_GATE_UP = 0, KIND_COL = 1, KIND_ROW = 2 };

constexpr int kStatusTimeout = -6;     // mirrors TP_ERR_TIMEOUT
// Waits on the way out (copies in flight landing, the last MMAs completing
// before tensor memory is freed) have their own limit, independent of the
// configurable one, so a short configured limit never cuts them short.
constexpr unsigned long long kTeardownNs = 20000000ull;
constexpr int kWBlockRows = 256;       // rows of one packed weight block
constexpr int kWBlockBytes = kWBlockRows * 128;  // 256 rows x 64 bf16

struct GemmParams {
  int T;             // tokens
  int m_tiles;       // tiles on the A (UMMA M) side
  int n_tiles;       // tiles on the B (UMMA N) side
  int splits;        // K splits per tile
  int units;         // m_tiles * n_tiles * splits
  int nkb;           // 64-wide k-blocks per tile (all shards for KIND_ROW)
  int kbs;           // k-blocks per shard (KIND_ROW)
  int nb;            // KIND_GATE_UP: 128-row gate blocks per shard
  int group_m;       // raster group along M (SWAP = false)
  int Is;            // KIND_GATE_UP: I / t
  int n_out;         // KIND_COL / KIND_ROW: output features
  int ws_out;        // KIND_COL: features per output shard (== n_out if unsplit)
  // KIND_GATE_UP / KIND_COL output of shard r, token m, feature c (within the shard):
  // out[r * out_sstride + m * out_rstride + c]. Shard-major [t][T][w]: (T * w, w);
  // gathered [T][t * w]: (w, t * w)
  long long out_sstride;
  int out_rstride;
  const uint8_t* w_packed;     // packed weight blocks
  __nv_bfloat16* out;
  __nv_bfloat16* out2;         // KIND_ROW: y + resid (nullable)
  const __nv_bfloat16* resid;  // KIND_ROW: residual [T][n_out]
  // Grouped problems (mixture of experts): token tile tm multiplies the weights of
  // expert tile_expert[tm] (expert_wbytes apart in w_packed), and only tiles
  // tm < *m_valid exist (both written on the device before the launch). Null for
  // one weight matrix. Only the unswapped, unsplit prefill engine takes them.
  const int* tile_expert;
  const int* m_valid;
  long long expert_wbytes;
  // CTA-pair engine on grouped problems: pair pm runs token tiles pair_tiles[2 pm]
  // and pair_tiles[2 pm + 1] (-1: no second tile), both of one expert; only pairs
  // pm < *pair_count exist
  const int* pair_tiles;
  const int* pair_count;
  // swapped KIND_GATE_UP only: per-token factor the gate and up accumulators are
  // multiplied by before SiLU*mul (the fused decode block's 1 / rms); null: none
  const float* inv;
  float* partials;             // split-K fp32 partials [tile][split][col][128 rows]
  unsigned* gbar;              // grid barrier {arrivals, generation}
  int* status;                 // device status word
  unsigned long long timeout_ns;
};

// Tail of a CTA-pair launch: the last `rem` pair units of the list are split into `s`
// parts along K, so that a last wave that would be less than half full runs as s
// shorter waves' worth of parts on more clusters. Each part writes its fp32 accumulator
// to `part` (per part and CTA rank: 128 rows x 256 columns); the last part of a unit to
// arrive (count in `cnt`, per unit and rank, reset by that part) adds the s partials in
// part order and applies the epilogue. s < 2: no split.
struct PairTail {
  int full;          // pair units run whole (the first `full` of the list)
  int rem;           // units split into parts
  int s;             // parts per split unit
  float* part;       // [rem][s][2][256 columns][128 rows] fp32
  unsigned* cnt;     // [rem][2]
};

// Parameters of the fused decode-shaped MLP block (mlp_decode.cu).
struct MlpDecodeParams {
  GemmParams g1;                 // KIND_GATE_UP, swapped operands
  GemmParams g2;                 // KIND_ROW, swapped operands
  const __nv_bfloat16* x_in;     // [T, H] (a, with the norm)
  const __nv_bfloat16* res_in;   // [T, H] or null
  const __nv_bfloat16* gamma;    // [H] (norm)
  __nv_bfloat16* res_out;        // [T, H] (norm)
  __nv_bfloat16* x_norm;         // [T, H] workspace (norm): y = bf16(r * gamma), gate_up's token operand
  float* inv;                    // [T] workspace (norm): 1 / rms of every row
  // Two sets of counters; a launch uses the set its launch count selects and clears the other.
  unsigned* bars;                // [0] norm arrivals, [1] CTAs that gave up waiting for the gate_up
                                 // CTAs to start, [2] gate_up tiles finished, [3] down units claimed;
                                 // set 1 at +4
  unsigned* cnt1;                // per gate_up tile: splits whose partial is written
  unsigned* hready;              // per gate_up tile: items of h written (complete at the tile's item count)
  unsigned* cnt2;                // per down tile: splits whose partial is written (low 16 bits) and the
                                 // splits that handed their slice of the sum to the last one (bit 16 + split)
  int cset;                      // words from set 0 to set 1 of cnt1 / hready / cnt2
  unsigned long long* epoch;     // completed launches in the high 32 bits (each CTA adds its share at exit)
  unsigned long long* ticket;    // CTAs started over all launches: a CTA's ticket mod grid is its place in
                                 // the start order of its launch (never cleared; grid fixed per workspace)
  int n_norm;                    // CTAs that own norm rows: the first n_norm to start
  float eps;
  int H;
  int has_norm;
};

template <bool SWAP, int KIND, int BN>
struct GemmShape {
  static constexpr int NA = SWAP ? 2 : 1;                // accumulators (128 rows each)
  static constexpr int kABytes = NA * 128 * 128;          // A tile: NA x 128 rows x 64 bf16
  static constexpr int kBBytes = BN * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kSmemBudget = 221 * 1024;
  static constexpr int kStagesRaw = kSmemBudget / kStageBytes;
  static constexpr int kStages = kStagesRaw > 12 ? 12 : kStagesRaw;
  static constexpr int kAccCols = NA * BN;  // tensor-memory columns per accumulator buffer
  static constexpr int kTmemNeed = 2 * kAccCols;
  static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256 : 512;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes;
  // epilogue segments: a segment is a run of kNG accumulator columns; GATE_UP
  // pairs each gate column with the up column kUOff further on
  static constexpr int kSeg = (SWAP && KIND != KIND_GATE_UP) ? 2 : 1;
  static constexpr int kNG = (KIND == KIND_GATE_UP && !SWAP) ? 128 : BN;
  static constexpr int kUOff = SWAP ? BN : 128;
  static constexpr int kCh = kNG >= 32 ? 32 : 16;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(128, BN);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128");
  static_assert(SWAP || BN == 256, "prefill tiles are 128 x 256");
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(kTmemNeed <= 512, "tensor memory");
};

// silu(g) = g * sigmoid(g). The fast division (2 ulp for denominators up to 2^126,
// 0 beyond, where silu is below 1e-36) costs a few instructions where the
// IEEE-rounded one costs a subroutine; the result is rounded to bf16 anyway.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Epilogue of N (multiple of 8) accumulator columns c0 .. c0+N-1 of segment
// `seg` in accumulator row `row`; g = values (gate for GATE_UP), u = up values.
// Writes N accumulator values of one row. For the swapped row-parallel kind,
// `rres` may hold the N residual values already loaded (else they are loaded
// here, all before the first store, so that they travel together).
template <bool SWAP, int KIND, int BN, int N>
__device__ __forceinline__ void emit_vals(const GemmParams& p, int tm, int tn, int seg, int row, int c0,
                                          const float* g, const float* u, const __nv_bfloat16* rres = nullptr) {
    if (!SWAP) {
      const int m = tm * 128 + row;
      if (m >= p.T) return;
      if (KIND == KIND_GATE_UP) {
        const int r = tn / p.nb, blk = tn - r * p.nb;
        const int i0 = blk * 128 + c0;
        __nv_bfloat16* dst = p.out + (size_t)r * p.out_sstride + (size_t)m * p.out_rstride + i0;
#pragma unroll
        for (int j = 0; j < N; j += 8) {
          if (i0 + j < p.Is) {
            uint4 v;
            v.x = pack_bf16x2(silu_f(g[j + 0]) * u[j + 0], silu_f(g[j + 1]) * u[j + 1]);
            v.y = pack_bf16x2(silu_f(g[j + 2]) * u[j + 2], silu_f(g[j + 3]) * u[j + 3]);
            v.z = pack_bf16x2(silu_f(g[j + 4]) * u[j + 4], silu_f(g[j + 5]) * u[j + 5]);
            v.w = pack_bf16x2(silu_f(g[j + 6]) * u[j + 6], silu_f(g[j + 7]) * u[j + 7]);
            *reinterpret_cast<uint4*>(dst + j) = v;
          }
        }
      } else if (KIND == KIND_COL) {
#pragma unroll
        for (int j = 0; j < N; j += 8) {
          const int n = tn * BN + c0 + j;
          if (n < p.n_out) {
            const int ro = n / p.ws_out, c = n - ro * p.ws_out;
            uint4 v;
            v.x = pack_bf16x2(g[j + 0], g[j + 1]);
            v.y = pack_bf16x2(g[j + 2], g[j + 3]);
            v.z = pack_bf16x2(g[j + 4], g[j + 5]);
            v.w = pack_bf16x2(g[j + 6], g[j + 7]);
            *reinterpret_cast<uint4*>(p.out + (size_t)ro * p.out_sstride + (size_t)m * p.out_rstride + c) = v;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < N; j += 8) {
          const int n = tn * BN + c0 + j;
          if (n < p.n_out) {
            const size_t off = (size_t)m * p.n_out + n;
            uint4 v;
            v.x = pack_bf16x2(g[j + 0], g[j + 1]);
            v.y = pack_bf16x2(g[j + 2], g[j + 3]);
            v.z = pack_bf16x2(g[j + 4], g[j + 5]);
            v.w = pack_bf16x2(g[j + 6], g[j + 7]);
            *reinterpret_cast<uint4*>(p.out + off) = v;
            if (p.out2 != nullptr) {
              const uint4 rv = *reinterpret_cast<const uint4*>(p.resid + off);
              const __nv_bfloat162* rb = reinterpret_cast<const __nv_bfloat162*>(&rv);
              const float2 r0 = __bfloat1622float2(rb[0]), r1 = __bfloat1622float2(rb[1]);
              const float2 r2 = __bfloat1622float2(rb[2]), r3 = __bfloat1622float2(rb[3]);
              uint4 w;
              w.x = pack_bf16x2(g[j + 0] + r0.x, g[j + 1] + r0.y);
              w.y = pack_bf16x2(g[j + 2] + r1.x, g[j + 3] + r1.y);
              w.z = pack_bf16x2(g[j + 4] + r2.x, g[j + 5] + r2.y);
              w.w = pack_bf16x2(g[j + 6] + r3.x, g[j + 7] + r3.y);
              *reinterpret_cast<uint4*>(p.out2 + off) = w;
            }
          }
        }
      }
    } else {
      // accumulator rows are output features, columns are tokens
      if (KIND == KIND_GATE_UP) {
        const int r = tm / p.nb, blk = tm - r * p.nb;
        const int i = blk * 128 + row;
        if (i >= p.Is) return;
        __nv_bfloat16* dst = p.out + (size_t)r * p.out_sstride + i;
#pragma unroll
        for (int j = 0; j < N; ++j) {
          const int tok = tn * BN + c0 + j;
          if (tok < p.T) {
            const float iv = p.inv != nullptr ? __ldcg(p.inv + tok) : 1.f;
            dst[(size_t)tok * p.out_rstride] = __float2bfloat16_rn(silu_f(g[j] * iv) * (u[j] * iv));
          }
        }
      } else if (KIND == KIND_COL) {
        const int f = tm * 256 + seg * 128 + row;
        if (f >= p.n_out) return;
        const int ro = f / p.ws_out, c = f - ro * p.ws_out;
        __nv_bfloat16* dst = p.out + (size_t)ro * p.out_sstride + c;
#pragma unroll
        for (int j = 0; j < N; ++j) {
          const int tok = tn * BN + c0 + j;
          if (tok < p.T) dst[(size_t)tok * p.out_rstride] = __float2bfloat16_rn(g[j]);
        }
      } else {
        const int f = tm * 256 + seg * 128 + row;
        if (f >= p.n_out) return;
        // residuals are loaded 8 tokens at a time, all before that group's stores
        static_assert(N % 8 == 0, "token groups");
        const __nv_bfloat16 z = __float2bfloat16_rn(0.f);
#pragma unroll
        for (int j0 = 0; j0 < N; j0 += 8) {
          __nv_bfloat162 rv[4];  // packed pairs keep registers low
          if (p.out2 != nullptr) {
#pragma unroll
            for (int j = j0; j < j0 + 8; j += 2) {
              const int tok = tn * BN + c0 + j;
              if (rres != nullptr) {
                rv[(j - j0) / 2] = __halves2bfloat162(rres[j], rres[j + 1]);
              } else {
                const __nv_bfloat16 a = tok < p.T ? p.resid[(size_t)tok * p.n_out + f] : z;
                const __nv_bfloat16 b = tok + 1 < p.T ? p.resid[(size_t)(tok + 1) * p.n_out + f] : z;
                rv[(j - j0) / 2] = __halves2bfloat162(a, b);
              }
            }
          }
#pragma unroll
          for (int j = j0; j < j0 + 8; ++j) {
            const int tok = tn * BN + c0 + j;
            if (tok < p.T) {
              const size_t off = (size_t)tok * p.n_out + f;
              p.out[off] = __float2bfloat16_rn(g[j]);
              if (p.out2 != nullptr) {
                const float r = ((j - j0) & 1) ? __high2float(rv[(j - j0) / 2]) : __low2float(rv[(j - j0) / 2]);
                p.out2[off] = __float2bfloat16_rn(g[j] + r);
              }
            }
          }
        }
      }
    }
}

// Split-K reduction of one tile's items [it_lo, it_hi): an item is 8 columns
// of one accumulator row (rows fastest). Adds the fp32 partials in ascending
// split order and applies the epilogue. Items are spread over `nthreads`
// threads, this one being `tid`; the loads of up to SC splits are all issued
// before they are added.
template <bool SWAP, int KIND, int BN>
__device__ __forceinline__ void reduce_tile_items(const GemmParams& p, int tile, int it_lo, int it_hi,
                                                  int tid, int nthreads) {
  using S = GemmShape<SWAP, KIND, BN>;
  constexpr int G = 8;
  constexpr int SC = (KIND == KIND_GATE_UP) ? 4 : 10;  // up to 10 splits in one round trip
  constexpr int ACC = S::kAccCols;
  constexpr bool kRes = SWAP && KIND == KIND_ROW;
  const float* tile_part = p.partials + (size_t)tile * p.splits * ACC * 128;
  const int tm = tile / p.n_tiles, tn = tile - tm * p.n_tiles;
  for (int it = it_lo + tid; it < it_hi; it += nthreads) {
    const int row = it & 127;
    const int c0 = (it >> 7) * G;
    const float* base_part = tile_part + row;
    // swapped row-parallel: the residual of the item's tokens is loaded along
    // with the partials instead of after them
    __nv_bfloat16 rres[G];
    if (kRes && p.out2 != nullptr) {
      const int seg = c0 / BN;
      const int f = tm * 256 + seg * 128 + row;
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const int tok = tn * BN + c0 - seg * BN + j;
        rres[j] = (f < p.n_out && tok < p.T) ? p.resid[(size_t)tok * p.n_out + f] : __float2bfloat16_rn(0.f);
      }
    }
    float g[G], u[G];
#pragma unroll
    for (int j = 0; j < G; ++j) g[j] = u[j] = 0.f;
    for (int s0 = 0; s0 < p.splits; s0 += SC) {
      float gv[SC][G], uv[SC][G];
#pragma unroll
      for (int s = 0; s < SC; ++s) {
        if (s0 + s < p.splits) {
          const float* ps = base_part + (size_t)(s0 + s) * ACC * 128;
#pragma unroll
          for (int j = 0; j < G; ++j) {
            gv[s][j] = __ldcg(ps + (size_t)(c0 + j) * 128);
            if (KIND == KIND_GATE_UP) uv[s][j] = __ldcg(ps + (size_t)(S::kUOff + c0 + j) * 128);
          }
        }
      }
#pragma unroll
      for (int s = 0; s < SC; ++s) {
        if (s0 + s < p.splits) {
#pragma unroll
          for (int j = 0; j < G; ++j) {
            g[j] += gv[s][j];
            if (KIND == KIND_GATE_UP) u[j] += uv[s][j];
          }
        }
      }
    }
    const int seg = (SWAP && KIND != KIND_GATE_UP) ? c0 / BN : 0;
    emit_vals<SWAP, KIND, BN, G>(p, tm, tn, seg, row, c0 - seg * BN, g, u,
                                 (kRes && p.out2 != nullptr) ? rres : nullptr);
  }
}
// Items of one tile: 8-column groups of the columns that own an output, x 128 rows.
template <bool SWAP, int KIND, int BN>
__host__ __device__ constexpr int tile_items() {
  using S = GemmShape<SWAP, KIND, BN>;
  return ((KIND == KIND_GATE_UP) ? S::kNG : S::kAccCols) / 8 * 128;
}

// Split-K reduction of every tile, spread over all threads of the grid.
template <bool SWAP, int KIND, int BN>
__device__ __forceinline__ void reduce_partials(const GemmParams& p, long long tid, long long nthreads) {
  constexpr int ITEMS = tile_items<SWAP, KIND, BN>();
  const long long total = (long long)p.m_tiles * p.n_tiles * ITEMS;
  for (long long it = tid; it < total; it += nthreads) {
    const int tile = (int)(it / ITEMS);
    const int i = (int)(it - (long long)tile * ITEMS);
    reduce_tile_items<SWAP, KIND, BN>(p, tile, i, i + 1, 0, 1);
  }
}

// Arrival counters used as grid-wide barriers between the phases of one
// launch. bar_arrive: one thread per CTA, after the CTA's writes (the
// fence makes them visible device-wide first). bar_wait: spin (with sleeps)
// until `n` CTAs have arrived; gives up after timeout_ns or when *abort is set.
__device__ __forceinline__ void bar_arrive(unsigned* c) {
  __threadfence();
  atomicAdd(c, 1u);
}
__device__ __forceinline__ bool bar_wait(const unsigned* c, unsigned n, unsigned long long timeout_ns,
                                         const volatile int* abort) {
  const volatile unsigned* v = c;
  if (*v >= n) {
    __threadfence();
    return true;
  }
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(32);
    if (*v >= n) {
      __threadfence();
      return true;
    }
    if ((it & 31u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
  }
}
// Order this thread's generic-proxy global writes before later async-proxy
// (TMA) reads of the same memory by other CTAs.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy reads of them (tensor-core operands).
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Grid-wide barrier for a cooperative launch, called by one thread per CTA.
// gbar[0] counts arrivals and is reset by the last CTA to arrive, which then
// bumps the generation gbar[1] that the others wait on. Bounded: returns
// false after timeout_ns.
__device__ __forceinline__ bool grid_barrier(unsigned* gbar, unsigned nblocks, unsigned long long timeout_ns) {
  volatile unsigned* vgen = gbar + 1;
  const unsigned gen = *vgen;
  __threadfence();
  const unsigned old = atomicAdd(gbar, 1u);
  if (old == nblocks - 1) {
    atomicExch(gbar, 0u);
    __threadfence();
    atomicAdd(gbar + 1, 1u);
    return true;
  }
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; *vgen == gen; ++it) {
    __nanosleep(64);
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > timeout_ns) return false;
  }
  __threadfence();
  return true;
}

// KIND2 >= 0 runs a second, independent problem (same operand shapes, split
// count 1) in the same launch: the units of both problems form one list that
// the persistent CTAs walk, so the two problems share the waves.
template <bool SWAP, int KIND, int BN, int KIND2 = -1>
__global__ void __launch_bounds__(192, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_act, const __grid_constant__ CUtensorMap map_act2,
                   const GemmParams p, const GemmParams p2) {
  using S = GemmShape<SWAP, KIND, BN>;
  constexpr bool kTwo = KIND2 >= 0;
  const int units_all = p.units + (kTwo ? p2.units : 0);
  constexpr int STAGES = S::kStages;
  constexpr int NA = S::NA;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t bar0 = base + STAGES * S::kStageBytes;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * STAGES + 4);
  uint8_t* misc = base_ptr + STAGES * S::kStageBytes + 8 * (2 * STAGES + 5);
  volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + 4);
  volatile int* s_ok = reinterpret_cast<volatile int*>(misc + 12);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 4);
    }
    mbar_init(done_bar, 1);
    *s_abort = 0;
    fence_barrier_init();
    prefetch_tensormap(&map_act);
    if (kTwo) prefetch_tensormap(&map_act2);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(s_tmem)), S::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  // unit of the combined list -> (problem, tile m, tile n, split)
  auto decode_unit = [&](int ug, bool& second, int& tm, int& tn, int& sp) {
    second = kTwo && ug >= p.units;
    const int u = second ? ug - p.units : ug;
    const GemmParams& q = second ? p2 : p;
    const int tile = u / q.splits;
    sp = u - tile * q.splits;
    if (!SWAP && q.group_m > 1) {
      const int group_size = q.group_m * q.n_tiles;
      const int g = tile / group_size;
      const int first_m = g * q.group_m;
      const int rem = q.m_tiles - first_m;
      const int gm = rem < q.group_m ? rem : q.group_m;
      const int in_g = tile - g * group_size;
      tm = first_m + in_g % gm;
      tn = in_g / gm;
    } else {
      tm = tile / q.n_tiles;
      tn = tile - tm * q.n_tiles;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // decode streams each weight byte once: keep it out of L2's way;
      // prefill re-reads weight blocks from L2 across token tiles
      const uint64_t pol_w = SWAP ? policy_evict_first() : policy_evict_normal();
      const uint64_t pol_a = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, last_phase_bits = 0;
      bool ok = true;
      for (int ug = blockIdx.x; ug < units_all && ok; ug += gridDim.x) {
        int tm, tn, sp;
        bool second;
        decode_unit(ug, second, tm, tn, sp);
        const GemmParams& q = second ? p2 : p;
        if (!SWAP && q.tile_expert != nullptr && tm >= *q.m_valid) continue;
        const CUtensorMap* map = second ? &map_act2 : &map_act;
        const bool row_kind = second ? (KIND2 == KIND_ROW) : (KIND == KIND_ROW);
        const int kb0 = (int)((long long)sp * q.nkb / q.splits);
        const int kb1 = (int)((long long)(sp + 1) * q.nkb / q.splits);
        const int wt = SWAP ? tm : tn;
        const uint8_t* wsrc = q.w_packed + (size_t)wt * q.nkb * kWBlockBytes;
        if (!SWAP && q.tile_expert != nullptr) wsrc += (size_t)q.tile_expert[tm] * (size_t)q.expert_wbytes;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, s_abort, p.timeout_ns)) {
            if (!*s_abort) {
              atomicExch(p.status, kStatusTimeout);
              *s_abort = 1;
            }
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * S::kStageBytes;
          const uint32_t sb = sa + S::kABytes;
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, S::kStageBytes);
          int kx = kb * 64, shard = 0;
          if (row_kind) {
            shard = kb / q.kbs;
            kx = (kb - shard * q.kbs) * 64;
          }
          const uint8_t* wblk = wsrc + (size_t)kb * kWBlockBytes;
          if (!SWAP) {
            tma_load_4d(sa, map, fb, kx, tm * 128, 0, shard, pol_a);        // 128 tokens
            bulk_load(sb, wblk, kWBlockBytes, fb, pol_w);                   // 256 weight rows
          } else {
            bulk_load(sa, wblk, kWBlockBytes, fb, pol_w);                   // 256 weight rows
            tma_load_4d(sb, map, fb, kx, tn * BN, 0, shard, pol_a);         // BN tokens
          }
          issued_mask |= 1u << stage;
          last_phase_bits = (last_phase_bits & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // drain: let copies already in flight land before the CTA exits
        for (int s = 0; s < STAGES; ++s)
          if (issued_mask & (1u << s))
            mbar_wait_bounded(full_bar(s), (last_phase_bits >> s) & 1u, nullptr, kTeardownNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and one elected lane issues each k-block's MMAs with
    // their commit, so descriptors and tensor-memory addresses stay warp-uniform
    // (elect.sync picks the same lane for the same mask: every commit follows the MMAs).
    {
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      auto timed_out = [&]() {
        if (lane == 0 && !*s_abort) {
          atomicExch(p.status, kStatusTimeout);
          *s_abort = 1;
        }
      };
      for (int ug = blockIdx.x; ug < units_all && ok; ug += gridDim.x) {
        int tm, tn, sp;
        bool second;
        decode_unit(ug, second, tm, tn, sp);
        const GemmParams& q = second ? p2 : p;
        if (!SWAP && q.tile_expert != nullptr && tm >= *q.m_valid) continue;
        const int kb0 = (int)((long long)sp * q.nkb / q.splits);
        const int kb1 = (int)((long long)(sp + 1) * q.nkb / q.splits);
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(tempty_bar(buf), acc_phase ^ 1u, s_abort, p.timeout_ns))) {
          timed_out();
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * S::kAccCols;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(full_bar(stage), phase, s_abort, p.timeout_ns))) {
            timed_out();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + stage * S::kStageBytes;
          const uint32_t sb = sa + S::kABytes;
          const uint64_t adesc = smem_desc_k128(sa);
          const uint64_t bdesc = smem_desc_k128(sb);
          if (elect_one()) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
              for (int a = 0; a < NA; ++a) {
                tc_mma_bf16(d_tmem + a * BN, adesc + (uint64_t)(a * (128 * 128 >> 4) + ks * 2),
                            bdesc + (uint64_t)(ks * 2), S::kIdesc, (kb > kb0 || ks > 0) ? 1u : 0u);
              }
            }
            tc_commit(empty_bar(stage));
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one()) tc_commit(tfull_bar(buf));
        __syncwarp();
        if (++buf == 2) {
          buf = 0;
          acc_phase ^= 1u;
        }
      }
      // all issued MMAs complete before tensor memory is released
      if (elect_one()) tc_commit(done_bar);
      __syncwarp();
      mbar_wait_bounded(done_bar, 0, nullptr, kTeardownNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;              // tensor-memory lane quadrant of this warp
    const int row = q * 32 + lane;       // row of the 128-row accumulator
    const int et = threadIdx.x - 64;     // 0..127
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    int buf = 0;
    uint32_t acc_phase = 0;
    constexpr int CH = S::kCh;
    constexpr int ACC = S::kAccCols;

    for (int ug = blockIdx.x; ug < units_all; ug += gridDim.x) {
      int tm, tn, sp;
      bool second;
      decode_unit(ug, second, tm, tn, sp);
      if (!SWAP && (second ? p2 : p).tile_expert != nullptr && tm >= *(second ? p2 : p).m_valid) continue;
      // one thread waits and the decision is shared, so all 128 epilogue
      // threads leave together and no named barrier is left half-joined
      if (et == 0) {
        const bool ok = mbar_wait_bounded(tfull_bar(buf), acc_phase, s_abort, p.timeout_ns);
        if (!ok && !*s_abort) {
          atomicExch(p.status, kStatusTimeout);
          *s_abort = 1;
        }
        *s_ok = ok ? 1 : 0;
      }
      named_bar_sync(1, 128);
      const int ok = *s_ok;
      named_bar_sync(1, 128);
      if (!ok) break;
      tc_fence_after();
      const uint32_t acc = lane_addr + buf * ACC;
      const int tile = tm * p.n_tiles + tn;
      float g[CH], uu[CH];
      // epilogue of one unit of problem kind K, straight from the accumulator
      auto direct = [&](auto kind_c, const GemmParams& q) {
        constexpr int K = decltype(kind_c)::value;
        using SK = GemmShape<SWAP, K, BN>;
#pragma unroll 1
        for (int seg = 0; seg < SK::kSeg; ++seg) {
#pragma unroll 1
          for (int c0 = 0; c0 < SK::kNG; c0 += CH) {
            const uint32_t col = seg * BN + c0;
            if (CH == 32) tmem_ld32(acc + col, g); else tmem_ld16(acc + col, g);
            if (K == KIND_GATE_UP) {
              if (CH == 32) tmem_ld32(acc + SK::kUOff + col, uu); else tmem_ld16(acc + SK::kUOff + col, uu);
            }
            tc_wait_ld();
            emit_vals<SWAP, K, BN, CH>(q, tm, tn, seg, row, c0, g, uu);
          }
        }
      };
      if (second) {
        direct(std::integral_constant<int, (kTwo ? KIND2 : KIND)>{}, p2);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(buf));
      } else if (p.splits == 1) {
        direct(std::integral_constant<int, KIND>{}, p);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(buf));
      } else {
        float* part = p.partials + ((size_t)tile * p.splits + sp) * ACC * 128;
#pragma unroll 1
        for (int c0 = 0; c0 < ACC; c0 += CH) {
          if (CH == 32) tmem_ld32(acc + c0, g); else tmem_ld16(acc + c0, g);
          tc_wait_ld();
#pragma unroll
          for (int j = 0; j < CH; ++j) __stcg(part + (size_t)(c0 + j) * 128 + row, g[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(buf));
      }
      if (++buf == 2) {
        buf = 0;
        acc_phase ^= 1u;
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::kTmemCols);
  }
  if (p.splits > 1) {
    // ---------------------------------------------------------- split-K reduction
    __threadfence();
    if (threadIdx.x == 0) {
      bool ok = !*s_abort && grid_barrier(p.gbar, gridDim.x, p.timeout_ns);
      if (!ok && !*s_abort) atomicExch(p.status, kStatusTimeout);
      *s_ok = ok ? 1 : 0;
    }
    __syncthreads();
    if (!*s_ok) return;
    reduce_partials<SWAP, KIND, BN>(p, (long long)blockIdx.x * blockDim.x + threadIdx.x,
                                    (long long)gridDim.x * blockDim.x);
  }
}

}  // namespace tpl
