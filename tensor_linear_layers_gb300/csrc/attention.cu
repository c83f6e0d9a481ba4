// Attention core between the column-parallel QKV projection and the
// row-parallel o_proj: causal scaled-dot-product attention of every shard's
// local q heads, each reading the kv head of its group, over sequences
// packed along the token axis ("vLLM Code Reading (Section 5)" §13: each
// rank runs attention on the heads it holds; "vLLM 源码完全拆解（十一）",
// QkvParallelLinear: which kv heads a shard holds under GQA).
//
// Input is the projection's own output, qkv [t][T][w_s] (shard r: its q
// heads | k heads | v heads, hd = 128 columns each); output is o_proj's
// input, attn [t][T][q_per * hd] (or both gathered). Flash-style, one CTA
// per SM, persistent:
//
//   unit     (sequence, 128-query tile, two q heads that read the same kv
//            head); a kv group of odd size leaves one single-head unit.
//            Units are handed out heaviest first (most key tiles) from a
//            counter, a CTA taking the next one as it frees up
//   warp 8   TMA: the unit's Q tiles (two 64-column boxes each, 128-byte
//            swizzle), then K tiles into a 3-stage ring and V tiles into a
//            2-stage ring; each K and V tile serves both heads
//   warp 9   tcgen05.mma, in the order S_A(0) S_B(0) | P_A V(j) S_A(j+1)
//            P_B V(j) S_B(j+1) | ..., so while one head's softmax runs the
//            tensor pipe computes the other head's products. S_A and S_B
//            have one tensor-memory buffer each; P is written by the softmax
//            over the first half of its S (bf16 pairs, the A operand of P V)
//            and the next S into that buffer is issued after the P V that
//            reads it (tcgen05.mma of one thread execute in issue order).
//            A single-head unit alternates its S between both buffers
//   warps 0-3 softmax of head A, warps 4-7 of head B: one query row per
//            thread, so every sub-partition runs two softmax warps. The
//            row of S from tensor memory, causal / sequence-end mask,
//            running max and sum in the exp2 domain, P = 2^(s*c - m) as
//            bf16 back into tensor memory. O is rescaled in tensor memory
//            only when the row max grows by more than 2^8 (until then the
//            stale max keeps every p <= 256); at the end O / l goes to
//            global memory as bf16
//
// Every wait is bounded (status word TP_ERR_TIMEOUT on timeout).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "gemm_tc.cuh"
#include "internal.h"

namespace tpl {


namespace {
constexpr int kTileBytes = 128 * 128 * 2;    // 128 rows x 128 bf16: two 64-column boxes
constexpr int kKStages = 3;                  // K ring
constexpr int kVStages = 2;                  // V ring
constexpr int kQOff = 0;                     // Q_A, then Q_B
constexpr int kKOff = 2 * kTileBytes;
constexpr int kVOff = kKOff + kKStages * kTileBytes;
constexpr int kBarOff = kVOff + kVStages * kTileBytes;
constexpr int kBarBytes = 512;
constexpr int kAttnSmem = 1024 + kBarOff + kBarBytes;
static_assert(kAttnSmem <= 227 * 1024, "shared memory per CTA");
constexpr int kUnitSlots = 4;                // units the producer may hand out ahead of the consumers
// warps 0-3 softmax of head A, 4-7 of head B, 8 producer, 9 MMA, 10-11 idle: three
// warpgroups, so the softmax warpgroups can take the registers the third gives back
constexpr int kThreads = 32 * 12;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kLaunchRegs = 65536 / kThreads / 8 * 8;   // 168: three warps per sub-partition
constexpr int kSoftmaxRegs = 200, kOtherRegs = 104;
static_assert(4 * kOtherRegs + 8 * kSoftmaxRegs <= 12 * kLaunchRegs, "register split fits the launch");
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128);
constexpr uint32_t kIdescO = idesc_bf16_f32(128, 128) | kIdescBMnMajor;
constexpr int kTmemCols = 512;               // S/P buffers [0,128) [128,256), O_A [256,384), O_B [384,512)
constexpr int kOCol = 256;
constexpr float kRescaleLog2 = 8.0f;         // rescale O when the row max grows by more than this
enum {
  Q_FULL = 0, Q_EMPTY,
  K_FULL, K_EMPTY = K_FULL + kKStages,
  V_FULL = K_EMPTY + kKStages, V_EMPTY = V_FULL + kVStages,
  S_FULL = V_EMPTY + kVStages,     // [2] S of a buffer computed
  P_READY = S_FULL + 2,            // [2] P of a buffer written (four softmax warps)
  PV_DONE = P_READY + 2,           // [2] a P V into O_A / O_B completed
  O_DONE = PV_DONE + 2,            // [2] the unit's last P V into O_A / O_B completed
  O_EMPTY = O_DONE + 2,            // [2] O_A / O_B read out (four softmax warps)
  DONE = O_EMPTY + 2,
  U_FULL,                          // a unit id published by the producer
  U_EMPTY = U_FULL + kUnitSlots,   // read by the MMA thread and the eight softmax warps
  NBARS = U_EMPTY + kUnitSlots
};
static_assert(8 * NBARS + 8 + 4 * kUnitSlots <= kBarBytes, "barrier area");
static_assert(S_FULL <= 32, "copy barriers fit the producer's bit masks");

struct Unit {
  int r, ia, ib, g, start, len, qt;   // ib < 0: single-head unit
};
__device__ __forceinline__ Unit decode_unit(const AttnParams& p, int u) {
  const int per = p.t * p.pairs_per_shard;
  const int e = u / per;
  const int hh = u - e * per;
  const int4 pr = p.pairs[e];
  Unit x;
  x.r = hh / p.pairs_per_shard;
  const int j = hh - x.r * p.pairs_per_shard;
  const int run = j / p.half, k = j - run * p.half;
  x.ia = run * p.run + 2 * k;
  x.ib = 2 * k + 1 < p.run ? x.ia + 1 : -1;
  const int first = p.rep > 1 ? x.r / p.rep : x.r * p.kv_per;  // first kv head the shard holds
  x.g = (x.r * p.q_per + x.ia) / p.group - first;
  x.start = pr.x;
  x.len = pr.y;
  x.qt = pr.z;
  return x;
}
}  // namespace

// Work table: for every sequence s and q tile q < ceil(len_s / 128) one entry,
// ordered by q descending (the number of key tiles), sequences ascending.
// Checks the offsets (0 first, T last, none falling, no length above
// max_tiles * 128); on a bad table it writes TP_ERR_SHAPE and no entries.
__global__ void attn_prep_kernel(const int* cu, int n_seqs, int T, int max_tiles, int4* pairs, int* n_pairs,
                                 int* next_unit, int* status) {
  extern __shared__ int off[];  // [max_tiles]
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_bad = (cu[0] != 0 || cu[n_seqs] != T) ? 1 : 0;
    *next_unit = 0;
  }
  __syncthreads();
  for (int s = tid; s < n_seqs; s += blockDim.x) {
    const int len = cu[s + 1] - cu[s];
    if (len < 0 || len > max_tiles * 128) atomicExch(&s_bad, 1);
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      *n_pairs = 0;
      atomicExch(status, -2);  // TP_ERR_SHAPE
    }
    return;
  }
  for (int q = tid; q < max_tiles; q += blockDim.x) {
    int c = 0;
    for (int s = 0; s < n_seqs; ++s) c += (cu[s + 1] - cu[s]) > q * 128 ? 1 : 0;
    off[q] = c;
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int q = max_tiles - 1; q >= 0; --q) {
      const int c = off[q];
      off[q] = acc;
      acc += c;
    }
    *n_pairs = acc;
  }
  __syncthreads();
  for (int q = tid; q < max_tiles; q += blockDim.x) {
    int pos = off[q];
    for (int s = 0; s < n_seqs; ++s) {
      const int len = cu[s + 1] - cu[s];
      if (len > q * 128) pairs[pos++] = make_int4(cu[s], len, q, 0);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap map_qkv, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t bar0 = base + kBarOff;
  auto bar = [&](int b) { return bar0 + 8u * b; };
  uint8_t* misc = base_ptr + kBarOff + 8 * NBARS;
  volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + 4);
  volatile int* s_units = reinterpret_cast<volatile int*>(misc + 8);  // [kUnitSlots] unit ids, -1 = no more
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int b = 0; b < NBARS; ++b) {
      int count = 1;
      if ((b >= P_READY && b < P_READY + 2) || (b >= O_EMPTY && b < O_EMPTY + 2)) count = 4;  // one warpgroup
      if (b >= U_EMPTY) count = 9;                          // the MMA thread and eight softmax warps
      mbar_init(bar(b), count);
    }
    *s_abort = 0;
    fence_barrier_init();
    prefetch_tensormap(&map_qkv);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(s_tmem)), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int n_units = *p.n_pairs * p.t * p.pairs_per_shard;
  const unsigned long long timeout = p.timeout_ns;
  auto set_abort = [&]() {
    if (!*s_abort) {
      atomicExch(p.status, kStatusTimeout);
      *s_abort = 1;
    }
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    regs_dec<kOtherRegs>();
    if (lane == 0) {
      const uint64_t pol = policy_evict_normal();
      uint32_t full_mask = 0, full_phase = 0;  // bit b: barrier b has a copy in flight, its phase
      auto issued = [&](int b, uint32_t ph) {
        full_mask |= 1u << b;
        full_phase = (full_phase & ~(1u << b)) | (ph << b);
      };
      auto load_box2 = [&](uint32_t dst, int b, int col, int row, int r) {
        tma_load_4d(dst, &map_qkv, bar(b), col, row, r, 0, pol);
        tma_load_4d(dst + kTileBytes / 2, &map_qkv, bar(b), col + 64, row, r, 0, pol);
      };
      bool ok = true;
      int kc = 0, vc = 0;  // K and V tiles loaded so far
      for (int nu = 0; ok; ++nu) {
        const int slot = nu % kUnitSlots;
        if (!mbar_wait_bounded(bar(U_EMPTY + slot), ((nu / kUnitSlots) & 1) ^ 1, s_abort, timeout)) {
          ok = false;
          break;
        }
        int u = atomicAdd(p.next_unit, 1);
        if (u >= n_units) u = -1;
        s_units[slot] = u;
        mbar_arrive(bar(U_FULL + slot));  // releases the id to the consumers
        if (u < 0) break;
        const Unit x = decode_unit(p, u);
        if (!mbar_wait_bounded(bar(Q_EMPTY), (nu & 1) ^ 1, s_abort, timeout)) {
          ok = false;
          break;
        }
        const int qrow = x.start + x.qt * 128;
        mbar_arrive_expect_tx(bar(Q_FULL), x.ib >= 0 ? 2 * kTileBytes : kTileBytes);
        load_box2(base + kQOff, Q_FULL, x.ia * 128, qrow, x.r);
        if (x.ib >= 0) load_box2(base + kQOff + kTileBytes, Q_FULL, x.ib * 128, qrow, x.r);
        issued(Q_FULL, nu & 1);
        const int kcol = (p.q_per + x.g) * 128, vcol = (p.q_per + p.kv_per + x.g) * 128;
        for (int kt = 0; kt <= x.qt; ++kt, ++kc, ++vc) {
          const int ks = kc % kKStages, vs = vc % kVStages;
          const uint32_t kph = (kc / kKStages) & 1, vph = (vc / kVStages) & 1;
          if (!mbar_wait_bounded(bar(K_EMPTY + ks), kph ^ 1, s_abort, timeout)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(K_FULL + ks), kTileBytes);
          load_box2(base + kKOff + ks * kTileBytes, K_FULL + ks, kcol, x.start + kt * 128, x.r);
          issued(K_FULL + ks, kph);
          if (!mbar_wait_bounded(bar(V_EMPTY + vs), vph ^ 1, s_abort, timeout)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(V_FULL + vs), kTileBytes);
          load_box2(base + kVOff + vs * kTileBytes, V_FULL + vs, vcol, x.start + kt * 128, x.r);
          issued(V_FULL + vs, vph);
        }
      }
      if (!ok) {
        set_abort();
        // no copy into this CTA's shared memory may outlive it
        for (int b = 0; b < S_FULL; ++b)
          if (full_mask & (1u << b)) mbar_wait_bounded(bar(b), (full_phase >> b) & 1u, nullptr, kTeardownNs);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    regs_dec<kOtherRegs>();
    if (lane == 0) {
      bool ok = true;
      auto wait = [&](int b, uint32_t ph) -> bool {
        if (mbar_wait_bounded(bar(b), ph, s_abort, timeout)) return true;
        set_abort();
        ok = false;
        return false;
      };
      // stage i's descriptor is stage 0's plus i tiles in the address field (address >> 4,
      // 14 bits; every shared address here is below 256 KB, so the field never carries)
      constexpr uint64_t kTileDesc = kTileBytes >> 4;
      const uint64_t q_desc0 = smem_desc_k128(base + kQOff);
      const uint64_t k_desc0 = smem_desc_k128(base + kKOff);
      const uint64_t v_desc0 = smem_desc_mn128(base + kVOff, kTileBytes / 2);
      int kc = 0, vc = 0;                  // K and V tiles consumed
      uint32_t use[2] = {0u, 0u};          // uses of each S/P buffer
      uint32_t oc[2] = {0u, 0u};           // units accumulated in O_A / O_B
      // S = Q K^T of head h (0 = A, 1 = B) for the next K tile into buffer b
      auto issue_s = [&](int h, int b) -> bool {
        const int ks = kc % kKStages;
        if (h == 0 && !wait(K_FULL + ks, (kc / kKStages) & 1)) return false;
        tc_fence_after();
        const uint64_t qd = q_desc0 + (uint64_t)h * kTileDesc;
        const uint64_t kd = k_desc0 + (uint64_t)ks * kTileDesc;
        const uint32_t d = tmem_base + b * 128;
        tc_mma_bf16_c<false>(d, qd, kd, kIdescS);
#pragma unroll
        for (int k = 1; k < 8; ++k) {
          const uint64_t o = (uint64_t)(((k >> 2) * (kTileBytes / 2) + (k & 3) * 32) >> 4);
          tc_mma_bf16_c<true>(d, qd + o, kd + o, kIdescS);
        }
        tc_commit(bar(S_FULL + b));
        return true;
      };
      auto release_k = [&]() {
        tc_commit(bar(K_EMPTY + kc % kKStages));
        ++kc;
      };
      // O_h += P V for the current V tile, P from buffer b; first = the unit's first tile
      auto issue_pv = [&](int h, int b, bool first) -> bool {
        if (!wait(P_READY + b, use[b] & 1)) return false;
        if (first && !wait(O_EMPTY + h, (oc[h] & 1) ^ 1)) return false;
        tc_fence_after();
        const uint64_t vd = v_desc0 + (uint64_t)(vc % kVStages) * kTileDesc;
        const uint32_t pa = tmem_base + b * 128, od = tmem_base + kOCol + h * 128;
        // 16 keys = two 8-row groups of V (2048 B) and 8 columns of P
        if (first)
          tc_mma_bf16_ta_c<false>(od, pa, vd, kIdescO);
        else
          tc_mma_bf16_ta_c<true>(od, pa, vd, kIdescO);
#pragma unroll
        for (int k = 1; k < 8; ++k)
          tc_mma_bf16_ta_c<true>(od, pa + k * 8, vd + (uint64_t)(k * (2048 >> 4)), kIdescO);
        tc_commit(bar(PV_DONE + h));
        ++use[b];
        return true;
      };
      auto wait_v = [&]() -> bool { return wait(V_FULL + vc % kVStages, (vc / kVStages) & 1); };
      auto release_v = [&]() {
        tc_commit(bar(V_EMPTY + vc % kVStages));
        ++vc;
      };
      for (int nu = 0; ok; ++nu) {
        const int slot = nu % kUnitSlots;
        if (!wait(U_FULL + slot, (nu / kUnitSlots) & 1)) break;
        const int u = s_units[slot];
        mbar_arrive(bar(U_EMPTY + slot));
        if (u < 0) break;
        const Unit x = decode_unit(p, u);
        const int n = x.qt + 1;
        if (!wait(Q_FULL, nu & 1)) break;
        if (x.ib >= 0) {
          // two heads: buffer 0 and O_A for head A, buffer 1 and O_B for head B
          if (!issue_s(0, 0) || !issue_s(1, 1)) break;
          release_k();
          if (n == 1) tc_commit(bar(Q_EMPTY));
          for (int j = 0; j < n; ++j) {
            if (!wait_v() || !issue_pv(0, 0, j == 0)) break;
            if (j + 1 < n && !issue_s(0, 0)) break;
            if (!issue_pv(1, 1, j == 0)) break;
            release_v();
            if (j + 1 < n) {
              if (!issue_s(1, 1)) break;
              release_k();
              if (j + 2 == n) tc_commit(bar(Q_EMPTY));
            }
          }
          if (!ok) break;
          tc_commit(bar(O_DONE + 0));
          tc_commit(bar(O_DONE + 1));
          ++oc[0];
          ++oc[1];
        } else {
          // one head: its S alternates between the two buffers, two tiles ahead of P V
          if (!issue_s(0, 0)) break;
          release_k();
          if (n > 1) {
            if (!issue_s(0, 1)) break;
            release_k();
          }
          if (n <= 2) tc_commit(bar(Q_EMPTY));
          for (int j = 0; j < n; ++j) {
            const int b = j & 1;
            if (!wait_v() || !issue_pv(0, b, j == 0)) break;
            release_v();
            if (j + 2 < n) {
              if (!issue_s(0, b)) break;
              release_k();
              if (j + 3 == n) tc_commit(bar(Q_EMPTY));
            }
          }
          if (!ok) break;
          tc_commit(bar(O_DONE + 0));
          ++oc[0];
        }
      }
      // this thread's MMAs complete before tensor memory is released
      tc_commit(bar(DONE));
      mbar_wait_bounded(bar(DONE), 0, nullptr, kTeardownNs);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax + epilogue
    regs_inc<kSoftmaxRegs>();
    const int wg = warp >> 2;                  // 0: head A, 1: head B
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;  // query row of the tile = tensor-memory lane
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16);
    const uint32_t o_addr = lane_addr + kOCol + wg * 128;
    const float c = p.scale_log2;
    uint32_t use[2] = {0u, 0u};   // uses of each S/P buffer, by either warpgroup
    uint32_t pv = 0;              // P V products into this warpgroup's O so far
    uint32_t oc = 0;              // units this warpgroup finished
    bool ok = true;
    auto wait_all = [&](int b, uint32_t ph) -> bool {
      bool w = mbar_wait_bounded(bar(b), ph, s_abort, timeout);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        if (lane == 0) set_abort();
        ok = false;
      }
      return w;
    };
    float s[128];
    for (int nu = 0; ok; ++nu) {
      const int slot = nu % kUnitSlots;
      if (!wait_all(U_FULL + slot, (nu / kUnitSlots) & 1)) break;
      const int u = s_units[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(U_EMPTY + slot));
      if (u < 0) break;
      const Unit x = decode_unit(p, u);
      const int n = x.qt + 1;
      const bool pair = x.ib >= 0;
      if (wg == 1 && !pair) {
        // head A alone: both buffers are its; count them
        use[0] += (n + 1) / 2;
        use[1] += n / 2;
        continue;
      }
      const int q_rel = x.qt * 128 + row;
      float m = -INFINITY, l = 0.f;
      for (int kt = 0; kt < n; ++kt) {
        const int b = pair ? wg : (kt & 1);
        if (!wait_all(S_FULL + b, use[b] & 1)) break;
        tc_fence_after();
        const uint32_t sa = lane_addr + b * 128;
        tmem_ld32(sa, s);
        tmem_ld32(sa + 32, s + 32);
        tmem_ld32(sa + 64, s + 64);
        tmem_ld32(sa + 96, s + 96);
        tc_wait_ld();
        if (kt == x.qt || (kt + 1) * 128 > x.len) {
          // diagonal tile and the tile holding the sequence end
#pragma unroll
          for (int n2 = 0; n2 < 128; ++n2) {
            const int key = kt * 128 + n2;
            if (key > q_rel || key >= x.len) s[n2] = -INFINITY;
          }
        }
        // row max (three-input max, eight independent chains)
        float mk[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) mk[j] = fmaxf(s[j], s[8 + j]);
#pragma unroll
        for (int n2 = 16; n2 < 128; n2 += 16)
#pragma unroll
          for (int j = 0; j < 8; ++j) mk[j] = fmax3(mk[j], s[n2 + j], s[n2 + 8 + j]);
        float mx = fmax3(fmax3(mk[0], mk[1], mk[2]), fmax3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7]));
        mx *= c;
        if (kt == 0) {
          m = mx;  // the first P V overwrites O
        } else if (mx > m + kRescaleLog2) {
          const float f = fast_exp2(m - mx);
          l *= f;
          m = mx;
          // O holds the products up to the previous key tile: let them land, then scale the row
          if (!wait_all(PV_DONE + wg, (pv - 1) & 1)) break;
          tc_fence_after();
          float o[16];
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 16) {
            tmem_ld16(o_addr + c0, o);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] *= f;
            tmem_st16(o_addr + c0, o);
          }
        }
        // P = 2^(s c - m) as bf16 pairs into the first 64 columns of the buffer
        const uint64_t c2 = f32x2_pack(c, c), nm2 = f32x2_pack(-m, -m);
        uint64_t lk[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float x0, x1;
            f32x2_unpack(f32x2_fma(f32x2_pack(s[h * 32 + 2 * j], s[h * 32 + 2 * j + 1]), c2, nm2), x0, x1);
            const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
            lk[j & 3] = f32x2_add(lk[j & 3], f32x2_pack(e0, e1));
            pk[j] = pack_bf16x2(e0, e1);
          }
          tmem_st16(sa + h * 16, reinterpret_cast<const float*>(pk));
        }
        float la[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) f32x2_unpack(lk[j], la[2 * j], la[2 * j + 1]);
        l += ((la[0] + la[1]) + (la[2] + la[3])) + ((la[4] + la[5]) + (la[6] + la[7]));
        tc_wait_st();      // P, and O as rescaled above, are in tensor memory
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(P_READY + b));
        ++use[b];
        ++pv;
      }
      if (!ok) break;
      if (pair) {
        use[wg ^ 1] += n;  // the other warpgroup's buffer
      }
      if (!wait_all(O_DONE + wg, oc & 1)) break;
      ++oc;
      tc_fence_after();
      const float inv = 1.0f / l;
      const int head = wg == 0 ? x.ia : x.ib;
      __nv_bfloat16* dst = p.out + (size_t)x.r * p.out_sstride + (size_t)(x.start + q_rel) * p.out_rstride + head * 128;
      float o[32];
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        tmem_ld32(o_addr + c0, o);
        tc_wait_ld();
        if (c0 == 96) {
          // O is in registers: the next unit's P V may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(O_EMPTY + wg));
        }
        if (q_rel < x.len) {
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint4 v;
            v.x = pack_bf16x2(o[j] * inv, o[j + 1] * inv);
            v.y = pack_bf16x2(o[j + 2] * inv, o[j + 3] * inv);
            v.z = pack_bf16x2(o[j + 4] * inv, o[j + 5] * inv);
            v.w = pack_bf16x2(o[j + 6] * inv, o[j + 7] * inv);
            *reinterpret_cast<uint4*>(dst + c0 + j) = v;
          }
        }
      }
    }
  } else {
    regs_dec<kOtherRegs>();  // warps 10-11: idle, their registers go to the softmax
  }

  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

cudaError_t launch_attention(const CUtensorMap& map_qkv, const AttnParams& p, const int* cu, int n_seqs,
                             int max_tiles, int4* pairs, int* n_pairs, int grid, cudaStream_t st) {
  attn_prep_kernel<<<1, 1024, max_tiles * (int)sizeof(int), st>>>(cu, n_seqs, p.T, max_tiles, pairs, n_pairs,
                                                                    p.next_unit, p.status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  attn_fwd_kernel<<<grid, kThreads, kAttnSmem, st>>>(map_qkv, p);
  return cudaGetLastError();
}

}  // namespace tpl
