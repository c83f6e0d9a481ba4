// Attention core between the column-parallel QKV projection and the
// row-parallel o_proj: causal scaled-dot-product attention of every shard's
// local q heads, each reading the kv head of its group, over sequences
// packed along the token axis ("vLLM Code Reading (Section 5)" §13: each
// rank runs attention on the heads it holds; "vLLM 源码完全拆解（十一）",
// QkvParallelLinear: which kv heads a shard holds under GQA).
//
// Input is the projection's own output, qkv [t][T][w_s] (shard r: its q
// heads | k heads | v heads, hd = 128 columns each); output is o_proj's
// input, attn [t][T][q_per * hd]. Flash-style, one CTA per SM, persistent:
//
//   unit     (q head, sequence, 128-query tile); units are handed out heaviest
//            first (most key tiles) from a counter, a CTA taking the next one
//            as it frees up; heads are innermost so the q heads of one kv head
//            run side by side and share its K/V tiles in L2
//   warp 0   TMA: the Q tile (two 64-column boxes, 128-byte swizzle), then
//            K and V tiles of 128 keys into a 3-stage ring
//   warp 2   tcgen05.mma: S = Q K^T into one of three tensor-memory buffers,
//            up to three key tiles ahead of O += P V
//   warp 1   tcgen05.mma: O += P V, once the softmax has written P. P is written by the softmax into
//            the buffer its S came from (bf16 pairs, the tensor-memory A
//            operand), so P never passes through shared memory; V is read
//            MN-major straight from its [key][hd] tile. A buffer is reused
//            once the P V that read it has completed
//   warps 4-7 softmax, one query row per thread: the row of S from tensor
//            memory, causal / sequence-end mask, running max and sum in the
//            exp2 domain, P = 2^(s*c - m) as bf16 back into tensor memory. O
//            is rescaled in tensor memory only when the row max grows by more
//            than 2^8 (until then the stale max keeps every p <= 256); at the
//            end of a unit the row sum l goes to the epilogue warps through
//            shared memory and the next unit starts at once
//   warps 8-11 epilogue: once the unit's last P V has completed, O out of tensor
//            memory (the buffer is released at once), O / l to global memory as
//            bf16, while the softmax warps work on the next unit
//   warp 3   idle; warps 0-3 run on 56 registers, the softmax warps on 232 and
//            the epilogue warps on 216
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
constexpr int kStages = 3;                   // K/V ring
constexpr int kSBufs = 3;                    // S/P buffers in tensor memory
constexpr int kQOff = 0;
constexpr int kKOff = kTileBytes;
constexpr int kVOff = kKOff + kStages * kTileBytes;
constexpr int kBarOff = kVOff + kStages * kTileBytes;
constexpr int kBarBytes = 512;
// row sums from the softmax to the epilogue warps: [2 units in flight][128 rows] fp32
constexpr int kLOff = kBarOff + kBarBytes;
constexpr int kAttnSmem = 1024 + kLOff + 2 * 128 * 4;
static_assert(kAttnSmem <= 232448, "shared memory of one CTA");
constexpr int kUnitSlots = 4;                // units the producer may hand out ahead of the consumers
constexpr int kSWarp = 2;                    // issues the S = Q K^T MMAs (warp 1 issues P V)
constexpr int kThreads = 384;                // three warpgroups: copies and MMAs, softmax, epilogue
constexpr int kOtherRegs = 56, kSoftRegs = 232, kEpiRegs = 216;
static_assert(128 * (kOtherRegs + kSoftRegs + kEpiRegs) <= kThreads * 168,
              "register split within the launch's 168 a thread");
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128);
constexpr uint32_t kIdescO = idesc_bf16_f32(128, 128) | kIdescBMnMajor;
constexpr int kTmemCols = 512;               // S/P buffers [0,128) [128,256) [256,384), O [384,512)
constexpr int kOCol = kSBufs * 128;
constexpr float kRescaleLog2 = 8.0f;         // rescale O when the row max grows by more than this
// Key tile j uses slot j % 3 of everything: K/V stage, S/P buffer and the barriers
// below. A wait costs an MMA issuer a few hundred cycles even when the barrier has
// already completed, so each issuer's inputs meet on one barrier per slot:
//   S_READY[i]  K landed (producer arrival + bytes) and the buffer is free (commit of
//               the P V three tiles back; armed once at start for the first three)
//   PV_READY[i] V landed (producer arrival + bytes) and P written (4 softmax warps)
static_assert(kStages == kSBufs, "K/V stages and S/P buffers advance together");
enum {
  Q_FULL = 0, Q_EMPTY,
  S_READY, K_EMPTY = S_READY + kStages, PV_READY = K_EMPTY + kStages, V_EMPTY = PV_READY + kStages,
  S_FULL = V_EMPTY + kStages,      // S of a buffer computed
  O_DONE = S_FULL + kSBufs, O_EMPTY, DONE, DONE_S,
  U_FULL,                          // a unit id published by the producer
  U_EMPTY = U_FULL + kUnitSlots,   // read by the two MMA warps, the softmax and the epilogue warps
  L_FULL = U_EMPTY + kUnitSlots,   // a unit's row sums written (per unit parity)
  L_EMPTY = L_FULL + 2,            // and read by the epilogue warps
  NBARS = L_EMPTY + 2
};
// barriers, tensor-memory address and abort flag, unit ids, then (16-byte aligned) their entries
static_assert(8 * NBARS + 8 + 4 * kUnitSlots + 15 + 16 * kUnitSlots <= kBarBytes, "barrier area");
static_assert(S_FULL <= 32, "copy barriers fit the producer's bit masks");

struct Unit {
  int r, i, g, start, len, qt;
};
// unit u from its work-table entry pr = pairs[u / heads]
__device__ __forceinline__ Unit decode_unit(const AttnParams& p, int u, int4 pr) {
  const int hh = u - (u / p.heads) * p.heads;
  Unit x;
  x.r = hh / p.q_per;
  x.i = hh - x.r * p.q_per;
  const int first = p.rep > 1 ? x.r / p.rep : x.r * p.kv_per;  // first kv head the shard holds
  x.g = (x.r * p.q_per + x.i) / p.group - first;
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
  // the attention grid may be scheduled now: it sets itself up, then waits for this
  // grid to complete before it reads the table
  if (tid == 0) griddep_launch_dependents();
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
  // [kUnitSlots] their work-table entries: the consumers read them here, not from global
  // memory, where a load would queue behind the output rows a softmax warp has just stored
  int4* s_pair = reinterpret_cast<int4*>((reinterpret_cast<uintptr_t>(misc + 8 + 4 * kUnitSlots) + 15) & ~uintptr_t(15));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int b = 0; b < NBARS; ++b) {
      int count = 1;
      if (b == O_EMPTY) count = 4;                          // the four epilogue warps
      if (b >= U_EMPTY && b < U_EMPTY + kUnitSlots) count = 10;  // 2 MMA, 4 softmax, 4 epilogue warps
      if (b >= L_FULL) count = 4;                           // the four softmax / epilogue warps
      if (b >= S_READY && b < S_READY + kStages) count = 2;  // producer + P V commit
      if (b >= PV_READY && b < PV_READY + kStages) count = 5;  // producer + four softmax warps
      mbar_init(bar(b), count);
    }
    // the buffers start free: arm the first use of every S_READY
    for (int i = 0; i < kStages; ++i) mbar_arrive(bar(S_READY + i));
    *s_abort = 0;
    fence_barrier_init();
    prefetch_tensormap(&map_qkv);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(s_tmem)), kTmemCols);
    tmem_relinquish();
  }
  // launched behind the table's preparation (programmatic dependent launch): the set-up
  // above overlaps it; the table, the unit counter and qkv are read only after this
  griddep_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int n_units = *p.n_pairs * p.heads;
  const unsigned long long timeout = p.timeout_ns;
  auto set_abort = [&]() {
    if (!*s_abort) {
      atomicExch(p.status, kStatusTimeout);
      *s_abort = 1;
    }
  };

  if (warp < 4) {
    // copies and MMAs (warp 3 idle) on few registers, so that the softmax and epilogue
    // warps can have more; each budget is set by a whole warpgroup and governs the
    // code it dominates
    regs_dec<kOtherRegs>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        const uint64_t pol = policy_evict_normal();
        uint32_t full_mask = 0, full_phase = 0;  // bit b: barrier b has a copy in flight, its phase
        auto issued = [&](int b, uint32_t ph) {
          full_mask |= 1u << b;
          full_phase = (full_phase & ~(1u << b)) | (ph << b);
        };
        auto load_tile = [&](uint32_t dst, int b, int col, int row, int r) {
          mbar_arrive_expect_tx(bar(b), kTileBytes);
          tma_load_4d(dst, &map_qkv, bar(b), col, row, r, 0, pol);
          tma_load_4d(dst + kTileBytes / 2, &map_qkv, bar(b), col + 64, row, r, 0, pol);
        };
        bool ok = true;
        int kv = 0;
        for (int nu = 0; ok; ++nu) {
          const int slot = nu % kUnitSlots;
          if (!mbar_wait_bounded(bar(U_EMPTY + slot), ((nu / kUnitSlots) & 1) ^ 1, s_abort, timeout)) {
            ok = false;
            break;
          }
          int u = atomicAdd(p.next_unit, 1);
          if (u >= n_units) u = -1;
          s_units[slot] = u;
          const int4 pr = u >= 0 ? p.pairs[u / p.heads] : make_int4(0, 0, 0, 0);
          s_pair[slot] = pr;
          mbar_arrive(bar(U_FULL + slot));  // releases the id and its entry to the consumers
          if (u < 0) break;
          const Unit x = decode_unit(p, u, pr);
          if (!mbar_wait_bounded(bar(Q_EMPTY), (nu & 1) ^ 1, s_abort, timeout)) {
            ok = false;
            break;
          }
          load_tile(base + kQOff, Q_FULL, x.i * 128, x.start + x.qt * 128, x.r);
          issued(Q_FULL, nu & 1);
          const int kcol = (p.q_per + x.g) * 128, vcol = (p.q_per + p.kv_per + x.g) * 128;
          for (int kt = 0; kt <= x.qt; ++kt, ++kv) {
            const int st = kv % kStages;
            const uint32_t ph = (kv / kStages) & 1;
            if (!mbar_wait_bounded(bar(K_EMPTY + st), ph ^ 1, s_abort, timeout)) {
              ok = false;
              break;
            }
            load_tile(base + kKOff + st * kTileBytes, S_READY + st, kcol, x.start + kt * 128, x.r);
            issued(S_READY + st, ph);
            if (!mbar_wait_bounded(bar(V_EMPTY + st), ph ^ 1, s_abort, timeout)) {
              ok = false;
              break;
            }
            load_tile(base + kVOff + st * kTileBytes, PV_READY + st, vcol, x.start + kt * 128, x.r);
            issued(PV_READY + st, ph);
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
    } else if (warp == 1 || warp == kSWarp) {
      // ------------------------------------------------------------ MMA issuers
      // Warp 2 issues S = Q K^T, warp 1 O += P V. Each shares its sub-partition with a
      // softmax warp, so every instruction saved keeps the tensor pipe fed: descriptors
      // are built once, a k-step adds a constant, ring positions advance without division.
      // The whole warp runs the loop (waits, unit ids, descriptors) and one elected lane
      // issues each group of MMAs with its commits: operands computed by a converged warp
      // are warp-uniform, where computed under a branch on the lane index they are not,
      // and each MMA then costs more to issue than its 64 cycles on the tensor pipe.
      // Ordering between the two goes through mbarriers: S_FULL (S done) -> softmax ->
      // PV_READY (P written, V in) -> P V -> S_READY (buffer free for the S three tiles
      // later, with its K).
      {
        const bool s_role = warp == kSWarp;
        bool ok = true;
        auto wait = [&](int b, uint32_t ph) -> bool {
          bool w = mbar_wait_bounded(bar(b), ph, s_abort, timeout);
          w = __all_sync(0xffffffffu, w);
          if (!w) {
            if (lane == 0) set_abort();
            ok = false;
          }
          return w;
        };
        auto advance = [](int& i, uint32_t& ph, int n) {
          if (++i == n) {
            i = 0;
            ph ^= 1u;
          }
        };
        // stage i's descriptor is stage 0's plus i tiles in the address field (address >> 4,
        // 14 bits; every shared address here is below 256 KB, so the field never carries)
        constexpr uint64_t kTileDesc = kTileBytes >> 4;
        const uint64_t q_desc = smem_desc_k128(base + kQOff);
        const uint64_t k_desc0 = smem_desc_k128(base + kKOff);
        const uint64_t v_desc0 = smem_desc_mn128(base + kVOff, kTileBytes / 2);
        int st = 0, buf = 0;        // K/V stage and S/P buffer of the next MMA group
        uint32_t st_ph = 0, buf_ph = 0;
        for (int nu = 0; ok; ++nu) {
          const int slot = nu % kUnitSlots;
          if (!wait(U_FULL + slot, (nu / kUnitSlots) & 1)) break;
          const int u = s_units[slot];
          const int4 pr = s_pair[slot];
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(U_EMPTY + slot));
          if (u < 0) break;
          const Unit x = decode_unit(p, u, pr);
          const int n = x.qt + 1;
          if (s_role) {
            if (!wait(Q_FULL, nu & 1)) break;
            for (int j = 0; j < n; ++j) {
              // K is in and the P V that last read this buffer has completed
              if (!wait(S_READY + st, st_ph)) break;
              tc_fence_after();
              const uint64_t kd = k_desc0 + (uint64_t)st * kTileDesc;
              const uint32_t d = tmem_base + buf * 128;
              if (elect_one()) {
                tc_mma_bf16_c<false>(d, q_desc, kd, kIdescS);
  #pragma unroll
                for (int k = 1; k < 8; ++k) {
                  const uint64_t o = (uint64_t)(((k >> 2) * (kTileBytes / 2) + (k & 3) * 32) >> 4);
                  tc_mma_bf16_c<true>(d, q_desc + o, kd + o, kIdescS);
                }
                tc_commit(bar(K_EMPTY + st));
                tc_commit(bar(S_FULL + buf));
                if (j == n - 1) tc_commit(bar(Q_EMPTY));
              }
              __syncwarp();
              advance(st, st_ph, kStages);
              advance(buf, buf_ph, kSBufs);
            }
          } else {
            for (int j = 0; j < n; ++j) {
              if (!wait(PV_READY + st, st_ph)) break;  // V is in and P written
              if (j == 0 && !wait(O_EMPTY, (nu & 1) ^ 1)) break;
              tc_fence_after();
              const uint64_t vd = v_desc0 + (uint64_t)st * kTileDesc;
              const uint32_t pa = tmem_base + buf * 128;
              if (elect_one()) {
                // 16 keys = two 8-row groups of V (2048 B) and 8 columns of P
                if (j == 0)
                  tc_mma_bf16_ta_c<false>(tmem_base + kOCol, pa, vd, kIdescO);
                else
                  tc_mma_bf16_ta_c<true>(tmem_base + kOCol, pa, vd, kIdescO);
  #pragma unroll
                for (int k = 1; k < 8; ++k)
                  tc_mma_bf16_ta_c<true>(tmem_base + kOCol, pa + k * 8, vd + (uint64_t)(k * (2048 >> 4)), kIdescO);
                tc_commit(bar(V_EMPTY + st));   // V consumed; O holds this tile (softmax rescale)
                tc_commit(bar(S_READY + st));   // the buffer's P is consumed
                if (j == n - 1) tc_commit(bar(O_DONE));
              }
              __syncwarp();
              advance(st, st_ph, kStages);
              advance(buf, buf_ph, kSBufs);
            }
          }
        }
        // this warp's MMAs complete before tensor memory is released
        const int done = s_role ? DONE_S : DONE;
        if (elect_one()) tc_commit(bar(done));
        __syncwarp();
        mbar_wait_bounded(bar(done), 0, nullptr, kTeardownNs);
        __syncwarp();
      }
    }
  } else if (warp < 8) {
    regs_inc<kSoftRegs>();
    // ------------------------------------------------------------ softmax
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;  // query row of the tile = tensor-memory lane
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16);
    const float c = p.scale_log2;
    float* xl = reinterpret_cast<float*>(base_ptr + kLOff);
    int sc = 0;  // S tiles consumed (= P tiles produced)
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
      const int4 pr = s_pair[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(U_EMPTY + slot));
      if (u < 0) break;
      const Unit x = decode_unit(p, u, pr);
      const int q_rel = x.qt * 128 + row;
      float m = -INFINITY, l = 0.f;
      for (int kt = 0; kt <= x.qt; ++kt) {
        const int b = sc % kSBufs;
        if (!wait_all(S_FULL + b, (sc / kSBufs) & 1)) break;
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
          for (int n = 0; n < 128; ++n) {
            const int key = kt * 128 + n;
            if (key > q_rel || key >= x.len) s[n] = -INFINITY;
          }
        }
        // row max (three-input max) and, below, the exponent and row sum on fp32 pairs:
        // the softmax issues every instruction of the tile from one warp per
        // sub-partition, so it is bound by their count. Independent chains (8 for the
        // max, 4 pairs for the sum) keep it from waiting on its own latency.
        float mk[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) mk[j] = fmaxf(s[j], s[8 + j]);
#pragma unroll
        for (int n = 16; n < 128; n += 16)
#pragma unroll
          for (int j = 0; j < 8; ++j) mk[j] = fmax3(mk[j], s[n + j], s[n + 8 + j]);
        float mx = fmax3(fmax3(mk[0], mk[1], mk[2]), fmax3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7]));
        mx *= c;
        if (kt == 0) {
          m = mx;  // the first P V overwrites O
        } else if (__any_sync(0xffffffffu, mx > m + kRescaleLog2)) {
          // the wait and the tensor-memory accesses below are warp-wide: the warp
          // rescales together, every row by its own factor (1 where the max held)
          float f = 1.0f;
          if (mx > m + kRescaleLog2) {
            f = fast_exp2(m - mx);
            l *= f;
            m = mx;
          }
          // O holds the products up to the previous key tile: let them land, then scale the rows
          const int pj = sc - 1;
          if (!wait_all(V_EMPTY + pj % kSBufs, (pj / kSBufs) & 1)) break;
          tc_fence_after();
          float o[32];
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 32) {
            tmem_ld32(lane_addr + kOCol + c0, o);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] *= f;
            tmem_st32(lane_addr + kOCol + c0, o);
          }
        }
        // P = 2^(s c - m) as bf16 pairs into the first 64 columns of the buffer
        const uint64_t c2 = f32x2_pack(c, c), nm2 = f32x2_pack(-m, -m);
        uint64_t lk[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float x0, x1;
            f32x2_unpack(f32x2_fma(f32x2_pack(s[h * 64 + 2 * j], s[h * 64 + 2 * j + 1]), c2, nm2), x0, x1);
            const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
            lk[j & 3] = f32x2_add(lk[j & 3], f32x2_pack(e0, e1));
            pk[j] = pack_bf16x2(e0, e1);
          }
          tmem_st32(sa + h * 32, reinterpret_cast<const float*>(pk));
        }
        float la[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) f32x2_unpack(lk[j], la[2 * j], la[2 * j + 1]);
        l += ((la[0] + la[1]) + (la[2] + la[3])) + ((la[4] + la[5]) + (la[6] + la[7]));
        tc_wait_st();      // P, and O as rescaled above, are in tensor memory
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(PV_READY + b));
        ++sc;
      }
      if (!ok) break;
      // the row sums go to the epilogue warps; the next unit starts at once
      const int lp = nu & 1;
      if (!wait_all(L_EMPTY + lp, ((nu >> 1) & 1) ^ 1)) break;
      xl[lp * 128 + row] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L_FULL + lp));
    }
  } else {
    regs_inc<kEpiRegs>();
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;  // query row of the tile = tensor-memory lane
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16);
    const float* xl = reinterpret_cast<const float*>(base_ptr + kLOff);
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
      const int4 pr = s_pair[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(U_EMPTY + slot));
      if (u < 0) break;
      const Unit x = decode_unit(p, u, pr);
      const int q_rel = x.qt * 128 + row;
      const int lp = nu & 1;
      if (!wait_all(L_FULL + lp, (nu >> 1) & 1)) break;
      const float l = xl[lp * 128 + row];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L_EMPTY + lp));
      if (!wait_all(O_DONE, nu & 1)) break;
      tc_fence_after();
      const float inv = 1.0f / l;
      __nv_bfloat16* dst = p.out + (size_t)x.r * p.out_sstride + (size_t)(x.start + q_rel) * p.out_rstride + x.i * 128;
      // O comes out of tensor memory whole (into the registers S used) and its buffer is
      // released before the rows are written.
      tmem_ld32(lane_addr + kOCol, s);
      tmem_ld32(lane_addr + kOCol + 32, s + 32);
      tmem_ld32(lane_addr + kOCol + 64, s + 64);
      tmem_ld32(lane_addr + kOCol + 96, s + 96);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(O_EMPTY));
      // Row q of the tile is this thread's: 256 bytes, eight 32-byte chunks. A store in
      // which each lane writes its own row touches 32 lines; instead each group of four
      // lanes transposes its 4 x 4 blocks of chunks (two shuffle stages per half row),
      // after which lane a of the group holds chunk a of the half of all four rows, and a
      // store has four lanes fill each line it touches (8 lines a store instead of 32).
      uint32_t w[64];
#pragma unroll
      for (int k = 0; k < 64; ++k) w[k] = pack_bf16x2(s[2 * k] * inv, s[2 * k + 1] * inv);
      const int a = lane & 3;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t* c = w + 32 * h;   // chunks 0..3 of this half: c[8 * i .. 8 * i + 7]
        // stage 1 (lanes a, a ^ 2): lanes 0, 1 give chunks 2, 3 and take the partner's 0, 1
        const bool hi2 = (a & 2) != 0;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int lo = 8 * i + e, up = 8 * (2 + i) + e;
            const uint32_t got = __shfl_xor_sync(0xffffffffu, hi2 ? c[lo] : c[up], 2);
            if (hi2) c[lo] = got; else c[up] = got;
          }
        // stage 2 (lanes a, a ^ 1), in each pair of chunks: even lanes give the second,
        // odd lanes the first
        const bool odd = (a & 1) != 0;
#pragma unroll
        for (int i = 0; i < 4; i += 2)
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int lo = 8 * i + e, up = 8 * (i + 1) + e;
            const uint32_t got = __shfl_xor_sync(0xffffffffu, odd ? c[lo] : c[up], 1);
            if (odd) c[lo] = got; else c[up] = got;
          }
        // c[8 k ..] is now chunk 4 h + a of row q - a + k
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (q_rel - a + k < x.len) {
            __nv_bfloat16* d = dst + (k - a) * p.out_rstride + (4 * h + a) * 16;
            const uint32_t* v = c + 8 * k;
            if (p.out_align32) {
              st_global_v8(d, *reinterpret_cast<const uint32_t(*)[8]>(v));
            } else {
              *reinterpret_cast<uint4*>(d) = make_uint4(v[0], v[1], v[2], v[3]);
              *reinterpret_cast<uint4*>(d + 8) = make_uint4(v[4], v[5], v[6], v[7]);
            }
          }
        }
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
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
    // The warpgroups' register budgets (setmaxnreg) come out of the registers the CTA is
    // launched with; were the kernel built with fewer, an increase would wait forever.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, attn_fwd_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * kThreads < 128 * (kOtherRegs + kSoftRegs + kEpiRegs)) return cudaErrorInvalidConfiguration;
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kAttnSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_fwd_kernel, map_qkv, p);
}

}  // namespace tpl
