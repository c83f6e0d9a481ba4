// Fused decode-shaped MLP block: one persistent launch runs the
// whole step for T <= 128 tokens.
//
//   norm     residual add + RMSNorm of the T rows by the epilogue warps of
//            the first n_norm CTAs to start; they arrive on bars[0]
//   gate_up  column-parallel units of 256 weight rows (128 gate + 128 up of
//            one shard) x a K range, owned by the CTAs that start next.
//            Without split-K the epilogue writes silu(g) * u to h [t][T][I/t]
//            straight from the accumulator; with split-K every split writes
//            its fp32 partial and the last split of a tile to arrive adds the
//            tile's partials in split order. hready[tile] counts written items
//   down     row-parallel units, claimed from a counter: K runs over the t
//            shards in turn, so the shards' partial sums meet in the
//            accumulator. The producer loads the h columns of a k-block as
//            soon as the gate_up tile that wrote them is complete, streaming
//            weight blocks meanwhile. Each split of a down tile adds its own
//            slice of the tile's partials once all have arrived; a split that
//            has waited too long hands its slice to the last one to arrive.
//            mlp_out = y, residual_stream = y + residual
//
// No CTA relies on the whole grid being resident. A CTA's place in the start
// order of its launch comes from a ticket counter, and it waits only on work
// owned by a CTA that has already started and that waits on nothing later:
// gate_up waits for the norm rows of CTAs with earlier tickets; down units are
// claimed only once every gate_up owner has started (a CTA that cannot claim
// for a while gives up and exits, freeing its SM; if any CTA gave up or had
// not started, CTAs keep claiming until no unit is left); and the splits of a
// down tile never wait on one another without a bound. Every wait is bounded
// (status word on timeout). There are two sets of counters: a launch uses the
// one its launch count (a word every CTA adds its share to at exit) selects,
// and clears the other for the next launch.
#include "gemm_launch.cuh"
#include <atomic>

namespace tpl {


// How long a CTA waits for the gate_up CTAs to start before it gives up its
// down work, and how long a down split waits for the other splits of its tile
// before it hands its slice of the sum to the last one. Neither is an error.
constexpr unsigned long long kStartPatienceNs = 50000ull;
constexpr unsigned long long kSplitPatienceNs = 50000ull;
constexpr int kUnitSlots = 4;

// Wait until *c >= n, reading it with acquire loads; false after timeout_ns or when
// *abort is set (bounded; a short sleep between reads).
__device__ __forceinline__ bool poll_acquire(const unsigned* c, unsigned n, unsigned long long timeout_ns,
                                             const volatile int* abort) {
  if (ld_acquire(c) >= n) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(32);
    if (ld_acquire(c) >= n) return true;
    if ((it & 31u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
  }
}   // down units handed from the producer to the MMA and epilogue roles

template <int BN>
__global__ void __launch_bounds__(192, 1)
    mlp_decode_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_h,
                      const MlpDecodeParams P) {
  using S1 = GemmShape<true, KIND_GATE_UP, BN>;
  using S2 = GemmShape<true, KIND_ROW, BN>;
  static_assert(S1::kStageBytes == S2::kStageBytes && S1::kAccCols == S2::kAccCols, "shared ring");
  using S = S1;
  constexpr int STAGES = S::kStages;
  constexpr int ACC = S::kAccCols;
  constexpr int CH = S::kCh;
  constexpr int kItems1 = tile_items<true, KIND_GATE_UP, BN>();  // h of a gate_up tile is complete at this count
  const unsigned grid = gridDim.x;

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
  volatile int* s_ok = reinterpret_cast<volatile int*>(misc + 8);
  float* s_red = reinterpret_cast<float*>(misc + 16);  // 4 floats: norm reduction
  // h tile of a gate_up unit, [token][128 columns] bf16, written out with 16-byte stores
  __nv_bfloat16* s_h = reinterpret_cast<__nv_bfloat16*>(base_ptr + STAGES * S::kStageBytes + S::kBarBytes);
  // after the h tile: this CTA's place in the start order, the down-unit hand-off ring
  uint8_t* xtra = base_ptr + STAGES * S::kStageBytes + S::kBarBytes + BN * 128 * 2;
  volatile int* s_me = reinterpret_cast<volatile int*>(xtra);
  volatile unsigned long long* s_tbase = reinterpret_cast<volatile unsigned long long*>(xtra + 8);
  volatile int* s_unit = reinterpret_cast<volatile int*>(xtra + 16);          // kUnitSlots
  const uint32_t ufull0 = smem_u32(xtra + 32);                                  // kUnitSlots mbarriers
  const uint32_t uempty0 = smem_u32(xtra + 64);                                 // kUnitSlots mbarriers
  volatile unsigned* s_word = reinterpret_cast<volatile unsigned*>(xtra + 96);  // epilogue decisions
  float* s_inv = reinterpret_cast<float*>(xtra + 128);                          // 1 / rms per token (BN)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // the ticket first, so that its round trip overlaps the set-up below
  if (threadIdx.x == 64) {
    const unsigned long long tk = atomicAdd(P.ticket, 1ull);
    const unsigned long long me = tk % grid;
    *s_me = (int)me;
    *s_tbase = tk - me;
  }
  // The block's activations (a, the residual and gamma: 2 T H + H elements) are fetched
  // into L2 while this launch waits for the one before it, so that the norm rows and the
  // first k-blocks of gate_up's token operand, loaded once the wait ends, do not queue in
  // HBM behind the weight ring's first fill. Each line is prefetched by one thread of the grid.
  if (threadIdx.x >= 64) {
    const long long lines = ((long long)P.g1.T * P.H * 2 + 127) / 128;
    const long long gl = ((long long)P.H * 2 + 127) / 128;
    const long long gt = (long long)blockIdx.x * 128 + (threadIdx.x - 64), nt = (long long)grid * 128;
    const char* a = reinterpret_cast<const char*>(P.x_in);
    const char* r = reinterpret_cast<const char*>(P.res_in);
    for (long long i = gt; i < lines; i += nt) {
      prefetch_l2(a + i * 128);
      if (r != nullptr) prefetch_l2(r + i * 128);
    }
    if (P.has_norm && gt < gl) prefetch_l2(reinterpret_cast<const char*>(P.gamma) + gt * 128);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 2);   // the producer, and whoever provides the token operand
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 4);
    }
    mbar_init(done_bar, 1);
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(ufull0 + 8u * i, 1);
      mbar_init(uempty0 + 8u * i, 2);   // the MMA issuer and the epilogue
    }
    *s_abort = 0;
    fence_barrier_init();
    prefetch_tensormap(&map_x);
    prefetch_tensormap(&map_h);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(s_tmem)), S::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const unsigned long long timeout = P.g1.timeout_ns;
  // Every CTA has taken its ticket before this point, so a launch that follows on
  // the same stream (and may be scheduled onto SMs this grid frees) takes tickets
  // only after all of this launch's; it touches nothing but constant weights before
  // its griddepcontrol.wait.
  if (threadIdx.x == 0) griddep_launch_dependents();

  const int me = *s_me;
  const unsigned long long tbase = *s_tbase;
  // roles by start order: norm rows on [0, n_norm), gate_up units on [n_norm, owners_end)
  const int n_norm = P.n_norm;
  const int G = P.g1.units, D = P.g2.units;
  const int owner_span = min(G, (int)grid - n_norm);
  const int owners_end = n_norm + owner_span;
  const int g_first = (me >= n_norm && me < owners_end) ? me - n_norm : G;
  // With the norm, gate_up's token operand is y = bf16(r * gamma), r = bf16(a + r0),
  // which the norm CTAs write with 1 / rms of every row; the accumulator is scaled by
  // 1 / rms per token in the epilogue. For T <= 32 the gate_up CTAs do not wait for it
  // to start: their epilogue warps build the operand of their first k-blocks into the
  // ring stages themselves (the weights arrive by bulk copy).
  constexpr bool kBuildX = BN <= 32;
  constexpr int kBuildKb = STAGES;    // k-blocks of a gate_up unit whose token operand is built here
  const bool build_x = kBuildX && P.has_norm && P.g1.splits == 1;
  auto started = [&]() -> unsigned long long {
    return *reinterpret_cast<const volatile unsigned long long*>(P.ticket) - tbase;
  };

  auto set_abort = [&]() {
    if (!*s_abort) {
      atomicExch(P.g1.status, kStatusTimeout);
      *s_abort = 1;
    }
  };
  // The counters of this launch: the set selected by the number of launches completed
  // before it (read after griddepcontrol.wait). The other set is the next launch's; this
  // launch clears it, so no CTA has to find out at exit whether it is the last one.
  auto launch_parity = [&]() -> int {
    return (int)((*reinterpret_cast<const volatile unsigned long long*>(P.epoch) >> 32) & 1ull);
  };
  auto krange = [](const GemmParams& p, int u, int& tm, int& kb0, int& kb1) {
    const int tile = u / p.splits;
    const int sp = u - tile * p.splits;
    tm = tile;  // one token tile: tile == weight tile
    kb0 = (int)((long long)sp * p.nkb / p.splits);
    kb1 = (int)((long long)(sp + 1) * p.nkb / p.splits);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      // weight blocks are constant: they stream before this launch waits for the one
      // before it (griddepcontrol.wait), which comes first whenever an activation
      // copy or a counter of the workspace is needed
      bool dep_waited = false;
      unsigned* c_bars = nullptr;           // this launch's counters, known after the dependency wait
      const unsigned* c_hready = nullptr;
      auto wait_dep = [&]() {
        griddep_wait();
        dep_waited = true;
        const int par = launch_parity();
        c_bars = P.bars + 4 * par;
        c_hready = P.hready + par * P.cset;
      };
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, last_phase_bits = 0;
      // activation halves waiting for their producer: FIFO of (stage, kx, shard, gate_up tile or -1)
      int q_stage[STAGES], q_kx[STAGES], q_sh[STAGES], q_dep[STAGES];
      int q_head = 0, q_n = 0;
      bool x_ready = !P.has_norm;
      bool ok = true;
      // gate_up tiles (the first 256) already seen complete, as four 64-bit register
      // words (no dynamically indexed array: local memory would go to L2, the shared
      // memory carve-out leaves almost no L1). A down unit reads the h of a dozen tiles,
      // two k-blocks each: a tile's counter is read until it shows the tile complete, and
      // with it the count of finished tiles; once that count is full nothing is read.
      uint64_t rdy0 = 0, rdy1 = 0, rdy2 = 0, rdy3 = 0;
      bool all_known = false;     // every gate_up tile is finished (bars[2] counts them)
      const int n_tiles1 = P.g1.m_tiles;
      auto tile_known = [&](int x) -> bool {
        const uint64_t w = x < 64 ? rdy0 : x < 128 ? rdy1 : x < 192 ? rdy2 : rdy3;
        return ((w >> (x & 63)) & 1ull) != 0ull;
      };
      auto mark_known = [&](int x) {
        const uint64_t b = 1ull << (x & 63);
        if (x < 64) rdy0 |= b;
        else if (x < 128) rdy1 |= b;
        else if (x < 192) rdy2 |= b;
        else rdy3 |= b;
      };
      auto dep_ready = [&](int dep) -> bool {
        if (dep < 0) {
          if (!x_ready) x_ready = ld_acquire(c_bars) >= (unsigned)n_norm;
          return x_ready;
        }
        if (dep >= 256) return ld_acquire(c_hready + dep) >= (unsigned)kItems1;
        if (all_known || tile_known(dep)) return true;
        // the tile's counter and the count of finished tiles, in one round trip
        const unsigned v = ld_acquire(c_hready + dep);
        const unsigned n_done = ld_acquire(c_bars + 2);
        if (n_done >= (unsigned)n_tiles1) {
          all_known = true;
          return true;
        }
        if (v < (unsigned)kItems1) return false;
        mark_known(dep);
        return true;
      };
      auto issue_front = [&]() {
        const int i = q_head;
        const uint32_t sb = base + q_stage[i] * S::kStageBytes + S::kABytes;
        fence_proxy_async_global();
        if (q_dep[i] < 0)
          tma_load_4d(sb, &map_x, full_bar(q_stage[i]), q_kx[i], 0, 0, 0, pol_a);
        else
          tma_load_4d(sb, &map_h, full_bar(q_stage[i]), q_kx[i], 0, 0, q_sh[i], pol_a);
        q_head = (q_head + 1) % STAGES;
        --q_n;
      };
      // issue every queued activation copy whose data is ready; block (bounded) on the
      // oldest one while more than `keep` entries remain queued
      auto drain = [&](int keep) -> bool {
        if (q_n <= keep && !dep_waited) return true;
        if (!dep_waited) wait_dep();
        while (q_n > 0) {
          if (dep_ready(q_dep[q_head])) {
            issue_front();
            continue;
          }
          if (q_n <= keep) return true;
          const int dep = q_dep[q_head];
          const unsigned* c = dep < 0 ? c_bars : c_hready + dep;
          if (!poll_acquire(c, dep < 0 ? (unsigned)n_norm : (unsigned)kItems1, timeout, s_abort)) return false;
          if (dep < 0) x_ready = true;
          else if (dep < 256) mark_known(dep);
          issue_front();
        }
        return true;
      };
      // the loads of one unit: weight blocks at once, activation halves as their data is ready
      auto issue_unit = [&](int ph, int u) -> bool {
        const GemmParams& p = ph == 0 ? P.g1 : P.g2;
        int tm, kb0, kb1;
        krange(p, u, tm, kb0, kb1);
        const uint8_t* wsrc = p.w_packed + (size_t)tm * p.nkb * kWBlockBytes;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, s_abort, timeout)) return false;
          const uint32_t sa = base + stage * S::kStageBytes;
          const uint32_t fb = full_bar(stage);
          if (ph == 0 && build_x && kb < kb0 + kBuildKb) {
            // the epilogue warps write the token operand and make the second arrival
            mbar_arrive_expect_tx(fb, S::kABytes);
            bulk_load(sa, wsrc + (size_t)kb * kWBlockBytes, kWBlockBytes, fb, pol_w);
            issued_mask |= 1u << stage;
            last_phase_bits = (last_phase_bits & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          mbar_arrive_expect_tx(fb, S::kStageBytes);
          mbar_arrive(fb);
          bulk_load(sa, wsrc + (size_t)kb * kWBlockBytes, kWBlockBytes, fb, pol_w);
          int kx = kb * 64, shard = 0, dep = -1;
          if (ph == 1) {
            shard = kb / p.kbs;
            const int kk = kb - shard * p.kbs;
            kx = kk * 64;
            dep = shard * P.g1.nb + (kk * 64) / 128;   // gate_up tile that wrote these h columns
          }
          const int slot = (q_head + q_n) % STAGES;
          q_stage[slot] = stage;
          q_kx[slot] = kx;
          q_sh[slot] = shard;
          q_dep[slot] = dep;
          ++q_n;
          if (!drain(STAGES - 1)) return false;
          issued_mask |= 1u << stage;
          last_phase_bits = (last_phase_bits & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        return true;
      };
      // ---- gate_up units of this CTA
      for (int u = g_first; u < G && ok; u += owner_span) {
        if (!issue_unit(0, u)) {
          set_abort();
          ok = false;
        }
      }
      // ---- down units, claimed from the launch's counter. A claimed unit waits on h
      // tiles, so nothing is claimed before every gate_up owner has started; a CTA that
      // has waited kStartPatienceNs for that gives up its down work (and says so) so
      // that its SM can take a CTA that has not started. When every CTA of the launch
      // has started and none gave up, every CTA makes one claim and together they claim
      // all units (there are no more units than CTAs); otherwise CTAs keep claiming.
      if (ok && !dep_waited) wait_dep();
      bool gave_up = false, first = true;
      int uslot = 0;
      uint32_t uphase = 0;
      for (;;) {
        int u = -1;
        if (ok && !gave_up) {
          bool claim = true;
          if (first) {
            if (started() < (unsigned long long)owners_end) {
              const uint64_t t0 = globaltimer_ns();
              while (started() < (unsigned long long)owners_end && globaltimer_ns() - t0 < kStartPatienceNs)
                __nanosleep(200);
              if (started() < (unsigned long long)owners_end) {
                // announce first, then look again: a CTA that later finds every CTA started
                // and nobody gone sees this count if this CTA does give up
                atomicAdd(c_bars + 1, 1u);
                __threadfence();
                if (started() < (unsigned long long)owners_end) gave_up = true;
                else atomicSub(c_bars + 1, 1u);
              }
            }
            claim = !gave_up;
          } else {
            const bool all_started = started() >= grid;
            __threadfence();
            const bool nobody_gone = *reinterpret_cast<const volatile unsigned*>(c_bars + 1) == 0u;
            claim = !(all_started && nobody_gone && D <= (int)grid);
          }
          if (claim) {
            u = (int)atomicAdd(c_bars + 3, 1u);
            if (u >= D) u = -1;
          }
          first = false;
        }
        if (!mbar_wait_bounded(uempty0 + 8u * uslot, uphase ^ 1u, s_abort, timeout)) {
          set_abort();
          ok = false;
          break;
        }
        s_unit[uslot] = u;
        mbar_arrive(ufull0 + 8u * uslot);
        if (++uslot == kUnitSlots) {
          uslot = 0;
          uphase ^= 1u;
        }
        if (u < 0) break;
        if (!issue_unit(1, u)) {
          set_abort();
          ok = false;
        }
      }
      if (!dep_waited) wait_dep();
      if (ok && !drain(0)) {
        set_abort();
        ok = false;
      }
      if (!ok) {
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
      auto wait_all = [&](uint32_t b, uint32_t ph) -> bool {
        return __all_sync(0xffffffffu, mbar_wait_bounded(b, ph, s_abort, timeout));
      };
      auto mma_unit = [&](int ph, int u) -> bool {
        const GemmParams& p = ph == 0 ? P.g1 : P.g2;
        int tm, kb0, kb1;
        krange(p, u, tm, kb0, kb1);
        if (!wait_all(tempty_bar(buf), acc_phase ^ 1u)) return false;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * ACC;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_all(full_bar(stage), phase)) return false;
          tc_fence_after();
          const uint32_t sa = base + stage * S::kStageBytes;
          const uint64_t adesc = smem_desc_k128(sa);
          const uint64_t bdesc = smem_desc_k128(sa + S::kABytes);
          if (elect_one()) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
              for (int a = 0; a < 2; ++a)
                tc_mma_bf16(d_tmem + a * BN, adesc + (uint64_t)(a * (128 * 128 >> 4) + ks * 2),
                            bdesc + (uint64_t)(ks * 2), S::kIdesc, (kb > kb0 || ks > 0) ? 1u : 0u);
            }
            tc_commit(empty_bar(stage));
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (elect_one()) tc_commit(tfull_bar(buf));
        __syncwarp();
        if (++buf == 2) {
          buf = 0;
          acc_phase ^= 1u;
        }
        return true;
      };
      for (int u = g_first; u < G && ok; u += owner_span) ok = mma_unit(0, u);
      int uslot = 0;
      uint32_t uphase = 0;
      while (ok) {
        if (!wait_all(ufull0 + 8u * uslot, uphase)) {
          ok = false;
          break;
        }
        const int u = s_unit[uslot];
        __syncwarp();
        if (lane == 0) mbar_arrive(uempty0 + 8u * uslot);
        if (++uslot == kUnitSlots) {
          uslot = 0;
          uphase ^= 1u;
        }
        if (u < 0) break;
        ok = mma_unit(1, u);
      }
      if (!ok && lane == 0) set_abort();
      if (elect_one()) tc_commit(done_bar);
      __syncwarp();
      mbar_wait_bounded(done_bar, 0, nullptr, kTeardownNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int et = threadIdx.x - 64;  // 0..127
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const long long etid = (long long)blockIdx.x * 128 + et, ethreads = (long long)grid * 128;
    int buf = 0;
    uint32_t acc_phase = 0;
    bool ok = true;

    // Barrier among the 128 epilogue threads that shares one thread's decision.
    auto agree = [&](bool mine_ok) -> bool {
      if (et == 0) *s_ok = mine_ok ? 1 : 0;
      named_bar_sync(1, 128);
      const bool r = *s_ok != 0;
      named_bar_sync(1, 128);
      return r;
    };
    auto share = [&](unsigned mine) -> unsigned {
      if (et == 0) *s_word = mine;
      named_bar_sync(1, 128);
      const unsigned r = *s_word;
      named_bar_sync(1, 128);
      return r;
    };
    griddep_wait();
    const int par = launch_parity();
    unsigned* const e_bars = P.bars + 4 * par;
    unsigned* const e_cnt1 = P.cnt1 + par * P.cset;
    unsigned* const e_hready = P.hready + par * P.cset;
    unsigned* const e_cnt2 = P.cnt2 + par * P.cset;
    {
      // the other set, used by the launch before this one, starts the next launch at zero
      unsigned* const o_bars = P.bars + 4 * (par ^ 1);
      unsigned* const o_cnt = P.cnt1 + (par ^ 1) * P.cset;
      for (long long i = etid; i < P.cset; i += ethreads) o_cnt[i] = 0u;
      if (blockIdx.x == 0 && et < 4) o_bars[et] = 0u;
    }
    // ---- phase 0: the rows of this CTA (the first n_norm CTAs to start): r = bf16(a + r0)
    // to residual_out, gate_up's token operand y = bf16(r * gamma) to the workspace, and
    // 1 / rms of r. The loads of a chunk (a, residual and gamma, up to 8 vectors per
    // thread each) are issued together before anything waits on them, so a row costs one
    // memory round trip (rows longer than 8 * 8 * 128 = 8192 take more chunks).
    if (P.has_norm && me < n_norm) {
      const int H = P.H, nvec = H >> 3;
      constexpr int NV = 8;
      const uint4* gv = reinterpret_cast<const uint4*>(P.gamma);
      for (int r = me; r < P.g1.T; r += n_norm) {
        const size_t roff = (size_t)r * H;
        const uint4* av = reinterpret_cast<const uint4*>(P.x_in + roff);
        const uint4* rv = reinterpret_cast<const uint4*>(P.res_in + roff);
        uint4* ro = reinterpret_cast<uint4*>(P.res_out + roff);
        uint4* yo = reinterpret_cast<uint4*>(P.x_norm + roff);
        float ss = 0.f;
        for (int v0 = 0; v0 < nvec; v0 += NV * 128) {
          uint4 a4[NV], r4[NV], g4[NV];
#pragma unroll
          for (int k = 0; k < NV; ++k) {
            const int v = v0 + k * 128 + et;
            if (v < nvec) {
              a4[k] = __ldcg(av + v);
              r4[k] = __ldcg(rv + v);
              g4[k] = __ldg(gv + v);
            }
          }
#pragma unroll
          for (int k = 0; k < NV; ++k) {
            const int v = v0 + k * 128 + et;
            if (v < nvec) {
              const __nv_bfloat162* ab = reinterpret_cast<const __nv_bfloat162*>(&a4[k]);
              const __nv_bfloat162* rb = reinterpret_cast<const __nv_bfloat162*>(&r4[k]);
              const __nv_bfloat162* gb = reinterpret_cast<const __nv_bfloat162*>(&g4[k]);
              uint4 o, y;
              __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
              __nv_bfloat162* yb = reinterpret_cast<__nv_bfloat162*>(&y);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 fa = __bfloat1622float2(ab[i]), fr = __bfloat1622float2(rb[i]);
                ob[i] = __floats2bfloat162_rn(fa.x + fr.x, fa.y + fr.y);
                const float2 q2 = __bfloat1622float2(ob[i]);  // the stored residual is what is normalised
                const float2 fg = __bfloat1622float2(gb[i]);
                ss += q2.x * q2.x + q2.y * q2.y;
                yb[i] = __floats2bfloat162_rn(q2.x * fg.x, q2.y * fg.y);
              }
              ro[v] = o;
              yo[v] = y;
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) s_red[q] = ss;
        named_bar_sync(1, 128);
        if (et == 0) P.inv[r] = rsqrtf((s_red[0] + s_red[1] + s_red[2] + s_red[3]) / (float)H + P.eps);
        named_bar_sync(1, 128);
      }
      // y is read by the tensor copies of gate_up (async proxy); the rows of all epilogue
      // threads are released by one release-add after the barrier
      fence_proxy_async_global();
      named_bar_sync(1, 128);
      if (et == 0) red_release_add(e_bars + 0, 1u);
    }

    float g[CH], uu[CH];
    // epilogue of one unit (ph 0: gate_up, 1: down)
    auto epi_unit = [&](int ph, int u) -> bool {
      const GemmParams& p = ph == 0 ? P.g1 : P.g2;
      int tm, kb0, kb1;
      krange(p, u, tm, kb0, kb1);
      const int sp = u - tm * p.splits;
      bool w_ok = true;
      if (et == 0) {
        w_ok = mbar_wait_bounded(tfull_bar(buf), acc_phase, s_abort, timeout);
        if (!w_ok) set_abort();
      }
      if (!agree(w_ok)) return false;
      tc_fence_after();
      const uint32_t acc = lane_addr + buf * ACC;
      if (++buf == 2) {
        buf = 0;
        acc_phase ^= 1u;
      }
      const uint32_t this_buf = (buf ^ 1);
      if (p.splits == 1) {
        if (ph == 0) {
          // silu(g) * u goes to shared memory as [token][column]; the tile is then
          // written row by row with 16-byte stores (one warp store covers 512 bytes,
          // where a column per thread would take a store per token)
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += CH) {
            if (CH == 32) { tmem_ld32(acc + c0, g); tmem_ld32(acc + BN + c0, uu); }
            else { tmem_ld16(acc + c0, g); tmem_ld16(acc + BN + c0, uu); }
            tc_wait_ld();
            if (P.has_norm) {
#pragma unroll
              for (int j = 0; j < CH; ++j) {
                const float iv = s_inv[c0 + j];
                s_h[(c0 + j) * 128 + row] = __float2bfloat16_rn(silu_f(g[j] * iv) * (uu[j] * iv));
              }
            } else {
#pragma unroll
              for (int j = 0; j < CH; ++j) s_h[(c0 + j) * 128 + row] = __float2bfloat16_rn(silu_f(g[j]) * uu[j]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(this_buf));
          named_bar_sync(1, 128);
          const int r = tm / p.nb, i0 = (tm - r * p.nb) * 128;
          __nv_bfloat16* dst = p.out + (size_t)r * p.T * p.Is + i0;
          for (int idx = et; idx < p.T * 16; idx += 128) {
            const int tok = idx >> 4, ch = idx & 15;
            if (i0 + ch * 8 < p.Is)
              *reinterpret_cast<uint4*>(dst + (size_t)tok * p.Is + ch * 8) =
                  *reinterpret_cast<const uint4*>(s_h + tok * 128 + ch * 8);
          }
          // this tile's h columns are complete (released by one thread after the barrier)
          fence_proxy_async_global();
          named_bar_sync(1, 128);
          if (et == 0) {
            red_release_add(e_hready + tm, (unsigned)kItems1);
            red_release_add(e_bars + 2, 1u);
          }
        } else {
#pragma unroll 1
          for (int seg = 0; seg < 2; ++seg) {
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += CH) {
              if (CH == 32) tmem_ld32(acc + seg * BN + c0, g); else tmem_ld16(acc + seg * BN + c0, g);
              tc_wait_ld();
              emit_vals<true, KIND_ROW, BN, CH>(p, tm, 0, seg, row, c0, g, uu);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(this_buf));
        }
        return true;
      }
      float* part = p.partials + ((size_t)tm * p.splits + sp) * ACC * 128;
#pragma unroll 1
      for (int c0 = 0; c0 < ACC; c0 += CH) {
        if (CH == 32) tmem_ld32(acc + c0, g); else tmem_ld16(acc + c0, g);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < CH; ++j) __stcg(part + (size_t)(c0 + j) * 128 + row, g[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(this_buf));
      // the partial of every epilogue thread is released by the arrival (acq_rel) after the barrier
      named_bar_sync(1, 128);
      if (ph == 0) {
        // gate_up split-K: the last split of the tile to arrive adds the tile's partials
        // (split order) and publishes its h columns; no split waits for another
        unsigned last = 0;
        if (et == 0) last = atom_acq_rel_add(e_cnt1 + tm, 1u) == (unsigned)(p.splits - 1) ? 1u : 0u;
        if (share(last)) {
          reduce_tile_items<true, KIND_GATE_UP, BN>(p, tm, 0, kItems1, et, 128);
          fence_proxy_async_global();
          named_bar_sync(1, 128);
          if (et == 0) {
            red_release_add(e_hready + tm, (unsigned)kItems1);
            red_release_add(e_bars + 2, 1u);
          }
        }
        return true;
      }
      // down split-K: the count word holds the arrivals (low 16 bits) and, in bit
      // 16 + s, the splits that handed their slice over. Each split adds its own slice
      // of the tile once all splits have arrived; a split that has waited
      // kSplitPatienceNs hands its slice to the last split to arrive, which adds its
      // own slice and every slice handed over before it arrived. Every slice is added
      // once, in split order, whoever adds it.
      constexpr int items = tile_items<true, KIND_ROW, BN>();
      const unsigned S2n = (unsigned)p.splits;
      unsigned mask = 0;
      if (et == 0) {
        unsigned* cnt = e_cnt2 + tm;
        const unsigned old = atom_acq_rel_add(cnt, 1u);
        if ((old & 0xFFFFu) == S2n - 1u) {
          mask = (1u << sp) | (old >> 16);
        } else {
          bool all = (ld_acquire(cnt) & 0xFFFFu) >= S2n;
          const uint64_t t0 = globaltimer_ns();
          while (!all && globaltimer_ns() - t0 < kSplitPatienceNs) {
            __nanosleep(64);
            all = (ld_acquire(cnt) & 0xFFFFu) >= S2n;
          }
          if (!all) {
            unsigned w = ld_acquire(cnt);
            for (;;) {
              if ((w & 0xFFFFu) >= S2n) {
                all = true;
                __threadfence();
                break;
              }
              const unsigned prev = atomicCAS(cnt, w, w | (1u << (16 + sp)));
              if (prev == w) break;      // handed over
              w = prev;
            }
          }
          if (all) mask = 1u << sp;
        }
      }
      mask = share(mask);
      for (int s = 0; s < (int)S2n; ++s)
        if (mask & (1u << s))
          reduce_tile_items<true, KIND_ROW, BN>(p, tm, (int)((long long)s * items / S2n),
                                                (int)((long long)(s + 1) * items / S2n), et, 128);
      return true;
    };
    // ---- the token operand of the first kBuildKb k-blocks of a gate_up unit (build_x):
    // y = bf16(bf16(a + r0) * gamma), the values the norm CTAs write for the rest, built
    // by this CTA's epilogue warps straight into the ring stages the producer filled
    // with those k-blocks' weights, so gate_up starts before the norm rows are published.
    // Loads run two k-blocks ahead. Each thread owns NC 16-byte chunks (8 features of one
    // token) of a k-block's [BN tokens][64] tile.
    constexpr int NC = kBuildX ? BN / 16 : 1;
    int bstage = 0;
    uint32_t bphase = 0;
    auto build_unit = [&](int u) -> bool {
      int tm, kb0, kb1;
      krange(P.g1, u, tm, kb0, kb1);
      const int kbb = min(kb1, kb0 + kBuildKb);
      const int H = P.H, T = P.g1.T;
      struct Chunks {
        uint4 a[NC], r[NC], g[NC];
      };
      auto load = [&](int kb, Chunks& c) {
#pragma unroll
        for (int m = 0; m < NC; ++m) {
          const int ci = et + 128 * m, t = ci >> 3, col = kb * 64 + (ci & 7) * 8;
          if (kb < kbb && t < T && col < H) {
            c.a[m] = __ldcg(reinterpret_cast<const uint4*>(P.x_in + (size_t)t * H + col));
            c.r[m] = __ldcg(reinterpret_cast<const uint4*>(P.res_in + (size_t)t * H + col));
            c.g[m] = __ldg(reinterpret_cast<const uint4*>(P.gamma + col));
          } else {
            c.a[m] = c.r[m] = c.g[m] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      };
      Chunks c0, c1, c2;
      load(kb0, c0);
      load(kb0 + 1, c1);
      for (int kb = kb0; kb < kbb; ++kb) {
        load(kb + 2, c2);
        uint4 y[NC];
#pragma unroll
        for (int m = 0; m < NC; ++m) {
          const __nv_bfloat162* ab = reinterpret_cast<const __nv_bfloat162*>(&c0.a[m]);
          const __nv_bfloat162* rb = reinterpret_cast<const __nv_bfloat162*>(&c0.r[m]);
          const __nv_bfloat162* gb = reinterpret_cast<const __nv_bfloat162*>(&c0.g[m]);
          __nv_bfloat162* yb = reinterpret_cast<__nv_bfloat162*>(&y[m]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 fa = __bfloat1622float2(ab[i]), fr = __bfloat1622float2(rb[i]);
            const float2 q2 = __bfloat1622float2(__floats2bfloat162_rn(fa.x + fr.x, fa.y + fr.y));
            const float2 fg = __bfloat1622float2(gb[i]);
            yb[i] = __floats2bfloat162_rn(q2.x * fg.x, q2.y * fg.y);
          }
        }
        bool w_ok = true;
        if (et == 0) {
          w_ok = mbar_wait_bounded(empty_bar(bstage), bphase ^ 1u, s_abort, timeout);
          if (!w_ok) set_abort();
        }
        if (!agree(w_ok)) return false;
        uint8_t* sb = base_ptr + bstage * S::kStageBytes + S::kABytes;   // [BN rows][128 B], 128-byte swizzle
#pragma unroll
        for (int m = 0; m < NC; ++m) {
          const int ci = et + 128 * m, t = ci >> 3, j = ci & 7;
          *reinterpret_cast<uint4*>(sb + t * 128 + ((j ^ (t & 7)) << 4)) = y[m];
        }
        fence_proxy_async_shared();
        named_bar_sync(1, 128);
        if (et == 0) mbar_arrive(full_bar(bstage));
        if (++bstage == STAGES) {
          bstage = 0;
          bphase ^= 1u;
        }
        c0 = c1;
        c1 = c2;
      }
      // the unit's other k-blocks are loaded by the producer: advance the ring past them
      for (int kb = kbb; kb < kb1; ++kb)
        if (++bstage == STAGES) {
          bstage = 0;
          bphase ^= 1u;
        }
      return true;
    };
    // the gate_up epilogue reads 1 / rms and down's residual epilogue residual_out, both
    // written by the norm CTAs (which wait on nothing)
    auto acquire_norm = [&]() -> bool {
      bool w_ok = true;
      if (et == 0) {
        w_ok = poll_acquire(e_bars + 0, (unsigned)n_norm, timeout, s_abort);
        if (!w_ok) set_abort();
      }
      if (!agree(w_ok)) return false;
      if (et < BN) s_inv[et] = et < P.g1.T ? __ldcg(P.inv + et) : 0.f;
      named_bar_sync(1, 128);
      return true;
    };
    bool norm_seen = !P.has_norm;
    // ---- gate_up units of this CTA, then the down units the producer hands over
    for (int u = g_first; u < G && ok; u += owner_span) {
      if (build_x && !build_unit(u)) {
        ok = false;
        break;
      }
      if (!norm_seen) {
        if (!acquire_norm()) {
          ok = false;
          break;
        }
        norm_seen = true;
      }
      ok = epi_unit(0, u);
    }
    if (ok && !norm_seen) ok = acquire_norm();
    int uslot = 0;
    uint32_t uphase = 0;
    while (ok) {
      bool w_ok = true;
      if (et == 0) {
        w_ok = mbar_wait_bounded(ufull0 + 8u * uslot, uphase, s_abort, timeout);
        if (!w_ok) set_abort();
      }
      if (!agree(w_ok)) break;
      const int u = s_unit[uslot];
      named_bar_sync(1, 128);
      if (et == 0) mbar_arrive(uempty0 + 8u * uslot);
      if (++uslot == kUnitSlots) {
        uslot = 0;
        uphase ^= 1u;
      }
      if (u < 0) break;
      ok = epi_unit(1, u);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::kTmemCols);
  }
  // this CTA's share of the launch count; the grid's shares add up to exactly 2^32, so the high
  // word counts completed launches whatever grid each launch had (no CTA waits for the sum)
  if (threadIdx.x == 0) {
    const unsigned long long share = (1ull << 32) / grid;
    atomicAdd(P.epoch, blockIdx.x == 0 ? (1ull << 32) - share * (grid - 1) : share);
  }
}

template <int BN>
cudaError_t launch_mlp_decode_bn(const CUtensorMap& mx, const CUtensorMap& mh, const MlpDecodeParams& P,
                                 int grid, cudaStream_t st) {
  using S = GemmShape<true, KIND_GATE_UP, BN>;
  auto kernel = mlp_decode_kernel<BN>;
  constexpr int kSmem = S::kSmemBytes + BN * 128 * 2 + 128 + BN * 4;  // ring, barriers, h tile, tickets and unit slots, 1/rms
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  // One CTA per SM (shared memory), grid == SM count. The kernel does not need its
  // CTAs to be resident together (their roles follow the order in which they start),
  // so other work may hold SMs meanwhile. Programmatic serialisation lets the next
  // launch on the stream be scheduled onto SMs this grid frees.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, mx, mh, P);
  return e;
}

// CTAs of the fused kernel for block_n = BN that fit on one SM (0: it cannot run here).
template <int BN>
int mlp_decode_ctas_per_sm_bn() {
  using S = GemmShape<true, KIND_GATE_UP, BN>;
  auto kernel = mlp_decode_kernel<BN>;
  constexpr int kSmem = S::kSmemBytes + BN * 128 * 2 + 128 + BN * 4;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 192, kSmem) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

int mlp_decode_ctas_per_sm(int bn) {
  // asked once per device and block_n (the answer cannot change)
  static std::atomic<int> cached[64][4];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const int slot = bn == 16 ? 0 : bn == 32 ? 1 : bn == 64 ? 2 : bn == 128 ? 3 : -1;
  if (slot < 0) return 0;
  const int v = cached[dev & 63][slot].load(std::memory_order_relaxed);
  if (v != 0) return v > 0 ? v : 0;
  int n = 0;
  switch (bn) {
    case 16: n = mlp_decode_ctas_per_sm_bn<16>(); break;
    case 32: n = mlp_decode_ctas_per_sm_bn<32>(); break;
    case 64: n = mlp_decode_ctas_per_sm_bn<64>(); break;
    default: n = mlp_decode_ctas_per_sm_bn<128>(); break;
  }
  cached[dev & 63][slot].store(n > 0 ? n : -1, std::memory_order_relaxed);
  return n;
}

cudaError_t launch_mlp_decode(int bn, const CUtensorMap& mx, const CUtensorMap& mh, const MlpDecodeParams& P,
                              int grid, cudaStream_t st) {
  switch (bn) {
    case 16: return launch_mlp_decode_bn<16>(mx, mh, P, grid, st);
    case 32: return launch_mlp_decode_bn<32>(mx, mh, P, grid, st);
    case 64: return launch_mlp_decode_bn<64>(mx, mh, P, grid, st);
    case 128: return launch_mlp_decode_bn<128>(mx, mh, P, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tpl
