// Fused decode-shaped MLP block: one persistent launch runs the
// whole step for T <= 128 tokens.
//
//   norm     residual add + RMSNorm of the T rows by the epilogue warps (rows
//            spread over CTAs); the CTAs that own rows arrive on bars[0]
//   gate_up  column-parallel units of 256 weight rows (128 gate + 128 up of
//            one shard) x a K range; with split-K every split writes its fp32
//            partial. After one grid-wide wait the CTAs add the partials tile
//            by tile (split order), in the order the down splits will read h,
//            write silu(g) * u to h [t][T][I/t] and count finished items in
//            hready[tile]
//   down     row-parallel units: K runs over the t shards in turn, so the
//            shards' partial sums meet in the accumulator. The producer loads
//            the h columns of a k-block as soon as the gate_up tile that
//            wrote them is complete, streaming weight blocks meanwhile. The
//            splits of a down tile (resident together) each add their slice
//            of the tile; mlp_out = y, residual_stream = y + residual
//
// Between the GEMMs, work flows through per-tile counters and flags in the
// workspace. Every wait is bounded (status word on timeout); with one CTA per SM
// every CTA of the grid is resident. There are two sets of counters: a launch
// uses the one its launch count (a word every CTA adds its share to at exit)
// selects, and clears the other for the next launch.
#include "gemm_launch.cuh"

namespace tpl {


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
  // CTAs that own norm rows (row r goes to CTA r % grid); only they arrive on bars[0]
  const unsigned norm_ctas = (unsigned)min((int)grid, P.g1.T);

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
  // the down unit this CTA takes at run time, and the barrier that publishes it to the roles
  const uint32_t unit_bar = smem_u32(misc + 32);
  volatile int* s_unit = reinterpret_cast<volatile int*>(misc + 40);
  // h tile of a gate_up unit, [token][128 columns] bf16, written out with 16-byte stores
  __nv_bfloat16* s_h = reinterpret_cast<__nv_bfloat16*>(base_ptr + STAGES * S::kStageBytes + S::kBarBytes);

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
    mbar_init(unit_bar, 1);
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
  // A launch that follows on the same stream may be scheduled onto SMs this grid
  // frees; it touches nothing but constant weights before its griddepcontrol.wait.
  if (threadIdx.x == 0) griddep_launch_dependents();

  auto set_abort = [&]() {
    if (!*s_abort) {
      atomicExch(P.g1.status, kStatusTimeout);
      *s_abort = 1;
    }
  };
  // gate_up units go to CTAs 0, 1, ... When there are no more down units than CTAs, each CTA
  // takes at most one down unit from a counter once its producer has issued its gate_up
  // work, so the CTAs that finish gate_up first (or have none) take the down units first.
  // Otherwise down units go to CTAs grid-1, grid-2, ..., so CTAs without gate_up work start
  // down at once.
  const bool dyn_down = P.g2.units <= (int)grid;
  auto first_unit = [&](int ph) -> int { return ph == 0 ? (int)blockIdx.x : (int)(grid - 1 - blockIdx.x); };
  auto step_unit = [&](int ph, int u, int units) -> int { return (ph == 1 && dyn_down) ? units : u + (int)grid; };
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
      const unsigned* c_bars = nullptr;     // this launch's counters, known after the dependency wait
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
      auto dep_ready = [&](int dep) -> bool {
        if (dep < 0) {
          if (!x_ready) x_ready = *reinterpret_cast<const volatile unsigned*>(c_bars) >= norm_ctas;
          return x_ready;
        }
        return *reinterpret_cast<const volatile unsigned*>(c_hready + dep) >= (unsigned)kItems1;
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
          if (!bar_wait(c, dep < 0 ? norm_ctas : (unsigned)kItems1, timeout, s_abort)) return false;
          if (dep < 0) x_ready = true;
          issue_front();
        }
        return true;
      };
      for (int ph = 0; ph < 2 && ok; ++ph) {
        const GemmParams& p = ph == 0 ? P.g1 : P.g2;
        int u0 = first_unit(ph);
        if (ph == 1 && dyn_down) {
          // the counter belongs to this launch once the previous one has completed
          if (!dep_waited) wait_dep();
          u0 = (int)atomicAdd(const_cast<unsigned*>(c_bars) + 3, 1u);
          *s_unit = u0;
          mbar_arrive(unit_bar);
        }
        for (int u = u0; u < p.units && ok; u = step_unit(ph, u, p.units)) {
          int tm, kb0, kb1;
          krange(p, u, tm, kb0, kb1);
          const uint8_t* wsrc = p.w_packed + (size_t)tm * p.nkb * kWBlockBytes;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, s_abort, timeout)) {
              set_abort();
              ok = false;
              break;
            }
            const uint32_t sa = base + stage * S::kStageBytes;
            const uint32_t fb = full_bar(stage);
            mbar_arrive_expect_tx(fb, S::kStageBytes);
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
            if (!drain(STAGES - 1)) {
              set_abort();
              ok = false;
              break;
            }
            issued_mask |= 1u << stage;
            last_phase_bits = (last_phase_bits & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
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
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int ph = 0; ph < 2 && ok; ++ph) {
        const GemmParams& p = ph == 0 ? P.g1 : P.g2;
        int u0 = first_unit(ph);
        if (ph == 1 && dyn_down) {
          if (!mbar_wait_bounded(unit_bar, 0, s_abort, timeout)) {
            set_abort();
            ok = false;
            break;
          }
          u0 = *s_unit;
        }
        for (int u = u0; u < p.units && ok; u = step_unit(ph, u, p.units)) {
          int tm, kb0, kb1;
          krange(p, u, tm, kb0, kb1);
          if (!mbar_wait_bounded(tempty_bar(buf), acc_phase ^ 1u, s_abort, timeout)) {
            set_abort();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * ACC;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait_bounded(full_bar(stage), phase, s_abort, timeout)) {
              set_abort();
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = base + stage * S::kStageBytes;
            const uint64_t adesc = smem_desc_k128(sa);
            const uint64_t bdesc = smem_desc_k128(sa + S::kABytes);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
              for (int a = 0; a < 2; ++a)
                tc_mma_bf16(d_tmem + a * BN, adesc + (uint64_t)(a * (128 * 128 >> 4) + ks * 2),
                            bdesc + (uint64_t)(ks * 2), S::kIdesc, (kb > kb0 || ks > 0) ? 1u : 0u);
            }
            tc_commit(empty_bar(stage));
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit(tfull_bar(buf));
          if (++buf == 2) {
            buf = 0;
            acc_phase ^= 1u;
          }
        }
      }
      tc_commit(done_bar);
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
    griddep_wait();
    const int par = launch_parity();
    unsigned* const e_bars = P.bars + 4 * par;
    unsigned* const e_hready = P.hready + par * P.cset;
    unsigned* const e_cnt2 = P.cnt2 + par * P.cset;
    {
      // the other set, used by the launch before this one, starts the next launch at zero
      unsigned* const o_bars = P.bars + 4 * (par ^ 1);
      unsigned* const o_cnt = P.cnt1 + (par ^ 1) * P.cset;
      for (long long i = etid; i < P.cset; i += ethreads) o_cnt[i] = 0u;
      if (blockIdx.x == 0 && et < 4) o_bars[et] = 0u;
    }
    // ---- phase 0: residual add + RMSNorm, one row per CTA in turn. The loads of
    // a chunk (a, residual and gamma, up to 8 vectors per thread each) are issued
    // together before anything waits on them, and the rounded residual stays in
    // registers, so a row costs one memory round trip (H <= 8 * 8 * 128 = 8192 in
    // one chunk; longer rows loop).
    if (P.has_norm) {
      const int H = P.H, nvec = H >> 3;
      constexpr int NV = 8;
      const uint4* gv = reinterpret_cast<const uint4*>(P.gamma);
      for (int r = blockIdx.x; r < P.g1.T; r += grid) {
        const size_t roff = (size_t)r * H;
        const uint4* av = reinterpret_cast<const uint4*>(P.x_in + roff);
        const uint4* rv = reinterpret_cast<const uint4*>(P.res_in + roff);
        uint4* ro = reinterpret_cast<uint4*>(P.res_out + roff);
        uint4* xo = reinterpret_cast<uint4*>(P.x_norm + roff);
        const bool one_chunk = nvec <= NV * 128;
        float ss = 0.f;
        uint4 a4[NV], r4[NV], g4[NV];
        for (int v0 = 0; v0 < nvec; v0 += NV * 128) {
#pragma unroll
          for (int k = 0; k < NV; ++k) {
            const int v = v0 + k * 128 + et;
            if (v < nvec) {
              a4[k] = __ldg(av + v);
              r4[k] = __ldg(rv + v);
              g4[k] = __ldg(gv + v);
            }
          }
#pragma unroll
          for (int k = 0; k < NV; ++k) {
            const int v = v0 + k * 128 + et;
            if (v < nvec) {
              const __nv_bfloat162* ab = reinterpret_cast<const __nv_bfloat162*>(&a4[k]);
              const __nv_bfloat162* rb = reinterpret_cast<const __nv_bfloat162*>(&r4[k]);
              __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&a4[k]);  // a4[k] becomes the residual
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 fa = __bfloat1622float2(ab[i]), fr = __bfloat1622float2(rb[i]);
                ob[i] = __floats2bfloat162_rn(fa.x + fr.x, fa.y + fr.y);
                const float2 q2 = __bfloat1622float2(ob[i]);  // the stored residual is what is normalised
                ss += q2.x * q2.x + q2.y * q2.y;
              }
              ro[v] = a4[k];
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) s_red[q] = ss;
        named_bar_sync(1, 128);
        const float inv = rsqrtf((s_red[0] + s_red[1] + s_red[2] + s_red[3]) / (float)H + P.eps);
        named_bar_sync(1, 128);
        for (int v0 = 0; v0 < nvec; v0 += NV * 128) {
          if (!one_chunk) {
            // rows longer than one chunk: the registers hold the last chunk only
#pragma unroll
            for (int k = 0; k < NV; ++k) {
              const int v = v0 + k * 128 + et;
              if (v < nvec) {
                a4[k] = ro[v];   // written by this thread above
                g4[k] = __ldg(gv + v);
              }
            }
          }
#pragma unroll
          for (int k = 0; k < NV; ++k) {
            const int v = v0 + k * 128 + et;
            if (v < nvec) {
              const __nv_bfloat162* rb = reinterpret_cast<const __nv_bfloat162*>(&a4[k]);
              const __nv_bfloat162* gb = reinterpret_cast<const __nv_bfloat162*>(&g4[k]);
              uint4 o;
              __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 fr = __bfloat1622float2(rb[i]), fg = __bfloat1622float2(gb[i]);
                ob[i] = __floats2bfloat162_rn(fr.x * inv * fg.x, fr.y * inv * fg.y);
              }
              xo[v] = o;
            }
          }
        }
      }
      // x_norm is read by the tensor copies of phase 1 (async proxy); the rows of all
      // epilogue threads are released by the one fence in bar_arrive after the barrier
      fence_proxy_async_global();
      named_bar_sync(1, 128);
      if (et == 0 && blockIdx.x < norm_ctas) bar_arrive(e_bars + 0);
    }

    float g[CH], uu[CH];
    // ---- gate_up units, then down units
    for (int ph = 0; ph < 2 && ok; ++ph) {
      const GemmParams& p = ph == 0 ? P.g1 : P.g2;
      int u0 = first_unit(ph);
      if (ph == 1 && dyn_down) {
        bool w_ok = true;
        if (et == 0) {
          w_ok = mbar_wait_bounded(unit_bar, 0, s_abort, timeout);
          if (!w_ok) set_abort();
        }
        if (!agree(w_ok)) {
          ok = false;
          break;
        }
        u0 = *s_unit;
      }
      for (int u = u0; u < p.units && ok; u = step_unit(ph, u, p.units)) {
        int tm, kb0, kb1;
        krange(p, u, tm, kb0, kb1);
        const int sp = u - tm * p.splits;
        bool w_ok = true;
        if (et == 0) {
          w_ok = mbar_wait_bounded(tfull_bar(buf), acc_phase, s_abort, timeout);
          if (!w_ok) set_abort();
        }
        if (!agree(w_ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = lane_addr + buf * ACC;
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
#pragma unroll
              for (int j = 0; j < CH; ++j) s_h[(c0 + j) * 128 + row] = __float2bfloat16_rn(silu_f(g[j]) * uu[j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(buf));
            named_bar_sync(1, 128);
            const int r = tm / p.nb, i0 = (tm - r * p.nb) * 128;
            __nv_bfloat16* dst = p.out + (size_t)r * p.T * p.Is + i0;
            for (int idx = et; idx < p.T * 16; idx += 128) {
              const int tok = idx >> 4, ch = idx & 15;
              if (i0 + ch * 8 < p.Is)
                *reinterpret_cast<uint4*>(dst + (size_t)tok * p.Is + ch * 8) =
                    *reinterpret_cast<const uint4*>(s_h + tok * 128 + ch * 8);
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
            if (lane == 0) mbar_arrive(tempty_bar(buf));
          }
          if (ph == 0) {
            // this tile's h columns are complete
            fence_proxy_async_global();
            __threadfence();
            named_bar_sync(1, 128);
            if (et == 0) atomicAdd(e_hready + tm, (unsigned)kItems1);
          }
        } else {
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
          if (lane == 0) mbar_arrive(tempty_bar(buf));
          if (ph == 1) {
            // down: the splits of a tile are resident at the same time when the
            // tile's units fall in one wave; each waits for the tile's partials
            // and adds its own slice. Otherwise the last split to arrive adds
            // the whole tile.
            __threadfence();
            named_bar_sync(1, 128);
            unsigned* cnt = e_cnt2 + tm;
            constexpr int items = tile_items<true, KIND_ROW, BN>();
            const bool together = (p.units <= (int)grid) || ((int)grid % p.splits == 0);
            unsigned old = 0;
            if (et == 0) old = atomicAdd(cnt, 1u);
            int lo = 0, hi = 0;
            if (together) {
              bool w2 = true;
              if (et == 0) {
                w2 = bar_wait(cnt, (unsigned)p.splits, timeout, s_abort);
                if (!w2) set_abort();
              }
              if (!agree(w2)) {
                ok = false;
                break;
              }
              lo = (int)((long long)sp * items / p.splits);
              hi = (int)((long long)(sp + 1) * items / p.splits);
            } else if (agree(old == (unsigned)(p.splits - 1))) {
              __threadfence();
              hi = items;
            }
            if (hi > lo) reduce_tile_items<true, KIND_ROW, BN>(p, tm, lo, hi, et, 128);
          }
        }
        if (++buf == 2) {
          buf = 0;
          acc_phase ^= 1u;
        }
      }
      if (ph == 0 && ok && P.g1.splits > 1) {
        // every CTA's gate_up partials are written: wait for all CTAs, then add
        // them up tile by tile, in the order the down splits will read h
        // (round-robin over the down splits, nearest k-block first), counting
        // finished items per tile so that down can start on a tile at once
        __threadfence();
        named_bar_sync(1, 128);
        bool w1 = true;
        if (et == 0) {
          bar_arrive(e_bars + 2);
          w1 = bar_wait(e_bars + 2, grid, timeout, s_abort);
          if (!w1) set_abort();
        }
        if (!agree(w1)) {
          ok = false;
          break;
        }
        const GemmParams& q1 = P.g1;
        const GemmParams& q2 = P.g2;
        const int n1 = q1.m_tiles;
        auto dep_of = [&](int kb) {
          const int sh = kb / q2.kbs, kk = kb - sh * q2.kbs;
          return sh * q1.nb + (kk * 64) / 128;
        };
        auto t0 = [&](int s) { return dep_of((int)((long long)s * q2.nkb / q2.splits)); };
        const int S2 = q2.splits;
        const int R = n1 / S2 + 2;
        constexpr int NCG = kItems1 / 128;
        const long long total = (long long)S2 * R * NCG * 128;
        for (long long it = (long long)blockIdx.x * 128 + et; it < total; it += (long long)grid * 128) {
          const int row = (int)(it & 127);
          const long long rest = it >> 7;
          const int cg = (int)(rest % NCG);
          const int n = (int)(rest / NCG);
          const int r = n / S2, s = n - r * S2;
          const int x = t0(s) + r;
          const bool valid = x < n1 && (s == S2 - 1 || x < t0(s + 1));  // same for the whole warp
          if (!valid) continue;
          reduce_tile_items<true, KIND_GATE_UP, BN>(q1, x, cg * 128 + row, cg * 128 + row + 1, 0, 1);
          fence_proxy_async_global();
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            atomicAdd(e_hready + x, 32u);
          }
        }
      }
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
  constexpr int kSmem = S::kSmemBytes + BN * 128 * 2;  // ring, barriers, h tile
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
  // One CTA per SM (shared memory) and grid == SM count: every CTA is resident
  // while nothing else occupies the GPU. Programmatic serialisation lets the next
  // launch on the stream be scheduled onto SMs this grid frees; it can only be
  // scheduled once every CTA of this grid has started (griddepcontrol.launch_dependents
  // is executed by all of them), so each grid still becomes fully resident. Waits
  // between CTAs are bounded: a grid that could not become resident ends with
  // TP_ERR_TIMEOUT in the status word instead of hanging.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, mx, mh, P);
  return e;
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
