// Fused decode-shaped MLP block: one persistent cooperative launch runs the
// whole step for T <= 128 tokens.
//
//   phase 0  residual add + RMSNorm of the T rows (epilogue warps; rows
//            spread over CTAs)                                -> bars[0]
//   phase 1  column-parallel gate_up: units of 256 weight rows (128 gate +
//            128 up of one shard) x a K range; fp32 partials
//                                                              -> bars[1]
//   phase 1b the partials of every tile are added in split order and
//            silu(g) * u is written to h [t][T][I/t]          -> bars[2]
//   phase 2  row-parallel down: K runs over the t shards in turn, so the
//            shards' partial sums meet in the accumulator; fp32 partials
//                                                              -> bars[3]
//   phase 2b partials added in split order; mlp_out = y, residual_stream =
//            y + residual
//
// The producer never waits for a phase boundary before it has to: it streams
// the next phase's weight blocks into free stages and only defers the
// activation half of those stages until the barrier that makes the
// activation valid has passed. All waits are bounded (status word on
// timeout); the cooperative launch guarantees every CTA is resident.
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

  auto set_abort = [&]() {
    if (!*s_abort) {
      atomicExch(P.g1.status, kStatusTimeout);
      *s_abort = 1;
    }
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
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, last_phase_bits = 0;
      int pend_stage[STAGES], pend_kx[STAGES], pend_sh[STAGES];
      int npend = 0;
      bool ok = true;
      for (int ph = 0; ph < 2 && ok; ++ph) {
        const GemmParams& p = ph == 0 ? P.g1 : P.g2;
        const CUtensorMap* map = ph == 0 ? &map_x : &map_h;
        const unsigned* flag = ph == 0 ? P.bars + 0 : P.bars + 2;
        bool ready = (ph == 0) ? !P.has_norm : false;
        auto flush = [&]() -> bool {
          if (!bar_wait(flag, grid, timeout, s_abort)) return false;
          fence_proxy_async_global();
          for (int i = 0; i < npend; ++i) {
            const uint32_t sb = base + pend_stage[i] * S::kStageBytes + S::kABytes;
            tma_load_4d(sb, map, full_bar(pend_stage[i]), pend_kx[i], 0, 0, pend_sh[i], pol_a);
          }
          npend = 0;
          ready = true;
          return true;
        };
        for (int u = blockIdx.x; u < p.units && ok; u += grid) {
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
            int kx = kb * 64, shard = 0;
            if (ph == 1) {
              shard = kb / p.kbs;
              kx = (kb - shard * p.kbs) * 64;
            }
            if (!ready) {
              const volatile unsigned* vf = flag;
              if (*vf >= grid && !flush()) {
                set_abort();
                ok = false;
                break;
              }
            }
            if (ready) {
              tma_load_4d(sa + S::kABytes, map, fb, kx, 0, 0, shard, pol_a);
            } else {
              pend_stage[npend] = stage;
              pend_kx[npend] = kx;
              pend_sh[npend] = shard;
              if (++npend == STAGES && !flush()) {
                set_abort();
                ok = false;
                break;
              }
            }
            issued_mask |= 1u << stage;
            last_phase_bits = (last_phase_bits & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (ok && npend > 0 && !flush()) {
          set_abort();
          ok = false;
        }
      }
      if (!ok) {
        for (int s = 0; s < STAGES; ++s)
          if (issued_mask & (1u << s))
            mbar_wait_bounded(full_bar(s), (last_phase_bits >> s) & 1u, nullptr, 20000000ull);
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
        for (int u = blockIdx.x; u < p.units && ok; u += grid) {
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
      mbar_wait_bounded(done_bar, 0, nullptr, timeout);
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

    // Barrier among the 128 epilogue threads that shares one thread's verdict.
    auto agree = [&](bool mine_ok) -> bool {
      if (et == 0) *s_ok = mine_ok ? 1 : 0;
      named_bar_sync(1, 128);
      const bool r = *s_ok != 0;
      named_bar_sync(1, 128);
      return r;
    };
    // All 128 epilogue threads: make this CTA's writes visible, arrive, wait for every CTA.
    auto grid_sync = [&](unsigned* c, bool proxy) -> bool {
      if (proxy) fence_proxy_async_global();
      __threadfence();
      named_bar_sync(1, 128);
      bool r = true;
      if (et == 0) {
        bar_arrive(c);
        r = bar_wait(c, grid, timeout, s_abort);
        if (!r) set_abort();
      }
      return agree(r);
    };

    // ---- phase 0: residual add + RMSNorm, one row per CTA in turn
    if (P.has_norm) {
      const int H = P.H, nvec = H >> 3;
      for (int r = blockIdx.x; r < P.g1.T; r += grid) {
        const size_t roff = (size_t)r * H;
        const uint4* av = reinterpret_cast<const uint4*>(P.x_in + roff);
        const uint4* rv = reinterpret_cast<const uint4*>(P.res_in + roff);
        uint4* ro = reinterpret_cast<uint4*>(P.res_out + roff);
        float ss = 0.f;
        for (int v = et; v < nvec; v += 128) {
          const uint4 a4 = __ldg(av + v), r4 = __ldg(rv + v);
          const __nv_bfloat162* ab = reinterpret_cast<const __nv_bfloat162*>(&a4);
          const __nv_bfloat162* rb = reinterpret_cast<const __nv_bfloat162*>(&r4);
          uint4 o;
          __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 fa = __bfloat1622float2(ab[i]), fr = __bfloat1622float2(rb[i]);
            ob[i] = __floats2bfloat162_rn(fa.x + fr.x, fa.y + fr.y);
            const float2 q2 = __bfloat1622float2(ob[i]);  // the stored residual is what is normalised
            ss += q2.x * q2.x + q2.y * q2.y;
          }
          ro[v] = o;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) s_red[q] = ss;
        named_bar_sync(1, 128);
        const float inv = rsqrtf((s_red[0] + s_red[1] + s_red[2] + s_red[3]) / (float)H + P.eps);
        named_bar_sync(1, 128);
        const uint4* gv = reinterpret_cast<const uint4*>(P.gamma);
        uint4* xo = reinterpret_cast<uint4*>(P.x_norm + roff);
        for (int v = et; v < nvec; v += 128) {
          const uint4 r4 = ro[v], g4 = __ldg(gv + v);
          const __nv_bfloat162* rb = reinterpret_cast<const __nv_bfloat162*>(&r4);
          const __nv_bfloat162* gb = reinterpret_cast<const __nv_bfloat162*>(&g4);
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
      // x_norm is read by the tensor copies of phase 1 (async proxy)
      fence_proxy_async_global();
      __threadfence();
      named_bar_sync(1, 128);
      if (et == 0) bar_arrive(P.bars + 0);
    }

    float g[CH], uu[CH];
    // ---- phases 1 and 2: units of the two GEMMs
    for (int ph = 0; ph < 2 && ok; ++ph) {
      const GemmParams& p = ph == 0 ? P.g1 : P.g2;
      for (int u = blockIdx.x; u < p.units && ok; u += grid) {
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
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += CH) {
              if (CH == 32) { tmem_ld32(acc + c0, g); tmem_ld32(acc + BN + c0, uu); }
              else { tmem_ld16(acc + c0, g); tmem_ld16(acc + BN + c0, uu); }
              tc_wait_ld();
              emit_vals<true, KIND_GATE_UP, BN, CH>(p, tm, 0, 0, row, c0, g, uu);
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
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(buf));
        if (++buf == 2) {
          buf = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) break;
      if (ph == 0) {
        if (P.g1.splits > 1) {
          if (!grid_sync(P.bars + 1, false)) { ok = false; break; }
          reduce_partials<true, KIND_GATE_UP, BN>(P.g1, etid, ethreads);
        }
        // h is read by the tensor copies of phase 2 (async proxy)
        fence_proxy_async_global();
        __threadfence();
        named_bar_sync(1, 128);
        if (et == 0) bar_arrive(P.bars + 2);
      } else if (P.g2.splits > 1) {
        if (!grid_sync(P.bars + 3, false)) { ok = false; break; }
        reduce_partials<true, KIND_ROW, BN>(P.g2, etid, ethreads);
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::kTmemCols);
  }
  // every wait of this CTA is behind it: the last CTA out resets the counters
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atomicAdd(P.bars + 4, 1u);
    if (old == grid - 1) {
      for (int i = 0; i < 5; ++i) atomicExch(P.bars + i, 0u);
    }
  }
}

template <int BN>
cudaError_t launch_mlp_decode_bn(const CUtensorMap& mx, const CUtensorMap& mh, const MlpDecodeParams& P,
                                 int grid, cudaStream_t st) {
  using S = GemmShape<true, KIND_GATE_UP, BN>;
  auto kernel = mlp_decode_kernel<BN>;
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
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
  return cudaLaunchKernelEx(&cfg, kernel, mx, mh, P);
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
