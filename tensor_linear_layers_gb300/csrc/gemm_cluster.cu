// Prefill-shaped GEMMs on CTA pairs (thread-block clusters of 2).
//
// The two CTAs of a cluster compute adjacent 128-token tiles against the same
// 256-row weight block. Each CTA loads its own token tile (TMA tensor copy)
// and half of the 32 KB weight block, multicast into both CTAs' shared memory,
// so every weight byte leaves L2 once per pair instead of once per CTA. The
// MMAs stay per CTA (tcgen05 cta_group::1, 128 x 256 accumulators in each
// CTA's tensor memory); a stage may be refilled only when both CTAs' MMAs have
// read it, so each MMA commit arrives on the empty barrier of both CTAs.
//
// Same epilogues as the one-CTA engine (gate_up with SiLU*mul, column-parallel
// store, row-parallel store + residual); no split-K. An optional second,
// independent problem shares the launch (the units of both form one list).
#include "gemm_launch.cuh"

namespace tpl {

template <int KIND, int KIND2>
__global__ void __launch_bounds__(192, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_act, const __grid_constant__ CUtensorMap map_act2,
                        const GemmParams p, const GemmParams p2) {
  using S = GemmShape<false, KIND, 256>;
  constexpr int STAGES = S::kStages;
  constexpr int BN = 256;
  constexpr bool kTwo = KIND2 >= 0;
  constexpr uint16_t kBoth = 0x3;
  constexpr uint32_t kHalfB = kWBlockBytes / 2;

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
  const int rank = (int)cluster_ctarank();          // 0 or 1 within the pair
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 2);   // both CTAs' MMAs release a stage
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
  // the peer multicasts into this CTA's stages and barriers: both must be initialised
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  const int pu1 = ((p.m_tiles + 1) >> 1) * p.n_tiles;
  const int pu_all = pu1 + (kTwo ? ((p2.m_tiles + 1) >> 1) * p2.n_tiles : 0);
  // pair unit -> (problem, token tile of this CTA, weight tile); grouped along M
  // pm: the pair of token tiles; grouped problems look the tiles up (false: pair skipped)
  auto decode = [&](int pu, bool& second, int& tm, int& tn, int& pm) -> bool {
    second = kTwo && pu >= pu1;
    const GemmParams& q = second ? p2 : p;
    const int u = second ? pu - pu1 : pu;
    const int m_pairs = (q.m_tiles + 1) >> 1;
    const int gm_pairs = q.group_m > 1 ? (q.group_m + 1) >> 1 : 1;
    const int group_size = gm_pairs * q.n_tiles;
    const int g = u / group_size;
    const int first = g * gm_pairs;
    const int rem = m_pairs - first;
    const int gm = rem < gm_pairs ? rem : gm_pairs;
    const int in_g = u - g * group_size;
    pm = first + in_g % gm;
    tn = in_g / gm;
    if (q.pair_tiles != nullptr) {
      if (pm >= *q.pair_count) return false;
      tm = q.pair_tiles[2 * pm + rank];
      if (tm < 0) tm = q.m_tiles;   // no second tile: rows past the buffer read as zero, none stored
      return true;
    }
    tm = 2 * pm + rank;     // may be a tile past T: its rows read as zero and are not stored
    return true;
  };
  auto fail = [&](const GemmParams& q) {
    if (!*s_abort) {
      atomicExch(q.status, kStatusTimeout);
      *s_abort = 1;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_normal();
      const uint64_t pol_a = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, last_phase_bits = 0;
      bool ok = true;
      for (int pu = cluster; pu < pu_all && ok; pu += nclusters) {
        int tm, tn, pm;
        bool second;
        if (!decode(pu, second, tm, tn, pm)) continue;
        const GemmParams& q = second ? p2 : p;
        const CUtensorMap* map = second ? &map_act2 : &map_act;
        const bool row_kind = second ? (KIND2 == KIND_ROW) : (KIND == KIND_ROW);
        const uint8_t* wsrc = q.w_packed + (size_t)tn * q.nkb * kWBlockBytes + rank * kHalfB;
        if (q.pair_tiles != nullptr)   // both tiles of a pair belong to the expert of its first
          wsrc += (size_t)q.tile_expert[q.pair_tiles[2 * pm]] * (size_t)q.expert_wbytes;
        for (int kb = 0; kb < q.nkb; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, s_abort, q.timeout_ns)) {
            fail(q);
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * S::kStageBytes;
          const uint32_t sb = sa + S::kABytes;
          const uint32_t fb = full_bar(stage);
          // own token tile (16 KB) + both halves of the weight block (2 x 16 KB, one from each CTA)
          mbar_arrive_expect_tx(fb, S::kStageBytes);
          int kx = kb * 64, shard = 0;
          if (row_kind) {
            shard = kb / q.kbs;
            kx = (kb - shard * q.kbs) * 64;
          }
          tma_load_4d(sa, map, fb, kx, tm * 128, 0, shard, pol_a);
          bulk_load_multicast(sb + rank * kHalfB, wsrc + (size_t)kb * kWBlockBytes, kHalfB, fb, kBoth, pol_w);
          issued_mask |= 1u << stage;
          last_phase_bits = (last_phase_bits & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
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
      for (int pu = cluster; pu < pu_all && ok; pu += nclusters) {
        int tm, tn, pm;
        bool second;
        if (!decode(pu, second, tm, tn, pm)) continue;
        const GemmParams& q = second ? p2 : p;
        if (!mbar_wait_bounded(tempty_bar(buf), acc_phase ^ 1u, s_abort, q.timeout_ns)) {
          fail(q);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * S::kAccCols;
        for (int kb = 0; kb < q.nkb; ++kb) {
          if (!mbar_wait_bounded(full_bar(stage), phase, s_abort, q.timeout_ns)) {
            fail(q);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + stage * S::kStageBytes;
          const uint64_t adesc = smem_desc_k128(sa);
          const uint64_t bdesc = smem_desc_k128(sa + S::kABytes);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc_mma_bf16(d_tmem, adesc + (uint64_t)(ks * 2), bdesc + (uint64_t)(ks * 2), S::kIdesc,
                        (kb > 0 || ks > 0) ? 1u : 0u);
          tc_commit_multicast(empty_bar(stage), kBoth);
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
      tc_commit(done_bar);
      mbar_wait_bounded(done_bar, 0, nullptr, kTeardownNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int qd = warp & 3;
    const int row = qd * 32 + lane;
    const int et = threadIdx.x - 64;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(qd * 32) << 16);
    int buf = 0;
    uint32_t acc_phase = 0;
    constexpr int CH = 32;
    float g[CH], uu[CH];
    for (int pu = cluster; pu < pu_all; pu += nclusters) {
      int tm, tn, pm;
      bool second;
      if (!decode(pu, second, tm, tn, pm)) continue;
      if (et == 0) {
        const bool ok = mbar_wait_bounded(tfull_bar(buf), acc_phase, s_abort, p.timeout_ns);
        if (!ok) fail(p);
        *s_ok = ok ? 1 : 0;
      }
      named_bar_sync(1, 128);
      const int ok = *s_ok;
      named_bar_sync(1, 128);
      if (!ok) break;
      tc_fence_after();
      const uint32_t acc = lane_addr + buf * S::kAccCols;
      auto direct = [&](auto kind_c, const GemmParams& q) {
        constexpr int K = decltype(kind_c)::value;
        using SK = GemmShape<false, K, BN>;
#pragma unroll 1
        for (int c0 = 0; c0 < SK::kNG; c0 += CH) {
          tmem_ld32(acc + c0, g);
          if (K == KIND_GATE_UP) tmem_ld32(acc + SK::kUOff + c0, uu);
          tc_wait_ld();
          emit_vals<false, K, BN, CH>(q, tm, tn, 0, row, c0, g, uu);
        }
      };
      if (second)
        direct(std::integral_constant<int, (kTwo ? KIND2 : KIND)>{}, p2);
      else
        direct(std::integral_constant<int, KIND>{}, p);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(buf));
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
  // the peer's multicast copies and MMA commits target this CTA's shared memory:
  // neither CTA leaves before both are done
  cluster_sync();
}

template <int KIND, int KIND2>
cudaError_t launch_pair(const CUtensorMap& a1, const GemmParams& p1, const CUtensorMap& a2, const GemmParams& p2,
                        int max_clusters, cudaStream_t st) {
  using S = GemmShape<false, KIND, 256>;
  auto kernel = tc_gemm_pair_kernel<KIND, KIND2>;
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
  const int pu = ((p1.m_tiles + 1) / 2) * p1.n_tiles + (KIND2 >= 0 ? ((p2.m_tiles + 1) / 2) * p2.n_tiles : 0);
  const int clusters = pu < max_clusters ? pu : max_clusters;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = S::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a1, a2, p1, p2);
}

// Number of 2-CTA clusters of this engine that fit on the device at once (0 if none).
int pair_max_clusters() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static std::atomic<int> cached[64];
  int v = cached[dev & 63].load();
  if (v != 0) return v > 0 ? v : 0;
  using S = GemmShape<false, KIND_GATE_UP, 256>;
  auto kernel = tc_gemm_pair_kernel<KIND_GATE_UP, -1>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes) != cudaSuccess) {
    cached[dev & 63].store(-1);
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = S::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    cached[dev & 63].store(-1);
    return 0;
  }
  cached[dev & 63].store(n);
  return n;
}

cudaError_t launch_gemm_pair(int kind, int kind2, const CUtensorMap& a1, const GemmParams& p1,
                             const CUtensorMap& a2, const GemmParams& p2, int max_clusters, cudaStream_t st) {
  if (kind2 < 0) {
    switch (kind) {
      case KIND_GATE_UP: return launch_pair<KIND_GATE_UP, -1>(a1, p1, a1, p1, max_clusters, st);
      case KIND_COL: return launch_pair<KIND_COL, -1>(a1, p1, a1, p1, max_clusters, st);
      case KIND_ROW: return launch_pair<KIND_ROW, -1>(a1, p1, a1, p1, max_clusters, st);
      default: return cudaErrorInvalidValue;
    }
  }
  if (kind == KIND_COL && kind2 == KIND_ROW) return launch_pair<KIND_COL, KIND_ROW>(a1, p1, a2, p2, max_clusters, st);
  return cudaErrorInvalidValue;
}

}  // namespace tpl
