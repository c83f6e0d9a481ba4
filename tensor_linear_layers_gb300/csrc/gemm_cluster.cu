// Prefill-shaped GEMMs on CTA pairs: tcgen05 cta_group::2 (two-SM) MMAs.
//
// The two CTAs of a cluster of 2 compute one 256-token x 256-weight-row tile
// together: CTA rank r holds token tile 2 pm + r (128 rows of A) and weight
// rows [128 r, 128 r + 128) of the 256-row weight block (half of B). One
// thread of the even CTA issues M = 256, N = 256 MMAs that read A and B from
// both CTAs' shared memory; each CTA's tensor memory receives its own 128
// tokens x all 256 weight rows. Every byte of a stage is therefore loaded
// once per pair, by the CTA that holds it, with plain TMA tensor copies (no
// multicast); the copies of both CTAs count on the even CTA's full barrier.
// The MMA commits arrive on both CTAs' empty and accumulator barriers; both
// CTAs' epilogue warps arrive on the even CTA's accumulator-empty barrier.
//
// Same epilogues as the one-CTA engine (gate_up with SiLU*mul, column-parallel
// store, row-parallel store + residual); no split-K. An optional second,
// independent problem shares the launch (the units of both form one list).
#include "gemm_launch.cuh"
#include <algorithm>

namespace tpl {

struct PairShape {
  static constexpr int kABytes = 128 * 128;   // 128 tokens x 64 bf16 of this CTA
  static constexpr int kBBytes = 128 * 128;   // this CTA's 128 of the block's 256 weight rows x 64 bf16
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = 7;
  static constexpr int kAccCols = 256;        // 128 lanes x 256 fp32 columns per accumulator
  static constexpr int kTmemCols = 512;       // two accumulators
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 256;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(256, 256);
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

template <int KIND, int KIND2>
__global__ void __launch_bounds__(192, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_act, const __grid_constant__ CUtensorMap map_w,
                        const __grid_constant__ CUtensorMap map_act2, const __grid_constant__ CUtensorMap map_w2,
                        const GemmParams p, const GemmParams p2, const PairTail tail) {
  using P = PairShape;
  constexpr int STAGES = P::kStages;
  constexpr int BN = 256;
  constexpr bool kTwo = KIND2 >= 0;
  constexpr uint16_t kBoth = 0x3;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t bar0 = base + STAGES * P::kStageBytes;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * STAGES + 4);
  uint8_t* misc = base_ptr + STAGES * P::kStageBytes + 8 * (2 * STAGES + 5);
  volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(misc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + 4);
  volatile int* s_ok = reinterpret_cast<volatile int*>(misc + 12);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = (int)(cluster_ctarank() & 1u);   // 0: the CTA that issues the MMAs
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);    // the even CTA's expect-tx arrival; both CTAs' bytes
      mbar_init(empty_bar(s), 1);   // the pair MMA's commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 8);  // four epilogue warps of each CTA
    }
    mbar_init(done_bar, 1);
    *s_abort = 0;
    fence_barrier_init();
    prefetch_tensormap(&map_act);
    prefetch_tensormap(&map_w);
    if (kTwo) {
      prefetch_tensormap(&map_act2);
      prefetch_tensormap(&map_w2);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(s_tmem)), P::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  // the peer's copies count on this CTA's barriers and the MMA commits arrive on
  // the peer's: both CTAs' barriers are initialised before either proceeds
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  const int pu1 = ((p.m_tiles + 1) >> 1) * p.n_tiles;
  const int pu_all_units = pu1 + (kTwo ? ((p2.m_tiles + 1) >> 1) * p2.n_tiles : 0);
  // the list the clusters walk: `full` whole units, then rem x s parts of the last units
  const bool split_tail = tail.s >= 2;
  const int pu_all = split_tail ? tail.full + tail.rem * tail.s : pu_all_units;
  // virtual unit -> (pair unit, part, split slot); part -1: whole
  auto vunit = [&](int v, int& pu, int& part, int& slot) {
    if (!split_tail || v < tail.full) {
      pu = v;
      part = -1;
      slot = -1;
      return;
    }
    const int w = v - tail.full;
    slot = w / tail.s;
    part = w - slot * tail.s;
    pu = tail.full + slot;
  };
  auto krange = [&](const GemmParams& q, int part, int& kb0, int& kb1) {
    if (part < 0) {
      kb0 = 0;
      kb1 = q.nkb;
    } else {
      kb0 = (int)((long long)part * q.nkb / tail.s);
      kb1 = (int)((long long)(part + 1) * q.nkb / tail.s);
    }
  };
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
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_normal();
      const uint64_t pol_a = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, last_phase_bits = 0;
      bool ok = true;
      for (int v = cluster; v < pu_all && ok; v += nclusters) {
        int pu, part, slot;
        vunit(v, pu, part, slot);
        int tm, tn, pm;
        bool second;
        if (!decode(pu, second, tm, tn, pm)) continue;
        const GemmParams& q = second ? p2 : p;
        int kb_lo, kb_hi;
        krange(q, part, kb_lo, kb_hi);
        const CUtensorMap* map = second ? &map_act2 : &map_act;
        const CUtensorMap* wmap = second ? &map_w2 : &map_w;
        const bool row_kind = second ? (KIND2 == KIND_ROW) : (KIND == KIND_ROW);
        int blk0 = tn * q.nkb;
        if (q.pair_tiles != nullptr)   // both tiles of a pair belong to the expert of its first
          blk0 += q.tile_expert[q.pair_tiles[2 * pm]] * (int)(q.expert_wbytes / kWBlockBytes);
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, s_abort, q.timeout_ns)) {
            fail(q);
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * P::kStageBytes;
          const uint32_t sb = sa + P::kABytes;
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          // the even CTA expects both CTAs' bytes: its own and the peer's token tile and weight half
          if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * P::kStageBytes);
          int kx = kb * 64, shard = 0;
          if (row_kind) {
            shard = kb / q.kbs;
            kx = (kb - shard * q.kbs) * 64;
          }
          tma_load_4d_pair(sa, map, fb, kx, tm * 128, 0, shard, pol_a);
          tma_load_3d_pair(sb, wmap, fb, 0, rank * 128, blk0 + kb, pol_w);
          issued_mask |= 1u << stage;
          last_phase_bits = (last_phase_bits & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let copies in flight land before the CTA exits: the even CTA sees them on its
        // full barriers; the peer's count there too, so it waits out a fixed bound instead
        if (leader) {
          for (int s = 0; s < STAGES; ++s)
            if (issued_mask & (1u << s))
              mbar_wait_bounded(full_bar(s), (last_phase_bits >> s) & 1u, nullptr, kTeardownNs);
        } else {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    // The whole warp runs the loop and one elected lane issues each k-block's MMAs
    // with their commit, so descriptors and tensor-memory addresses stay warp-uniform.
    if (leader) {
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int v = cluster; v < pu_all && ok; v += nclusters) {
        int pu, part, slot;
        vunit(v, pu, part, slot);
        int tm, tn, pm;
        bool second;
        if (!decode(pu, second, tm, tn, pm)) continue;
        const GemmParams& q = second ? p2 : p;
        int kb_lo, kb_hi;
        krange(q, part, kb_lo, kb_hi);
        if (!__all_sync(0xffffffffu, mbar_wait_bounded_cluster(tempty_bar(buf), acc_phase ^ 1u, s_abort, q.timeout_ns))) {
          if (lane == 0) fail(q);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * P::kAccCols;
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(full_bar(stage), phase, s_abort, q.timeout_ns))) {
            if (lane == 0) fail(q);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + stage * P::kStageBytes;
          const uint64_t adesc = smem_desc_k128(sa);
          const uint64_t bdesc = smem_desc_k128(sa + P::kABytes);
          if (elect_one()) {
            if (kb == kb_lo)
              tc_mma_bf16_pair<false>(d_tmem, adesc, bdesc, P::kIdesc);
            else
              tc_mma_bf16_pair<true>(d_tmem, adesc, bdesc, P::kIdesc);
#pragma unroll
            for (int ks = 1; ks < 4; ++ks)
              tc_mma_bf16_pair<true>(d_tmem, adesc + (uint64_t)(ks * 2), bdesc + (uint64_t)(ks * 2), P::kIdesc);
            tc_commit_pair_multicast(empty_bar(stage), kBoth);
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // elect.sync picks the same lane for the same mask, so this commit follows the
        // MMAs above
        if (elect_one()) tc_commit_pair_multicast(tfull_bar(buf), kBoth);
        __syncwarp();
        if (++buf == 2) {
          buf = 0;
          acc_phase ^= 1u;
        }
      }
      // every issued MMA completes before either CTA frees tensor memory or exits
      if (elect_one()) tc_commit_pair(done_bar);
      __syncwarp();
      mbar_wait_bounded(done_bar, 0, nullptr, kTeardownNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int qd = warp & 3;
    const int row = qd * 32 + lane;
    const int et = threadIdx.x - 64;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(qd * 32) << 16);
    int buf = 0;
    uint32_t acc_phase = 0;
    constexpr int CH = 32;
    float g[CH], uu[CH];
    for (int v = cluster; v < pu_all; v += nclusters) {
      int pu, part, slot;
      vunit(v, pu, part, slot);
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
      const uint32_t acc = lane_addr + buf * P::kAccCols;
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
      if (part < 0) {
        if (second)
          direct(std::integral_constant<int, (kTwo ? KIND2 : KIND)>{}, p2);
        else
          direct(std::integral_constant<int, KIND>{}, p);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(buf), 0));
      } else {
        // a part of a split unit: its fp32 accumulator goes to the workspace (columns
        // fastest across threads: row `row` of column c at c * 128 + row)
        float* mine = tail.part + ((size_t)(slot * tail.s + part) * 2 + rank) * (256 * 128);
#pragma unroll 1
        for (int c0 = 0; c0 < 256; c0 += CH) {
          tmem_ld32(acc + c0, g);
          tc_wait_ld();
#pragma unroll
          for (int j = 0; j < CH; ++j) __stcg(mine + (size_t)(c0 + j) * 128 + row, g[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(buf), 0));
        // the last part to arrive adds the parts in order and applies the epilogue
        named_bar_sync(1, 128);
        if (et == 0) *s_ok = atom_acq_rel_add(tail.cnt + slot * 2 + rank, 1u) == (unsigned)(tail.s - 1) ? 1 : 0;
        named_bar_sync(1, 128);
        const bool last = *s_ok != 0;
        named_bar_sync(1, 128);
        if (last) {
          if (et == 0) atomicExch(tail.cnt + slot * 2 + rank, 0u);   // ready for the next launch
          const float* base_p = tail.part + (size_t)slot * tail.s * 2 * (256 * 128) + (size_t)rank * (256 * 128);
          auto summed = [&](auto kind_c, const GemmParams& q) {
            constexpr int K = decltype(kind_c)::value;
            using SK = GemmShape<false, K, BN>;
#pragma unroll 1
            for (int c0 = 0; c0 < SK::kNG; c0 += CH) {
#pragma unroll
              for (int j = 0; j < CH; ++j) {
                g[j] = 0.f;
                if (K == KIND_GATE_UP) uu[j] = 0.f;
              }
              for (int pp = 0; pp < tail.s; ++pp) {
                const float* src = base_p + (size_t)pp * 2 * (256 * 128);
#pragma unroll
                for (int j = 0; j < CH; ++j) {
                  g[j] += __ldcg(src + (size_t)(c0 + j) * 128 + row);
                  if (K == KIND_GATE_UP) uu[j] += __ldcg(src + (size_t)(SK::kUOff + c0 + j) * 128 + row);
                }
              }
              emit_vals<false, K, BN, CH>(q, tm, tn, 0, row, c0, g, uu);
            }
          };
          if (second)
            summed(std::integral_constant<int, (kTwo ? KIND2 : KIND)>{}, p2);
          else
            summed(std::integral_constant<int, KIND>{}, p);
        }
      }
      if (++buf == 2) {
        buf = 0;
        acc_phase ^= 1u;
      }
    }
  }

  __syncthreads();
  // the even CTA's MMAs are complete and both epilogues have read their accumulators
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, P::kTmemCols);
  }
  // neither CTA leaves while the other may still touch its shared or tensor memory
  cluster_sync();
}

// How a launch of pu pair units on `clusters` clusters splits its tail (see PairTail):
// when the last wave would be at most half full, its units are split into
// s = min(4, clusters / rem, max_s) parts, max_s the fewest k-blocks of a problem (every
// part keeps at least one). Grouped (expert) problems are not split.
PairTail plan_pair_tail(int pu, int clusters, bool grouped, float* part, unsigned* cnt, int max_s) {
  PairTail t{};
  t.full = pu;
  t.s = 1;
  if (grouped || part == nullptr || cnt == nullptr || clusters < 2 || pu < 1) return t;
  const int waves = (pu + clusters - 1) / clusters;
  const int rem = pu - (waves - 1) * clusters;
  const int s = std::min(std::min(4, clusters / rem), max_s);
  if (s < 2) return t;
  t.full = pu - rem;
  t.rem = rem;
  t.s = s;
  t.part = part;
  t.cnt = cnt;
  return t;
}

// Waves (in whole-unit times) a launch of pu pair units takes on `clusters` clusters,
// counting a split tail's parts as 1 / s of a unit.
double pair_waves(int pu, int clusters) {
  if (clusters < 1 || pu < 1) return 0.0;
  const PairTail t = plan_pair_tail(pu, clusters, false, reinterpret_cast<float*>(1), reinterpret_cast<unsigned*>(1), 4);
  if (t.s < 2) return (double)((pu + clusters - 1) / clusters);
  return (double)(t.full / clusters) + 1.0 / t.s;
}

template <int KIND, int KIND2>
cudaError_t launch_pair(const CUtensorMap& a1, const CUtensorMap& w1, const GemmParams& p1, const CUtensorMap& a2,
                        const CUtensorMap& w2, const GemmParams& p2, int max_clusters, float* tail_part,
                        unsigned* tail_cnt, cudaStream_t st) {
  using P = PairShape;
  auto kernel = tc_gemm_pair_kernel<KIND, KIND2>;
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  const int pu = ((p1.m_tiles + 1) / 2) * p1.n_tiles + (KIND2 >= 0 ? ((p2.m_tiles + 1) / 2) * p2.n_tiles : 0);
  const int min_nkb = KIND2 >= 0 ? std::min(p1.nkb, p2.nkb) : p1.nkb;
  const PairTail tail = plan_pair_tail(pu, max_clusters, p1.pair_tiles != nullptr, tail_part, tail_cnt, min_nkb);
  const int vunits = tail.s >= 2 ? tail.full + tail.rem * tail.s : pu;
  const int clusters = vunits < max_clusters ? vunits : max_clusters;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = P::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a1, w1, a2, w2, p1, p2, tail);
}

int pair_stages() { return PairShape::kStages; }

// Number of 2-CTA clusters of this engine that fit on the device at once (0 if none).
int pair_max_clusters() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static std::atomic<int> cached[64];
  int v = cached[dev & 63].load();
  if (v != 0) return v > 0 ? v : 0;
  using P = PairShape;
  auto kernel = tc_gemm_pair_kernel<KIND_GATE_UP, -1>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P::kSmemBytes) != cudaSuccess) {
    cached[dev & 63].store(-1);
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = P::kSmemBytes;
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

cudaError_t launch_gemm_pair(int kind, int kind2, const CUtensorMap& a1, const CUtensorMap& w1, const GemmParams& p1,
                             const CUtensorMap& a2, const CUtensorMap& w2, const GemmParams& p2, int max_clusters,
                             float* tail_part, unsigned* tail_cnt, cudaStream_t st) {
  float* tp = tail_part;
  unsigned* tc = tail_cnt;
  if (kind2 < 0) {
    switch (kind) {
      case KIND_GATE_UP: return launch_pair<KIND_GATE_UP, -1>(a1, w1, p1, a1, w1, p1, max_clusters, tp, tc, st);
      case KIND_COL: return launch_pair<KIND_COL, -1>(a1, w1, p1, a1, w1, p1, max_clusters, tp, tc, st);
      case KIND_ROW: return launch_pair<KIND_ROW, -1>(a1, w1, p1, a1, w1, p1, max_clusters, tp, tc, st);
      default: return cudaErrorInvalidValue;
    }
  }
  if (kind == KIND_COL && kind2 == KIND_ROW)
    return launch_pair<KIND_COL, KIND_ROW>(a1, w1, p1, a2, w2, p2, max_clusters, tp, tc, st);
  return cudaErrorInvalidValue;
}

// Workspace of a pair launch's split tail on a device with `nsm` SMs: at most nsm / 2
// parts (one per cluster) of 2 x 128 KB, then the counters.
int64_t pair_tail_bytes(int nsm) {
  const int64_t parts = std::max(1, nsm / 2);
  return parts * 2 * 256 * 128 * 4 + ((parts * 2 * 4 + 255) & ~int64_t(255));
}

}  // namespace tpl
