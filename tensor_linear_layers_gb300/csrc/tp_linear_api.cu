// Host side of libtplinear.so: argument validation, shard packing, tensor
// maps, launch plans and the C ABI declared in include/tp_linear.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <atomic>
#include <cstdlib>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "gemm_tc.cuh"
#include "internal.h"
#include "tp_linear.h"

namespace tpl {
cudaError_t launch_gemm_prefill(int kind, const CUtensorMap& a, const GemmParams& p, int grid,
                                cudaStream_t st);
cudaError_t launch_gemm_decode_gate_up(int bn, const CUtensorMap& a, const GemmParams& p, int grid,
                                       cudaStream_t st);
cudaError_t launch_gemm_decode_col(int bn, const CUtensorMap& a, const GemmParams& p, int grid,
                                   cudaStream_t st);
cudaError_t launch_gemm_decode_row(int bn, const CUtensorMap& a, const GemmParams& p, int grid,
                                   cudaStream_t st);
int gemm_stages_prefill(int kind);
cudaError_t launch_gemm_prefill_col_row(const CUtensorMap& a1, const GemmParams& p1, const CUtensorMap& a2,
                                        const GemmParams& p2, int grid, cudaStream_t st);
cudaError_t launch_gemm_pair(int kind, int kind2, const CUtensorMap& a1, const CUtensorMap& w1, const GemmParams& p1,
                             const CUtensorMap& a2, const CUtensorMap& w2, const GemmParams& p2, int max_clusters,
                             float* tail_part, unsigned* tail_cnt, cudaStream_t st);
int64_t pair_tail_bytes(int nsm);
double pair_waves(int pu, int clusters);
int pair_max_clusters();
int pair_stages();
int gemm_stages_decode_gate_up(int bn);
int gemm_stages_decode_col(int bn);
int gemm_stages_decode_row(int bn);

cudaError_t launch_gemm(bool swap, int kind, int bn, const CUtensorMap& a, const GemmParams& p,
                        int grid, cudaStream_t st) {
  if (!swap) return launch_gemm_prefill(kind, a, p, grid, st);
  switch (kind) {
    case KIND_GATE_UP: return launch_gemm_decode_gate_up(bn, a, p, grid, st);
    case KIND_COL: return launch_gemm_decode_col(bn, a, p, grid, st);
    case KIND_ROW: return launch_gemm_decode_row(bn, a, p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}
int gemm_stages(bool swap, int kind, int bn) {
  if (!swap) return gemm_stages_prefill(kind);
  switch (kind) {
    case KIND_GATE_UP: return gemm_stages_decode_gate_up(bn);
    case KIND_COL: return gemm_stages_decode_col(bn);
    case KIND_ROW: return gemm_stages_decode_row(bn);
    default: return 0;
  }
}
}  // namespace tpl

using namespace tpl;

// ============================================================================ errors
namespace {
thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}
int ok() {
  g_err[0] = '\0';
  return TP_OK;
}
int cuda_fail(cudaError_t e, const char* what) {
  return fail(TP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
constexpr int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

// ============================================================================ driver entry
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 4-D bf16 tensor map: dims (d0 innermost .. d3), dense strides, box (64, box_rows, 1, 1),
// 128-byte swizzle, out-of-bounds elements read as zero.
int make_map(CUtensorMap* m, const void* ptr, int64_t d0, int64_t d1, int64_t d2, int64_t d3,
             int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[4] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2, (cuuint64_t)d3};
  const cuuint64_t strides[3] = {(cuuint64_t)(d0 * 2), (cuuint64_t)(d0 * d1 * 2),
                                 (cuuint64_t)(d0 * d1 * d2 * 2)};
  const cuuint32_t box[4] = {64u, (cuuint32_t)box_rows, 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for dims %lld x %lld x %lld x %lld",
                (int)r, (long long)d0, (long long)d1, (long long)d2, (long long)d3);
  return TP_OK;
}

// Tensor map of a t-shard activation with per-shard width w and T rows:
// shard-major [t][T][w] (each shard's rows contiguous, as a rank holds them) or
// gathered [T][t * w] (the shards' columns side by side in every row). The shard
// index is dimension 2 (shard_dim == 2) or 3 (shard_dim == 3) of the map.
int make_shard_map(CUtensorMap* m, const void* ptr, int64_t w, int64_t T, int64_t t, int shard_dim,
                   bool gathered, int box_rows) {
  if (!gathered) return shard_dim == 2 ? make_map(m, ptr, w, T, t, 1, box_rows) : make_map(m, ptr, w, T, 1, t, box_rows);
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t row = (cuuint64_t)(t * w * 2), shard = (cuuint64_t)(w * 2);
  cuuint64_t dims[4], strides[3];
  dims[0] = (cuuint64_t)w;
  dims[1] = (cuuint64_t)T;
  strides[0] = row;
  if (shard_dim == 2) {
    dims[2] = (cuuint64_t)t;
    dims[3] = 1;
    strides[1] = shard;
    strides[2] = row * (cuuint64_t)T;
  } else {
    dims[2] = 1;
    dims[3] = (cuuint64_t)t;
    strides[1] = row * (cuuint64_t)T;
    strides[2] = shard;
  }
  const cuuint32_t box[4] = {64u, (cuuint32_t)box_rows, 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a gathered %lld x %lld x %lld map",
                (int)r, (long long)w, (long long)T, (long long)t);
  return TP_OK;
}

// Tensor map of packed weight blocks for the CTA-pair engine: dims (64 elements,
// 256 rows, n_blocks), each block 32 KB, boxes of 64 x 128 rows (one half of a
// block, 16 KB). The blocks are already in the swizzled image the MMA reads, so
// the copy itself does not swizzle.
int make_wmap(CUtensorMap* m, const void* ptr, int64_t n_blocks) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[3] = {64u, 256u, (cuuint64_t)n_blocks};
  const cuuint64_t strides[2] = {128u, (cuuint64_t)kWBlockBytes};
  const cuuint32_t box[3] = {64u, 128u, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for %lld packed weight blocks", (int)r,
                (long long)n_blocks);
  return TP_OK;
}

// ============================================================================ workspace layout
// header: [0] status word; [64] grid barrier of the column-parallel GEMM;
// [128] grid barrier of the row-parallel GEMM; [192] counters of the fused
// decode block (two sets of four words), [224] its launch count (64 bits),
// [232] its ticket counter (CTAs started, 64 bits). Then the fused block's two
// sets of per-tile counters and flags (fixed size per handle), then the
// buffers whose size depends on T.
constexpr int64_t kGbarColOff = 64;
constexpr int64_t kGbarRowOff = 128;
constexpr int64_t kDecodeBarsOff = 192;
constexpr int64_t kTileCountersOff = 256;
constexpr int64_t kFusedMaxT = 128;
constexpr int64_t kCaptureOff = 256;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per on-chip wait
std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};

// A decoder-layer call runs the MLP half in its own part of the layer's
// workspace; while it enqueues, every kernel it launches writes device errors
// to the layer's status word instead of that part's own first word.
thread_local int* t_status = nullptr;
struct StatusRedirect {
  explicit StatusRedirect(int* s) { t_status = s; }
  ~StatusRedirect() { t_status = nullptr; }
};

}  // namespace

// ============================================================================ handle
struct tp_linear {
  tp_config_t cfg;
  int device;
  int nsm;
  int64_t H;
  // MLP
  int64_t I, Is;
  // ATTN
  int q_per, kv_per, rep;
  int64_t ws_qkv;  // packed rows per QKV shard
  int64_t Ks;      // row-parallel input features per shard (Is or nq*hd/t)
  int64_t n_col;   // column-parallel output rows in total
  // packed weight blocks (256 rows x 64 K each)
  int nb;          // MLP: 128-row gate blocks per shard
  int wt_col, nkb_col, wt_row, nkb_row, kbs_row;
  void* w_col;
  void* w_row;
  const void* gamma;
  // the packed blocks of w_col / w_row (all experts) as tensor maps, for the CTA-pair engine
  CUtensorMap wmap_col, wmap_row;
  uint64_t uid;    // unique per handle created in this process (never reused)
};

namespace {

// start of the T-dependent part of a forward workspace: after the header and
// the fused block's two sets of per-tile counters (cnt1 and hready per gate_up
// tile, cnt2 per down tile)
int64_t tile_counter_words(const tp_linear* h) { return 2 * (int64_t)h->wt_col + (int64_t)h->wt_row; }
int64_t dyn_off(const tp_linear* h) { return align256(kTileCountersOff + 4 * 2 * tile_counter_words(h)); }

struct Plan {
  bool swap;
  int kind;
  int bn;
  int m_tiles, n_tiles, splits, units, nkb, kbs, nb, grid, acc_cols;
  int64_t partial_bytes;
};

// Pick the operand orientation, tile width and K split of one GEMM.
// force_splits > 0 overrides the split count.
Plan make_plan(const tp_linear* h, int which, int64_t T, int force_splits = 0) {
  Plan pl{};
  const bool mlp = h->cfg.kind != TP_BLOCK_ATTN_PROJ;
  pl.kind = which == 0 ? (mlp ? KIND_GATE_UP : KIND_COL) : KIND_ROW;
  pl.swap = T <= 128;
  pl.bn = pl.swap ? (T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : 128) : 256;
  const int t = h->cfg.t;
  (void)t;
  int64_t w_tiles;
  if (which == 0) {
    pl.nkb = h->nkb_col;
    pl.kbs = 0;
    pl.nb = h->nb;
    w_tiles = h->wt_col;   // MLP: 128 gate + 128 up rows per tile
  } else {
    pl.kbs = h->kbs_row;
    pl.nkb = h->nkb_row;
    w_tiles = h->wt_row;
  }
  if (pl.swap) {
    pl.m_tiles = (int)w_tiles;
    pl.n_tiles = (int)ceil_div(T, pl.bn);
  } else {
    pl.m_tiles = (int)ceil_div(T, 128);
    pl.n_tiles = (int)w_tiles;
  }
  pl.acc_cols = pl.swap ? 2 * pl.bn : pl.bn;
  const int64_t tiles = (int64_t)pl.m_tiles * pl.n_tiles;
  // time ~ waves * (k-blocks per unit + per-unit overhead); the overhead of a
  // split unit includes writing and re-reading its fp32 partial tile
  const double c1 = pl.swap ? 4.0 : 8.0;
  const double cs = pl.swap ? 2.0 : 16.0;
  int best = 1;
  double best_cost = 1e30;
  const int max_s = std::min(16, std::max(1, pl.nkb / 2));
  for (int s = 1; s <= max_s; ++s) {
    const double waves = (double)ceil_div(tiles * s, h->nsm);
    const double cost = waves * ((double)pl.nkb / s + c1 + (s > 1 ? cs : 0.0));
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  pl.splits = force_splits > 0 ? std::min(force_splits, std::max(1, pl.nkb)) : best;
  pl.units = (int)(tiles * pl.splits);
  pl.grid = (int)std::min<int64_t>(pl.units, h->nsm);   // one CTA per SM (shared memory)
  pl.partial_bytes = pl.splits > 1 ? tiles * pl.splits * pl.acc_cols * 128 * 4 : 0;
  return pl;
}

struct Layout {
  int64_t x_norm, inv, h, part_col, part_row, pair_tail, total;
};

// Split count of the gate_up GEMM inside the fused decode block. Decode streams
// weights from HBM, and a few more than half the SMs keep it busy, so a unit
// takes a tile's whole K (h comes straight out of the accumulator, no partials)
// unless there are too few tiles for that.
int fused_gate_up_splits(const tp_linear* h) {
  const int tiles = h->wt_col;
  // with split-K, leave at least 8 CTAs for the norm rows
  return tiles * 2 >= h->nsm ? 1 : std::max(1, (h->nsm - 8) / tiles);
}

// Split count of the down GEMM inside the fused decode block: the stand-alone plan's, capped
// so that there are no more down units than SMs. Each CTA then takes at most one down unit
// at run time, in the order the CTAs finish their gate_up work, and every split of a tile is
// resident at once. (Fewer, larger units, leaving the CTAs that finish gate_up last without
// down work, measured slower: a unit then needs more bandwidth than one SM draws.)
int fused_down_splits(const tp_linear* h, int64_t T) {
  const Plan p = make_plan(h, 1, T);
  const int tiles = p.m_tiles * p.n_tiles;
  return std::min(p.splits, std::max(1, h->nsm / std::max(tiles, 1)));
}

Layout make_layout(const tp_linear* h, int64_t T) {
  Layout L{};
  int64_t off = dyn_off(h);
  const bool mlp = h->cfg.kind == TP_BLOCK_MLP;
  if (mlp && (h->cfg.flags & TP_FLAG_HAS_NORM)) {
    L.x_norm = off;
    off = align256(off + T * h->H * 2);
    L.inv = off;                       // the fused decode block's 1 / rms per row
    off = align256(off + T * 4);
  }
  if (mlp) {
    L.h = off;
    off = align256(off + (int64_t)h->cfg.t * T * h->Is * 2);
  }
  L.part_col = off;
  int64_t pc = make_plan(h, 0, T).partial_bytes;
  if (T <= kFusedMaxT) pc = std::max(pc, make_plan(h, 0, T, fused_gate_up_splits(h)).partial_bytes);
  off = align256(off + pc);
  L.part_row = off;
  off = align256(off + make_plan(h, 1, T).partial_bytes);
  if (T > kFusedMaxT) {
    L.pair_tail = off;   // the CTA-pair launches' split tail: partials, then counters
    off = align256(off + pair_tail_bytes(h->nsm));
  }
  L.total = off;
  return L;
}

// The partials and counters of a pair launch's split tail in workspace `ws` (null: no split).
float* tail_part(const tp_linear* h, void* ws, const Layout& L) {
  return L.pair_tail ? reinterpret_cast<float*>(static_cast<char*>(ws) + L.pair_tail) : nullptr;
}
unsigned* tail_cnt(const tp_linear* h, void* ws, const Layout& L) {
  if (!L.pair_tail) return nullptr;
  const int64_t parts = std::max(1, h->nsm / 2);
  return reinterpret_cast<unsigned*>(static_cast<char*>(ws) + L.pair_tail + parts * 2 * 256 * 128 * 4);
}

// Attention core workspace: after the handle's persistent counters and flags,
// [256) the table size, [260) the unit counter, [512) the (sequence, q tile)
// table, 16 B per entry.
int64_t attn_ws_bytes(const tp_linear* h, int64_t T, int64_t n_seqs) {
  return dyn_off(h) + 512 + 16 * (ceil_div(T, 128) + n_seqs + 1);
}

// Mixture-of-experts workspace for n_entries routed (token, expert) entries:
// after the header, the valid tile count, per-entry ranks and rows, the token of
// every row, the expert of every 128-row tile, then x, h and y in row order.
// Each expert's rows start on a 128-row boundary: at most n_entries + 127 E rows.
struct MoeLayout {
  int64_t max_rows, max_pairs, m_valid, pair_count, rank, perm_row, row_src, tile_expert, pair_tiles, x_perm, h_perm,
      y_perm, total;
};
MoeLayout moe_layout(const tp_linear* h, int64_t n_entries) {
  MoeLayout L{};
  L.max_rows = ceil_div(n_entries + (int64_t)h->cfg.n_experts * 127, 128) * 128;
  L.max_pairs = L.max_rows / 256 + h->cfg.n_experts;   // each expert leaves at most one lone tile
  int64_t off = dyn_off(h);
  L.m_valid = off;
  L.pair_count = off + 4;
  off = align256(off + 8);
  L.rank = off;
  off = align256(off + 4 * n_entries);
  L.perm_row = off;
  off = align256(off + 4 * n_entries);
  L.row_src = off;
  off = align256(off + 4 * L.max_rows);
  L.tile_expert = off;
  off = align256(off + 4 * (L.max_rows / 128));
  L.pair_tiles = off;
  off = align256(off + 8 * L.max_pairs);
  L.x_perm = off;
  off = align256(off + 2 * L.max_rows * h->H);
  L.h_perm = off;
  off = align256(off + 2 * (int64_t)h->cfg.t * L.max_rows * h->Is);
  L.y_perm = off;
  off = align256(off + 2 * L.max_rows * h->H);
  L.total = off;
  return L;
}

int check_device(const tp_linear* h) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != h->device)
    return fail(TP_ERR_ARG, "current device %d is not the handle's device %d", dev, h->device);
  return TP_OK;
}

// Prefill GEMMs may run on CTA pairs (two-SM MMAs over 256-token tiles, each
// CTA loading half of every weight block); TPL_GEMM_PAIR=0 in the environment
// keeps them on single CTAs.
bool pair_engine_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("TPL_GEMM_PAIR");
    return v == nullptr || v[0] != '0';
  }();
  return on;
}
// Estimated cost (in k-block times of one CTA) of running prefill units of full K on
// pairs vs. the single-CTA plan; a pair k-block is assumed to take 0.8 of a single one
// because it pulls a third less from L2.
bool prefer_pair(const tp_linear* h, const Plan* pls, int n, int ncl) {
  if (!pair_engine_enabled() || ncl <= 0) return false;
  long long pu = 0, units = 0;
  double one = 0;
  for (int i = 0; i < n; ++i) {
    const Plan& pl = pls[i];
    if (pl.swap) return false;
    pu += (long long)((pl.m_tiles + 1) / 2) * pl.n_tiles;
    units += pl.units;
  }
  // single-CTA cost of the same plans (as launched)
  if (n == 1)
    one = (double)ceil_div(pls[0].units, h->nsm) * ((double)pls[0].nkb / pls[0].splits + (pls[0].splits > 1 ? 16.0 : 0.0));
  else
    one = (double)ceil_div(units, h->nsm) * pls[0].nkb;
  const double pair = pair_waves((int)pu, ncl) * pls[0].nkb * 0.8;
  return pair < one;
}

GemmParams base_params(const Plan& pl, int64_t T, void* ws, int64_t part_off, int64_t gbar_off) {
  GemmParams p{};
  p.T = (int)T;
  p.m_tiles = pl.m_tiles;
  p.n_tiles = pl.n_tiles;
  p.splits = pl.splits;
  p.units = pl.units;
  p.nkb = pl.nkb;
  p.kbs = pl.kbs;
  p.nb = pl.nb;
  // raster groups of 32 token tiles (16 CTA pairs): each weight tile is read from DRAM
  // once per group while the group's token tiles stay in L2 (Llama-3-70B gate_up: 12.9 GB
  // of DRAM reads per launch with groups of 8, 8.6 GB with 32; 3.6 % faster)
  p.group_m = 32;
  char* w = static_cast<char*>(ws);
  p.partials = reinterpret_cast<float*>(w + part_off);
  p.gbar = reinterpret_cast<unsigned*>(w + gbar_off);
  p.status = t_status != nullptr ? t_status : reinterpret_cast<int*>(w);
  p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  return p;
}

bool gathered(const tp_linear* h) { return (h->cfg.flags & TP_FLAG_GATHERED) != 0; }

// where the column-parallel GEMM writes shard r, token m: per-shard width w
void set_col_out(GemmParams& p, const tp_linear* h, int64_t T, int64_t w, bool gath) {
  p.out_sstride = gath ? w : T * w;
  p.out_rstride = (int)(gath ? h->cfg.t * w : w);
}

// column-parallel GEMM: gate_up (MLP) or QKV (ATTN)
int run_col(const tp_linear* h, int64_t T, const void* x, void* out, void* ws, const Layout& L,
            cudaStream_t st) {
  const Plan pl = make_plan(h, 0, T);
  CUtensorMap map_x;
  int rc = make_map(&map_x, x, h->H, T, 1, 1, pl.swap ? pl.bn : 128);
  if (rc) return rc;
  GemmParams p = base_params(pl, T, ws, L.part_col, kGbarColOff);
  p.out = static_cast<__nv_bfloat16*>(out);
  if (h->cfg.kind == TP_BLOCK_MLP) {
    p.Is = (int)h->Is;
  } else {
    p.n_out = (int)h->n_col;
    p.ws_out = (int)h->ws_qkv;
  }
  set_col_out(p, h, T, h->cfg.kind == TP_BLOCK_MLP ? h->Is : h->ws_qkv, gathered(h));
  p.w_packed = static_cast<const uint8_t*>(h->w_col);
  const int ncl = pl.swap ? 0 : pair_max_clusters();
  if (!pl.swap && prefer_pair(h, &pl, 1, ncl)) {
    const Plan p1 = make_plan(h, 0, T, 1);
    GemmParams q = p;
    q.splits = 1;
    q.units = p1.units;
    cudaError_t e = launch_gemm_pair(pl.kind, -1, map_x, h->wmap_col, q, map_x, h->wmap_col, q, ncl,
                                     tail_part(h, ws, L), tail_cnt(h, ws, L), st);
    if (e != cudaSuccess) return cuda_fail(e, "column-parallel GEMM launch (pairs)");
    return TP_OK;
  }
  cudaError_t e = launch_gemm(pl.swap, pl.kind, pl.bn, map_x, p, pl.grid, st);
  if (e != cudaSuccess) return cuda_fail(e, "column-parallel GEMM launch");
  return TP_OK;
}

// row-parallel GEMM with the cross-shard reduction: down (MLP) or o_proj (ATTN)
int run_row(const tp_linear* h, int64_t T, const void* in_shards, const void* resid, void* out,
            void* out2, void* ws, const Layout& L, cudaStream_t st) {
  const Plan pl = make_plan(h, 1, T);
  CUtensorMap map_in;
  int rc = make_shard_map(&map_in, in_shards, h->Ks, T, h->cfg.t, 3, gathered(h), pl.swap ? pl.bn : 128);
  if (rc) return rc;
  GemmParams p = base_params(pl, T, ws, L.part_row, kGbarRowOff);
  p.n_out = (int)h->H;
  p.ws_out = (int)h->H;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.out2 = static_cast<__nv_bfloat16*>(out2);
  p.resid = static_cast<const __nv_bfloat16*>(resid);
  p.w_packed = static_cast<const uint8_t*>(h->w_row);
  const int ncl = pl.swap ? 0 : pair_max_clusters();
  if (!pl.swap && prefer_pair(h, &pl, 1, ncl)) {
    const Plan p1 = make_plan(h, 1, T, 1);
    GemmParams q = p;
    q.splits = 1;
    q.units = p1.units;
    cudaError_t e = launch_gemm_pair(pl.kind, -1, map_in, h->wmap_row, q, map_in, h->wmap_row, q, ncl,
                                     tail_part(h, ws, L), tail_cnt(h, ws, L), st);
    if (e != cudaSuccess) return cuda_fail(e, "row-parallel GEMM launch (pairs)");
    return TP_OK;
  }
  cudaError_t e = launch_gemm(pl.swap, pl.kind, pl.bn, map_in, p, pl.grid, st);
  if (e != cudaSuccess) return cuda_fail(e, "row-parallel GEMM launch");
  return TP_OK;
}

// QKV and o_proj of one attention block at prefill size: the two GEMMs are
// independent (o_proj reads the caller's attention output), so one launch walks
// both problems' tiles and they share the waves.
int run_col_row_together(const tp_linear* h, int64_t T, const void* x, void* qkv_out, const void* attn_in,
                         void* o_out, void* ws, const Layout& L, cudaStream_t st) {
  const Plan pc = make_plan(h, 0, T, 1), pr = make_plan(h, 1, T, 1);
  CUtensorMap map_x, map_a;
  int rc = make_map(&map_x, x, h->H, T, 1, 1, 128);
  if (!rc) rc = make_shard_map(&map_a, attn_in, h->Ks, T, h->cfg.t, 3, gathered(h), 128);
  if (rc) return rc;
  GemmParams p1 = base_params(pc, T, ws, L.part_col, kGbarColOff);
  p1.out = static_cast<__nv_bfloat16*>(qkv_out);
  p1.n_out = (int)h->n_col;
  p1.ws_out = (int)h->ws_qkv;
  set_col_out(p1, h, T, h->ws_qkv, gathered(h));
  p1.w_packed = static_cast<const uint8_t*>(h->w_col);
  GemmParams p2 = base_params(pr, T, ws, L.part_row, kGbarRowOff);
  p2.out = static_cast<__nv_bfloat16*>(o_out);
  p2.n_out = (int)h->H;
  p2.ws_out = (int)h->H;
  p2.w_packed = static_cast<const uint8_t*>(h->w_row);
  const int ncl = pair_max_clusters();
  const Plan both[2] = {pc, pr};
  cudaError_t e;
  if (prefer_pair(h, both, 2, ncl)) {
    e = launch_gemm_pair(KIND_COL, KIND_ROW, map_x, h->wmap_col, p1, map_a, h->wmap_row, p2, ncl,
                         tail_part(h, ws, L), tail_cnt(h, ws, L), st);
  } else {
    const int grid = (int)std::min<int64_t>((int64_t)pc.units + pr.units, h->nsm);
    e = launch_gemm_prefill_col_row(map_x, p1, map_a, p2, grid, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "attention projections launch");
  return TP_OK;
}

int check_ws(const tp_linear* h, int64_t T, const void* ws, int64_t ws_bytes, Layout* L) {
  if (ws == nullptr || !aligned16(ws)) return fail(TP_ERR_ARG, "workspace is null or not 16-byte aligned");
  *L = make_layout(h, T);
  if (ws_bytes < L->total)
    return fail(TP_ERR_ARG, "workspace too small: %lld bytes, %lld needed for T=%lld",
                (long long)ws_bytes, (long long)L->total, (long long)T);
  return TP_OK;
}

int check_T(int64_t T) {
  if (T < 0) return fail(TP_ERR_SHAPE, "T must be >= 0 (got %lld)", (long long)T);
  if (T > (1 << 24)) return fail(TP_ERR_UNSUPPORTED, "T > 16777216 tokens in one call");
  return TP_OK;
}

#define TP_CHECK_PTR(p, name)                                                        \
  do {                                                                               \
    if ((p) == nullptr) return fail(TP_ERR_ARG, "%s is null", name);                \
    if (!aligned16(p)) return fail(TP_ERR_ARG, "%s is not 16-byte aligned", name);  \
  } while (0)

int validate_cfg(const tp_config_t* c) {
  if (c == nullptr) return fail(TP_ERR_ARG, "config is null");
  if (c->kind != TP_BLOCK_MLP && c->kind != TP_BLOCK_ATTN_PROJ && c->kind != TP_BLOCK_MOE)
    return fail(TP_ERR_ARG, "unknown block kind %d", c->kind);
  if (c->kind == TP_BLOCK_MOE) {
    if (c->n_experts < 1 || c->n_experts > 256)
      return fail(TP_ERR_UNSUPPORTED, "n_experts must be in [1, 256] (got %d)", c->n_experts);
    if (c->flags != 0) return fail(TP_ERR_ARG, "flags must be 0 for the MoE block");
  } else if (c->n_experts != 0) {
    return fail(TP_ERR_ARG, "n_experts must be 0 unless kind is TP_BLOCK_MOE");
  }
  if (c->t <= 0) return fail(TP_ERR_SHAPE, "t must be positive (got %d)", c->t);
  if ((c->t & (c->t - 1)) != 0 || c->t > 8)
    return fail(TP_ERR_UNSUPPORTED, "t must be a power of 2 in [1, 8] (got %d)", c->t);
  if (c->hidden <= 0 || c->hidden > (1 << 20)) return fail(TP_ERR_SHAPE, "hidden out of range");
  if (c->hidden % 8 != 0) return fail(TP_ERR_UNSUPPORTED, "hidden must be a multiple of 8");
  if (c->kind != TP_BLOCK_ATTN_PROJ) {
    if (c->intermediate <= 0 || c->intermediate > (1 << 22))
      return fail(TP_ERR_SHAPE, "intermediate out of range");
    if (c->intermediate % c->t != 0)
      return fail(TP_ERR_SHAPE, "intermediate %lld is not divisible by t=%d",
                  (long long)c->intermediate, c->t);
    if ((c->intermediate / c->t) % 8 != 0)
      return fail(TP_ERR_UNSUPPORTED, "intermediate / t must be a multiple of 8");
  } else {
    if (c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0)
      return fail(TP_ERR_SHAPE, "head counts must be positive");
    if (c->n_q_heads % c->t != 0)
      return fail(TP_ERR_SHAPE, "n_q_heads %d is not divisible by t=%d", c->n_q_heads, c->t);
    if (c->n_kv_heads % c->t != 0 && c->t % c->n_kv_heads != 0)
      return fail(TP_ERR_SHAPE, "n_kv_heads %d and t=%d: neither divides the other", c->n_kv_heads, c->t);
    if (c->n_q_heads % c->n_kv_heads != 0)
      return fail(TP_ERR_SHAPE, "n_q_heads must be a multiple of n_kv_heads");
    if (c->head_dim % 8 != 0) return fail(TP_ERR_UNSUPPORTED, "head_dim must be a multiple of 8");
  }
  if (c->flags & ~(TP_FLAG_HAS_NORM | TP_FLAG_GATHERED)) return fail(TP_ERR_ARG, "unknown flags 0x%x", c->flags);
  if ((c->flags & TP_FLAG_HAS_NORM) && !(c->rms_eps >= 0.0f))
    return fail(TP_ERR_ARG, "rms_eps must be >= 0");
  if ((c->flags & TP_FLAG_HAS_NORM) && c->hidden > max_norm_hidden())
    return fail(TP_ERR_UNSUPPORTED, "hidden > %d with the fused norm", max_norm_hidden());
  return TP_OK;
}

void derive(tp_linear* h) {
  const tp_config_t& c = h->cfg;
  h->H = c.hidden;
  const int t = c.t;
  if (c.kind != TP_BLOCK_ATTN_PROJ) {
    h->I = c.intermediate;
    h->Is = c.intermediate / t;
    h->Ks = h->Is;
    h->n_col = 2 * h->I;
  } else {
    h->q_per = c.n_q_heads / t;
    if (t >= c.n_kv_heads) {
      h->kv_per = 1;
      h->rep = t / c.n_kv_heads;
    } else {
      h->kv_per = c.n_kv_heads / t;
      h->rep = 1;
    }
    h->ws_qkv = (int64_t)(h->q_per + 2 * h->kv_per) * c.head_dim;
    h->n_col = t * h->ws_qkv;
    h->Ks = (int64_t)c.n_q_heads * c.head_dim / t;
  }
  h->nkb_col = (int)ceil_div(h->H, 64);
  if (c.kind != TP_BLOCK_ATTN_PROJ) {
    h->nb = (int)ceil_div(h->Is, 128);
    h->wt_col = t * h->nb;
  } else {
    h->nb = 0;
    h->wt_col = (int)ceil_div(h->n_col, 256);
  }
  h->kbs_row = (int)ceil_div(h->Ks, 64);
  h->nkb_row = t * h->kbs_row;
  h->wt_row = (int)ceil_div(h->H, 256);
}

}  // namespace

// ============================================================================ C ABI
extern "C" {

const char* tp_last_error(void) { return g_err; }

int tp_packed_weight_bytes(const tp_config_t* cfg, int64_t* col_bytes, int64_t* row_bytes) {
  int rc = validate_cfg(cfg);
  if (rc) return rc;
  if (col_bytes == nullptr || row_bytes == nullptr) return fail(TP_ERR_ARG, "null output pointer");
  tp_linear tmp{};
  tmp.cfg = *cfg;
  derive(&tmp);
  const int64_t E = cfg->kind == TP_BLOCK_MOE ? cfg->n_experts : 1;
  *col_bytes = E * tmp.wt_col * tmp.nkb_col * kWBlockBytes;
  *row_bytes = E * tmp.wt_row * tmp.nkb_row * kWBlockBytes;
  return ok();
}

int tp_linear_create(const tp_config_t* cfg, const void* const* w_full, int32_t n_w,
                     void* w_col_packed, void* w_row_packed, const void* gamma, tp_stream_t stream,
                     tp_linear_t** out) {
  if (out == nullptr) return fail(TP_ERR_ARG, "out is null");
  *out = nullptr;
  int rc = validate_cfg(cfg);
  if (rc) return rc;
  const bool mlp = cfg->kind != TP_BLOCK_ATTN_PROJ;
  const int n_exp = cfg->kind == TP_BLOCK_MOE ? cfg->n_experts : 1;
  const int need = mlp ? 3 * n_exp : 4;
  if (w_full == nullptr || n_w != need)
    return fail(TP_ERR_ARG, "expected %d full weight pointers, got %d", need, n_w);
  for (int i = 0; i < need; ++i) TP_CHECK_PTR(w_full[i], "w_full[i]");
  TP_CHECK_PTR(w_col_packed, "w_col_packed");
  TP_CHECK_PTR(w_row_packed, "w_row_packed");
  if (cfg->flags & TP_FLAG_HAS_NORM) TP_CHECK_PTR(gamma, "gamma");

  tp_linear* h = new (std::nothrow) tp_linear();
  if (h == nullptr) return fail(TP_ERR_ARG, "out of host memory");
  h->cfg = *cfg;
  derive(h);
  static std::atomic<uint64_t> next_uid{1};
  h->uid = next_uid.fetch_add(1);
  h->w_col = w_col_packed;
  h->w_row = w_row_packed;
  h->gamma = (cfg->flags & TP_FLAG_HAS_NORM) ? gamma : nullptr;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->nsm, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "device query");
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int t = cfg->t;
  // pack the shards ("weight_loader": narrow the full tensor to each rank's slice),
  // tiled into swizzled 32 KB blocks
  PackSpec pc{}, pr{};
  pc.t = pr.t = t;
  pc.H = pr.H = h->H;
  pc.nkb = h->nkb_col;
  if (mlp) {
    pc.mode = PACK_GATE_UP;
    pc.src[0] = static_cast<const __nv_bfloat16*>(w_full[0]);
    pc.src[1] = static_cast<const __nv_bfloat16*>(w_full[1]);
    pc.Is = h->Is;
    pc.nb = h->nb;
    pr.src[0] = static_cast<const __nv_bfloat16*>(w_full[2]);
  } else {
    pc.mode = PACK_QKV;
    for (int i = 0; i < 3; ++i) pc.src[i] = static_cast<const __nv_bfloat16*>(w_full[i]);
    pc.n_col = h->n_col;
    pc.ws = h->ws_qkv;
    pc.q_per = h->q_per;
    pc.kv_per = h->kv_per;
    pc.rep = h->rep;
    pc.hd = cfg->head_dim;
    pr.src[0] = static_cast<const __nv_bfloat16*>(w_full[3]);
  }
  pr.mode = PACK_ROW;
  pr.Is = h->Ks;
  pr.kbs = h->kbs_row;
  pr.nkb = h->nkb_row;
  // experts one after another, each in the dense layout
  const int64_t col_blocks = (int64_t)h->wt_col * h->nkb_col, row_blocks = (int64_t)h->wt_row * h->nkb_row;
  e = cudaSuccess;
  for (int x = 0; x < n_exp && e == cudaSuccess; ++x) {
    if (mlp) {
      pc.src[0] = static_cast<const __nv_bfloat16*>(w_full[3 * x]);
      pc.src[1] = static_cast<const __nv_bfloat16*>(w_full[3 * x + 1]);
      pr.src[0] = static_cast<const __nv_bfloat16*>(w_full[3 * x + 2]);
    }
    e = launch_pack(pc, col_blocks, static_cast<uint8_t*>(w_col_packed) + x * col_blocks * kWBlockBytes, st);
    if (e == cudaSuccess)
      e = launch_pack(pr, row_blocks, static_cast<uint8_t*>(w_row_packed) + x * row_blocks * kWBlockBytes, st);
  }
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "weight packing");
  }
  if ((rc = make_wmap(&h->wmap_col, w_col_packed, n_exp * col_blocks)) ||
      (rc = make_wmap(&h->wmap_row, w_row_packed, n_exp * row_blocks))) {
    delete h;
    return rc;
  }
  *out = h;
  return ok();
}

int tp_linear_destroy(tp_linear_t* h) {
  delete h;
  return ok();
}

int tp_workspace_size(const tp_linear_t* h, int64_t max_tokens, int64_t* bytes) {
  if (h == nullptr || bytes == nullptr) return fail(TP_ERR_ARG, "null argument");
  int rc = check_T(max_tokens);
  if (rc) return rc;
  // Up to 128 tokens every T has its own plan; beyond, a plan depends on T only
  // through the number of 128-token tiles, and the buffers grow with T, so the
  // largest T of each tile count bounds that count.
  if (h->cfg.kind == TP_BLOCK_MOE) {   // max_tokens counts routed entries (tokens x top_k)
    *bytes = moe_layout(h, max_tokens).total;
    return ok();
  }
  int64_t best = dyn_off(h);
  for (int64_t T = 1; T <= std::min<int64_t>(max_tokens, kFusedMaxT); ++T)
    best = std::max(best, make_layout(h, T).total);
  for (int64_t m = 2; (m - 1) * 128 < max_tokens; ++m)
    best = std::max(best, make_layout(h, std::min<int64_t>(max_tokens, m * 128)).total);
  // the attention core's work table, for up to max_tokens sequences
  if (h->cfg.kind == TP_BLOCK_ATTN_PROJ) best = std::max(best, attn_ws_bytes(h, max_tokens, max_tokens));
  *bytes = best;
  return ok();
}

int tp_describe_plan(const tp_linear_t* h, int64_t T, tp_gemm_plan_t* plans, int32_t max_plans) {
  if (h == nullptr || plans == nullptr || max_plans < 0) return fail(TP_ERR_ARG, "null argument");
  if (check_T(T) || T == 0) return 0;
  int n = 0;
  for (int which = 0; which < 2 && n < max_plans; ++which, ++n) {
    const Plan pl = make_plan(h, which, T);
    plans[n].swap_ab = pl.swap;
    plans[n].block_n = pl.bn;
    plans[n].splits = pl.splits;
    plans[n].units = pl.units;
    plans[n].grid = pl.grid;
    plans[n].stages = gemm_stages(pl.swap, pl.kind, pl.bn);
    plans[n].engine = 0;
    if (h->cfg.kind == TP_BLOCK_MLP && T <= kFusedMaxT) {
      plans[n].engine = 2;
    } else if (!pl.swap) {
      const int ncl = pair_max_clusters();
      bool pair;
      if (h->cfg.kind == TP_BLOCK_ATTN_PROJ && T > kFusedMaxT) {
        const Plan both[2] = {make_plan(h, 0, T, 1), make_plan(h, 1, T, 1)};
        pair = prefer_pair(h, both, 2, ncl);
      } else {
        pair = prefer_pair(h, &pl, 1, ncl);
      }
      if (pair) {
        plans[n].engine = 1;
        plans[n].splits = 1;
        plans[n].units = ((pl.m_tiles + 1) / 2) * pl.n_tiles;
        plans[n].grid = 2 * std::min(plans[n].units, ncl);
        plans[n].stages = pair_stages();
      }
    }
  }
  g_err[0] = '\0';
  return n;
}

int tp_add_rms_norm(int64_t T, int64_t H, const void* a, const void* residual_in, const void* gamma,
                    float eps, void* residual_out, void* x_out, tp_stream_t stream) {
  int rc = check_T(T);
  if (rc) return rc;
  if (H <= 0 || H % 8 != 0) return fail(TP_ERR_UNSUPPORTED, "H must be a positive multiple of 8");
  if (H > max_norm_hidden()) return fail(TP_ERR_UNSUPPORTED, "H > %d", max_norm_hidden());
  if (!(eps >= 0.0f)) return fail(TP_ERR_ARG, "eps must be >= 0");
  if (T == 0) return ok();
  TP_CHECK_PTR(a, "a");
  if (residual_in != nullptr) TP_CHECK_PTR(residual_in, "residual_in");
  TP_CHECK_PTR(gamma, "gamma");
  TP_CHECK_PTR(residual_out, "residual_out");
  TP_CHECK_PTR(x_out, "x_out");
  if (T == 0) return ok();
  cudaError_t e = launch_add_rms_norm((int)T, (int)H, a, residual_in, gamma, eps, residual_out,
                                      x_out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "add_rms_norm launch");
  return ok();
}

int tp_gate_up_forward(tp_linear_t* h, int64_t T, const void* x, void* h_out, void* workspace,
                       int64_t workspace_bytes, tp_stream_t stream) {
  if (h == nullptr) return fail(TP_ERR_ARG, "handle is null");
  if (h->cfg.kind != TP_BLOCK_MLP) return fail(TP_ERR_ARG, "not an MLP handle");
  int rc = check_T(T);
  if (rc) return rc;
  if (T == 0) return ok();
  TP_CHECK_PTR(x, "x");
  TP_CHECK_PTR(h_out, "h_out");
  Layout L;
  if ((rc = check_ws(h, T, workspace, workspace_bytes, &L))) return rc;
  if ((rc = check_device(h))) return rc;
  if (T == 0) return ok();
  if ((rc = run_col(h, T, x, h_out, workspace, L, static_cast<cudaStream_t>(stream)))) return rc;
  return ok();
}

int tp_down_forward(tp_linear_t* h, int64_t T, const void* h_in, const void* residual,
                    void* mlp_out, void* residual_stream, void* workspace, int64_t workspace_bytes,
                    tp_stream_t stream) {
  if (h == nullptr) return fail(TP_ERR_ARG, "handle is null");
  if (h->cfg.kind != TP_BLOCK_MLP) return fail(TP_ERR_ARG, "not an MLP handle");
  int rc = check_T(T);
  if (rc) return rc;
  if (T == 0) return ok();
  TP_CHECK_PTR(h_in, "h_in");
  TP_CHECK_PTR(mlp_out, "mlp_out");
  if (residual_stream != nullptr) {
    TP_CHECK_PTR(residual_stream, "residual_stream");
    TP_CHECK_PTR(residual, "residual");
  }
  Layout L;
  if ((rc = check_ws(h, T, workspace, workspace_bytes, &L))) return rc;
  if ((rc = check_device(h))) return rc;
  if (T == 0) return ok();
  if ((rc = run_row(h, T, h_in, residual, mlp_out, residual_stream, workspace, L,
                    static_cast<cudaStream_t>(stream))))
    return rc;
  return ok();
}

// The fused decode-shaped block (T <= 128) over the workspace `ws` laid out as L:
// norm, gate_up, h, down and both reductions in one launch. status: where device
// errors go (null: the workspace's status word).
int run_fused_decode(const tp_linear* h, int64_t T, char* ws, const Layout& L, const void* x_in,
                     const void* residual_in, void* residual_out, void* mlp_out, void* residual_stream,
                     int32_t* status, cudaStream_t st) {
  const bool norm = (h->cfg.flags & TP_FLAG_HAS_NORM) != 0;
  const Plan p1 = make_plan(h, 0, T, fused_gate_up_splits(h)), p2 = make_plan(h, 1, T, fused_down_splits(h, T));
  if (mlp_decode_ctas_per_sm(p1.bn) < 1)
    return fail(TP_ERR_UNSUPPORTED, "the fused decode block (block_n %d) does not fit on an SM of this device",
                p1.bn);
  void* hbuf = ws + L.h;
  const void* xsrc = norm ? static_cast<const void*>(ws + L.x_norm) : x_in;
  CUtensorMap map_x, map_h;
  int rc;
  if ((rc = make_map(&map_x, xsrc, h->H, T, 1, 1, p1.bn))) return rc;
  if ((rc = make_map(&map_h, hbuf, h->Ks, T, 1, h->cfg.t, p2.bn))) return rc;
  MlpDecodeParams P{};
  P.g1 = base_params(p1, T, ws, L.part_col, kGbarColOff);
  P.g1.out = static_cast<__nv_bfloat16*>(hbuf);
  P.g1.Is = (int)h->Is;
  set_col_out(P.g1, h, T, h->Is, false);   // h stays inside the launch: shard-major
  P.g1.w_packed = static_cast<const uint8_t*>(h->w_col);
  P.g2 = base_params(p2, T, ws, L.part_row, kGbarRowOff);
  P.g2.n_out = (int)h->H;
  P.g2.ws_out = (int)h->H;
  P.g2.out = static_cast<__nv_bfloat16*>(mlp_out);
  P.g2.out2 = static_cast<__nv_bfloat16*>(residual_stream);
  P.g2.resid = static_cast<const __nv_bfloat16*>(norm ? residual_out : residual_in);
  P.g2.w_packed = static_cast<const uint8_t*>(h->w_row);
  if (status != nullptr) P.g1.status = P.g2.status = status;
  P.x_in = static_cast<const __nv_bfloat16*>(x_in);
  P.res_in = static_cast<const __nv_bfloat16*>(residual_in);
  P.gamma = static_cast<const __nv_bfloat16*>(h->gamma);
  P.res_out = static_cast<__nv_bfloat16*>(residual_out);
  P.x_norm = reinterpret_cast<__nv_bfloat16*>(ws + L.x_norm);
  P.inv = norm ? reinterpret_cast<float*>(ws + L.inv) : nullptr;
  P.g1.inv = P.inv;   // gate_up with split-K scales in the reduction
  P.bars = reinterpret_cast<unsigned*>(ws + kDecodeBarsOff);
  P.cnt1 = reinterpret_cast<unsigned*>(ws + kTileCountersOff);
  P.hready = P.cnt1 + h->wt_col;
  P.cnt2 = P.hready + h->wt_col;
  P.cset = (int)tile_counter_words(h);
  P.epoch = reinterpret_cast<unsigned long long*>(ws + kDecodeBarsOff + 32);
  P.ticket = reinterpret_cast<unsigned long long*>(ws + kDecodeBarsOff + 40);
  // the first CTAs to start own the norm rows; the gate_up units go to the CTAs after them
  const int grid = h->nsm;
  P.n_norm = norm ? (int)std::max<int64_t>(1, std::min<int64_t>(T, grid - p1.units)) : 0;
  P.eps = h->cfg.rms_eps;
  P.H = (int)h->H;
  P.has_norm = norm ? 1 : 0;
  const cudaError_t e = launch_mlp_decode(p1.bn, map_x, map_h, P, grid, st);
  if (e != cudaSuccess) return cuda_fail(e, "fused decode MLP launch");
  return TP_OK;
}

int tp_mlp_forward(tp_linear_t* h, int64_t T, const void* x_in, const void* residual_in,
                   void* residual_out, void* mlp_out, void* residual_stream, void* workspace,
                   int64_t workspace_bytes, tp_stream_t stream) {
  if (h == nullptr) return fail(TP_ERR_ARG, "handle is null");
  if (h->cfg.kind != TP_BLOCK_MLP) return fail(TP_ERR_ARG, "not an MLP handle");
  int rc = check_T(T);
  if (rc) return rc;
  if (T == 0) return ok();
  const bool norm = (h->cfg.flags & TP_FLAG_HAS_NORM) != 0;
  TP_CHECK_PTR(x_in, "x_in");
  TP_CHECK_PTR(mlp_out, "mlp_out");
  if (norm) {
    TP_CHECK_PTR(residual_in, "residual_in");
    TP_CHECK_PTR(residual_out, "residual_out");
  }
  if (residual_in != nullptr) TP_CHECK_PTR(residual_in, "residual_in");
  if (residual_stream != nullptr) {
    TP_CHECK_PTR(residual_stream, "residual_stream");
    if (residual_in == nullptr) return fail(TP_ERR_ARG, "residual_stream needs a residual");
  }
  Layout L;
  if ((rc = check_ws(h, T, workspace, workspace_bytes, &L))) return rc;
  if ((rc = check_device(h))) return rc;
  if (T == 0) return ok();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const void* x = x_in;
  const void* resid = residual_in;
  if (norm) {
    x = ws + L.x_norm;
    resid = residual_out;
  }
  void* hbuf = ws + L.h;
  if (T <= kFusedMaxT) {
    // decode-shaped step: norm, gate_up, h, down and both reductions in one launch
    if ((rc = run_fused_decode(h, T, ws, L, x_in, residual_in, residual_out, mlp_out, residual_stream, nullptr,
                               st)))
      return rc;
    return ok();
  }
  if (norm) {
    cudaError_t e = launch_add_rms_norm((int)T, (int)h->H, x_in, residual_in, h->gamma,
                                        h->cfg.rms_eps, residual_out, ws + L.x_norm, st);
    if (e != cudaSuccess) return cuda_fail(e, "add_rms_norm launch");
  }
  if ((rc = run_col(h, T, x, hbuf, workspace, L, st))) return rc;
  if ((rc = run_row(h, T, hbuf, resid, mlp_out, residual_stream, workspace, L, st))) return rc;
  return ok();
}

int tp_attn_proj_forward(tp_linear_t* h, int64_t T, const void* x, void* qkv_out,
                         const void* attn_in, void* o_out, void* workspace, int64_t workspace_bytes,
                         tp_stream_t stream) {
  if (h == nullptr) return fail(TP_ERR_ARG, "handle is null");
  if (h->cfg.kind != TP_BLOCK_ATTN_PROJ) return fail(TP_ERR_ARG, "not an attention handle");
  int rc = check_T(T);
  if (rc) return rc;
  if (T == 0) return ok();
  const bool do_qkv = x != nullptr || qkv_out != nullptr;
  const bool do_o = attn_in != nullptr || o_out != nullptr;
  if (do_qkv) {
    TP_CHECK_PTR(x, "x");
    TP_CHECK_PTR(qkv_out, "qkv_out");
  }
  if (do_o) {
    TP_CHECK_PTR(attn_in, "attn_in");
    TP_CHECK_PTR(o_out, "o_out");
  }
  Layout L;
  if ((rc = check_ws(h, T, workspace, workspace_bytes, &L))) return rc;
  if ((rc = check_device(h))) return rc;
  if (T == 0) return ok();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (do_qkv && do_o && T > kFusedMaxT) {
    if ((rc = run_col_row_together(h, T, x, qkv_out, attn_in, o_out, workspace, L, st))) return rc;
    return ok();
  }
  if (do_qkv && (rc = run_col(h, T, x, qkv_out, workspace, L, st))) return rc;
  if (do_o && (rc = run_row(h, T, attn_in, nullptr, o_out, nullptr, workspace, L, st))) return rc;
  return ok();
}

int tp_attention_forward(tp_linear_t* h, int64_t T, const void* qkv, const int32_t* cu_seqlens,
                         int32_t n_seqs, int32_t max_seqlen, void* attn_out, void* workspace,
                         int64_t workspace_bytes, tp_stream_t stream) {
  if (h == nullptr) return fail(TP_ERR_ARG, "handle is null");
  if (h->cfg.kind != TP_BLOCK_ATTN_PROJ) return fail(TP_ERR_ARG, "not an attention handle");
  int rc = check_T(T);
  if (rc) return rc;
  if (T == 0) return ok();
  if (h->cfg.head_dim != 128) return fail(TP_ERR_UNSUPPORTED, "the attention core is built for head_dim 128");
  TP_CHECK_PTR(qkv, "qkv");
  TP_CHECK_PTR(attn_out, "attn_out");
  if (cu_seqlens == nullptr || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
    return fail(TP_ERR_ARG, "cu_seqlens is null or not 4-byte aligned");
  if (n_seqs < 1 || n_seqs > T) return fail(TP_ERR_SHAPE, "n_seqs must be in [1, T] (got %d)", n_seqs);
  if (max_seqlen < 1 || max_seqlen > T)
    return fail(TP_ERR_SHAPE, "max_seqlen must be in [1, T] (got %d)", max_seqlen);
  const int max_tiles = (int)ceil_div(max_seqlen, 128);
  if (max_tiles > 8192) return fail(TP_ERR_UNSUPPORTED, "max_seqlen > 1048576");
  if (workspace == nullptr || !aligned16(workspace)) return fail(TP_ERR_ARG, "workspace is null or not 16-byte aligned");
  if (workspace_bytes < attn_ws_bytes(h, T, n_seqs))
    return fail(TP_ERR_ARG, "workspace too small: %lld bytes, %lld needed", (long long)workspace_bytes,
                (long long)attn_ws_bytes(h, T, n_seqs));
  if ((rc = check_device(h))) return rc;
  CUtensorMap map_qkv;
  if ((rc = make_shard_map(&map_qkv, qkv, h->ws_qkv, T, h->cfg.t, 2, gathered(h), 128))) return rc;
  char* ws = static_cast<char*>(workspace);
  AttnParams p{};
  p.pairs = reinterpret_cast<const int4*>(ws + dyn_off(h) + 512);
  p.n_pairs = reinterpret_cast<const int*>(ws + dyn_off(h) + 256);
  p.next_unit = reinterpret_cast<int*>(ws + dyn_off(h) + 260);
  p.out = static_cast<__nv_bfloat16*>(attn_out);
  p.out_align32 = (reinterpret_cast<uintptr_t>(attn_out) & 31u) == 0 ? 1 : 0;
  p.out_sstride = gathered(h) ? h->Ks : T * h->Ks;
  p.out_rstride = (int)(gathered(h) ? h->cfg.t * h->Ks : h->Ks);
  p.status = t_status != nullptr ? t_status : reinterpret_cast<int*>(ws);
  p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  p.T = (int)T;
  p.q_per = h->q_per;
  p.kv_per = h->kv_per;
  p.rep = h->rep;
  p.group = h->cfg.n_q_heads / h->cfg.n_kv_heads;
  p.heads = h->cfg.t * h->q_per;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)h->cfg.head_dim));
  const int64_t max_units = (ceil_div(T, 128) + n_seqs) * p.heads;
  const int grid = (int)std::min<int64_t>(h->nsm, max_units);
  const cudaError_t e =
      launch_attention(map_qkv, p, cu_seqlens, n_seqs, max_tiles, const_cast<int4*>(p.pairs),
                       const_cast<int*>(p.n_pairs), grid, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return ok();
}

// Paged attention: splits along each request's keys so that about twelve CTAs per SM are
// launched, at most 512 splits and at most 256 MiB of partial results. Workspace: the status
// word, then the splits' partial results.
struct PagedPlan {
  int split_len, n_splits, q_stride;
  int64_t partials_off, ws_bytes;
};
PagedPlan paged_plan(const tp_linear* h, int n_reqs, int max_query_len, int max_seq_len) {
  PagedPlan pl{};
  const int gq = h->q_per / (h->rep > 1 ? 1 : h->kv_per);
  const int64_t per_split = (int64_t)n_reqs * h->cfg.t * h->kv_per;
  const int max_chunks = (int)ceil_div(std::max(max_seq_len, 1), 128);
  // the partial results are q_stride * (128 + 2) floats per item: at most 256 MiB of them
  // unless a single split already needs more (long chunks of new tokens)
  const int64_t item_bytes = (int64_t)max_query_len * gq * (128 + 2) * 4;
  const int64_t cap = std::max<int64_t>(1, (int64_t(256) << 20) / std::max<int64_t>(per_split * item_bytes, 1));
  const int want = (int)std::max<int64_t>(
      1, std::min<int64_t>({max_chunks, 512, cap, ceil_div(12LL * h->nsm, std::max<int64_t>(per_split, 1))}));
  pl.split_len = (int)ceil_div(ceil_div(std::max(max_seq_len, 1), want), 128) * 128;
  pl.n_splits = (int)ceil_div(std::max(max_seq_len, 1), pl.split_len);
  pl.q_stride = max_query_len * gq;
  pl.partials_off = 256;
  pl.ws_bytes = pl.partials_off + per_split * pl.n_splits * pl.q_stride * (128 + 2) * 4;
  return pl;
}

int tp_kv_cache_write(tp_linear_t* h, int64_t T, const void* qkv, const int32_t* slot_mapping, void* cache_k,
                      void* cache_v, int64_t num_blocks, int32_t block_size, void* workspace, int64_t workspace_bytes,
                      tp_stream_t stream) {
  if (h == nullptr) return fail(TP_ERR_ARG, "handle is null");
  if (h->cfg.kind != TP_BLOCK_ATTN_PROJ) return fail(TP_ERR_ARG, "not an attention handle");
  int rc = check_T(T);
  if (rc) return rc;
  if (h->cfg.head_dim != 128) return fail(TP_ERR_UNSUPPORTED, "the KV cache is built for head_dim 128");
  if (num_blocks < 1 || block_size < 1) return fail(TP_ERR_SHAPE, "num_blocks and block_size must be >= 1");
  if (T == 0) return ok();
  TP_CHECK_PTR(qkv, "qkv");
  TP_CHECK_PTR(cache_k, "cache_k");
  TP_CHECK_PTR(cache_v, "cache_v");
  if (slot_mapping == nullptr || (reinterpret_cast<uintptr_t>(slot_mapping) & 3u) != 0)
    return fail(TP_ERR_ARG, "slot_mapping is null or not 4-byte aligned");
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < 16)
    return fail(TP_ERR_ARG, "workspace is null, not 16-byte aligned or under 16 bytes");
  if ((rc = check_device(h))) return rc;
  const bool gath = gathered(h);
  const cudaError_t e = launch_kv_write(qkv, (int)T, h->cfg.t, gath ? h->ws_qkv : T * h->ws_qkv,
                                        (int)(gath ? h->cfg.t * h->ws_qkv : h->ws_qkv), h->q_per, h->kv_per,
                                        slot_mapping, num_blocks * (long long)block_size, cache_k, cache_v,
                                        reinterpret_cast<int*>(workspace), h->nsm, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "KV cache write launch");
  return ok();
}

int tp_paged_attention_workspace_size(const tp_linear_t* h, int32_t n_reqs, int32_t max_query_len,
                                      int32_t max_seq_len, int64_t* bytes) {
  if (h == nullptr || bytes == nullptr) return fail(TP_ERR_ARG, "null argument");
  if (h->cfg.kind != TP_BLOCK_ATTN_PROJ) return fail(TP_ERR_ARG, "not an attention handle");
  if (n_reqs < 1 || max_query_len < 1 || max_seq_len < max_query_len)
    return fail(TP_ERR_SHAPE, "need n_reqs >= 1 and 1 <= max_query_len <= max_seq_len");
  *bytes = paged_plan(h, n_reqs, max_query_len, max_seq_len).ws_bytes;
  return ok();
}

int tp_paged_attention(tp_linear_t* h, int64_t T, const void* qkv, const int32_t* query_start_loc,
                       const int32_t* seq_lens, int32_t n_reqs, int32_t max_query_len, int32_t max_seq_len,
                       const int32_t* block_tables, int32_t max_blocks_per_req, const int32_t* slot_mapping,
                       void* cache_k, void* cache_v, int64_t num_blocks, int32_t block_size, void* attn_out,
                       void* workspace, int64_t workspace_bytes, tp_stream_t stream) {
  if (h == nullptr) return fail(TP_ERR_ARG, "handle is null");
  if (h->cfg.kind != TP_BLOCK_ATTN_PROJ) return fail(TP_ERR_ARG, "not an attention handle");
  int rc = check_T(T);
  if (rc) return rc;
  if (h->cfg.head_dim != 128) return fail(TP_ERR_UNSUPPORTED, "the KV cache is built for head_dim 128");
  if (T == 0) return ok();
  if (n_reqs < 1 || max_query_len < 1 || max_seq_len < max_query_len || max_query_len > T)
    return fail(TP_ERR_SHAPE, "need n_reqs >= 1 and 1 <= max_query_len <= min(T, max_seq_len)");
  if (num_blocks < 1 || block_size < 1 || max_blocks_per_req < 1 ||
      (int64_t)max_blocks_per_req * block_size < max_seq_len)
    return fail(TP_ERR_SHAPE, "the block tables cannot hold max_seq_len tokens");
  if (num_blocks > INT32_MAX) return fail(TP_ERR_UNSUPPORTED, "more than 2^31 - 1 cache blocks");
  if (num_blocks * (int64_t)block_size * h->kv_per * 128 > (int64_t(1) << 40))
    return fail(TP_ERR_UNSUPPORTED, "cache larger than 2^40 elements per shard");
  if (num_blocks * (int64_t)block_size * h->cfg.t > INT32_MAX)
    return fail(TP_ERR_UNSUPPORTED, "more than 2^31 - 1 cache slots over all shards");
  TP_CHECK_PTR(qkv, "qkv");
  TP_CHECK_PTR(cache_k, "cache_k");
  TP_CHECK_PTR(cache_v, "cache_v");
  TP_CHECK_PTR(attn_out, "attn_out");
  for (const int32_t* q : {query_start_loc, seq_lens, block_tables})
    if (q == nullptr || (reinterpret_cast<uintptr_t>(q) & 3u) != 0)
      return fail(TP_ERR_ARG, "query_start_loc, seq_lens and block_tables must be 4-byte aligned device arrays");
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 3u) != 0)
    return fail(TP_ERR_ARG, "slot_mapping must be null or a 4-byte aligned device array");
  const PagedPlan pl = paged_plan(h, n_reqs, max_query_len, max_seq_len);
  if (workspace == nullptr || !aligned16(workspace)) return fail(TP_ERR_ARG, "workspace is null or not 16-byte aligned");
  if (workspace_bytes < pl.ws_bytes)
    return fail(TP_ERR_ARG, "workspace too small: %lld bytes, %lld needed", (long long)workspace_bytes,
                (long long)pl.ws_bytes);
  if ((rc = check_device(h))) return rc;
  const bool gath = gathered(h);
  PagedAttnParams p{};
  p.qkv = static_cast<const __nv_bfloat16*>(qkv);
  p.sstride_in = gath ? h->ws_qkv : T * h->ws_qkv;
  p.rstride_in = (int)(gath ? h->cfg.t * h->ws_qkv : h->ws_qkv);
  p.qsl = query_start_loc;
  p.seq_lens = seq_lens;
  p.block_tables = block_tables;
  p.slots = slot_mapping;
  p.n_slots = num_blocks * (int64_t)block_size;
  p.cache_k = static_cast<__nv_bfloat16*>(cache_k);
  p.cache_v = static_cast<__nv_bfloat16*>(cache_v);
  p.out = static_cast<__nv_bfloat16*>(attn_out);
  p.sstride_out = gath ? h->Ks : T * h->Ks;
  p.rstride_out = (int)(gath ? h->cfg.t * h->Ks : h->Ks);
  p.partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + pl.partials_off);
  p.status = reinterpret_cast<int*>(workspace);
  p.t = h->cfg.t;
  p.q_per = h->q_per;
  p.kv_per = h->kv_per;
  p.rep = h->rep;
  p.max_blocks = max_blocks_per_req;
  p.num_blocks = (int)num_blocks;
  p.block_size = block_size;
  p.max_query_len = max_query_len;
  p.max_seq_len = max_seq_len;
  p.split_len = pl.split_len;
  p.n_splits = pl.n_splits;
  p.q_stride = pl.q_stride;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt(128.0));
  const cudaError_t e = launch_paged_attention(p, n_reqs, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "paged attention launch");
  return ok();
}

int tp_moe_forward(tp_linear_t* h, int64_t T, int32_t top_k, const void* x, const int32_t* expert_ids,
                   const float* gates, void* y, void* workspace, int64_t workspace_bytes, tp_stream_t stream) {
  if (h == nullptr) return fail(TP_ERR_ARG, "handle is null");
  if (h->cfg.kind != TP_BLOCK_MOE) return fail(TP_ERR_ARG, "not an MoE handle");
  int rc = check_T(T);
  if (rc) return rc;
  const int E = h->cfg.n_experts;
  if (top_k < 1 || top_k > E) return fail(TP_ERR_SHAPE, "top_k must be in [1, n_experts] (got %d)", top_k);
  if (T == 0) return ok();
  const int64_t N = T * top_k;
  if (N > (1 << 24)) return fail(TP_ERR_UNSUPPORTED, "more than 16777216 routed entries");
  TP_CHECK_PTR(x, "x");
  TP_CHECK_PTR(y, "y");
  if (expert_ids == nullptr || (reinterpret_cast<uintptr_t>(expert_ids) & 3u) != 0)
    return fail(TP_ERR_ARG, "expert_ids is null or not 4-byte aligned");
  if (gates == nullptr || (reinterpret_cast<uintptr_t>(gates) & 3u) != 0)
    return fail(TP_ERR_ARG, "gates is null or not 4-byte aligned");
  if (workspace == nullptr || !aligned16(workspace)) return fail(TP_ERR_ARG, "workspace is null or not 16-byte aligned");
  const MoeLayout L = moe_layout(h, N);
  if (workspace_bytes < L.total)
    return fail(TP_ERR_ARG, "workspace too small: %lld bytes, %lld needed for %lld routed entries",
                (long long)workspace_bytes, (long long)L.total, (long long)N);
  if ((rc = check_device(h))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* m_valid = reinterpret_cast<int*>(ws + L.m_valid);
  int* tile_expert = reinterpret_cast<int*>(ws + L.tile_expert);
  int* perm_row = reinterpret_cast<int*>(ws + L.perm_row);
  const int64_t R = L.max_rows;
  int* pair_tiles = reinterpret_cast<int*>(ws + L.pair_tiles);
  int* pair_count = reinterpret_cast<int*>(ws + L.pair_count);
  cudaError_t e = launch_moe_route(expert_ids, (int)N, top_k, E, (int)R, reinterpret_cast<int*>(ws + L.rank), perm_row,
                                   reinterpret_cast<int*>(ws + L.row_src), tile_expert, m_valid, pair_tiles,
                                   pair_count, reinterpret_cast<int*>(ws), st);
  if (e == cudaSuccess)
    e = launch_moe_gather(x, (int)h->H, reinterpret_cast<int*>(ws + L.row_src), m_valid, (int)R, ws + L.x_perm,
                          h->nsm, st);
  if (e != cudaSuccess) return cuda_fail(e, "MoE routing launch");
  // grouped GEMMs: every 128-row tile belongs to one expert; tiles past *m_valid are skipped.
  // With about a tile or more per expert the CTA-pair engine takes them, two tiles of one
  // expert sharing each weight block.
  const int ncl = pair_max_clusters();
  const bool pairs = pair_engine_enabled() && ncl > 0 && N >= 128LL * E;
  for (int which = 0; which < 2; ++which) {
    Plan pl{};
    pl.swap = false;
    pl.kind = which == 0 ? KIND_GATE_UP : KIND_ROW;
    pl.bn = 256;
    pl.splits = 1;
    pl.m_tiles = (int)(R / 128);
    pl.n_tiles = which == 0 ? h->wt_col : h->wt_row;
    pl.nkb = which == 0 ? h->nkb_col : h->nkb_row;
    pl.kbs = which == 0 ? 0 : h->kbs_row;
    pl.nb = which == 0 ? h->nb : 0;
    pl.units = pl.m_tiles * pl.n_tiles;
    pl.grid = std::min(pl.units, h->nsm);
    CUtensorMap map_a;
    rc = which == 0 ? make_map(&map_a, ws + L.x_perm, h->H, R, 1, 1, 128)
                    : make_shard_map(&map_a, ws + L.h_perm, h->Is, R, h->cfg.t, 3, false, 128);
    if (rc) return rc;
    GemmParams p = base_params(pl, R, workspace, 0, which == 0 ? kGbarColOff : kGbarRowOff);
    p.tile_expert = tile_expert;
    p.m_valid = m_valid;
    p.expert_wbytes = (long long)pl.n_tiles * pl.nkb * kWBlockBytes;
    if (which == 0) {
      p.out = reinterpret_cast<__nv_bfloat16*>(ws + L.h_perm);
      p.Is = (int)h->Is;
      set_col_out(p, h, R, h->Is, false);
      p.w_packed = static_cast<const uint8_t*>(h->w_col);
    } else {
      p.n_out = (int)h->H;
      p.ws_out = (int)h->H;
      p.out = reinterpret_cast<__nv_bfloat16*>(ws + L.y_perm);
      p.w_packed = static_cast<const uint8_t*>(h->w_row);
    }
    if (pairs) {
      p.m_tiles = (int)(2 * L.max_pairs);
      p.pair_tiles = pair_tiles;
      p.pair_count = pair_count;
      const CUtensorMap& wm = which == 0 ? h->wmap_col : h->wmap_row;
      e = launch_gemm_pair(pl.kind, -1, map_a, wm, p, map_a, wm, p, ncl, nullptr, nullptr, st);
    } else {
      e = launch_gemm(false, pl.kind, pl.bn, map_a, p, pl.grid, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "grouped expert GEMM launch");
  }
  e = launch_moe_combine(ws + L.y_perm, (int)h->H, (int)T, top_k, perm_row, gates, y, h->nsm, st);
  if (e != cudaSuccess) return cuda_fail(e, "MoE combine launch");
  return ok();
}

int tp_set_wait_timeout(int64_t ns) {
  if (ns <= 0) return fail(TP_ERR_ARG, "wait limit must be positive (got %lld ns)", (long long)ns);
  g_timeout_ns.store((unsigned long long)ns, std::memory_order_relaxed);
  return ok();
}

// ---------------------------------------------------------------------------- no-allocation variant
// Scratch of tp_mlp_forward_no_alloc: a file-scope device array, so callers that
// must not allocate device memory still get the fused decode block. Every GPU
// that loads this library holds these 16 MiB until the process exits.
namespace {
constexpr int64_t kNoAllocScratchBytes = int64_t(16) << 20;
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

// Device address of g_no_alloc_scratch per device ordinal, looked up once per
// device with that device current (in host code the symbol itself is only a
// host-side stand-in and must never be handed to a kernel).
constexpr int kMaxDevices = 64;
std::mutex g_no_alloc_mu;
void* g_no_alloc_ptr[kMaxDevices] = {};
// handle (uid) whose counters the array holds on each device; 0: none yet
uint64_t g_no_alloc_owner[kMaxDevices] = {};

// Scratch the fused decode kernel itself uses: the counters, x_norm, h and the
// split-K partials of its own two plans.
Layout no_alloc_layout(const tp_linear* h, int64_t T) {
  Layout L{};
  int64_t off = dyn_off(h);
  if (h->cfg.flags & TP_FLAG_HAS_NORM) {
    L.x_norm = off;
    off = align256(off + T * h->H * 2);
    L.inv = off;
    off = align256(off + T * 4);
  }
  L.h = off;
  off = align256(off + (int64_t)h->cfg.t * T * h->Is * 2);
  L.part_col = off;
  off = align256(off + make_plan(h, 0, T, fused_gate_up_splits(h)).partial_bytes);
  L.part_row = off;
  off = align256(off + make_plan(h, 1, T).partial_bytes);
  L.total = off;
  return L;
}

// The array's device address on `device` (looked up on the first call there) and
// whether its counters must be cleared because another handle (or none) used it last.
int no_alloc_scratch(int device, uint64_t uid, void** out, bool* clear) {
  if (device < 0 || device >= kMaxDevices) return fail(TP_ERR_UNSUPPORTED, "device ordinal %d", device);
  std::lock_guard<std::mutex> lock(g_no_alloc_mu);
  if (g_no_alloc_ptr[device] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_no_alloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    g_no_alloc_ptr[device] = ptr;
  }
  *out = g_no_alloc_ptr[device];
  *clear = g_no_alloc_owner[device] != uid;
  g_no_alloc_owner[device] = uid;
  return TP_OK;
}
}  // namespace

extern "C" int tp_mlp_forward_no_alloc(tp_linear_t* h, int64_t T, const void* x_in, const void* residual_in,
                                       void* residual_out, void* mlp_out, void* residual_stream,
                                       int32_t* status_dev, tp_stream_t stream) {
  if (h == nullptr) return fail(TP_ERR_ARG, "handle is null");
  if (h->cfg.kind != TP_BLOCK_MLP) return fail(TP_ERR_ARG, "not an MLP handle");
  int rc = check_T(T);
  if (rc) return rc;
  if (T == 0) return ok();
  if (T > kFusedMaxT)
    return fail(TP_ERR_UNSUPPORTED, "tp_mlp_forward_no_alloc runs the decode-shaped block only: T=%lld > %lld",
                (long long)T, (long long)kFusedMaxT);
  const bool norm = (h->cfg.flags & TP_FLAG_HAS_NORM) != 0;
  TP_CHECK_PTR(x_in, "x_in");
  TP_CHECK_PTR(mlp_out, "mlp_out");
  if (norm) {
    TP_CHECK_PTR(residual_in, "residual_in");
    TP_CHECK_PTR(residual_out, "residual_out");
  }
  if (residual_in != nullptr) TP_CHECK_PTR(residual_in, "residual_in");
  if (residual_stream != nullptr) {
    TP_CHECK_PTR(residual_stream, "residual_stream");
    if (residual_in == nullptr) return fail(TP_ERR_ARG, "residual_stream needs a residual");
  }
  if (status_dev != nullptr && (reinterpret_cast<uintptr_t>(status_dev) & 3u) != 0)
    return fail(TP_ERR_ARG, "status_dev is not 4-byte aligned");
  if ((rc = check_device(h))) return rc;
  const Layout L = no_alloc_layout(h, T);
  if (L.total > kNoAllocScratchBytes)
    return fail(TP_ERR_UNSUPPORTED,
                "tp_mlp_forward_no_alloc: this shape needs %lld bytes of scratch, the fixed scratch holds %lld",
                (long long)L.total, (long long)kNoAllocScratchBytes);
  void* scratch = nullptr;
  bool clear = true;
  if ((rc = no_alloc_scratch(h->device, h->uid, &scratch, &clear))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(scratch);
  // The counters start at zero for a handle that did not make the last call here (their
  // layout is the handle's): a memset, not an allocation. Between calls of one handle
  // the kernel keeps them consistent itself (each launch clears the set the next one
  // uses, even a launch that gave up), so those calls keep overlapping one another.
  if (clear) {
    const cudaError_t e = cudaMemsetAsync(ws, 0, (size_t)dyn_off(h), st);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the no-alloc scratch counters");
  }
  if ((rc = run_fused_decode(h, T, ws, L, x_in, residual_in, residual_out, mlp_out, residual_stream, status_dev,
                             st)))
    return rc;
  return ok();
}

// ---------------------------------------------------------------------------- capture
namespace {
constexpr int kSmemTableMaxLog2 = 13;  // 8192 slots = 64 KB of shared memory
struct CaptureLayout {
  int cap_log2;
  bool global_table;
  int64_t n_match, rows, table, total;
};
CaptureLayout capture_layout(int64_t T, int64_t n_sel) {
  CaptureLayout c{};
  int lg = 6;
  while ((int64_t(1) << lg) < 2 * n_sel) ++lg;
  c.cap_log2 = lg;
  c.global_table = lg > kSmemTableMaxLog2;
  c.n_match = kCaptureOff;
  c.rows = kCaptureOff + 256;
  c.table = align256(c.rows + 4 * std::max<int64_t>(T, 1));
  c.total = c.global_table ? align256(c.table + (int64_t(8) << lg)) : c.table;
  return c;
}
}  // namespace

int tp_capture_workspace_size(int64_t T, int64_t n_sel, int64_t* bytes) {
  if (bytes == nullptr) return fail(TP_ERR_ARG, "bytes is null");
  int rc = check_T(T);
  if (rc) return rc;
  if (n_sel < 0 || n_sel > (int64_t(1) << 26)) return fail(TP_ERR_SHAPE, "n_sel out of range");
  *bytes = capture_layout(T, n_sel).total;
  return ok();
}

int tp_capture_rows(int64_t T, int64_t H, const int32_t* row_req, const int32_t* row_pos,
                    const int64_t* sel_keys, int64_t n_sel, int32_t n_tensors,
                    const void* const* tensors, const int32_t* tensor_types, int32_t layer,
                    tp_record_hdr_t* hdr_out, void* rows_out, int64_t capacity, int64_t* n_out_dev,
                    void* workspace, int64_t workspace_bytes, tp_stream_t stream) {
  int rc = check_T(T);
  if (rc) return rc;
  if (H <= 0 || H % 8 != 0) return fail(TP_ERR_UNSUPPORTED, "H must be a positive multiple of 8");
  if (n_sel < 0 || n_sel > (int64_t(1) << 26)) return fail(TP_ERR_SHAPE, "n_sel out of range");
  if (n_tensors < 1 || n_tensors > kCaptureMaxTensors)
    return fail(TP_ERR_UNSUPPORTED, "n_tensors must be in [1, %d]", kCaptureMaxTensors);
  if (capacity < 0) return fail(TP_ERR_SHAPE, "capacity must be >= 0");
  if (T == 0) return ok();
  if (tensors == nullptr || tensor_types == nullptr) return fail(TP_ERR_ARG, "tensor list is null");
  TP_CHECK_PTR(row_req, "row_req");
  TP_CHECK_PTR(row_pos, "row_pos");
  if (n_sel > 0) TP_CHECK_PTR(sel_keys, "sel_keys");
  TP_CHECK_PTR(n_out_dev, "n_out_dev");
  if (capacity > 0) {
    TP_CHECK_PTR(hdr_out, "hdr_out");
    TP_CHECK_PTR(rows_out, "rows_out");
  }
  CaptureMeta meta{};
  for (int k = 0; k < n_tensors; ++k) {
    TP_CHECK_PTR(tensors[k], "tensors[k]");
    meta.tensors[k] = static_cast<const __nv_bfloat16*>(tensors[k]);
    meta.types[k] = tensor_types[k];
  }
  meta.n_tensors = n_tensors;
  meta.layer = layer;
  meta.hdr = reinterpret_cast<int32_t*>(hdr_out);
  meta.rows_out = rows_out;
  if (workspace == nullptr || !aligned16(workspace))
    return fail(TP_ERR_ARG, "workspace is null or not 16-byte aligned");
  const CaptureLayout c = capture_layout(T, n_sel);
  if (workspace_bytes < c.total)
    return fail(TP_ERR_ARG, "capture workspace too small: %lld < %lld", (long long)workspace_bytes,
                (long long)c.total);
  if (T == 0) return ok();
  int dev = 0, nsm = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  char* ws = static_cast<char*>(workspace);
  const int64_t recs = std::min<int64_t>(capacity, (int64_t)n_tensors * T);
  const int copy_grid = (int)std::max<int64_t>(1, std::min<int64_t>(recs, 4 * nsm));
  cudaError_t e = launch_capture(
      (int)T, (int)H, row_req, row_pos, sel_keys, (int)n_sel,
      c.global_table ? reinterpret_cast<uint64_t*>(ws + c.table) : nullptr, c.cap_log2,
      c.global_table ? 0 : (size_t(8) << c.cap_log2), meta, capacity, n_out_dev,
      reinterpret_cast<int32_t*>(ws + c.rows), reinterpret_cast<int32_t*>(ws + c.n_match),
      reinterpret_cast<int*>(ws), copy_grid, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "capture launch");
  return ok();
}

}  // extern "C"

// ============================================================================ decoder layer
// One layer = the attention handle's half, then the MLP handle's half, on one
// stream. The workspace layout is fixed by max_tokens: the attention half's
// workspace from byte 0 (its status word is the layer's), the MLP half's, then
// x1 [T][H], qkv [t][T][w_s] and the attention output A [t][T][nq*hd/t].
struct tp_layer {
  tp_linear* attn;
  tp_linear* mlp;
  int64_t max_tokens;
  int64_t attn_ws, mlp_off, mlp_ws, x1_off, qkv_off, a_off, total;
};

extern "C" {

int tp_layer_create(tp_linear_t* attn, tp_linear_t* mlp, int64_t max_tokens, tp_layer_t** out) {
  if (out == nullptr) return fail(TP_ERR_ARG, "out is null");
  *out = nullptr;
  if (attn == nullptr || mlp == nullptr) return fail(TP_ERR_ARG, "handle is null");
  if (attn->cfg.kind != TP_BLOCK_ATTN_PROJ) return fail(TP_ERR_ARG, "first handle is not an attention handle");
  if (mlp->cfg.kind != TP_BLOCK_MLP) return fail(TP_ERR_ARG, "second handle is not an MLP handle");
  if (!(attn->cfg.flags & TP_FLAG_HAS_NORM) || !(mlp->cfg.flags & TP_FLAG_HAS_NORM))
    return fail(TP_ERR_ARG, "both handles need TP_FLAG_HAS_NORM (input and post-attention norms)");
  if (attn->H != mlp->H)
    return fail(TP_ERR_SHAPE, "hidden sizes differ (%lld vs %lld)", (long long)attn->H, (long long)mlp->H);
  if (attn->device != mlp->device) return fail(TP_ERR_ARG, "handles are on different devices");
  if (attn->cfg.head_dim != 128) return fail(TP_ERR_UNSUPPORTED, "the attention core is built for head_dim 128");
  if (max_tokens < 1) return fail(TP_ERR_SHAPE, "max_tokens must be >= 1");
  int rc = check_T(max_tokens);
  if (rc) return rc;
  tp_layer* L = new (std::nothrow) tp_layer();
  if (L == nullptr) return fail(TP_ERR_ARG, "out of host memory");
  L->attn = attn;
  L->mlp = mlp;
  L->max_tokens = max_tokens;
  if ((rc = tp_workspace_size(attn, max_tokens, &L->attn_ws)) ||
      (rc = tp_workspace_size(mlp, max_tokens, &L->mlp_ws))) {
    delete L;
    return rc;
  }
  L->mlp_off = align256(L->attn_ws);
  L->x1_off = align256(L->mlp_off + L->mlp_ws);
  L->qkv_off = align256(L->x1_off + max_tokens * attn->H * 2);
  L->a_off = align256(L->qkv_off + (int64_t)attn->cfg.t * max_tokens * attn->ws_qkv * 2);
  L->total = align256(L->a_off + (int64_t)attn->cfg.t * max_tokens * attn->Ks * 2);
  *out = L;
  return ok();
}

int tp_layer_destroy(tp_layer_t* layer) {
  delete layer;
  return ok();
}

int tp_layer_workspace_size(const tp_layer_t* layer, int64_t* bytes) {
  if (layer == nullptr || bytes == nullptr) return fail(TP_ERR_ARG, "null argument");
  *bytes = layer->total;
  return ok();
}

int tp_decoder_layer_forward(tp_layer_t* layer, int64_t T, const tp_layer_io_t* io, void* workspace,
                             int64_t workspace_bytes, tp_stream_t stream) {
  if (layer == nullptr || io == nullptr) return fail(TP_ERR_ARG, "null argument");
  int rc = check_T(T);
  if (rc) return rc;
  if (T > layer->max_tokens)
    return fail(TP_ERR_SHAPE, "T=%lld exceeds the layer's max_tokens=%lld", (long long)T,
                (long long)layer->max_tokens);
  if (T == 0) return ok();
  tp_linear* at = layer->attn;
  TP_CHECK_PTR(io->hidden_in, "hidden_in");
  if (io->residual_in != nullptr) TP_CHECK_PTR(io->residual_in, "residual_in");
  TP_CHECK_PTR(io->residual_attn, "residual_attn");
  TP_CHECK_PTR(io->attn_out, "attn_out");
  TP_CHECK_PTR(io->residual_mlp, "residual_mlp");
  TP_CHECK_PTR(io->mlp_out, "mlp_out");
  if (io->residual_stream != nullptr) TP_CHECK_PTR(io->residual_stream, "residual_stream");
  if (io->cu_seqlens == nullptr || (reinterpret_cast<uintptr_t>(io->cu_seqlens) & 3u) != 0)
    return fail(TP_ERR_ARG, "cu_seqlens is null or not 4-byte aligned");
  if (io->n_seqs < 1 || io->n_seqs > T) return fail(TP_ERR_SHAPE, "n_seqs must be in [1, T] (got %d)", io->n_seqs);
  if (io->max_seqlen < 1 || io->max_seqlen > T)
    return fail(TP_ERR_SHAPE, "max_seqlen must be in [1, T] (got %d)", io->max_seqlen);
  if (ceil_div(io->max_seqlen, 128) > 8192) return fail(TP_ERR_UNSUPPORTED, "max_seqlen > 1048576");
  if (workspace == nullptr || !aligned16(workspace))
    return fail(TP_ERR_ARG, "workspace is null or not 16-byte aligned");
  if (workspace_bytes < layer->total)
    return fail(TP_ERR_ARG, "workspace too small: %lld bytes, %lld needed", (long long)workspace_bytes,
                (long long)layer->total);
  if ((rc = check_device(at))) return rc;
  char* ws = static_cast<char*>(workspace);
  void* x1 = ws + layer->x1_off;
  void* qkv = ws + layer->qkv_off;
  void* A = ws + layer->a_off;
  StatusRedirect redirect(reinterpret_cast<int*>(ws));
  if ((rc = tp_add_rms_norm(T, at->H, io->hidden_in, io->residual_in, at->gamma, at->cfg.rms_eps,
                            io->residual_attn, x1, stream)))
    return rc;
  if ((rc = tp_attn_proj_forward(at, T, x1, qkv, nullptr, nullptr, ws, layer->attn_ws, stream))) return rc;
  if ((rc = tp_attention_forward(at, T, qkv, io->cu_seqlens, io->n_seqs, io->max_seqlen, A, ws,
                                 layer->attn_ws, stream)))
    return rc;
  if ((rc = tp_attn_proj_forward(at, T, nullptr, nullptr, A, io->attn_out, ws, layer->attn_ws, stream)))
    return rc;
  if ((rc = tp_mlp_forward(layer->mlp, T, io->attn_out, io->residual_attn, io->residual_mlp, io->mlp_out,
                           io->residual_stream, ws + layer->mlp_off, layer->mlp_ws, stream)))
    return rc;
  return ok();
}

}  // extern "C"
