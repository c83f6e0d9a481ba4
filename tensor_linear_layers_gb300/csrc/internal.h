// Declarations shared by the library's translation units (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

namespace tpl {

constexpr int kStatusCapacity = -5;

// ---------------------------------------------------------------- capture
constexpr int kCaptureMaxTensors = 8;
struct CaptureMeta {
  const __nv_bfloat16* tensors[kCaptureMaxTensors];
  int32_t types[kCaptureMaxTensors];
  int32_t n_tensors;
  int32_t layer;
  int32_t* hdr;        // [capacity][6]
  void* rows_out;      // [capacity][H] bf16
};

cudaError_t launch_capture(int T, int H, const int32_t* row_req, const int32_t* row_pos,
                           const int64_t* sel, int n_sel, uint64_t* gtable, int cap_log2,
                           size_t table_smem, const CaptureMeta& meta, int64_t capacity,
                           int64_t* n_out_dev, int32_t* match_rows, int32_t* n_match_ws, int* status,
                           int copy_grid, cudaStream_t st);

// ---------------------------------------------------------------- RMSNorm
cudaError_t launch_add_rms_norm(int T, int H, const void* a, const void* res, const void* gamma,
                                float eps, void* res_out, void* x_out, cudaStream_t st);
int max_norm_hidden();

// ---------------------------------------------------------------- packing
// Weights are packed as blocks of 256 rows x 64 K elements (32 KB) in the
// 128-byte-swizzled K-major image the MMA reads; block (w_tile, kb) sits at
// (w_tile * nkb + kb) * 32 KB. Rows or K past the end are zero.
enum PackMode : int { PACK_GATE_UP = 0, PACK_ROW = 1, PACK_QKV = 2 };
struct PackSpec {
  int mode;
  const __nv_bfloat16* src[3];
  int64_t H;       // hidden: K of the column kinds, output rows of PACK_ROW
  int64_t Is;      // PACK_GATE_UP: rows per shard; PACK_ROW: K per shard
  int64_t t;
  int64_t nb;      // PACK_GATE_UP: 128-row blocks per shard
  int64_t nkb;     // k-blocks per weight tile
  int64_t kbs;     // PACK_ROW: k-blocks per shard
  int64_t n_col;   // PACK_QKV: packed rows in total
  int64_t ws;      // PACK_QKV: packed rows per shard
  int q_per, kv_per, rep, hd;
};
cudaError_t launch_pack(const PackSpec& s, int64_t n_blocks, void* dst, cudaStream_t st);

// ---------------------------------------------------------------- attention core
struct AttnParams {
  const int4* pairs;       // [n_pairs] {sequence start, length, q tile, 0}, heaviest first
  const int* n_pairs;      // written by the preparation kernel
  int* next_unit;          // units handed out so far (CTAs take the next one when free); zeroed by the preparation kernel
  __nv_bfloat16* out;      // shard r, token m at out + r * out_sstride + m * out_rstride
  long long out_sstride;   // [t][T][q_per * 128]: T * q_per * 128; gathered [T][t * q_per * 128]: q_per * 128
  int out_rstride;         // q_per * 128, or t * q_per * 128 gathered
  int* status;
  unsigned long long timeout_ns;
  int T, q_per, kv_per, rep, group, heads;  // group = nq / nkv, heads = t * q_per
  float scale_log2;        // log2(e) / sqrt(hd)
  int out_align32;         // out is 32-byte aligned (rows are then written with 32-byte stores)
};
// Builds the (sequence, q tile) table from cu_seqlens (device) into `pairs` and
// runs the attention kernel on `grid` CTAs; map_qkv covers qkv as
// (w_s, T, t, 1) with 64 x 128 boxes.
cudaError_t launch_attention(const CUtensorMap& map_qkv, const AttnParams& p, const int* cu, int n_seqs,
                             int max_tiles, int4* pairs, int* n_pairs, int grid, cudaStream_t st);

// ---------------------------------------------------------------- GEMM
struct GemmParams;
// Launch the GEMM instantiation for (swap, kind, bn); cudaErrorInvalidValue
// when no such instantiation exists.
cudaError_t launch_gemm(bool swap, int kind, int bn, const CUtensorMap& map_act, const GemmParams& p,
                        int grid, cudaStream_t st);
int gemm_stages(bool swap, int kind, int bn);
struct MlpDecodeParams;
// The fused decode-shaped MLP block (T <= 128): one launch.
cudaError_t launch_mlp_decode(int bn, const CUtensorMap& map_x, const CUtensorMap& map_h,
                              const MlpDecodeParams& P, int grid, cudaStream_t st);
// CTAs of the fused kernel that fit on one SM (0 when it cannot run on this device).
int mlp_decode_ctas_per_sm(int bn);

// Paged KV cache (kv_cache.cu).
struct PagedAttnParams {
  const __nv_bfloat16* qkv;          // new tokens: shard r, token i at qkv + r * sstride_in + i * rstride_in
  long long sstride_in;
  int rstride_in;
  const int* qsl;                    // [n_reqs + 1] new-token offsets
  const int* seq_lens;               // [n_reqs] tokens of each request, new ones included
  const int* block_tables;           // [n_reqs][max_blocks]
  const int* slots;                  // [T] cache slot of each new token, written before it is read (null: none)
  long long n_slots;                 // num_blocks * block_size
  __nv_bfloat16* cache_k;            // [t][num_blocks][block_size][kv_per][128]
  __nv_bfloat16* cache_v;
  __nv_bfloat16* out;                // shard r, token i at out + r * sstride_out + i * rstride_out
  long long sstride_out;
  int rstride_out;
  float* partials;                   // [item][q_stride][128 + 2]: o, max, sum of each split
  int* status;
  int t, q_per, kv_per, rep, max_blocks, num_blocks, block_size, max_query_len, max_seq_len;
  int split_len, n_splits;           // keys per split, splits per (request, shard, kv head)
  int q_stride;                      // query slots of one item: max_query_len * (q heads per kv head)
  float scale_log2;
};
cudaError_t launch_kv_write(const void* qkv, int T, int t, long long sstride, int rstride, int q_per, int kv_per,
                            const int* slots, long long n_slots, void* ck, void* cv, int* status, int nsm,
                            cudaStream_t st);
cudaError_t launch_paged_attention(const PagedAttnParams& p, int n_reqs, cudaStream_t st);

// Mixture of experts (moe.cu): routing sort, row gather, weighted combine.
cudaError_t launch_moe_route(const int* ids, int n_entries, int k, int E, int max_rows, int* rank, int* perm_row,
                             int* row_src, int* tile_expert, int* m_valid, int* pair_tiles, int* pair_count,
                             int* status, cudaStream_t st);
cudaError_t launch_moe_gather(const void* x, int H, const int* row_src, const int* m_valid, int max_rows,
                              void* x_perm, int nsm, cudaStream_t st);
cudaError_t launch_moe_combine(const void* y_perm, int H, int T, int k, const int* perm_row, const float* gates,
                               void* y, int nsm, cudaStream_t st);

}  // namespace tpl
