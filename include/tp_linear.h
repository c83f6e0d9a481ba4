/*
 * tp_linear.h -- C ABI of libtplinear.so: a Megatron-style tensor-parallel
 * decoder linear block on one GB300 (sm_103a).
 *
 * The block is the column-parallel / row-parallel pair the pages describe:
 *   - "vLLM 源码完全拆解（十一）：模型并行与 Worker 层" (sections on the split
 *     of one matmul, ColumnParallelLinear, MergedColumnParallelLinear /
 *     QkvParallelLinear, RowParallelLinear and the column-row block);
 *   - "vLLM Code Reading (Section 5)", sections 11-14 (column/row split
 *     identities; attention and MLP TP data flow);
 *   - "Tensor & pipeline parallelism" (Undercurrent internals): what the
 *     capture hooks see (post-reduce, full tensors) and how records are keyed.
 *
 * The t tensor-parallel shards are a logical weight layout held on one GPU.
 * The all-reduce that follows a row-parallel layer on t GPUs becomes an
 * on-chip reduction of the t per-shard partial sums (tensor-memory
 * accumulation across the shards' K ranges, or a deterministic split-K fix-up
 * in fp32); there is no inter-GPU collective.
 *
 * Conventions shared by every call:
 *   - Weights are bf16 in nn.Linear layout [out_features, in_features],
 *     row-major; activations are bf16 row-major. All GEMMs multiply bf16,
 *     accumulate in fp32 and round the result to bf16 (nearest-even).
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise,
 *     and must be 16-byte aligned (tensor-memory-access copies need it).
 *   - The library never allocates, frees or synchronises. Calls only enqueue
 *     work on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *     Errors found on the host are returned; errors found by a kernel are
 *     written to the workspace status word (see tp_workspace_size) and
 *     become visible after the caller synchronises.
 *   - Return value: TP_OK (0) or a negative TP_ERR_* code; tp_last_error()
 *     then holds a message (thread-local).
 *   - T = 0 tokens is legal everywhere and enqueues nothing (a step with no
 *     scheduled tokens runs no forward pass).
 */
#ifndef TP_LINEAR_H
#define TP_LINEAR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TP_OK 0
#define TP_ERR_ARG (-1)         /* null / misaligned pointer, bad enum, workspace too small */
#define TP_ERR_SHAPE (-2)       /* a size that does not divide (the pages' divide()), T < 0 */
#define TP_ERR_UNSUPPORTED (-3) /* legal per the pages but not built (e.g. t not a power of 2) */
#define TP_ERR_CUDA (-4)        /* a CUDA runtime/driver call failed */
#define TP_ERR_CAPACITY (-5)    /* device status: capture records exceeded capacity */
#define TP_ERR_TIMEOUT (-6)     /* device status: a bounded on-chip wait gave up */

typedef struct tp_linear tp_linear_t; /* opaque handle: shapes, plans, packed-weight pointers */
typedef void* tp_stream_t;            /* cudaStream_t */

enum { TP_BLOCK_MLP = 0, TP_BLOCK_ATTN_PROJ = 1, TP_BLOCK_MOE = 2 };
enum {
  TP_FLAG_HAS_NORM = 1, /* MLP: fused residual add + RMSNorm in front of gate_up;
                           ATTN: the handle carries the layer's input RMSNorm */
  /* Gathered activations ("vLLM 源码完全拆解（十一）" ColumnParallelLinear gather_output=True,
   * RowParallelLinear input_is_parallel=False): the column-parallel output and the
   * row-parallel input are [T][t * w] (the t shards' columns side by side in each row,
   * i.e. the unsharded tensor) instead of shard-major [t][T][w]. Applies to h_out /
   * h_in of the stage calls, qkv_out / attn_in of tp_attn_proj_forward and qkv /
   * attn_out of tp_attention_forward. Results are bit-identical to the shard-major
   * layout: only the addresses change. */
  TP_FLAG_GATHERED = 2
};

typedef struct {
  int32_t kind;          /* TP_BLOCK_MLP, TP_BLOCK_ATTN_PROJ or TP_BLOCK_MOE */
  int32_t t;             /* logical tensor-parallel size: 1, 2, 4 or 8 */
  int64_t hidden;        /* H */
  int64_t intermediate;  /* MLP, MOE (per expert): I, I % t == 0, (I / t) % 8 == 0 */
  int32_t n_q_heads;     /* ATTN: nq % t == 0 */
  int32_t n_kv_heads;    /* ATTN: nkv % t == 0, or t % nkv == 0 (kv heads replicated) */
  int32_t head_dim;      /* ATTN: hd % 8 == 0 */
  float rms_eps;         /* with TP_FLAG_HAS_NORM */
  int32_t flags;         /* TP_FLAG_* */
  int32_t n_experts;     /* MOE: experts, 1..256; 0 for the other kinds */
} tp_config_t;

/*
 * Sizes of the two packed weight buffers the caller allocates for a handle.
 * Logically each buffer holds the t shards the pages describe
 * ("MergedColumnParallelLinear" / "QkvParallelLinear" / "RowParallelLinear",
 * weight_loader: narrow(dim, rank * shard, shard)):
 *   MLP : col = gate_up  shard r: its gate rows, then its up rows
 *         row = down     shard r: input columns r*I/t .. (r+1)*I/t of W_down
 *   ATTN: col = qkv      shard r: its q heads | k heads | v heads
 *                        (w_s = (nq/t + 2*kv_per_shard) * hd rows)
 *         row = o_proj   shard r: input columns of its heads
 * Physically they are stored as 32 KB blocks of 256 rows x 64 input features
 * in the 128-byte-swizzled image the tensor cores read (gate_up: 128 gate +
 * the matching 128 up rows of one shard per block; row-parallel weights: K
 * running over shard 0, then shard 1, ...). Rows or K past the end are zero,
 * so the sizes are those of the padded block grid.
 */
int tp_packed_weight_bytes(const tp_config_t* cfg, int64_t* col_bytes, int64_t* row_bytes);

/*
 * Validate `cfg`, pack the unsharded weights into the shard layout above (on
 * `stream`) and return a handle. w_full: MLP {W_gate [I,H], W_up [I,H],
 * W_down [H,I]}, n_w = 3; ATTN {W_q [nq*hd,H], W_k [nkv*hd,H], W_v [nkv*hd,H],
 * W_o [H,nq*hd]}, n_w = 4. gamma: RMSNorm weight [H] bf16 (MLP with
 * TP_FLAG_HAS_NORM; ATTN with TP_FLAG_HAS_NORM: the layer's input_layernorm,
 * used by tp_decoder_layer_forward), else NULL. The handle borrows w_col_packed, w_row_packed
 * and gamma for its lifetime; w_full may be freed once `stream` has passed the
 * packing. The shard count follows divide(): a remainder is TP_ERR_SHAPE.
 */
int tp_linear_create(const tp_config_t* cfg, const void* const* w_full, int32_t n_w,
                     void* w_col_packed, void* w_row_packed, const void* gamma,
                     tp_stream_t stream, tp_linear_t** out);
int tp_linear_destroy(tp_linear_t* h);

/*
 * Workspace bytes a forward call with at most `max_tokens` tokens needs.
 * The workspace is caller-owned device memory that must be ZERO-FILLED before
 * its first use with a handle; afterwards the kernels leave it consistent
 * (split-K arrival counters reset themselves). Bytes [0, 4) are the device
 * status word: int32, 0 = ok, else a TP_ERR_* code written by a kernel
 * (sticky until the caller clears it). Holds the normalised input, the
 * shard-major intermediate h [t][T][I/t] and fp32 split-K partials.
 * One workspace must not be used by two calls that may run concurrently.
 */
int tp_workspace_size(const tp_linear_t* h, int64_t max_tokens, int64_t* bytes);

/*
 * MLP half of a decoder layer ("Tensor & pipeline parallelism": mlp_out,
 * residual_stream; "vLLM Code Reading (Section 5)" §14):
 *   with TP_FLAG_HAS_NORM: r = x_in + residual_in; x = RMSNorm(r) * gamma
 *   else:                  x = x_in;  r = residual_in (may be NULL)
 *   h_r = silu(x W_gate,r^T) * (x W_up,r^T)            (column-parallel, per shard)
 *   mlp_out = sum_r h_r W_down,r^T                      (row-parallel, reduced on chip)
 *   residual_stream = mlp_out + r                       (if residual_stream != NULL)
 * x_in, residual_in, residual_out, mlp_out, residual_stream: [T, H] bf16.
 * residual_out (required with norm, ignored without) receives r in bf16.
 */
int tp_mlp_forward(tp_linear_t* h, int64_t T, const void* x_in, const void* residual_in,
                   void* residual_out, void* mlp_out, void* residual_stream,
                   void* workspace, int64_t workspace_bytes, tp_stream_t stream);

/*
 * tp_mlp_forward for callers that cannot allocate device memory. The pages
 * have no counterpart: it is a service of this library, not a step of the
 * method. Some callers may not call cudaMalloc at all, or not at the moment
 * they run the block: plug-ins whose host hands them only memory it planned
 * ahead, runtimes whose own allocator owns all device memory, real-time loops
 * that forbid allocation after start-up. This entry point allocates nothing; it
 * runs the same fused decode-shaped block as tp_mlp_forward (same arguments,
 * same results) with its scratch in a fixed 16 MiB array inside the library
 * (each GPU that loads the library holds it until the process exits).
 *   - T <= 128 only, and only shapes whose scratch fits in 16 MiB; anything
 *     larger returns TP_ERR_UNSUPPORTED with the size in tp_last_error().
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is kept for the life of the process: it does not survive a
 *     device or context reset (cudaDeviceReset), after which this entry point
 *     must not be called.
 *   - Every call shares the one array, which keeps the last call's contents:
 *     calls that may overlap on the GPU (two streams, two handles) race and
 *     must be serialised by the caller. When the previous call on the device
 *     came from another handle (or this is the first), the call clears the
 *     counters first (a memset on `stream`, not an allocation); calls of one
 *     handle in a row need no clearing.
 *   - status_dev: optional device int32 the caller owns and zeroes; kernels
 *     write a TP_ERR_* code there on a device-side failure. NULL: errors go to a
 *     word of the shared array and are not reported to the caller.
 * Calls no cudaMalloc, cudaFree or other allocating routine.
 */
int tp_mlp_forward_no_alloc(tp_linear_t* h, int64_t T, const void* x_in, const void* residual_in,
                            void* residual_out, void* mlp_out, void* residual_stream,
                            int32_t* status_dev, tp_stream_t stream);

/*
 * The steps of tp_mlp_forward, one call each (same semantics, same kernels):
 *   tp_add_rms_norm : residual_out = a + residual_in (NULL: a); x_out = RMSNorm(residual_out) * gamma.
 *                     a, residual_in, residual_out, x_out [T, H]; gamma [H]. Any H % 8 == 0.
 *   tp_gate_up_forward: h_out [t][T][I/t] = silu(x W_gate,r^T) * (x W_up,r^T) per shard r.
 *   tp_down_forward : mlp_out = sum_r h_in[r] W_down,r^T; residual_stream = mlp_out + residual.
 */
int tp_add_rms_norm(int64_t T, int64_t H, const void* a, const void* residual_in, const void* gamma,
                    float eps, void* residual_out, void* x_out, tp_stream_t stream);
/*
 * Sequence parallelism ("Tensor Parallelism", collectives: reduce-scatter;
 * "Tensor & pipeline parallelism", residual_stream: the residual split across
 * the TP ranks by token): the reduce-scatter that ends a row-parallel layer
 * keeps rank r's rows [r*Tp/t, (r+1)*Tp/t) of the reduced output, Tp = T padded
 * up to a multiple of t. Here the reduction happens on chip and the scatter is
 * a view: give mlp_out / o_out a buffer of Tp rows whose last Tp - T rows are
 * zero and read it as [t][Tp/t][H]; rank r's slice is slice r.
 */
int tp_gate_up_forward(tp_linear_t* h, int64_t T, const void* x, void* h_out,
                       void* workspace, int64_t workspace_bytes, tp_stream_t stream);
int tp_down_forward(tp_linear_t* h, int64_t T, const void* h_in, const void* residual,
                    void* mlp_out, void* residual_stream,
                    void* workspace, int64_t workspace_bytes, tp_stream_t stream);

/*
 * Attention projections ("vLLM Code Reading (Section 5)" §13;
 * "Tensor & pipeline parallelism": attn_out):
 *   qkv_out [t][T][w_s] = per shard r: x [Wq_r; Wk_r; Wv_r]^T    (not gathered)
 *   o_out   [T, H]      = sum_r attn_in[r] Wo_r^T                 (reduced on chip)
 * x [T, H]; attn_in [t][T][nq*hd/t] (shard r's local heads). Either half may be
 * skipped by passing NULL for both of its pointers.
 */
int tp_attn_proj_forward(tp_linear_t* h, int64_t T, const void* x, void* qkv_out,
                         const void* attn_in, void* o_out,
                         void* workspace, int64_t workspace_bytes, tp_stream_t stream);

/*
 * Attention core between the two projections ("vLLM Code Reading (Section 5)"
 * §13: each rank runs attention on the heads it holds; "vLLM 源码完全拆解
 * （十一）" QkvParallelLinear: which kv head a shard holds under GQA):
 *   for every shard r and local q head i (global head h = r*nq/t + i):
 *     attn_out[r][:, i*hd:(i+1)*hd] = softmax(q_h k_g^T / sqrt(hd) + causal) v_g,
 *     g = the kv head of h's group (h / (nq/nkv)), held by shard r
 *   sequence s is tokens [cu_seqlens[s], cu_seqlens[s+1]); a query sees the keys of
 *   its own sequence at or before it. q and k are used as given (no positional
 *   rotation is applied).
 * qkv: [t][T][w_s] bf16, tp_attn_proj_forward's qkv_out. attn_out: [t][T][nq*hd/t]
 * bf16, the layout of tp_attn_proj_forward's attn_in. cu_seqlens: DEVICE int32
 * [n_seqs + 1], 0 = cu_seqlens[0] <= ... <= cu_seqlens[n_seqs] = T, 4-byte aligned.
 * n_seqs in [1, T]; max_seqlen (host) >= every sequence length, <= T. head_dim 128
 * (else TP_ERR_UNSUPPORTED). Scores and softmax in fp32, P rounded to bf16 for the
 * P V product, output rounded to bf16. Offsets that do not rise from 0 to T, or a
 * length above max_seqlen rounded up to 128, write TP_ERR_SHAPE to the workspace
 * status word and leave attn_out unwritten. The workspace (tp_workspace_size of the
 * handle covers up to max_tokens sequences) holds the per-call work table.
 */
int tp_attention_forward(tp_linear_t* h, int64_t T, const void* qkv, const int32_t* cu_seqlens,
                         int32_t n_seqs, int32_t max_seqlen, void* attn_out, void* workspace,
                         int64_t workspace_bytes, tp_stream_t stream);

/*
 * Paged KV cache ("vLLM Code Reading (Section 5)" §13: each rank's attention kernel
 * writes the KV cache of the heads it holds; the model runner's slot mapping comes
 * from the block table). Layout, per shard r: cache_k[r], cache_v[r] are
 * [num_blocks][block_size][kv_per][128] bf16 (kv_per = the shard's kv heads), so a
 * cache is t * num_blocks * block_size * kv_per * 128 elements; slot s is block
 * s / block_size, offset s % block_size.
 *
 * tp_kv_cache_write: for every token i of qkv ([t][T][w_s], or gathered) with
 *   slot_mapping[i] >= 0, copies the k and v heads of every shard into that slot.
 *   A slot past the cache writes TP_ERR_SHAPE to the status word (workspace bytes
 *   [0, 4); the workspace needs 16 bytes here) and is skipped; negative = padding.
 * tp_paged_attention: the new tokens of request b are rows [query_start_loc[b],
 *   query_start_loc[b+1]) of qkv and the last positions of its seq_lens[b] tokens;
 *   the token at position p attends (causally) to positions 0..p of its request,
 *   read from the cache through block_tables[b][p / block_size] (int32, row length
 *   max_blocks_per_req). The new tokens' k and v must be in the cache: either
 *   written before (tp_kv_cache_write), or written by this call when slot_mapping
 *   (int32 [T], device, may be null) is given: token i goes to slot_mapping[i] as
 *   tp_kv_cache_write would put it (negative = padding, past the cache =
 *   TP_ERR_SHAPE), by the attention kernel itself, before it reads that position.
 *   The slot of a new token must be the one its request's block table names for its
 *   position, and no other request of the call may read it. attn_out has the
 *   attention core's layout. Scores, softmax and the split merge in fp32, output
 *   rounded to bf16. Device arrays: query_start_loc [n_reqs + 1], seq_lens [n_reqs],
 *   block_tables [n_reqs][max_blocks_per_req], all int32. Host bounds: every request
 *   has at most max_query_len new tokens and max_seq_len tokens (else TP_ERR_SHAPE in
 *   the status word); block ids outside [0, num_blocks) likewise. The workspace
 *   (tp_paged_attention_workspace_size) holds the status word and the per-split
 *   partial results. head_dim 128; t * num_blocks * block_size < 2^31
 *   (TP_ERR_UNSUPPORTED otherwise). qkv, the caches and attn_out 16-byte aligned.
 */
int tp_kv_cache_write(tp_linear_t* h, int64_t T, const void* qkv, const int32_t* slot_mapping, void* cache_k,
                      void* cache_v, int64_t num_blocks, int32_t block_size, void* workspace,
                      int64_t workspace_bytes, tp_stream_t stream);
int tp_paged_attention_workspace_size(const tp_linear_t* h, int32_t n_reqs, int32_t max_query_len,
                                      int32_t max_seq_len, int64_t* bytes);
int tp_paged_attention(tp_linear_t* h, int64_t T, const void* qkv, const int32_t* query_start_loc,
                       const int32_t* seq_lens, int32_t n_reqs, int32_t max_query_len, int32_t max_seq_len,
                       const int32_t* block_tables, int32_t max_blocks_per_req, const int32_t* slot_mapping,
                       void* cache_k, void* cache_v, int64_t num_blocks, int32_t block_size, void* attn_out,
                       void* workspace, int64_t workspace_bytes, tp_stream_t stream);

/*
 * Mixture-of-experts block with within-expert tensor parallelism ("Tensor
 * Parallelism", MoE Expert Parallelism, Within-Expert Parallel: every expert's
 * FFN is split with the dense column-parallel gate/up and row-parallel down
 * pattern). A TP_BLOCK_MOE handle holds n_experts experts, created from
 * w_full = {W_gate_0, W_up_0, W_down_0, W_gate_1, ...} (n_w = 3 * n_experts,
 * shapes as for the MLP, I per expert); the packed buffers hold the experts one
 * after another. The routing is the caller's:
 *   y[i] = sum_{j < top_k} gates[i][j] * FFN_{expert_ids[i][j]}(x[i]),
 *   FFN_e(x) = sum_r h_r Wdown_e,r^T,  h_r = silu(x Wg_e,r^T) * (x Wu_e,r^T)
 * x, y: [T, H] bf16; expert_ids: int32 [T][top_k] in [0, n_experts); gates: fp32
 * [T][top_k] (both device, 4-byte aligned). The slots of a token are added in
 * order, in fp32, and y is rounded once. Rows go to experts by a stable sort, each
 * expert's rows padded to 128; every expert's h and output are rounded to bf16.
 * For an MoE handle, tp_workspace_size's max_tokens counts routed entries
 * (T * top_k). An id out of range writes TP_ERR_SHAPE to the status word and
 * y = 0. top_k in [1, n_experts] (else TP_ERR_SHAPE).
 */
int tp_moe_forward(tp_linear_t* h, int64_t T, int32_t top_k, const void* x, const int32_t* expert_ids,
                   const float* gates, void* y, void* workspace, int64_t workspace_bytes, tp_stream_t stream);

/*
 * One whole decoder layer, in the order "vLLM Code Reading (Section 5)" §13-§14
 * gives (QKV split by head, attention on each shard's heads, o_proj reduced, then
 * the MLP) with the fused add + norm of "Tensor & pipeline parallelism"
 * (residual_stream; the attn_out and mlp_out hook points):
 *   r1 = hidden_in + residual_in          (residual_in NULL: r1 = hidden_in, a first layer)
 *   x1 = RMSNorm(r1) * gamma_attn         (input_layernorm: the attention handle's gamma and eps)
 *   qkv = x1 [Wq_r; Wk_r; Wv_r]^T          (per shard, as tp_attn_proj_forward)
 *   A   = attention core                  (as tp_attention_forward, over cu_seqlens)
 *   attn_out = sum_r A_r Wo_r^T            (o_proj, reduced on chip)
 *   r2 = attn_out + r1; x2 = RMSNorm(r2) * gamma_mlp   (the MLP handle's norm)
 *   mlp_out = sum_r h_r Wdown_r^T, h_r = silu(x2 Wg_r^T) * (x2 Wu_r^T)
 *   residual_stream = mlp_out + r2        (if residual_stream != NULL)
 * Every intermediate is rounded to bf16, as between separate calls.
 *
 * tp_layer_create binds an attention handle and an MLP handle, both created with
 * TP_FLAG_HAS_NORM, of the same hidden size, on the current device, head_dim 128;
 * it borrows both for its lifetime (destroy the layer first). max_tokens fixes the
 * workspace layout: every call takes T <= max_tokens. The workspace
 * (tp_layer_workspace_size bytes, caller-owned, ZERO-FILLED before first use)
 * holds both halves' working storage and the intermediates x1, qkv and A; bytes
 * [0, 4) are the status word of every kernel of the layer (TP_ERR_SHAPE for bad
 * offsets, TP_ERR_TIMEOUT for a wait that gave up). Pointers in io: [T, H] bf16
 * device tensors, 16-byte aligned; cu_seqlens as for tp_attention_forward. All
 * host-side checks run before anything is enqueued.
 */
typedef struct tp_layer tp_layer_t;
typedef struct {
  const void* hidden_in;      /* [T, H] hidden states entering the layer */
  const void* residual_in;    /* [T, H] or NULL */
  const int32_t* cu_seqlens;  /* device int32 [n_seqs + 1] */
  int32_t n_seqs;
  int32_t max_seqlen;         /* host: >= every sequence length, <= T */
  void* residual_attn;        /* out r1 [T, H] */
  void* attn_out;             /* out [T, H] */
  void* residual_mlp;         /* out r2 [T, H] */
  void* mlp_out;              /* out [T, H] */
  void* residual_stream;      /* out [T, H] or NULL */
} tp_layer_io_t;

int tp_layer_create(tp_linear_t* attn, tp_linear_t* mlp, int64_t max_tokens, tp_layer_t** out);
int tp_layer_destroy(tp_layer_t* layer);
int tp_layer_workspace_size(const tp_layer_t* layer, int64_t* bytes);
int tp_decoder_layer_forward(tp_layer_t* layer, int64_t T, const tp_layer_io_t* io, void* workspace,
                             int64_t workspace_bytes, tp_stream_t stream);

/*
 * Activation capture ("Tensor & pipeline parallelism": What the adapter hooks,
 * Duplicate records across TP ranks, Merging records): records every row i of
 * each tensor whose key (row_req[i] << 32) | (uint32)row_pos[i] is among the
 * n_sel selector keys (any order; duplicates give one record; keys that match
 * no row give none). Records are grouped by tensor in the order given, rows
 * ascending within a tensor. Record j: hdr_out[j] = {request_id, token_pos,
 * tensor_type, layer, row, 0} and rows_out[j] = tensors[k][row] (H bf16,
 * bit-exact). *n_out_dev (device int64) receives the total number of records
 * n_tensors * n_match, even when it exceeds `capacity`; only records with
 * j < capacity are written, and TP_ERR_CAPACITY is written to the status word
 * (workspace bytes [0,4)) when it overflows. Call it after the reducing layer
 * has been enqueued: stream order makes it read the reduced tensors.
 * row_req, row_pos: [T] int32; sel_keys: [n_sel] int64; tensors: HOST array
 * of n_tensors device pointers to [T, H] bf16; tensor_types: HOST array.
 */
typedef struct {
  int32_t request_id, token_pos, tensor_type, layer, row, pad;
} tp_record_hdr_t;

int tp_capture_workspace_size(int64_t T, int64_t n_sel, int64_t* bytes);
int tp_capture_rows(int64_t T, int64_t H, const int32_t* row_req, const int32_t* row_pos,
                    const int64_t* sel_keys, int64_t n_sel, int32_t n_tensors,
                    const void* const* tensors, const int32_t* tensor_types, int32_t layer,
                    tp_record_hdr_t* hdr_out, void* rows_out, int64_t capacity,
                    int64_t* n_out_dev, void* workspace, int64_t workspace_bytes,
                    tp_stream_t stream);

/*
 * Wall-clock limit of every on-chip wait of the kernels launched after this
 * call (process-wide; default 2 s). Every wait between pipeline roles and
 * between CTAs is bounded: when one runs out, the kernel writes TP_ERR_TIMEOUT
 * to the status word, lets its copies in flight land, frees tensor memory and
 * returns, leaving the CUDA context usable (the workspace must then be zeroed
 * again). A short limit makes waits run out on purpose, which is how the
 * failure path is tested without faulting the GPU. ns <= 0 is TP_ERR_ARG.
 */
int tp_set_wait_timeout(int64_t ns);

/* Thread-local message describing the last non-zero return on this thread. */
const char* tp_last_error(void);

/*
 * Plan of the GEMM launches a forward call with T tokens would make, for
 * inspection and benchmarks: writes up to 2 entries of
 * {swap_ab, block_n, splits, units, grid, stages, engine} for the
 * column-parallel and the row-parallel GEMM. engine: 0 = one CTA per unit
 * (the other fields describe that launch), 1 = CTA pairs (two-SM MMAs over
 * 256-token x 256-row tiles, no split-K; an attention handle reports the
 * launch that runs QKV and o_proj together), 2 = the fused decode-shaped MLP
 * block (T <= 128, both GEMMs in one launch). The pair choice needs the
 * device: without one it reports engine 0. Returns the number written.
 */
typedef struct {
  int32_t swap_ab, block_n, splits, units, grid, stages, engine;
} tp_gemm_plan_t;
int tp_describe_plan(const tp_linear_t* h, int64_t T, tp_gemm_plan_t* plans, int32_t max_plans);

#ifdef __cplusplus
}
#endif
#endif /* TP_LINEAR_H */
