/*
 * tp.h -- C ABI of libtpshard.so: the Megatron tensor-parallel transformer
 * block with t logical shards resident on one GPU (sm_103a).
 *
 * The partition math follows the pages this library implements:
 *   - "02 — Tensor Parallelism" (project-fortress roadmap), sections
 *     "Column-parallel vs row-parallel — the derivation", "The MLP pairing",
 *     "The attention pairing", "Sequence parallelism (Megatron-3)";
 *   - "Tensor and sequence parallelism" (ai-infra handbooks), sections
 *     "How Megatron partitions" (the f / g operator table), "Sequence
 *     parallelism" and "The implementation";
 *   - "Tensor Parallelism's Communication Boundary" (aryanputta.com),
 *     sections "Follow the coordinates" and "Count the object, then the
 *     collective" (bias added once);
 *   - "Parallelism Strategies #1 - Tensor Parallelism" (substack), the
 *     sharded backward and the local weight-shard gradients;
 *   - "Megatron-LM: Tensor Parallelism" (vanos001), sections "Attention
 *     Block" and "MLP Block".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - tp_bf16 is the raw bit pattern of an IEEE bfloat16.  Accumulation is fp32.
 *  - Activations multiply weights from the left: Y = X W, W stored (in, out)
 *    in its UNPACKED form.  The t shards own contiguous, rank-ordered blocks
 *    C_i = [i*F/t, (i+1)*F/t) of the split dimension; t must divide it.
 *  - PACKED weights are per-shard slices stored (out, in), K contiguous:
 *      column-parallel W (h, F)  -> [t][F/t][h]      (tp_pack_col)
 *      row-parallel    W (F, h)  -> [t][h][F/t]      (tp_pack_row)
 *      SwiGLU gate/up  (h, F)    -> [t][F/t/128][2][128][h]   (tp_pack_swiglu)
 *      W_qkv (d, 3d) = [Q|K|V]   -> [t][3d/t][d] rows [Q_i|K_i|V_i] (tp_pack_qkv_heads)
 *      W_o (d, d), rows by head  -> [t][d][d/t]      (tp_pack_row)
 *    Weight gradients come back in the same packed layouts, in fp32.
 *  - Memory: every pointer is a DEVICE pointer owned by the caller (the
 *    library never allocates, never frees and keeps no pointer after a call
 *    returns).  Pointers must be 16-byte aligned (else TP_ERR_ALIGN); the
 *    innermost dimension of every matrix must be a multiple of 8 elements.
 *  - Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and the call returns without synchronising.  Argument
 *    errors are detected on the host before anything is launched and leave
 *    outputs untouched.  Device-side errors (a bounded wait that expired) are
 *    recorded in a per-device error word that tp_get_device_status() reads.
 *  - Workspace: entry points that need scratch take (ws, ws_bytes); the
 *    matching *_workspace_size() gives the minimum.  Too small -> TP_ERR_WORKSPACE.
 *  - Thread safety: calls on different streams may run concurrently; they
 *    share only the device error word.
 *  - Environment variables (for tuning and tests; none is needed):
 *      TP_WAIT_TIMEOUT_MS  limit of every bounded wait inside a kernel, 1..60000 ms
 *                          (default 2000; read once per process);
 *      TP_GEMM_PAIR=0      single-CTA GEMM kernel instead of the CTA-pair kernel;
 *      TP_SPLITK=S         K ranges per tile of the M <= 128 cluster split (1 = none);
 *      TP_SPLITC_NARROW=0|1  256- or 128-column tiles of that split (default: by size);
 *      TP_STREAMK=0        no split K across CTA pairs even with a workspace;
 *      TP_SPLIT_CHAIN=0    split K across CTA pairs by counted ranges only.
 *    All but the first are read at each call.
 */
#ifndef TPSHARD_TP_H
#define TPSHARD_TP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TP_ABI_VERSION 1

typedef enum {
  TP_OK = 0,
  TP_ERR_INVALID_ARG = 1, /* null required pointer, bad enum, t < 1, negative size */
  TP_ERR_SHAPE = 2,       /* t does not divide the split dim, unsupported size */
  TP_ERR_ALIGN = 3,       /* pointer not 16-byte aligned, row length not a multiple of 8 */
  TP_ERR_WORKSPACE = 4,   /* ws_bytes smaller than the *_workspace_size() result */
  TP_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
  TP_ERR_TIMEOUT = 6,     /* device: a bounded wait inside a kernel expired */
  TP_ERR_UNSUPPORTED = 7  /* no sm_103a device, or a combination not built */
} tp_status;

typedef enum {
  TP_ACT_IDENTITY = 0,
  TP_ACT_RELU = 1,
  TP_ACT_GELU_TANH = 2, /* 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))) */
  TP_ACT_GELU_ERF = 3,  /* 0.5 z (1 + erf(z / sqrt 2)) */
  TP_ACT_SWIGLU = 4     /* silu(X W_gate) * (X W_up); tp_mlp_forward / tp_mlp_backward and the decode
                           entry point (not tp_column_parallel_forward) */
} tp_act;

/* Flags for tp_mlp_forward / tp_mlp_backward. */
#define TP_FLAG_UNFUSED_REDUCE 1u /* materialise the t partial sums P_i (fp32, in ws) and
                                     reduce them in a separate kernel instead of in the
                                     row-parallel GEMM's accumulator */
#define TP_FLAG_OVERLAP_REDUCE 2u /* materialise the P_i tile by tile and reduce every
                                     finished tile while later tiles compute, inside the
                                     row-parallel GEMM (tp_row_parallel_forward_overlap);
                                     M > 128, t <= 8; takes precedence over UNFUSED */

/* Flag of the attention entry points (tp_attn_forward / backward and their grouped-query
 * forms): the attention input X and the packed W_qkv hold IEEE fp16 bits instead of bf16
 * (tp_sp_layernorm_forward_f16 and tp_convert_bf16_to_f16 produce them), and the backward
 * keeps dQKV in fp16 too.  A wide model's attention logits spread over several units (about
 * 5 at d = 12288 with N(0, 0.02) weights), so the 2^-9 rounding of a bf16 X becomes a
 * logit error of a few hundredths and a relative error of the softmax of a few percent;
 * fp16 keeps 3 more mantissa bits at the same cost. */
#define TP_ATTN_F16_INPUT 1u

typedef uint16_t tp_bf16;
typedef struct CUstream_st* tp_stream; /* identical to cudaStream_t */

/* ------------------------------------------------------------------ misc */
int tp_abi_version(void);
const char* tp_status_string(tp_status s);

/* Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns TP_OK, TP_ERR_TIMEOUT (a bounded wait expired), TP_ERR_SHAPE
 * (a kernel found an argument that lives in device memory out of range, e.g.
 * a decode position >= L_max or a token id >= V), or TP_ERR_CUDA if the
 * synchronisation itself failed. */
tp_status tp_get_device_status(tp_stream stream);

/* Fault-path self test: launches one CTA that waits on an mbarrier nothing
 * will ever complete, with a limit of `timeout_us` microseconds (1..10^7).
 * The wait gives up, records TP_ERR_TIMEOUT in the error word and the kernel
 * returns normally; the context stays usable.  tp_get_device_status() then
 * reports TP_ERR_TIMEOUT. */
tp_status tp_selftest_bounded_wait(int64_t timeout_us, tp_stream stream);

/* Where the most recent TP_ERR_CUDA returned on this thread came from:
 * "file:line: cudaErrorName (description)" or a tensor-map failure; "" if
 * none.  The string belongs to the library and stays valid until this
 * thread's next failing call. */
const char* tp_last_error_detail(void);

/* Number of CUDA kernels this library has enqueued in this process so far
 * (all devices, all streams).  Host-side counter; never synchronises. */
uint64_t tp_kernel_launch_count(void);

/* -------------------------------------------------------------- packing
 * Bit-exact permutations of bf16 weights into the per-shard layouts listed
 * above ("Tensor and sequence parallelism", section "The implementation":
 * each rank keeps w1[cols] and w2[:, cols]; "02 — Tensor Parallelism",
 * section "The attention pairing": each rank owns n_heads/t heads of Q, K, V).
 * Src and dst must not overlap.  The unpack_* calls are exact inverses, so a
 * checkpoint sharded t ways is re-sharded t' ways as unpack(t) then pack(t'). */
tp_status tp_pack_col(const tp_bf16* W, int64_t h, int64_t F, int t, tp_bf16* Wp, tp_stream stream);
tp_status tp_unpack_col(const tp_bf16* Wp, int64_t h, int64_t F, int t, tp_bf16* W, tp_stream stream);
tp_status tp_pack_row(const tp_bf16* W, int64_t F, int64_t h, int t, tp_bf16* Wp, tp_stream stream);
tp_status tp_unpack_row(const tp_bf16* Wp, int64_t F, int64_t h, int t, tp_bf16* W, tp_stream stream);
/* Wg, Wu: (h, F); (F/t) % 128 == 0. */
tp_status tp_pack_swiglu(const tp_bf16* Wg, const tp_bf16* Wu, int64_t h, int64_t F, int t, tp_bf16* Wp,
                         tp_stream stream);
/* Wqkv: (d, 3d), columns [Q|K|V], head j at columns j*head_dim of each block.
 * n_heads*head_dim == d, t | n_heads, head_dim % 8 == 0. */
tp_status tp_pack_qkv_heads(const tp_bf16* Wqkv, int64_t d, int n_heads, int head_dim, int t, tp_bf16* Wp,
                            tp_stream stream);
tp_status tp_unpack_qkv_heads(const tp_bf16* Wp, int64_t d, int n_heads, int head_dim, int t, tp_bf16* Wqkv,
                              tp_stream stream);
/* b: (3d) -> [t][3d/t] in the same head order. */
tp_status tp_pack_qkv_bias(const tp_bf16* b, int64_t d, int n_heads, int head_dim, int t, tp_bf16* bp,
                           tp_stream stream);

/* Grouped-query attention ("02 — Tensor Parallelism", "The attention
 * pairing": with GQA/MQA the heads shard by KV group; "Tensor and sequence
 * parallelism", exercise 1: with fewer KV heads than shards each KV head is
 * replicated on t/n_kv shards).
 * Wqkv: (d, (n_heads + 2 n_kv) * head_dim), columns [Q heads | K heads | V
 * heads]; query head j reads KV head j / (n_heads / n_kv).
 * Packed: [t][R][d], R = (n_heads/t + 2 kv_t) * head_dim, rows [shard i's Q
 * heads | its kv_t K heads | its kv_t V heads], kv_t = n_kv/t when n_kv >= t
 * (the groups of its query heads), else 1 (KV head i*n_kv/t, a copy).
 * Requires t | n_heads, n_kv | n_heads, and n_kv % t == 0 or t % n_kv == 0.
 * Unpack writes every copy of a replicated column (the same bits). */
tp_status tp_pack_qkv_gqa(const tp_bf16* Wqkv, int64_t d, int n_heads, int n_kv_heads, int head_dim, int t,
                          tp_bf16* Wp, tp_stream stream);
tp_status tp_unpack_qkv_gqa(const tp_bf16* Wp, int64_t d, int n_heads, int n_kv_heads, int head_dim, int t,
                            tp_bf16* Wqkv, tp_stream stream);
/* b: ((n_heads + 2 n_kv) * head_dim) -> [t][R] in the same order. */
tp_status tp_pack_qkv_gqa_bias(const tp_bf16* b, int n_heads, int n_kv_heads, int head_dim, int t, tp_bf16* bp,
                               tp_stream stream);

/* ------------------------------------------- column / row parallel linear
 * The two halves of the pairing, each ONE kernel launch ("02 — Tensor
 * Parallelism", "Column-parallel" and "Row-parallel"):
 *
 * Column-parallel (W split along its output dim; f forward = identity, X read
 * by every shard): Z_i = X W_i + b[C_i];  A_i = act(Z_i).
 *   X [M][h]; W_p [t][N/t][h] (tp_pack_col of W (h, N)); b [N] nullable;
 *   Z [t][M][N/t] nullable; A [t][M][N/t] required.  h, N/t multiples of 8. */
tp_status tp_column_parallel_forward(const tp_bf16* X, int64_t M, int64_t h, int64_t N, int t, tp_act act,
                                     const tp_bf16* W_p, const tp_bf16* b, tp_bf16* Z, tp_bf16* A,
                                     tp_stream stream);

/* Row-parallel (W split along its input dim) followed by g: the t partial
 * products of the sharded input are summed in shard order inside the GEMM's
 * accumulator, then the bias is added once and the residual after it:
 *   Y = sum_{i=0..t-1} A_i W_i + b + residual.
 *   A [t][M][K/t]; W_p [t][h][K/t] (tp_pack_row of W (K, h)); b [h] nullable;
 *   residual [M][h] nullable; Y [M][h].  h, K/t multiples of 8. */
tp_status tp_row_parallel_forward(const tp_bf16* A, int64_t M, int64_t K, int64_t h, int t, const tp_bf16* W_p,
                                  const tp_bf16* b, const tp_bf16* residual, tp_bf16* Y, tp_stream stream);
/* Few tokens (M <= 128, a single 128-row output tile) leave most SMs idle: there, these
 * two calls, the MLP and the attention blocks split each output tile's K steps -- for the
 * row-parallel GEMM the t shards' K ranges laid end to end -- over the 2..16 CTAs of a
 * thread-block cluster, which sum their fp32 partials on chip (distributed shared memory)
 * in range order before the epilogue; output tiles are 128 columns wide when 256-column
 * tiles would keep under a quarter of the SMs busy.  No workspace is needed and the result
 * does not depend on timing; only the rounding of the fp32 sum differs from the unsplit
 * GEMM. */

/* The same two calls with a workspace (tp_*_workspace_size() bytes, 256-byte aligned; a
 * smaller one is used as far as it goes, NULL runs the calls above).  It lets a GEMM of
 * more than 128 rows split K where its 256 x 256 output tiles do not fill the GPU's CTA
 * pairs evenly: the full rounds of whole tiles stay whole, and the remaining tiles (all of
 * them, when they are fewer than the pairs) are cut into S equal ranges of k-steps (a
 * row-parallel GEMM's t shard ranges laid end to end) at the same cut points for every
 * tile, dealt to all pairs -- S is chosen by a time model to finish first, and no cut is
 * made when it would save too little.  bf16 outputs (the row-parallel GEMM, the f-reduced
 * dX) chain their ranges when at most half a round of tiles is split: range 0 stores its
 * fp32 partial into the tile's running sum in ws, each next range adds into it after the
 * previous range's flag (a bounded wait on a range dealt earlier), and the last range adds
 * its accumulator and applies the epilogue.  The other outputs count their ranges: every
 * range leaves its fp32 partial in ws and counts itself; the range that completes a tile's
 * count adds the tile's partials in range order and applies the epilogue.  Either way the
 * sums run in range order, so they are deterministic for a given device (the plan depends
 * on its SM count) and only the rounding of the fp32 sum differs from the data-parallel
 * schedule.  Flags and counters reset themselves (CUDA-graph replay is fine; any initial
 * contents are).  The MLP and attention calls take the same room at the end of their
 * workspaces.  Workspaces must not be shared by calls that may run at the same time. */
size_t tp_column_parallel_workspace_size(int64_t M, int64_t h, int64_t N, int t);
tp_status tp_column_parallel_forward_ws(const tp_bf16* X, int64_t M, int64_t h, int64_t N, int t, tp_act act,
                                        const tp_bf16* W_p, const tp_bf16* b, tp_bf16* Z, tp_bf16* A, void* ws,
                                        size_t ws_bytes, tp_stream stream);
size_t tp_row_parallel_workspace_size(int64_t M, int64_t K, int64_t h, int t);
tp_status tp_row_parallel_forward_ws(const tp_bf16* A, int64_t M, int64_t K, int64_t h, int t, const tp_bf16* W_p,
                                     const tp_bf16* b, const tp_bf16* residual, tp_bf16* Y, void* ws,
                                     size_t ws_bytes, tp_stream stream);

/* Row-parallel GEMM with the g all-reduce overlapped, tile by tile ("Tensor
 * and sequence parallelism", section "Volume and scale": the matrix multiply is
 * cut into blocks and each block is communicated while the next computes --
 * Megatron's tp-comm-overlap).  Every shard's partial P_i = A_i W_i is written
 * tile by tile to an explicit fp32 buffer in ws (the data a multi-GPU run would
 * send): each 256 x 256 output tile's t shard products are separate work items.
 * The CTA pairs' full rounds walk a tile's shards one after another (so the
 * operand panels of one shard are shared by all pairs, as in the fused GEMM), the
 * remaining tiles' shards are dealt to all pairs, and the item that completes a
 * tile's set of t (per 32-row block) sums its partials in shard order, adds b once
 * and the residual after it, and writes that block of Y -- while the tensor cores
 * go on with the next tiles.  Same bits as TP_FLAG_UNFUSED_REDUCE.
 *   A [t][M][K/t]; W_p [t][h][K/t]; b [h], residual [M][h] nullable; Y [M][h] bf16;
 *   partials_out [t][M][h] fp32 (nullable: receives a copy of the exchanged
 *   partials after the call);
 *   ws: tp_row_parallel_overlap_workspace_size() bytes, 256-byte aligned: the
 *   partials [t][M][h] fp32, then 64 bytes of counters per output tile (any initial
 *   contents; they reset themselves).
 *   M > 128 (TP_ERR_UNSUPPORTED otherwise), 1 <= t <= 8 (t > 8: TP_ERR_SHAPE),
 *   h and K/t multiples of 8. */
size_t tp_row_parallel_overlap_workspace_size(int64_t M, int64_t K, int64_t h, int t);
tp_status tp_row_parallel_forward_overlap(const tp_bf16* A, int64_t M, int64_t K, int64_t h, int t,
                                          const tp_bf16* W_p, const tp_bf16* b, const tp_bf16* residual, tp_bf16* Y,
                                          float* partials_out, void* ws, size_t ws_bytes, tp_stream stream);

/* -------------------------------------------------------------- TP MLP
 * Forward ("02 — Tensor Parallelism", "The MLP pairing"; "Tensor and
 * sequence parallelism", f/g table):
 *   f forward (identity): every shard reads the same X [M][h].
 *   shard i: Z_i = X W_up,i + b_up[C_i];  A_i = act(Z_i)            (column-parallel)
 *            P_i = A_i W_down,i                                      (row-parallel)
 *   g forward (all-reduce): Y = sum_{i=0..t-1} P_i + b_down (+ residual), bias ONCE.
 * On one GPU the all-reduce is fused: the row-parallel GEMM accumulates the
 * shards' K ranges one after another into a single fp32 accumulator, i = 0..t-1
 * in order, and adds b_down once in its epilogue.  With TP_FLAG_UNFUSED_REDUCE
 * the t partials are written to ws ([t][M][h] fp32) and summed by a separate
 * fixed-order reduction kernel; with TP_FLAG_OVERLAP_REDUCE the partials are
 * reduced tile by tile while the GEMM runs (see tp_row_parallel_forward_overlap).
 *   X [M][h]; Wup_p [t][F/t][h]; bup [F] (nullable); Wdown_p [t][h][F/t];
 *   bdown [h] (nullable); residual [M][h] (nullable, added after the sum);
 *   Y [M][h]; Z_save [t][M][F/t] (nullable: inference); A_save [t][M][F/t] (required).
 * act: IDENTITY, RELU, GELU_TANH, GELU_ERF or SWIGLU.  h % 8 == 0, (F/t) % 8 == 0.
 * SWIGLU ("02 — Tensor Parallelism", "The core observation": the up-projection
 * is twice as wide; gate and up split by the same C_i, so the product is local):
 *   Wup_p is tp_pack_swiglu's [t][2F/t][h] (gate and up rows in alternating groups
 *   of 128); Z_i = X [W_gate | W_up]_i is saved in the same interleaved order,
 *   Z_save [t][M][2F/t] (required); A_i = silu(gate) * up [t][M][F/t], formed in the
 *   GEMM's epilogue from the fp32 accumulators.  bup must be NULL (TP_ERR_UNSUPPORTED
 *   otherwise); (F/t) % 128 == 0 (TP_ERR_SHAPE).
 * ws: tp_mlp_workspace_size() bytes: the two flags' partials (required with them; NULL,
 * 0 otherwise), then room for the GEMMs' split-K partials (see
 * tp_row_parallel_forward_ws), used when present. */
size_t tp_mlp_workspace_size(int64_t M, int64_t h, int64_t F, int t, unsigned flags);
tp_status tp_mlp_forward(const tp_bf16* X, int64_t M, int64_t h, int64_t F, int t, tp_act act,
                         const tp_bf16* Wup_p, const tp_bf16* bup, const tp_bf16* Wdown_p, const tp_bf16* bdown,
                         const tp_bf16* residual, tp_bf16* Y, tp_bf16* Z_save, tp_bf16* A_save, unsigned flags,
                         void* ws, size_t ws_bytes, tp_stream stream);

/* Backward of L = <Y, dY> ("Parallelism Strategies #1 - Tensor Parallelism",
 * sharded backward; "Tensor and sequence parallelism", f/g table):
 *   g backward (identity): every shard receives dY unchanged; db_down = sum_rows dY once.
 *   shard i: dZ_i = (dY W_down,i^T) * act'(Z_i);  db_up[C_i] = sum_rows dZ_i
 *            dW_down,i = A_i^T dY;  dW_up,i = dZ_i^T X      (local, no reduction)
 *   f backward (all-reduce): dX = sum_{i=0..t-1} dZ_i W_up,i^T (fused as in the forward).
 * Outputs: dX [M][h] bf16; dWup_p [t][F/t][h] and dWdown_p [t][h][F/t] fp32
 * (overwritten, or added to when `accumulate` != 0); dbup [F], dbdown [h] fp32
 * (nullable).  SWIGLU: dA_i = dY W_down,i^T stays in the GEMM's fp32 accumulators; its
 * epilogue writes d gate = dA u silu'(gate) and d up = dA silu(gate), interleaved like
 * Z_save; dWup_p is [t][2F/t][h] in tp_pack_swiglu's layout; dbup must be NULL.  ws (the
 * size query covers every activation) holds dZ and column-sum scratch -- the required
 * part -- then room for the GEMMs' split-K partials, used when present. */
size_t tp_mlp_backward_workspace_size(int64_t M, int64_t h, int64_t F, int t, unsigned flags);
tp_status tp_mlp_backward(const tp_bf16* dY, const tp_bf16* X, const tp_bf16* Z_save, const tp_bf16* A_save,
                          int64_t M, int64_t h, int64_t F, int t, tp_act act, const tp_bf16* Wup_p,
                          const tp_bf16* Wdown_p, tp_bf16* dX, float* dWup_p, float* dWdown_p, float* dbup,
                          float* dbdown, int accumulate, unsigned flags, void* ws, size_t ws_bytes,
                          tp_stream stream);

/* -------------------------------------------------------- decode SwiGLU
 * Memory-bound decode step of a SwiGLU MLP ("02 — Tensor Parallelism",
 * "The core observation" (times 2 for SwiGLU) and "When to use TP": decode is
 * bandwidth-bound):
 *   shard i: a_i = silu(x W_gate,i) * (x W_up,i);   y = sum_{i=0..t-1} a_i W_down,i.
 * x [M][h] with 1 <= M <= 8; Wgu_p from tp_pack_swiglu; Wdown_p from
 * tp_pack_row; y [M][h]; a_save [M][F] bf16 (required: shard i's hidden
 * vector at columns C_i; the down projection reads it).  No biases. */
tp_status tp_decode_swiglu_forward(const tp_bf16* x, int64_t M, int64_t h, int64_t F, int t,
                                   const tp_bf16* Wgu_p, const tp_bf16* Wdown_p, tp_bf16* y, tp_bf16* a_save,
                                   tp_stream stream);

/* ------------------------------------ decode attention, sharded KV cache
 * One decode step of the attention block for B sequences ("02 — Tensor
 * Parallelism", "The critical inference-time subtlety: KV cache also shards":
 * each shard holds the KV heads of its own query heads, so the cache splits
 * with the heads; "The count: two all-reduces per block per direction": the
 * block ends in one all-reduce of B x d elements per token):
 *   shard i: qkv_i = x W_qkv,i + b_qkv,i                 (column-parallel GEMV)
 *            K_cache[i][jl][b][pos[b]] = k, V_cache[...] = v  (append, fp16)
 *            per query head: o = softmax(scale q K[0..pos[b]]^T) V[0..pos[b]]
 *   g:       y = sum_{i=0..t-1} O_i W_o,i + b_o          (fixed order, bias once)
 * x [B][d] bf16, 1 <= B <= 256; Wqkv_p / bqkv_p from tp_pack_qkv_gqa(_bias)
 * (bqkv_p nullable); Wo_p [t][d][n_heads*head_dim/t] from tp_pack_row of W_o
 * (n_heads*head_dim, d); bo [d] nullable; y [B][d] bf16.
 * K_cache, V_cache: IEEE fp16 bits, [t][kv_t][B][L_max][head_dim] (kv_t as for
 * tp_pack_qkv_gqa); a replicated KV head has one copy per shard that holds
 * it.  Positions 0..pos[b]-1 must hold the sequence's earlier keys/values;
 * the call writes position pos[b] and attends to keys 0..pos[b].  Bytes past
 * pos[b] are never used (they may hold anything, even non-finite values).
 * pos: DEVICE int32 [B], 0 <= pos[b] < L_max; a position out of range is
 * clamped, its cache write skipped, and tp_get_device_status() reports
 * TP_ERR_SHAPE.  head_dim == 128; query heads per KV group on one shard
 * (min(n_heads/n_kv, n_heads/t)) <= 32.  ws: 256-byte aligned,
 * tp_decode_attn_workspace_size() bytes (Q, the tile plan, split-KV partials
 * and O); the call allocates nothing.  Four to five kernels: the QKV GEMV
 * (per group of 8 sequences), the split-KV attention, the combine, and the
 * W_o GEMV (per group of 8 sequences). */
size_t tp_decode_attn_workspace_size(int64_t B, int64_t d, int n_heads, int n_kv_heads, int head_dim, int t,
                                     int64_t L_max);
tp_status tp_decode_attn_forward(const tp_bf16* x, int64_t B, int64_t d, int n_heads, int n_kv_heads, int head_dim,
                                 int t, float scale, const tp_bf16* Wqkv_p, const tp_bf16* bqkv_p,
                                 const tp_bf16* Wo_p, const tp_bf16* bo, uint16_t* K_cache, uint16_t* V_cache,
                                 int64_t L_max, const int32_t* pos, tp_bf16* y, void* ws, size_t ws_bytes,
                                 tp_stream stream);

/* -------------------------------------------------- head-sharded attention
 * ("02 — Tensor Parallelism", "The attention pairing"; "Megatron-LM: Tensor
 * Parallelism", "Attention Block"):
 *   shard i: QKV_i = X W_qkv,i + b_qkv,i   -> [N][3d/t] = [Q_i|K_i|V_i]
 *            per local head: S = scale Q K^T, causal mask (key > query), P = softmax(S), O = P V
 *            O_i = local heads side by side [N][d/t];   partial Y_i = O_i W_o,i
 *   g: Y = sum_i Y_i + b_o (+ residual), bias once.
 * X [N][d] (already normalised); Wqkv_p [t][3d/t][d]; bqkv_p [t][3d/t]
 * (nullable); Wo_p [t][d][d/t]; bo [d] (nullable); residual [N][d] (nullable);
 * Y [N][d]; QKV_save [t][N][3d/t] holds IEEE fp16 bits (not bf16: with
 * logits spread over several units, fp16's 3 extra mantissa bits keep the
 * softmax of wide models within tolerance); O_save
 * [t][N][d/t] bf16; lse_save [t][H/t][N] fp32 (natural-log log-sum-exp of
 * each scaled score row).  head_dim == 128.
 * flags: 0 or TP_ATTN_F16_INPUT (X and Wqkv_p in IEEE fp16; other bits: TP_ERR_UNSUPPORTED).
 * ws is optional: NULL, 0 runs
 * the GEMMs' data-parallel schedule; tp_attn_forward_workspace_size() bytes (256-byte
 * aligned) let them split K (see tp_row_parallel_forward_ws).  The attention
 * kernel runs one CTA per (head, pair of 128-query tiles) with an online softmax; no
 * N x N score matrix is ever stored. */
size_t tp_attn_forward_workspace_size(int64_t N, int64_t d, int n_heads, int head_dim, int t, unsigned flags);
tp_status tp_attn_forward(const tp_bf16* X, int64_t N, int64_t d, int n_heads, int head_dim, int t, int causal,
                          float scale, const tp_bf16* Wqkv_p, const tp_bf16* bqkv_p, const tp_bf16* Wo_p,
                          const tp_bf16* bo, const tp_bf16* residual, tp_bf16* Y, tp_bf16* QKV_save,
                          tp_bf16* O_save, float* lse_save, unsigned flags, void* ws, size_t ws_bytes,
                          tp_stream stream);

/* Grouped-query form of tp_attn_forward ("02 — Tensor Parallelism", "The
 * attention pairing": GQA/MQA shard by KV group; "Tensor and sequence
 * parallelism", exercise 1: fewer KV heads than shards -> replicated KV heads).
 * Wqkv_p / bqkv_p from tp_pack_qkv_gqa(_bias); QKV_save [t][N][R] IEEE fp16 with
 * R = (n_heads/t + 2 kv_t) * head_dim (rows [Q heads | K heads | V heads] of the
 * shard); query head j of a shard reads the shard's KV head j / min(n_heads/n_kv,
 * n_heads/t).  Everything else as tp_attn_forward (which is this call with
 * n_kv_heads = n_heads). */
tp_status tp_attn_gqa_forward(const tp_bf16* X, int64_t N, int64_t d, int n_heads, int n_kv_heads, int head_dim,
                              int t, int causal, float scale, const tp_bf16* Wqkv_p, const tp_bf16* bqkv_p,
                              const tp_bf16* Wo_p, const tp_bf16* bo, const tp_bf16* residual, tp_bf16* Y,
                              uint16_t* QKV_save, tp_bf16* O_save, float* lse_save, unsigned flags, void* ws,
                              size_t ws_bytes, tp_stream stream);

/* Backward of L = <Y, dY>: g backward identity; per shard dO_i = dY W_o,i^T,
 * head-local softmax backward, dQKV_i; dW_o,i = O_i^T dY; dW_qkv,i = dQKV_i^T X;
 * f backward: dX = sum_i dQKV_i W_qkv,i^T (fused).  dWqkv_p [t][3d/t][d],
 * dbqkv_p [t][3d/t], dWo_p [t][d][d/t], dbo [d]: fp32 (overwritten, or added to when
 * accumulate != 0; dbqkv_p / dbo nullable).  Inputs are the forward's saved
 * QKV_save, O_save, lse_save.  flags: 0, or TP_ATTN_F16_INPUT when the forward had it (X and
 * Wqkv_p fp16; dQKV in ws is then fp16).  ws (see the size query) holds,
 * in order, each 256-byte aligned: dO [t][N][d/t] fp16, D = rowsum(dO * O)
 * [t][H/t][N] fp32, dQKV [t][N][3d/t] bf16, column-sum scratch -- the required part
 * (TP_ERR_WORKSPACE below it) -- then room for the GEMMs' split-K partials, used
 * when present.  The
 * attention gradient runs as two deterministic kernels (dK/dV per key block,
 * dQ per query block); scores are recomputed from the saved log-sum-exp. */
size_t tp_attn_backward_workspace_size(int64_t N, int64_t d, int n_heads, int head_dim, int t, unsigned flags);
tp_status tp_attn_backward(const tp_bf16* dY, const tp_bf16* X, const tp_bf16* QKV_save, const tp_bf16* O_save,
                           const float* lse_save, int64_t N, int64_t d, int n_heads, int head_dim, int t,
                           int causal, float scale, const tp_bf16* Wqkv_p, const tp_bf16* Wo_p, tp_bf16* dX,
                           float* dWqkv_p, float* dbqkv_p, float* dWo_p, float* dbo, int accumulate,
                           unsigned flags, void* ws, size_t ws_bytes, tp_stream stream);

/* Grouped-query backward: as tp_attn_backward with the layouts of
 * tp_attn_gqa_forward.  A KV head's dK / dV sum over the query heads of its
 * group on the shard; dWqkv_p [t][R][d] and dbqkv_p [t][R] hold each shard's
 * gradient for its own copy of the columns (a replicated KV head has t/n_kv
 * copies); tp_reduce_qkv_gqa_grad sums them into the unsplit gradient.
 * ws: tp_attn_gqa_backward_workspace_size() bytes (dO, D, dQKV [t][N][R] bf16,
 * column-sum scratch). */
size_t tp_attn_gqa_backward_workspace_size(int64_t N, int64_t d, int n_heads, int n_kv_heads, int head_dim, int t,
                                           unsigned flags);
tp_status tp_attn_gqa_backward(const tp_bf16* dY, const tp_bf16* X, const uint16_t* QKV_save, const tp_bf16* O_save,
                               const float* lse_save, int64_t N, int64_t d, int n_heads, int n_kv_heads,
                               int head_dim, int t, int causal, float scale, const tp_bf16* Wqkv_p,
                               const tp_bf16* Wo_p, tp_bf16* dX, float* dWqkv_p, float* dbqkv_p, float* dWo_p,
                               float* dbo, int accumulate, unsigned flags, void* ws, size_t ws_bytes,
                               tp_stream stream);

/* The head-local attention core alone, between the two projections ("02 —
 * Tensor Parallelism", "The attention pairing": each shard's heads run with no
 * communication).  For callers that form QKV themselves, and for timing the
 * kernels on their own.
 * Forward: QKV [t][N][R] IEEE fp16 in the layout of tp_attn_gqa_forward's
 * QKV_save (R = (n_heads/t + 2 kv_t) * head_dim); writes O [t][N][d/t] bf16 and
 * lse [t][n_heads/t][N] fp32 (natural log).  One kernel launch.
 * Backward: dO [t][N][d/t] IEEE fp16, O and lse from the forward; Dvec
 * [t][n_heads/t][N] fp32 is caller-owned scratch (receives rowsum(dO * O));
 * writes dQKV [t][N][R] bf16 (every element: dQ, dK and dV of each head).
 * Three launches: the row dot product, dK/dV per key block, dQ per query block.
 * Pointers 16-byte aligned (TP_ERR_ALIGN); shape rules of tp_attn_gqa_forward
 * (TP_ERR_SHAPE); N == 0 is a no-op.  Asynchronous on `stream`. */
tp_status tp_attn_core_forward(const uint16_t* QKV, int64_t N, int64_t d, int n_heads, int n_kv_heads, int head_dim,
                               int t, int causal, float scale, tp_bf16* O, float* lse, tp_stream stream);
tp_status tp_attn_core_backward(const uint16_t* QKV, const tp_bf16* O, const uint16_t* dO, const float* lse,
                                int64_t N, int64_t d, int n_heads, int n_kv_heads, int head_dim, int t, int causal,
                                float scale, float* Dvec, tp_bf16* dQKV, tp_stream stream);

/* The replica-group reduction of grouped-query weight gradients: dW (d,
 * (n_heads + 2 n_kv) head_dim) fp32, unsplit layout, gets for every column the
 * sum, in shard order, of the packed gradients dWp [t][R][d] (fp32) of all shard
 * copies holding it -- one copy for query columns and when n_kv >= t, t/n_kv
 * copies for a replicated KV head's columns (the copies' gradients must be
 * summed, as the LayerNorm weights shared by sequence shards are).  accumulate
 * != 0 adds to dW.  Src and dst must not overlap. */
tp_status tp_reduce_qkv_gqa_grad(const float* dWp, int64_t d, int n_heads, int n_kv_heads, int head_dim, int t,
                                 float* dW, int accumulate, tp_stream stream);

/* --------------------------------------------- vocab-parallel embedding
 * ("Megatron-LM: Tensor Parallelism", "Common Pitfalls" item 5: the embedding
 * lookup is sharded by vocabulary.)  Shard i owns rows [i V/t, (i+1) V/t) of
 * E (V, h); the packed table E_p [t][V/t][h] bf16 is E's own row-major layout.
 * Forward: f hands every shard all ids; shard i's partial is E_p[i][id - i V/t]
 * for the ids it owns and zero elsewhere; g sums the partials (one of them is
 * non-zero per token, so the fused sum reads only the owning shard).
 *   ids [N] int32 (device), 0 <= id < V; Y [N][h] bf16.  V % t == 0,
 *   V < 2^19, h % 8 == 0.  An id out of range gives a zero row and
 *   tp_get_device_status() reports TP_ERR_SHAPE.
 * Backward: g backward hands dY to every shard; shard i adds dY[n] into
 * dE_p[i][id - i V/t] for every token it owns.  Deterministic: the tokens of a
 * row are added in a fixed order (chunks of 8192 tokens are grouped by id on the
 * device, the ids in order of first occurrence and each id's tokens in token order).  dE_p [t][V/t][h] fp32, overwritten (zeroed first) or added
 * to when accumulate != 0; ws: tp_vocab_embedding_backward_workspace_size(N)
 * bytes.  The LM head on the same split is the column-parallel GEMM against
 * E^T (tp_column_parallel_forward); the pages define no loss, none is built. */
tp_status tp_vocab_embedding_forward(const int32_t* ids, int64_t N, int64_t V, int64_t h, int t, const tp_bf16* E_p,
                                     tp_bf16* Y, tp_stream stream);
size_t tp_vocab_embedding_backward_workspace_size(int64_t N);
tp_status tp_vocab_embedding_backward(const int32_t* ids, const tp_bf16* dY, int64_t N, int64_t V, int64_t h, int t,
                                      float* dE_p, int accumulate, void* ws, size_t ws_bytes, tp_stream stream);

/* ------------------------------------------- sequence-parallel LayerNorm
 * ("Tensor and sequence parallelism", section "Sequence parallelism";
 * "02 — Tensor Parallelism", "Sequence parallelism (Megatron-3)"):
 * X_sh [t][s/t][h]: shard j normalises only its own s/t rows,
 *   y = (x - mean) * rstd * gamma + beta,  rstd = 1/sqrt(biased var + eps).
 * The all-gather that enters the TP region is zero-copy: [t][s/t][h] is the
 * same bytes as [s][h].  mean, rstd: [s] fp32 (saved for backward).
 * t = 1 is an ordinary replicated LayerNorm. */
tp_status tp_sp_layernorm_forward(const tp_bf16* X_sh, int64_t s, int64_t h, int t, const tp_bf16* gamma,
                                  const tp_bf16* beta, float eps, tp_bf16* Y_sh, float* mean, float* rstd,
                                  tp_stream stream);

/* Backward: dX rows per shard (plus dres [s][h] if non-null: the residual
 * branch's gradient, added in the same pass); per-shard partial weight grads
 * dgamma_part[j] = sum over shard j's rows of dy*xhat, dbeta_part[j] = sum dy
 * ([t][h] fp32); then the LayerNorm weight-gradient all-reduce:
 * dgamma = sum_{j=0..t-1} dgamma_part[j] (fixed order), same for dbeta. */
/* tp_sp_layernorm_forward with Y_sh written as IEEE fp16 bits (the attention block's input
 * under TP_ATTN_F16_INPUT); same arguments and statistics. */
tp_status tp_sp_layernorm_forward_f16(const tp_bf16* X_sh, int64_t s, int64_t h, int t, const tp_bf16* gamma,
                                      const tp_bf16* beta, float eps, uint16_t* Y_sh, float* mean, float* rstd,
                                      tp_stream stream);

/* dst[i] = fp16(src[i]) for n bf16 values, round to nearest even: exact for bf16 values in
 * fp16's normal range (2^-14 .. 65504); smaller ones become fp16 subnormals (zero below
 * 2^-25), larger ones infinity.  For weights packed once (e.g. W_qkv under
 * TP_ATTN_F16_INPUT).  src, dst 16-byte aligned, not overlapping. */
tp_status tp_convert_bf16_to_f16(const tp_bf16* src, int64_t n, uint16_t* dst, tp_stream stream);

tp_status tp_sp_layernorm_backward(const tp_bf16* dY_sh, const tp_bf16* X_sh, const tp_bf16* gamma,
                                   const float* mean, const float* rstd, const tp_bf16* dres, int64_t s, int64_t h,
                                   int t, tp_bf16* dX_sh, float* dgamma_part, float* dbeta_part, float* dgamma,
                                   float* dbeta, tp_stream stream);

/* ------------------------------------------------------------ utilities
 * Fixed-order reduction of t partial buffers (the on-device stand-in for an
 * all-reduce, unfused form): out[r][c] = sum_{i=0..t-1} P[i][r][c] + bias[c]
 * (once, nullable) + residual[r][c] (nullable).  P fp32 [t][rows][cols];
 * out_bf16 and/or out_f32 (at least one non-null). */
tp_status tp_shard_reduce(const float* P, int64_t rows, int64_t cols, int t, const tp_bf16* bias,
                          const tp_bf16* residual, tp_bf16* out_bf16, float* out_f32, tp_stream stream);

/* Column sums of a bf16 matrix [rows][cols] -> fp32 [cols] in a fixed order
 * (bias gradients).  ws: tp_colsum_workspace_size(rows, cols) bytes.  cols even;
 * rows are summed in 64-row chunks, and any row count whose chunk count fits in
 * 2^31 - 1 is accepted (the chunks are spread over the grid's x dimension). */
size_t tp_colsum_workspace_size(int64_t rows, int64_t cols);
tp_status tp_colsum(const tp_bf16* G, int64_t rows, int64_t cols, float* out, int accumulate, void* ws,
                    size_t ws_bytes, tp_stream stream);

/* Column sums like tp_colsum, for callers that cannot allocate device memory
 * and so cannot hand over a workspace (code that must not call cudaMalloc,
 * code whose device memory is all held by another allocator's pool, plugins
 * that only receive their input and output pointers).  The pages have no
 * counterpart to this entry point.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *     The partial sums live in a 4 MiB array inside the library's device image,
 *     which every GPU that loads the library keeps until the process exits.
 *   - Limit: ceil(rows / 64) * cols <= 1048576 (e.g. 2048 rows x 32768 columns);
 *     larger sizes return TP_ERR_SHAPE and touch nothing.
 *   - The first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress, with the device current); make that first
 *     call before any stream capture.
 *   - All calls share the one array: calls that may run at the same time on the
 *     GPU (different streams without ordering between them) race and give
 *     wrong sums.  Calls ordered on one stream are fine; each call overwrites
 *     every partial it reads, so nothing from a previous call leaks in.
 *   - G [rows][cols] bf16, cols even; out [cols] fp32 (added to when accumulate != 0). */
tp_status tp_colsum_noalloc(const tp_bf16* G, int64_t rows, int64_t cols, float* out, int accumulate,
                            tp_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* TPSHARD_TP_H */
