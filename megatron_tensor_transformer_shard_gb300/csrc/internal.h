// Host-side interfaces shared between the translation units of libtpshard.so.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

#include "tp.h"

namespace tp {

// ------------------------------------------------------------ device state
int* device_error_word();          // device address of the error word of the current device
uint64_t wait_timeout_ns();        // limit for every bounded wait in the library's kernels
int device_sm_count();             // SMs of the current device
bool device_is_sm103();            // compute capability 10.3
tp_status ready();                 // TP_OK if the current device can run this library's kernels
void count_launch(int n = 1);      // every kernel launch of the library is counted
uint64_t launches_so_far();
const char* error_detail();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define TP_RETURN_IF(expr)        \
  do {                            \
    tp_status _s = (expr);        \
    if (_s != TP_OK) return _s;   \
  } while (0)

// Records a human-readable cause of the next TP_ERR_CUDA (thread-local; read
// with tp_last_error_detail()).
void set_error_detail(const char* file, int line, const char* what);
tp_status cuda_failure(const char* file, int line, cudaError_t e);

#define TP_CUDA_CHECK(expr)                                                  \
  do {                                                                       \
    cudaError_t _e = (expr);                                                 \
    if (_e != cudaSuccess) return ::tp::cuda_failure(__FILE__, __LINE__, _e); \
  } while (0)

// After a <<<...>>> launch: count it and surface launch errors.
#define TP_LAUNCHED()                                                        \
  do {                                                                       \
    count_launch();                                                          \
    cudaError_t _e = cudaGetLastError();                                     \
    if (_e != cudaSuccess) return ::tp::cuda_failure(__FILE__, __LINE__, _e); \
  } while (0)

#define TP_FAIL_DETAIL(what) (::tp::set_error_detail(__FILE__, __LINE__, what), TP_ERR_CUDA)

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel on the stream drains; it must execute
// griddepcontrol.wait before touching anything that kernel writes.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ----------------------------------------------------------------- GEMM
// One launch computes, for every output batch b in [0, nbatch):
//   D[b] (M x N) = sum_{s < nsum} A_sel (M x K) * B_sel (N x K)^T     (fp32 accumulate)
// where the operand shard selected is (nsum > 1 ? s : b) for a sharded
// operand and 0 otherwise.  nsum > 1 is the fused shard reduction: the K
// ranges of the t shards accumulate one after another, in shard order, into
// the same accumulator.  Operands are bf16 matrices, either K-major (stored
// [rows][K], K contiguous) or MN-major (stored [K][rows], rows contiguous).
struct GemmOperand {
  const uint16_t* ptr = nullptr;
  int64_t ld = 0;            // elements between consecutive stored rows
  int64_t shard_stride = 0;  // elements between shards
  bool sharded = false;
  bool mn_major = false;
};

enum GemmEpilogue : int {
  EPI_BF16 = 0,   // D = bf16(acc + bias[n] + residual[m][n])      (bias/residual nullable)
  EPI_ACT = 1,    // Z = acc + bias_b[n];  D = bf16(Z) (nullable);  D2 = bf16(act(Z))
  EPI_DACT = 2,   // D = bf16(acc * act'(aux_b[m][n]))
  EPI_F32 = 3,    // D = acc (+ D if accumulate), fp32
  // SwiGLU over the interleaved gate / up layout of tp_pack_swiglu (groups of 128 columns:
  // gate, then up).  EPI_GLU: acc columns are Z's; D = bf16(Z) (nullable), D2 = bf16(silu(g) u)
  // with its own stride (ldd2, d2_batch_stride).  EPI_DGLU: acc columns are dA's (N = the
  // A width); aux = Z; D = dZ (gate and up interleaved like Z, row stride ldd):
  // d gate = dA u silu'(g), d up = dA silu(g).
  EPI_GLU = 4,
  EPI_DGLU = 5,
};

struct GemmProblem {
  int64_t M = 0, N = 0, K = 0;
  int nbatch = 1, nsum = 1;
  GemmOperand a, b;
  int f16_ab = 0;  // both operands IEEE fp16 instead of bf16 (the MMA takes one type for both)
  int epi = EPI_BF16;
  int act = TP_ACT_IDENTITY;
  void* d = nullptr;
  int64_t ldd = 0, d_batch_stride = 0;
  void* d2 = nullptr;  // EPI_ACT: activation output, same layout as d; EPI_GLU: silu(g) u
  int64_t ldd2 = 0, d2_batch_stride = 0;  // EPI_GLU only (EPI_ACT's d2 shares d's strides)
  const uint16_t* bias = nullptr;
  int64_t bias_batch_stride = 0;
  const uint16_t* aux = nullptr;  // EPI_DACT: Z
  int64_t ld_aux = 0, aux_batch_stride = 0;
  // EPI_DACT (nullable): column sums of D before rounding, one row per 32-row block of M,
  // colsum[b][(M + 31) / 32][N] fp32 -- the partial pass of a fused column sum (bias gradient)
  float* colsum = nullptr;
  const uint16_t* residual = nullptr;
  int64_t ld_res = 0;
  int accumulate = 0;
  int out_f16 = 0;  // EPI_ACT only: write D / D2 as IEEE fp16 instead of bf16
  // Overlapped shard reduction (CTA-pair kernel, EPI_BF16, nbatch = 1, nsum = t shards):
  // each tile's t shard K ranges are separate work items (shard-major order), whose fp32
  // partials P_i go to ovl_part [t][M][N] (the data a multi-GPU run would
  // exchange) and are summed in shard order in an fp32 running sum per tile (ovl_run:
  // gemm_overlap_scratch_bytes(M, N) bytes, 16-byte aligned, any contents) while the tensor
  // cores go on; the last shard adds its accumulator, then the epilogue adds the bias once
  // and the residual after it.
  float* ovl_part = nullptr;
  float* ovl_run = nullptr;
  // Split-K workspace (nullable, 256-byte aligned): lets the CTA-pair kernel cut the tiles
  // past its last full round into K ranges dealt to every cluster (BF16, ACT, F32 without
  // accumulate, DACT epilogues).  gemm_sk_ws_bytes() bytes cover any plan; less limits the
  // ranges.
  void* sk_ws = nullptr;
  size_t sk_ws_bytes = 0;
};
// Split-K workspace: up to kSkMaxSlots 256 x 256 fp32 partials, then per split tile 8
// counters of 8 bytes (kSkCounterBytes per slot over-provisions them).
constexpr int64_t kSkMaxSlots = 256;
constexpr size_t kSkSlotBytes = 256 * 256 * 4;
constexpr size_t kSkCounterBytes = 8 * 8;
inline size_t gemm_sk_ws_bytes() { return kSkMaxSlots * (kSkSlotBytes + kSkCounterBytes); }
// Scratch of the overlapped reduction: a 256 x 256 fp32 running sum per output tile, then 8
// flags of 8 bytes (two CTAs x four warps) per tile.
inline size_t gemm_overlap_scratch_bytes(int64_t M, int64_t N) {
  const int64_t tiles = ((M + 255) / 256) * ((N + 255) / 256);
  return static_cast<size_t>(tiles) * (256 * 256 * 4 + 64);
}

tp_status run_gemm(const GemmProblem& p, cudaStream_t s);

// ------------------------------------------------------------- others
tp_status run_colsum(const uint16_t* G, int64_t rows, int64_t cols, int64_t ld, float* out, int accumulate,
                     float* ws, size_t ws_floats, cudaStream_t s);
size_t colsum_ws_floats(int64_t rows, int64_t cols);
tp_status run_colsum_batched(const uint16_t* G, int64_t rows, int64_t cols, int64_t ld, int nbatch,
                             int64_t batch_stride, float* out, int accumulate, float* ws, size_t ws_floats,
                             cudaStream_t s);
// Two column-sum jobs fused into one partial and one final launch.
struct ColsumJob {
  const uint16_t* G = nullptr;
  int64_t rows = 0, cols = 0, ld = 0, bs = 0;
  int nbatch = 1;
  float* out = nullptr;
  float* ws = nullptr;  // colsum2_ws_floats(rows, cols, nbatch) floats
  int accumulate = 0;
  int f16 = 0;  // G holds IEEE fp16 values (else bf16)
  // ws already holds [nbatch][nchunks][cols] partials (written by a GEMM epilogue): only the
  // final in-order sum runs, over the caller's nchunks
  int partials_ready = 0;
  int nchunks = 0;      // set by run_colsum2 (by the caller when partials_ready)
  int64_t cblocks = 0;  // set by run_colsum2
};
size_t colsum2_ws_floats(int64_t rows, int64_t cols, int nbatch);
tp_status run_colsum2(ColsumJob a, ColsumJob b, cudaStream_t s);
tp_status run_shard_reduce(const float* P, int64_t rows, int64_t cols, int t, const uint16_t* bias,
                           const uint16_t* residual, uint16_t* out_bf16, float* out_f32, cudaStream_t s);

// packing (pack.cu).  dir 0: src unpacked -> dst packed; dir 1: src packed -> dst unpacked.
tp_status pack_col(const uint16_t* src, int64_t h, int64_t F, int t, uint16_t* dst, int dir, cudaStream_t s);
tp_status pack_row(const uint16_t* src, int64_t F, int64_t h, int t, uint16_t* dst, int dir, cudaStream_t s);
tp_status pack_swiglu(const uint16_t* Wg, const uint16_t* Wu, int64_t h, int64_t F, int t, uint16_t* Wp,
                      cudaStream_t s);
tp_status pack_qkv(const uint16_t* src, int64_t d, int n_heads, int head_dim, int t, uint16_t* dst, int dir,
                   cudaStream_t s);
tp_status pack_qkv_bias(const uint16_t* b, int64_t d, int n_heads, int head_dim, int t, uint16_t* bp,
                        cudaStream_t s);

tp_status pack_qkv_gqa(const uint16_t* src, int64_t d, int n_heads, int n_kv, int head_dim, int t, uint16_t* dst,
                       int dir, cudaStream_t s);
tp_status pack_qkv_gqa_bias(const uint16_t* b, int n_heads, int n_kv, int head_dim, int t, uint16_t* bp,
                            cudaStream_t s);

// skinny GEMM (skinny_gemm.cu): y[b][r] = sum_k W[r][k] x[b][k] for 1..32 rows of x.
enum SkEpilogue : int { SK_EPI_BF16 = 0, SK_EPI_QKV = 1 };
struct SkGemmJob {
  const uint16_t* W = nullptr;  // [slabs][R][Kt] bf16, Kt = 128 * ku_per_slab
  int slabs = 1;
  int64_t R = 0;
  int ku_per_slab = 0;
  const uint16_t* x = nullptr;  // [B][ldx] bf16, K = slabs * Kt columns used
  int64_t ldx = 0;
  int B = 0;
  float* part = nullptr;        // skinny_part_floats(R, B) floats
  int nrb = 0, nku = 0;         // set by run_skinny_gemm
  int epi = SK_EPI_BF16;
  const uint16_t* bias = nullptr;  // [R] nullable, added once after the full K sum
  uint16_t* y = nullptr;           // SK_EPI_BF16: y[b * ldy + r]
  int64_t ldy = 0;
  // SK_EPI_QKV: packed decode QKV rows [t][R_t], routed to q (fp16) or the cache copies
  int64_t R_t = 0, L_max = 0;
  int q_t = 0, kv_t = 0, nh = 0;
  int* cnt = nullptr;  // SK_EPI_BF16: [R/128] counters, zero on entry -> the reduction runs inside the GEMM
  const int32_t* pos = nullptr;
  uint16_t* q = nullptr;
  uint16_t* Kc = nullptr;
  uint16_t* Vc = nullptr;
  int* err = nullptr;
};
size_t skinny_part_floats(int64_t R, int B);
bool skinny_ok(int64_t R, int64_t Kt, int B);
tp_status run_skinny_gemm(SkGemmJob j, cudaStream_t s);

tp_status reduce_qkv_gqa_grad(const float* dWp, int64_t d, int n_heads, int n_kv, int head_dim, int t, float* dW,
                              int accumulate, cudaStream_t s);

// vocab-parallel embedding (embedding.cu)
size_t emb_bwd_ws_bytes(int64_t N);
tp_status run_emb_forward(const int32_t* ids, int64_t N, int64_t V, int64_t h, int t, const uint16_t* E, uint16_t* Y,
                          cudaStream_t s);
tp_status run_emb_backward(const int32_t* ids, const uint16_t* dY, int64_t N, int64_t V, int64_t h, int t, float* dE,
                           int accumulate, void* ws, size_t ws_bytes, cudaStream_t s);

// decode attention (decode_attn.cu)
size_t decode_attn_ws_bytes(int64_t B, int64_t d, int n_heads, int n_kv, int head_dim, int t, int64_t L_max);
tp_status run_decode_attn(const uint16_t* x, int64_t B, int64_t d, int n_heads, int n_kv, int head_dim, int t,
                          float scale, const uint16_t* Wqkv_p, const uint16_t* bqkv_p, const uint16_t* Wo_p,
                          const uint16_t* bo, uint16_t* Kc, uint16_t* Vc, int64_t L_max, const int32_t* pos,
                          uint16_t* y, void* ws, size_t ws_bytes, cudaStream_t s);
tp_status run_row_gemv(const uint16_t* a, int64_t M, int64_t K, int64_t h, int t, const uint16_t* Wd,
                       const uint16_t* bias, uint16_t* y, cudaStream_t s);

// decode GEMV (gemv.cu), LayerNorm (layernorm.cu)
tp_status run_decode_swiglu(const uint16_t* x, int64_t M, int64_t h, int64_t F, int t, const uint16_t* Wgu,
                            const uint16_t* Wd, uint16_t* y, uint16_t* a, cudaStream_t s);
// out_f16: Y is written as IEEE fp16 (else bf16).
tp_status run_ln_forward(const uint16_t* X, int64_t s, int64_t h, int t, const uint16_t* gamma,
                         const uint16_t* beta, float eps, uint16_t* Y, float* mean, float* rstd, cudaStream_t st,
                         int out_f16 = 0);
// dst[i] = fp16(src[i]) for n bf16 values (round to nearest even).
tp_status run_bf16_to_f16(const uint16_t* src, int64_t n, uint16_t* dst, cudaStream_t s);
tp_status run_ln_backward(const uint16_t* dY, const uint16_t* X, const uint16_t* gamma, const float* mean,
                          const float* rstd, const uint16_t* dres, int64_t s, int64_t h, int t, uint16_t* dX,
                          float* dg_part, float* db_part, float* dgamma, float* dbeta, cudaStream_t st);

// attention (attention.cu)
// n_kv: KV heads (n_kv = n_heads for multi-head attention); QKV rows per shard are
// [q_t query heads | kv_t K heads | kv_t V heads], 128 columns each.
// SwiGLU of the token-parallel MLP (Z over the interleaved packed gate / up weights).

tp_status run_attention_fwd(const uint16_t* QKV, int64_t N, int64_t d, int n_heads, int n_kv, int head_dim, int t,
                            int causal, float scale, uint16_t* O, float* lse, cudaStream_t s);
// dqkv_f16: dQKV is written as IEEE fp16 (else bf16).
tp_status run_attention_bwd(const uint16_t* QKV, const uint16_t* O, const uint16_t* dO, const float* lse, int64_t N,
                            int64_t d, int n_heads, int n_kv, int head_dim, int t, int causal, float scale, float* Dvec,
                            uint16_t* dQKV, cudaStream_t s, int dqkv_f16 = 0);

}  // namespace tp
