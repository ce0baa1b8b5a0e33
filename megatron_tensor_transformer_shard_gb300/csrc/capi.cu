// extern "C" entry points of libtpshard.so (declared in include/tp.h), the
// per-device error word, and the fault-path self test.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "trace.h"
#include "ptx.cuh"

namespace tp {

// Written by any kernel whose bounded wait expired (first error wins).
__device__ int g_tp_error_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int* g_err_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
int g_is_sm103[kMaxDevices] = {};

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

// Per-device set-up, once, with that device current.
bool ensure_device(int dev) {
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_err_ptr[dev]) return true;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_tp_error_word) != cudaSuccess) return false;
  int sms = 0, major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return false;
  g_sm_count[dev] = sms;
  g_is_sm103[dev] = (major == 10 && minor == 3);
  g_err_ptr[dev] = static_cast<int*>(p);
  return true;
}

__global__ void selftest_wait_kernel(int* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nothing ever arrives on `bar`: the wait must give up by itself.
    ptx::mbar_wait(&bar, 0, &abort_flag, err, 0x1FF, timeout_ns);
  }
  __syncthreads();
}

}  // namespace

int* device_error_word() {
  const int dev = current_device();
  if (dev < 0 || !ensure_device(dev)) return nullptr;
  return g_err_ptr[dev];
}

int device_sm_count() {
  const int dev = current_device();
  if (dev < 0 || !ensure_device(dev)) return 1;
  return g_sm_count[dev] > 0 ? g_sm_count[dev] : 1;
}

bool device_is_sm103() {
  const int dev = current_device();
  if (dev < 0 || !ensure_device(dev)) return false;
  return g_is_sm103[dev] != 0;
}

namespace {
std::atomic<uint64_t> g_launches{0};
}

namespace {
thread_local char g_detail[256] = "";
}

void set_error_detail(const char* file, int line, const char* what) {
  const char* f = std::strrchr(file, '/');
  std::snprintf(g_detail, sizeof(g_detail), "%s:%d: %s", f ? f + 1 : file, line, what);
}

tp_status cuda_failure(const char* file, int line, cudaError_t e) {
  char buf[160];
  std::snprintf(buf, sizeof(buf), "%s (%s)", cudaGetErrorName(e), cudaGetErrorString(e));
  set_error_detail(file, line, buf);
  return TP_ERR_CUDA;
}

const char* error_detail() { return g_detail; }

void count_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }
uint64_t launches_so_far() { return g_launches.load(std::memory_order_relaxed); }

tp_status ready() {
  // Driver-API calls (tensor-map encoding) need the device's primary context
  // current on this thread; threads that reach the library first (e.g. an
  // autograd worker) may not have it yet.
  thread_local int ctx_dev = -1;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TP_FAIL_DETAIL("cudaGetDevice failed");
  if (dev != ctx_dev) {
    TP_CUDA_CHECK(cudaSetDevice(dev));
    ctx_dev = dev;
  }
  if (!device_error_word()) return TP_ERR_CUDA;
  if (!device_is_sm103()) return TP_ERR_UNSUPPORTED;
  return TP_OK;
}

uint64_t wait_timeout_ns() {
  static uint64_t ns = [] {
    const char* e = std::getenv("TP_WAIT_TIMEOUT_MS");
    long ms = e ? std::atol(e) : 0;
    if (ms <= 0 || ms > 60000) ms = 2000;
    return static_cast<uint64_t>(ms) * 1000000ull;
  }();
  return ns;
}

}  // namespace tp

using namespace tp;

namespace {

inline cudaStream_t S(tp_stream s) { return reinterpret_cast<cudaStream_t>(s); }

bool act_ok(int a) { return a >= TP_ACT_IDENTITY && a <= TP_ACT_GELU_ERF; }
bool mlp_act_ok(int a) { return act_ok(a) || a == TP_ACT_SWIGLU; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace of tp_attn_backward (each piece 256-byte aligned).
struct AttnBwdWs {
  uint16_t* dO;
  float* Dvec;
  uint16_t* dQKV;
  float* cs;
  size_t cs_floats;
  size_t total;
};

// QKV row width of one shard: [q_t query heads | kv_t K heads | kv_t V heads] x head_dim.
int64_t qkv_row_width(int n_heads, int n_kv, int head_dim, int t) {
  const int kv_t = n_kv >= t ? n_kv / t : 1;
  return static_cast<int64_t>(n_heads / t + 2 * kv_t) * head_dim;
}

bool gqa_ok(int64_t d, int n_heads, int n_kv, int head_dim, int t) {
  if (head_dim != 128 || static_cast<int64_t>(n_heads) * head_dim != d || n_heads % t != 0) return false;
  if (n_kv < 1 || n_heads % n_kv != 0) return false;
  return n_kv >= t ? n_kv % t == 0 : t % n_kv == 0;
}

AttnBwdWs attn_bwd_layout(void* ws, int64_t N, int64_t d, int n_heads, int64_t row_w, int t) {
  AttnBwdWs w{};
  uint8_t* b = static_cast<uint8_t*>(ws);
  size_t off = 0;
  w.dO = reinterpret_cast<uint16_t*>(b + off);
  off += round_up(static_cast<size_t>(N) * d * 2, 256);
  w.Dvec = reinterpret_cast<float*>(b + off);
  off += round_up(static_cast<size_t>(N) * n_heads * 4, 256);
  w.dQKV = reinterpret_cast<uint16_t*>(b + off);
  off += round_up(static_cast<size_t>(N) * t * row_w * 2, 256);
  w.cs = reinterpret_cast<float*>(b + off);
  w.cs_floats = colsum2_ws_floats(N, d, 1) + colsum2_ws_floats(N, row_w, t);
  off += round_up(w.cs_floats * 4, 256);
  w.total = off;
  return w;
}

}  // namespace

namespace {

// Partials [t][M][h] fp32, then (overlapped reduction) the CTA pairs' running sums.
size_t row_partials_ws(int64_t M, int64_t h, int t, bool overlap) {
  size_t sz = round_up(static_cast<size_t>(t) * M * h * sizeof(float), 256);
  if (overlap) sz += round_up(gemm_overlap_scratch_bytes(M, h), 256);
  return sz;
}

tp_status column_parallel(const tp_bf16* X, int64_t M, int64_t h, int64_t N, int t, tp_act act, const tp_bf16* W_p,
                          const tp_bf16* b, tp_bf16* Z, tp_bf16* A, void* sk_ws, size_t sk_bytes, cudaStream_t s) {
  if (M < 0 || h < 1 || N < 1 || t < 1 || !act_ok(act)) return TP_ERR_INVALID_ARG;
  if (N % t != 0) return TP_ERR_SHAPE;
  const int64_t Nt = N / t;
  if (h % 8 != 0 || Nt % 8 != 0) return TP_ERR_ALIGN;
  if (M == 0) return TP_OK;
  if (!X || !W_p || !A) return TP_ERR_INVALID_ARG;
  GemmProblem c;
  c.M = M; c.N = Nt; c.K = h; c.nbatch = t; c.nsum = 1;
  c.a.ptr = X; c.a.ld = h;
  c.b.ptr = W_p; c.b.ld = h; c.b.sharded = true; c.b.shard_stride = Nt * h;
  c.epi = EPI_ACT; c.act = act;
  c.d = Z; c.d2 = A; c.ldd = Nt; c.d_batch_stride = M * Nt;
  c.bias = b; c.bias_batch_stride = Nt;
  c.sk_ws = sk_ws; c.sk_ws_bytes = sk_bytes;
  return run_gemm(c, s);
}

tp_status row_parallel(const tp_bf16* A, int64_t M, int64_t K, int64_t h, int t, const tp_bf16* W_p,
                       const tp_bf16* b, const tp_bf16* residual, tp_bf16* Y, void* sk_ws, size_t sk_bytes,
                       cudaStream_t s) {
  if (M < 0 || h < 1 || K < 1 || t < 1) return TP_ERR_INVALID_ARG;
  if (K % t != 0) return TP_ERR_SHAPE;
  const int64_t Kt = K / t;
  if (h % 8 != 0 || Kt % 8 != 0) return TP_ERR_ALIGN;
  if (M == 0) return TP_OK;
  if (!A || !W_p || !Y) return TP_ERR_INVALID_ARG;
  GemmProblem r;
  r.M = M; r.N = h; r.K = Kt; r.nbatch = 1; r.nsum = t;
  r.a.ptr = A; r.a.ld = Kt; r.a.sharded = true; r.a.shard_stride = M * Kt;
  r.b.ptr = W_p; r.b.ld = Kt; r.b.sharded = true; r.b.shard_stride = h * Kt;
  r.epi = EPI_BF16; r.d = Y; r.ldd = h; r.bias = b; r.residual = residual; r.ld_res = h;
  r.sk_ws = sk_ws; r.sk_ws_bytes = sk_bytes;
  return run_gemm(r, s);
}

// The forward's required scratch: the partials of the unfused / overlapped reduction.  A
// workspace that also holds gemm_sk_ws_bytes() after it lets the GEMMs split K.
size_t mlp_fwd_base_ws(int64_t M, int64_t h, int t, unsigned flags) {
  if (flags & TP_FLAG_OVERLAP_REDUCE) return row_partials_ws(M, h, t, true);
  return (flags & TP_FLAG_UNFUSED_REDUCE) ? round_up(static_cast<size_t>(t) * M * h * sizeof(float), 256) : 0;
}

// The part of a caller's workspace past `base` bytes, 256-byte aligned, for split K (NULL
// when there is none).
void* sk_part_of(void* ws, size_t ws_bytes, size_t base, size_t* sk_bytes) {
  *sk_bytes = 0;
  if (!ws || ws_bytes <= base) return nullptr;
  uint8_t* p = static_cast<uint8_t*>(ws) + base;
  const size_t skew = (256 - (reinterpret_cast<uintptr_t>(p) & 255u)) & 255u;
  if (ws_bytes - base <= skew) return nullptr;
  *sk_bytes = ws_bytes - base - skew;
  return p + skew;
}

}  // namespace

extern "C" {

size_t tp_attn_gqa_backward_workspace_size(int64_t N, int64_t d, int n_heads, int n_kv_heads, int head_dim, int t,
                                           unsigned flags) {
  (void)flags;
  if (N < 0 || d < 1 || n_heads < 1 || t < 1 || !gqa_ok(d, n_heads, n_kv_heads, head_dim, t)) return 0;
  // the required part, then room for the GEMMs' split-K partials
  return attn_bwd_layout(nullptr, N, d, n_heads, qkv_row_width(n_heads, n_kv_heads, head_dim, t), t).total +
         gemm_sk_ws_bytes();
}

size_t tp_attn_backward_workspace_size(int64_t N, int64_t d, int n_heads, int head_dim, int t, unsigned flags) {
  (void)head_dim;
  (void)flags;
  if (N < 0 || d < 1 || n_heads < 1 || t < 1) return 0;
  return attn_bwd_layout(nullptr, N, d, n_heads, 3 * d / t, t).total + gemm_sk_ws_bytes();
}

tp_status tp_attn_gqa_backward(const tp_bf16* dY, const tp_bf16* X, const uint16_t* QKV_save, const tp_bf16* O_save,
                               const float* lse_save, int64_t N, int64_t d, int n_heads, int n_kv_heads,
                               int head_dim, int t, int causal, float scale, const tp_bf16* Wqkv_p,
                               const tp_bf16* Wo_p, tp_bf16* dX, float* dWqkv_p, float* dbqkv_p, float* dWo_p,
                               float* dbo, int accumulate, unsigned flags, void* ws, size_t ws_bytes,
                               tp_stream stream) {
  TP_TRACE();
  if (N < 0 || d < 1 || n_heads < 1 || n_kv_heads < 1 || t < 1 || head_dim < 1) return TP_ERR_INVALID_ARG;
  if ((flags & ~TP_ATTN_F16_INPUT) != 0) return TP_ERR_UNSUPPORTED;
  const int f16in = (flags & TP_ATTN_F16_INPUT) ? 1 : 0;  // X, W_qkv and so dQKV in IEEE fp16
  if (!gqa_ok(d, n_heads, n_kv_heads, head_dim, t)) return TP_ERR_SHAPE;
  if (!dWqkv_p || !dWo_p) return TP_ERR_INVALID_ARG;
  if (N > 0 && (!dY || !X || !QKV_save || !O_save || !lse_save || !Wqkv_p || !Wo_p || !dX)) return TP_ERR_INVALID_ARG;
  const int64_t rw = qkv_row_width(n_heads, n_kv_heads, head_dim, t);  // one shard's QKV row
  const AttnBwdWs w = attn_bwd_layout(ws, N, d, n_heads, rw, t);
  if (!ws || ws_bytes < w.total) return TP_ERR_WORKSPACE;
  if (!aligned16(ws)) return TP_ERR_ALIGN;
  size_t sk_bytes = 0;
  void* sk_ws = sk_part_of(ws, ws_bytes, w.total, &sk_bytes);  // split K, when the workspace has room
  const cudaStream_t s = S(stream);
  const int64_t dt = d / t;
  if (N == 0) {
    TP_RETURN_IF(ready());
    if (!accumulate) {
      TP_CUDA_CHECK(cudaMemsetAsync(dWqkv_p, 0, sizeof(float) * t * rw * d, s));
      TP_CUDA_CHECK(cudaMemsetAsync(dWo_p, 0, sizeof(float) * d * d, s));
      if (dbqkv_p) TP_CUDA_CHECK(cudaMemsetAsync(dbqkv_p, 0, sizeof(float) * t * rw, s));
      if (dbo) TP_CUDA_CHECK(cudaMemsetAsync(dbo, 0, sizeof(float) * d, s));
    }
    return TP_OK;
  }
  // dO_i = dY W_o,i^T  (row-parallel W_o, input grad stays sharded).
  GemmProblem g;
  g.M = N; g.N = dt; g.K = d; g.nbatch = t;
  g.a.ptr = dY; g.a.ld = d;
  g.b.ptr = Wo_p; g.b.ld = dt; g.b.sharded = true; g.b.shard_stride = d * dt; g.b.mn_major = true;
  g.epi = EPI_ACT; g.act = TP_ACT_IDENTITY; g.out_f16 = 1;  // dO feeds the fp16 attention kernels
  g.d = nullptr; g.d2 = w.dO; g.ldd = dt; g.d_batch_stride = N * dt;
  g.sk_ws = sk_ws; g.sk_ws_bytes = sk_bytes;
  TP_RETURN_IF(run_gemm(g, s));
  // dW_o,i = O_i^T dY  -> packed [t][d][dt] (local).
  GemmProblem wo;
  wo.M = d; wo.N = dt; wo.K = N; wo.nbatch = t;
  wo.a.ptr = dY; wo.a.ld = d; wo.a.mn_major = true;
  wo.b.ptr = O_save; wo.b.ld = dt; wo.b.sharded = true; wo.b.shard_stride = N * dt; wo.b.mn_major = true;
  wo.epi = EPI_F32; wo.d = dWo_p; wo.ldd = dt; wo.d_batch_stride = d * dt; wo.accumulate = accumulate;
  wo.sk_ws = sk_ws; wo.sk_ws_bytes = sk_bytes;
  TP_RETURN_IF(run_gemm(wo, s));
  // Head-local softmax-attention backward -> dQKV_i.
  TP_RETURN_IF(run_attention_bwd(QKV_save, O_save, w.dO, lse_save, N, d, n_heads, n_kv_heads, head_dim, t, causal,
                                 scale, w.Dvec, w.dQKV, s, f16in));
  // Bias gradients in one fused pass: db_o once (g backward is the identity), db_qkv per shard.
  if (dbo || dbqkv_p) {
    ColsumJob jo, jq;
    if (dbo) {
      jo.G = dY; jo.rows = N; jo.cols = d; jo.ld = d; jo.bs = N * d; jo.nbatch = 1;
      jo.out = dbo; jo.ws = w.cs; jo.accumulate = accumulate;
    }
    if (dbqkv_p) {
      jq.G = w.dQKV; jq.rows = N; jq.cols = rw; jq.ld = rw; jq.bs = N * rw; jq.nbatch = t;
      jq.out = dbqkv_p; jq.ws = w.cs + colsum2_ws_floats(N, d, 1); jq.accumulate = accumulate; jq.f16 = f16in;
    }
    TP_RETURN_IF(run_colsum2(jo, jq, s));
  }
  // dW_qkv,i = dQKV_i^T X -> packed [t][rw][d] (local; a replicated KV head gets one gradient per copy).
  GemmProblem wq;
  wq.M = rw; wq.N = d; wq.K = N; wq.nbatch = t;
  wq.a.ptr = w.dQKV; wq.a.ld = rw; wq.a.sharded = true; wq.a.shard_stride = N * rw; wq.a.mn_major = true;
  wq.b.ptr = X; wq.b.ld = d; wq.b.mn_major = true;
  wq.epi = EPI_F32; wq.d = dWqkv_p; wq.ldd = d; wq.d_batch_stride = rw * d; wq.accumulate = accumulate;
  wq.f16_ab = f16in;
  wq.sk_ws = sk_ws; wq.sk_ws_bytes = sk_bytes;
  TP_RETURN_IF(run_gemm(wq, s));
  // f backward: dX = sum_i dQKV_i W_qkv,i (fixed shard order, fused).
  GemmProblem dx;
  dx.M = N; dx.N = d; dx.K = rw; dx.nsum = t;
  dx.a.ptr = w.dQKV; dx.a.ld = rw; dx.a.sharded = true; dx.a.shard_stride = N * rw;
  dx.b.ptr = Wqkv_p; dx.b.ld = d; dx.b.sharded = true; dx.b.shard_stride = rw * d; dx.b.mn_major = true;
  dx.epi = EPI_BF16; dx.d = dX; dx.ldd = d;
  dx.f16_ab = f16in;
  dx.sk_ws = sk_ws; dx.sk_ws_bytes = sk_bytes;
  return run_gemm(dx, s);
}

tp_status tp_attn_backward(const tp_bf16* dY, const tp_bf16* X, const tp_bf16* QKV_save, const tp_bf16* O_save,
                           const float* lse_save, int64_t N, int64_t d, int n_heads, int head_dim, int t,
                           int causal, float scale, const tp_bf16* Wqkv_p, const tp_bf16* Wo_p, tp_bf16* dX,
                           float* dWqkv_p, float* dbqkv_p, float* dWo_p, float* dbo, int accumulate,
                           unsigned flags, void* ws, size_t ws_bytes, tp_stream stream) {
  TP_TRACE();
  if (N < 0 || d < 1 || n_heads < 1 || t < 1 || head_dim < 1) return TP_ERR_INVALID_ARG;
  if ((flags & ~TP_ATTN_F16_INPUT) != 0) return TP_ERR_UNSUPPORTED;
  if (head_dim != 128 || static_cast<int64_t>(n_heads) * head_dim != d || n_heads % t != 0) return TP_ERR_SHAPE;
  return tp_attn_gqa_backward(dY, X, QKV_save, O_save, lse_save, N, d, n_heads, n_heads, head_dim, t, causal, scale,
                              Wqkv_p, Wo_p, dX, dWqkv_p, dbqkv_p, dWo_p, dbo, accumulate, flags, ws, ws_bytes, stream);
}

int tp_abi_version(void) { return TP_ABI_VERSION; }

uint64_t tp_kernel_launch_count(void) { return launches_so_far(); }

const char* tp_last_error_detail(void) { return error_detail(); }

const char* tp_status_string(tp_status s) {
  switch (s) {
    case TP_OK: return "TP_OK";
    case TP_ERR_INVALID_ARG: return "TP_ERR_INVALID_ARG: null pointer, bad enum or negative size";
    case TP_ERR_SHAPE: return "TP_ERR_SHAPE: t does not divide the split dimension, or unsupported size";
    case TP_ERR_ALIGN: return "TP_ERR_ALIGN: pointer not 16-byte aligned or row length not a multiple of 8";
    case TP_ERR_WORKSPACE: return "TP_ERR_WORKSPACE: workspace smaller than the *_workspace_size() result";
    case TP_ERR_CUDA: return "TP_ERR_CUDA: CUDA runtime call or kernel launch failed";
    case TP_ERR_TIMEOUT: return "TP_ERR_TIMEOUT: a bounded wait inside a kernel expired";
    case TP_ERR_UNSUPPORTED: return "TP_ERR_UNSUPPORTED: needs an sm_103a device / combination not built";
  }
  return "unknown tp_status";
}

tp_status tp_get_device_status(tp_stream stream) {
  TP_TRACE();
  if (!device_error_word()) return TP_ERR_CUDA;
  if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return TP_ERR_CUDA;
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_tp_error_word, sizeof(int)) != cudaSuccess) return TP_ERR_CUDA;
  if (word == 0) return TP_OK;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_tp_error_word, &zero, sizeof(int)) != cudaSuccess) return TP_ERR_CUDA;
  // codes 0x200-0x2ff: an argument the host could not check (it lives in device memory)
  return (word >= 0x200 && word < 0x300) ? TP_ERR_SHAPE : TP_ERR_TIMEOUT;
}

tp_status tp_selftest_bounded_wait(int64_t timeout_us, tp_stream stream) {
  TP_TRACE();
  if (timeout_us < 1 || timeout_us > 10000000) return TP_ERR_INVALID_ARG;
  TP_RETURN_IF(ready());
  selftest_wait_kernel<<<1, 32, 0, S(stream)>>>(device_error_word(), static_cast<uint64_t>(timeout_us) * 1000ull);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

// ------------------------------------------------------------------ packing
tp_status tp_pack_col(const tp_bf16* W, int64_t h, int64_t F, int t, tp_bf16* Wp, tp_stream stream) {
  TP_TRACE();
  return pack_col(W, h, F, t, Wp, 0, S(stream));
}
tp_status tp_unpack_col(const tp_bf16* Wp, int64_t h, int64_t F, int t, tp_bf16* W, tp_stream stream) {
  TP_TRACE();
  return pack_col(Wp, h, F, t, W, 1, S(stream));
}
tp_status tp_pack_row(const tp_bf16* W, int64_t F, int64_t h, int t, tp_bf16* Wp, tp_stream stream) {
  TP_TRACE();
  return pack_row(W, F, h, t, Wp, 0, S(stream));
}
tp_status tp_unpack_row(const tp_bf16* Wp, int64_t F, int64_t h, int t, tp_bf16* W, tp_stream stream) {
  TP_TRACE();
  return pack_row(Wp, F, h, t, W, 1, S(stream));
}
tp_status tp_pack_swiglu(const tp_bf16* Wg, const tp_bf16* Wu, int64_t h, int64_t F, int t, tp_bf16* Wp,
                         tp_stream stream) {
  TP_TRACE();
  return pack_swiglu(Wg, Wu, h, F, t, Wp, S(stream));
}
tp_status tp_pack_qkv_heads(const tp_bf16* Wqkv, int64_t d, int n_heads, int head_dim, int t, tp_bf16* Wp,
                            tp_stream stream) {
  TP_TRACE();
  return pack_qkv(Wqkv, d, n_heads, head_dim, t, Wp, 0, S(stream));
}
tp_status tp_unpack_qkv_heads(const tp_bf16* Wp, int64_t d, int n_heads, int head_dim, int t, tp_bf16* Wqkv,
                              tp_stream stream) {
  TP_TRACE();
  return pack_qkv(Wp, d, n_heads, head_dim, t, Wqkv, 1, S(stream));
}
tp_status tp_pack_qkv_bias(const tp_bf16* b, int64_t d, int n_heads, int head_dim, int t, tp_bf16* bp,
                           tp_stream stream) {
  TP_TRACE();
  return pack_qkv_bias(b, d, n_heads, head_dim, t, bp, S(stream));
}

tp_status tp_pack_qkv_gqa(const tp_bf16* Wqkv, int64_t d, int n_heads, int n_kv_heads, int head_dim, int t,
                          tp_bf16* Wp, tp_stream stream) {
  TP_TRACE();
  return pack_qkv_gqa(Wqkv, d, n_heads, n_kv_heads, head_dim, t, Wp, 0, S(stream));
}
tp_status tp_unpack_qkv_gqa(const tp_bf16* Wp, int64_t d, int n_heads, int n_kv_heads, int head_dim, int t,
                            tp_bf16* Wqkv, tp_stream stream) {
  TP_TRACE();
  return pack_qkv_gqa(Wp, d, n_heads, n_kv_heads, head_dim, t, Wqkv, 1, S(stream));
}
tp_status tp_pack_qkv_gqa_bias(const tp_bf16* b, int n_heads, int n_kv_heads, int head_dim, int t, tp_bf16* bp,
                               tp_stream stream) {
  TP_TRACE();
  return pack_qkv_gqa_bias(b, n_heads, n_kv_heads, head_dim, t, bp, S(stream));
}

// ------------------------------------------------------------------ TP MLP

size_t tp_mlp_workspace_size(int64_t M, int64_t h, int64_t F, int t, unsigned flags) {
  if (M < 0 || h < 0 || F < 0 || t < 1) return 0;
  return mlp_fwd_base_ws(M, h, t, flags) + gemm_sk_ws_bytes();
}

size_t tp_row_parallel_overlap_workspace_size(int64_t M, int64_t K, int64_t h, int t) {
  (void)K;
  if (M < 0 || h < 0 || t < 1) return 0;
  return row_partials_ws(M, h, t, true);
}

tp_status tp_row_parallel_forward_overlap(const tp_bf16* A, int64_t M, int64_t K, int64_t h, int t,
                                          const tp_bf16* W_p, const tp_bf16* b, const tp_bf16* residual, tp_bf16* Y,
                                          float* partials_out, void* ws, size_t ws_bytes, tp_stream stream) {
  TP_TRACE();
  if (M < 0 || h < 1 || K < 1 || t < 1) return TP_ERR_INVALID_ARG;
  if (K % t != 0 || t > 8) return TP_ERR_SHAPE;
  const int64_t Kt = K / t;
  if (h % 8 != 0 || Kt % 8 != 0) return TP_ERR_ALIGN;
  if (M == 0) return TP_OK;
  if (!A || !W_p || !Y) return TP_ERR_INVALID_ARG;
  if (M <= 128) return TP_ERR_UNSUPPORTED;  // CTA-pair kernel (M > 128)
  const size_t need = row_partials_ws(M, h, t, true);
  if (!ws || ws_bytes < need) return TP_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return TP_ERR_ALIGN;
  float* P = static_cast<float*>(ws);
  float* run = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + round_up(static_cast<size_t>(t) * M * h * 4, 256));
  GemmProblem r;
  r.M = M; r.N = h; r.K = Kt; r.nbatch = 1; r.nsum = t;
  r.a.ptr = A; r.a.ld = Kt; r.a.sharded = true; r.a.shard_stride = M * Kt;
  r.b.ptr = W_p; r.b.ld = Kt; r.b.sharded = true; r.b.shard_stride = h * Kt;
  r.epi = EPI_BF16; r.d = Y; r.ldd = h; r.bias = b; r.residual = residual; r.ld_res = h;
  r.ovl_part = P; r.ovl_run = run;
  TP_RETURN_IF(run_gemm(r, S(stream)));
  if (partials_out)
    TP_CUDA_CHECK(cudaMemcpyAsync(partials_out, P, static_cast<size_t>(t) * M * h * sizeof(float),
                                  cudaMemcpyDeviceToDevice, S(stream)));
  return TP_OK;
}

tp_status tp_column_parallel_forward(const tp_bf16* X, int64_t M, int64_t h, int64_t N, int t, tp_act act,
                                     const tp_bf16* W_p, const tp_bf16* b, tp_bf16* Z, tp_bf16* A,
                                     tp_stream stream) {
  TP_TRACE();
  return column_parallel(X, M, h, N, t, act, W_p, b, Z, A, nullptr, 0, S(stream));
}

tp_status tp_row_parallel_forward(const tp_bf16* A, int64_t M, int64_t K, int64_t h, int t, const tp_bf16* W_p,
                                  const tp_bf16* b, const tp_bf16* residual, tp_bf16* Y, tp_stream stream) {
  TP_TRACE();
  return row_parallel(A, M, K, h, t, W_p, b, residual, Y, nullptr, 0, S(stream));
}

size_t tp_column_parallel_workspace_size(int64_t M, int64_t h, int64_t N, int t) {
  (void)M; (void)h; (void)N; (void)t;
  return gemm_sk_ws_bytes();
}

tp_status tp_column_parallel_forward_ws(const tp_bf16* X, int64_t M, int64_t h, int64_t N, int t, tp_act act,
                                        const tp_bf16* W_p, const tp_bf16* b, tp_bf16* Z, tp_bf16* A, void* ws,
                                        size_t ws_bytes, tp_stream stream) {
  TP_TRACE();
  size_t sk = 0;
  void* skp = sk_part_of(ws, ws_bytes, 0, &sk);
  return column_parallel(X, M, h, N, t, act, W_p, b, Z, A, skp, sk, S(stream));
}

size_t tp_row_parallel_workspace_size(int64_t M, int64_t K, int64_t h, int t) {
  (void)M; (void)K; (void)h; (void)t;
  return gemm_sk_ws_bytes();
}

tp_status tp_row_parallel_forward_ws(const tp_bf16* A, int64_t M, int64_t K, int64_t h, int t, const tp_bf16* W_p,
                                     const tp_bf16* b, const tp_bf16* residual, tp_bf16* Y, void* ws,
                                     size_t ws_bytes, tp_stream stream) {
  TP_TRACE();
  size_t sk = 0;
  void* skp = sk_part_of(ws, ws_bytes, 0, &sk);
  return row_parallel(A, M, K, h, t, W_p, b, residual, Y, skp, sk, S(stream));
}

tp_status tp_mlp_forward(const tp_bf16* X, int64_t M, int64_t h, int64_t F, int t, tp_act act,
                         const tp_bf16* Wup_p, const tp_bf16* bup, const tp_bf16* Wdown_p, const tp_bf16* bdown,
                         const tp_bf16* residual, tp_bf16* Y, tp_bf16* Z_save, tp_bf16* A_save, unsigned flags,
                         void* ws, size_t ws_bytes, tp_stream stream) {
  TP_TRACE();
  if (M < 0 || h < 1 || F < 1 || t < 1 || !mlp_act_ok(act)) return TP_ERR_INVALID_ARG;
  if (F % t != 0) return TP_ERR_SHAPE;
  const int64_t Ft = F / t;
  if (h % 8 != 0 || Ft % 8 != 0) return TP_ERR_ALIGN;
  const bool swiglu = act == TP_ACT_SWIGLU;
  if (swiglu && Ft % 128 != 0) return TP_ERR_SHAPE;
  if (swiglu && bup) return TP_ERR_UNSUPPORTED;
  if (M == 0) return TP_OK;  // no tokens: nothing to compute (buffers may be NULL)
  if (!X || !Wup_p || !Wdown_p || !Y || !A_save || (swiglu && !Z_save)) return TP_ERR_INVALID_ARG;
  const bool overlap = (flags & TP_FLAG_OVERLAP_REDUCE) != 0;
  const bool unfused = !overlap && (flags & TP_FLAG_UNFUSED_REDUCE) != 0;
  const size_t base_ws = mlp_fwd_base_ws(M, h, t, flags);
  if (ws_bytes < base_ws || ((unfused || overlap) && !ws)) return TP_ERR_WORKSPACE;
  size_t sk_bytes = 0;
  void* sk_ws = sk_part_of(ws, ws_bytes, base_ws, &sk_bytes);  // split K, when the workspace has room
  if (overlap && t > 8) return TP_ERR_SHAPE;
  if (overlap && M <= 128) return TP_ERR_UNSUPPORTED;
  const cudaStream_t s = S(stream);

  if (swiglu) {
    // f (identity) + column-parallel over the interleaved gate / up weights: Z_i = X [W_gate | W_up]_i,
    // and A_i = silu(gate) * up in the same epilogue (a 256-column tile is one gate / up group).
    GemmProblem c;
    c.M = M; c.N = 2 * Ft; c.K = h; c.nbatch = t; c.nsum = 1;
    c.a.ptr = X; c.a.ld = h;
    c.b.ptr = Wup_p; c.b.ld = h; c.b.sharded = true; c.b.shard_stride = 2 * Ft * h;
    c.epi = EPI_GLU;
    c.d = Z_save; c.ldd = 2 * Ft; c.d_batch_stride = M * 2 * Ft;
    c.d2 = A_save; c.ldd2 = Ft; c.d2_batch_stride = M * Ft;
    TP_RETURN_IF(run_gemm(c, s));
  } else {
    // f (identity) + column-parallel: Z_i = X W_up,i + b_up[C_i]; A_i = act(Z_i).
    TP_RETURN_IF(column_parallel(X, M, h, F, t, act, Wup_p, bup, Z_save, A_save, sk_ws, sk_bytes, s));
  }
  if (overlap)
    return tp_row_parallel_forward_overlap(A_save, M, F, h, t, Wdown_p, bdown, residual, Y, nullptr, ws, ws_bytes,
                                           stream);

  // Row-parallel + g: Y = sum_i A_i W_down,i + b_down (once) + residual.
  if (!unfused) return row_parallel(A_save, M, F, h, t, Wdown_p, bdown, residual, Y, sk_ws, sk_bytes, s);
  GemmProblem r;
  r.M = M; r.N = h; r.K = Ft; r.nbatch = t; r.nsum = 1;
  r.a.ptr = A_save; r.a.ld = Ft; r.a.sharded = true; r.a.shard_stride = M * Ft;
  r.b.ptr = Wdown_p; r.b.ld = Ft; r.b.sharded = true; r.b.shard_stride = h * Ft;
  float* P = static_cast<float*>(ws);
  r.epi = EPI_F32; r.d = P; r.ldd = h; r.d_batch_stride = M * h;
  // data-parallel schedule: the partials are then the same bits as the overlapped path's
  TP_RETURN_IF(run_gemm(r, s));
  return run_shard_reduce(P, M, h, t, bdown, residual, Y, nullptr, s);
}

// Column-sum scratch of the MLP backward: db_down's partial pass over dY, then db_up's
// partials, one row per 32-row block of each shard's dZ, written by the dgrad epilogue.
size_t mlp_cs_floats(int64_t M, int64_t h, int64_t Ft, int t) {
  const int64_t blocks = (M + 31) / 32;
  return colsum2_ws_floats(M, h, 1) + static_cast<size_t>(t) * (blocks > 0 ? blocks : 1) * Ft;
}

// Required scratch of the MLP backward: dZ (twice as wide under SwiGLU: gate and up),
// column-sum scratch, partials; sized for every activation.
size_t mlp_bwd_base_ws(int64_t M, int64_t h, int64_t F, int t, unsigned flags) {
  const int64_t Ft = F / t;
  size_t sz = round_up(static_cast<size_t>(M) * F * 2 * 2, 256);
  const size_t cs = mlp_cs_floats(M, h, Ft, t);
  sz += round_up(cs * sizeof(float), 256);
  if (flags & TP_FLAG_UNFUSED_REDUCE) sz += static_cast<size_t>(t) * M * h * sizeof(float);
  return sz;
}

size_t tp_mlp_backward_workspace_size(int64_t M, int64_t h, int64_t F, int t, unsigned flags) {
  if (M < 0 || h < 0 || F < 0 || t < 1) return 0;
  // the required part, then room for the GEMMs' split-K partials
  return round_up(mlp_bwd_base_ws(M, h, F, t, flags), 256) + gemm_sk_ws_bytes();
}

tp_status tp_mlp_backward(const tp_bf16* dY, const tp_bf16* X, const tp_bf16* Z_save, const tp_bf16* A_save,
                          int64_t M, int64_t h, int64_t F, int t, tp_act act, const tp_bf16* Wup_p,
                          const tp_bf16* Wdown_p, tp_bf16* dX, float* dWup_p, float* dWdown_p, float* dbup,
                          float* dbdown, int accumulate, unsigned flags, void* ws, size_t ws_bytes,
                          tp_stream stream) {
  TP_TRACE();
  if (M < 0 || h < 1 || F < 1 || t < 1 || !mlp_act_ok(act)) return TP_ERR_INVALID_ARG;
  if (!dWup_p || !dWdown_p) return TP_ERR_INVALID_ARG;
  const bool swiglu = act == TP_ACT_SWIGLU;
  if (swiglu && (F / t) % 128 != 0) return TP_ERR_SHAPE;
  if (swiglu && dbup) return TP_ERR_UNSUPPORTED;
  if (M > 0 && (!dY || !X || !A_save || !Wup_p || !Wdown_p || !dX)) return TP_ERR_INVALID_ARG;
  if (M > 0 && act != TP_ACT_IDENTITY && !Z_save) return TP_ERR_INVALID_ARG;
  if (F % t != 0) return TP_ERR_SHAPE;
  const int64_t Ft = F / t;
  if (h % 8 != 0 || Ft % 8 != 0) return TP_ERR_ALIGN;
  const size_t base_ws = mlp_bwd_base_ws(M, h, F, t, flags);
  if (!ws || ws_bytes < base_ws) return TP_ERR_WORKSPACE;
  size_t sk_bytes = 0;
  void* sk_ws = sk_part_of(ws, ws_bytes, base_ws, &sk_bytes);  // split K, when the workspace has room
  if (!aligned16(ws)) return TP_ERR_ALIGN;
  const cudaStream_t s = S(stream);
  const bool unfused = (flags & TP_FLAG_UNFUSED_REDUCE) != 0;

  const int64_t Fzt = swiglu ? 2 * Ft : Ft;  // columns of a shard's Z / dZ
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* dZ = reinterpret_cast<uint16_t*>(w);
  w += round_up(static_cast<size_t>(M) * F * 2 * 2, 256);
  float* cs_ws = reinterpret_cast<float*>(w);
  const size_t cs_floats = mlp_cs_floats(M, h, Ft, t);
  float* dbup_part = cs_ws + colsum2_ws_floats(M, h, 1);  // [t][(M + 31) / 32][Ft]
  w += round_up(cs_floats * sizeof(float), 256);
  float* P = reinterpret_cast<float*>(w);

  if (M == 0) {  // no tokens: every gradient is zero (or unchanged when accumulating)
    if (!accumulate) {
      TP_RETURN_IF(ready());
      TP_CUDA_CHECK(cudaMemsetAsync(dWup_p, 0, sizeof(float) * Fzt * t * h, s));
      TP_CUDA_CHECK(cudaMemsetAsync(dWdown_p, 0, sizeof(float) * F * h, s));
      if (dbup) TP_CUDA_CHECK(cudaMemsetAsync(dbup, 0, sizeof(float) * F, s));
      if (dbdown) TP_CUDA_CHECK(cudaMemsetAsync(dbdown, 0, sizeof(float) * h, s));
    }
    return TP_OK;
  }

  // dgrad + act': dZ_i = (dY W_down,i^T) * act'(Z_i).  SwiGLU: the epilogue turns dA_i =
  // dY W_down,i^T into d gate = dA u silu'(gate) and d up = dA silu(gate), interleaved like Z.
  GemmProblem g;
  g.M = M; g.N = Ft; g.K = h; g.nbatch = t;
  g.a.ptr = dY; g.a.ld = h;
  g.b.ptr = Wdown_p; g.b.ld = Ft; g.b.sharded = true; g.b.shard_stride = h * Ft; g.b.mn_major = true;
  if (swiglu) {
    g.epi = EPI_DGLU; g.aux = Z_save; g.ld_aux = 2 * Ft; g.aux_batch_stride = M * 2 * Ft;
    g.d = dZ; g.ldd = 2 * Ft; g.d_batch_stride = M * 2 * Ft;
  } else {
    g.epi = EPI_DACT; g.act = act; g.aux = Z_save ? Z_save : A_save; g.ld_aux = Ft; g.aux_batch_stride = M * Ft;
    g.d = dZ; g.ldd = Ft; g.d_batch_stride = M * Ft;
    g.colsum = dbup ? dbup_part : nullptr;  // db_up's partial column sums from the epilogue
  }
  g.sk_ws = sk_ws; g.sk_ws_bytes = sk_bytes;
  TP_RETURN_IF(run_gemm(g, s));

  // Bias gradients: db_down = sum_rows dY, taken once (g backward is the identity), by a
  // partial and a final pass; db_up[C_i] = sum_rows dZ_i for every shard, whose per-32-row
  // partials the dgrad epilogue wrote, by the final pass alone (one launch for both sums).
  if (dbdown || dbup) {
    ColsumJob jd, ju;
    if (dbdown) {
      jd.G = dY; jd.rows = M; jd.cols = h; jd.ld = h; jd.bs = M * h; jd.nbatch = 1;
      jd.out = dbdown; jd.ws = cs_ws; jd.accumulate = accumulate;
    }
    if (dbup) {  // the dgrad epilogue wrote the partials: only their in-order sum is left
      ju.rows = M; ju.cols = Ft; ju.nbatch = t;
      ju.out = dbup; ju.ws = dbup_part; ju.accumulate = accumulate;
      ju.partials_ready = 1; ju.nchunks = static_cast<int>((M + 31) / 32);
    }
    TP_RETURN_IF(run_colsum2(jd, ju, s));
  }

  // Local weight gradients (no reduction): dW_down,i = A_i^T dY  -> packed [t][h][Ft].
  GemmProblem wd;
  wd.M = h; wd.N = Ft; wd.K = M; wd.nbatch = t;
  wd.a.ptr = dY; wd.a.ld = h; wd.a.mn_major = true;
  wd.b.ptr = A_save; wd.b.ld = Ft; wd.b.sharded = true; wd.b.shard_stride = M * Ft; wd.b.mn_major = true;
  wd.epi = EPI_F32; wd.d = dWdown_p; wd.ldd = Ft; wd.d_batch_stride = h * Ft; wd.accumulate = accumulate;
  wd.sk_ws = sk_ws; wd.sk_ws_bytes = sk_bytes;  // split K needs the TMA-store (non-accumulating) epilogue
  TP_RETURN_IF(run_gemm(wd, s));

  // dW_up,i = dZ_i^T X -> packed [t][Ft][h] (SwiGLU: [t][2 Ft][h], tp_pack_swiglu's layout).
  GemmProblem wu;
  wu.M = Fzt; wu.N = h; wu.K = M; wu.nbatch = t;
  wu.a.ptr = dZ; wu.a.ld = Fzt; wu.a.sharded = true; wu.a.shard_stride = M * Fzt; wu.a.mn_major = true;
  wu.b.ptr = X; wu.b.ld = h; wu.b.mn_major = true;
  wu.epi = EPI_F32; wu.d = dWup_p; wu.ldd = h; wu.d_batch_stride = Fzt * h; wu.accumulate = accumulate;
  wu.sk_ws = sk_ws; wu.sk_ws_bytes = sk_bytes;
  TP_RETURN_IF(run_gemm(wu, s));

  // f backward: dX = sum_i dZ_i W_up,i^T.
  GemmProblem dx;
  dx.M = M; dx.N = h; dx.K = Fzt;
  dx.a.ptr = dZ; dx.a.ld = Fzt; dx.a.sharded = true; dx.a.shard_stride = M * Fzt;
  dx.b.ptr = Wup_p; dx.b.ld = h; dx.b.sharded = true; dx.b.shard_stride = Fzt * h; dx.b.mn_major = true;
  dx.sk_ws = sk_ws; dx.sk_ws_bytes = sk_bytes;
  if (!unfused) {
    dx.nsum = t;
    dx.epi = EPI_BF16; dx.d = dX; dx.ldd = h;
    return run_gemm(dx, s);
  }
  dx.nbatch = t;
  dx.epi = EPI_F32; dx.d = P; dx.ldd = h; dx.d_batch_stride = M * h;
  TP_RETURN_IF(run_gemm(dx, s));
  return run_shard_reduce(P, M, h, t, nullptr, nullptr, dX, nullptr, s);
}

// ------------------------------------------------------------------ decode
tp_status tp_decode_swiglu_forward(const tp_bf16* x, int64_t M, int64_t h, int64_t F, int t,
                                   const tp_bf16* Wgu_p, const tp_bf16* Wdown_p, tp_bf16* y, tp_bf16* a_save,
                                   tp_stream stream) {
  TP_TRACE();
  return run_decode_swiglu(x, M, h, F, t, Wgu_p, Wdown_p, y, a_save, S(stream));
}

// ----------------------------------------------------------- vocab embedding
tp_status tp_vocab_embedding_forward(const int32_t* ids, int64_t N, int64_t V, int64_t h, int t, const tp_bf16* E_p,
                                     tp_bf16* Y, tp_stream stream) {
  TP_TRACE();
  return run_emb_forward(ids, N, V, h, t, E_p, Y, S(stream));
}

size_t tp_vocab_embedding_backward_workspace_size(int64_t N) { return N < 0 ? 0 : emb_bwd_ws_bytes(N); }

tp_status tp_vocab_embedding_backward(const int32_t* ids, const tp_bf16* dY, int64_t N, int64_t V, int64_t h, int t,
                                      float* dE_p, int accumulate, void* ws, size_t ws_bytes, tp_stream stream) {
  TP_TRACE();
  return run_emb_backward(ids, dY, N, V, h, t, dE_p, accumulate, ws, ws_bytes, S(stream));
}

// ----------------------------------------------------------- decode attention
size_t tp_decode_attn_workspace_size(int64_t B, int64_t d, int n_heads, int n_kv_heads, int head_dim, int t,
                                     int64_t L_max) {
  return decode_attn_ws_bytes(B, d, n_heads, n_kv_heads, head_dim, t, L_max);
}

tp_status tp_decode_attn_forward(const tp_bf16* x, int64_t B, int64_t d, int n_heads, int n_kv_heads, int head_dim,
                                 int t, float scale, const tp_bf16* Wqkv_p, const tp_bf16* bqkv_p,
                                 const tp_bf16* Wo_p, const tp_bf16* bo, uint16_t* K_cache, uint16_t* V_cache,
                                 int64_t L_max, const int32_t* pos, tp_bf16* y, void* ws, size_t ws_bytes,
                                 tp_stream stream) {
  TP_TRACE();
  return run_decode_attn(x, B, d, n_heads, n_kv_heads, head_dim, t, scale, Wqkv_p, bqkv_p, Wo_p, bo, K_cache, V_cache,
                         L_max, pos, y, ws, ws_bytes, S(stream));
}

// ------------------------------------------------------------------ attention
tp_status tp_attn_gqa_forward(const tp_bf16* X, int64_t N, int64_t d, int n_heads, int n_kv_heads, int head_dim,
                              int t, int causal, float scale, const tp_bf16* Wqkv_p, const tp_bf16* bqkv_p,
                              const tp_bf16* Wo_p, const tp_bf16* bo, const tp_bf16* residual, tp_bf16* Y,
                              uint16_t* QKV_save, tp_bf16* O_save, float* lse_save, unsigned flags, void* ws,
                              size_t ws_bytes, tp_stream stream) {
  TP_TRACE();
  if (N < 0 || d < 1 || n_heads < 1 || n_kv_heads < 1 || t < 1 || head_dim < 1) return TP_ERR_INVALID_ARG;
  if ((flags & ~TP_ATTN_F16_INPUT) != 0) return TP_ERR_UNSUPPORTED;
  if (!gqa_ok(d, n_heads, n_kv_heads, head_dim, t)) return TP_ERR_SHAPE;
  if (N == 0) return TP_OK;
  if (!X || !Wqkv_p || !Wo_p || !Y || !QKV_save || !O_save || !lse_save) return TP_ERR_INVALID_ARG;
  // f (identity) + column-parallel W_qkv by KV group: QKV_i = X W_qkv,i + b_qkv,i, stored fp16.
  const int64_t rw = qkv_row_width(n_heads, n_kv_heads, head_dim, t);
  GemmProblem c;
  c.M = N; c.N = rw; c.K = d; c.nbatch = t;
  c.a.ptr = X; c.a.ld = d;
  c.b.ptr = Wqkv_p; c.b.ld = d; c.b.sharded = true; c.b.shard_stride = rw * d;
  c.epi = EPI_ACT; c.act = TP_ACT_IDENTITY; c.out_f16 = 1;
  c.f16_ab = (flags & TP_ATTN_F16_INPUT) ? 1 : 0;  // X and W_qkv in IEEE fp16
  c.d = nullptr; c.d2 = QKV_save; c.ldd = rw; c.d_batch_stride = N * rw;
  c.bias = bqkv_p; c.bias_batch_stride = rw;
  size_t sk_bytes = 0;
  void* sk_ws = sk_part_of(ws, ws_bytes, 0, &sk_bytes);  // optional: the GEMMs' split-K partials
  c.sk_ws = sk_ws; c.sk_ws_bytes = sk_bytes;
  TP_RETURN_IF(run_gemm(c, S(stream)));
  // Attention on each shard's own query heads, no communication.
  TP_RETURN_IF(run_attention_fwd(QKV_save, N, d, n_heads, n_kv_heads, head_dim, t, causal, scale, O_save, lse_save,
                                 S(stream)));
  // Row-parallel W_o + g: Y = sum_i O_i W_o,i + b_o (once) + residual.
  return row_parallel(O_save, N, d, d, t, Wo_p, bo, residual, Y, sk_ws, sk_bytes, S(stream));
}

size_t tp_attn_forward_workspace_size(int64_t N, int64_t d, int n_heads, int head_dim, int t, unsigned flags) {
  (void)N; (void)d; (void)n_heads; (void)head_dim; (void)t; (void)flags;
  return gemm_sk_ws_bytes();
}

tp_status tp_attn_forward(const tp_bf16* X, int64_t N, int64_t d, int n_heads, int head_dim, int t, int causal,
                          float scale, const tp_bf16* Wqkv_p, const tp_bf16* bqkv_p, const tp_bf16* Wo_p,
                          const tp_bf16* bo, const tp_bf16* residual, tp_bf16* Y, tp_bf16* QKV_save,
                          tp_bf16* O_save, float* lse_save, unsigned flags, void* ws, size_t ws_bytes,
                          tp_stream stream) {
  TP_TRACE();
  if (N < 0 || d < 1 || n_heads < 1 || t < 1 || head_dim < 1) return TP_ERR_INVALID_ARG;
  if ((flags & ~TP_ATTN_F16_INPUT) != 0) return TP_ERR_UNSUPPORTED;
  if (head_dim != 128 || static_cast<int64_t>(n_heads) * head_dim != d || n_heads % t != 0) return TP_ERR_SHAPE;
  return tp_attn_gqa_forward(X, N, d, n_heads, n_heads, head_dim, t, causal, scale, Wqkv_p, bqkv_p, Wo_p, bo, residual,
                             Y, QKV_save, O_save, lse_save, flags, ws, ws_bytes, stream);
}

tp_status tp_attn_core_forward(const uint16_t* QKV, int64_t N, int64_t d, int n_heads, int n_kv_heads, int head_dim,
                               int t, int causal, float scale, tp_bf16* O, float* lse, tp_stream stream) {
  TP_TRACE();
  return run_attention_fwd(QKV, N, d, n_heads, n_kv_heads, head_dim, t, causal, scale, O, lse, S(stream));
}

tp_status tp_attn_core_backward(const uint16_t* QKV, const tp_bf16* O, const uint16_t* dO, const float* lse,
                                int64_t N, int64_t d, int n_heads, int n_kv_heads, int head_dim, int t, int causal,
                                float scale, float* Dvec, tp_bf16* dQKV, tp_stream stream) {
  TP_TRACE();
  return run_attention_bwd(QKV, O, dO, lse, N, d, n_heads, n_kv_heads, head_dim, t, causal, scale, Dvec, dQKV,
                           S(stream));
}

// Sum of the t shards' packed W_qkv gradients into the unsplit (d, (n_heads + 2 n_kv) head_dim)
// gradient: every column receives the gradient of each shard copy that holds it, added in
// shard order (the replica-group all-reduce of a replicated KV head's weights).
tp_status tp_reduce_qkv_gqa_grad(const float* dWp, int64_t d, int n_heads, int n_kv_heads, int head_dim, int t,
                                 float* dW, int accumulate, tp_stream stream) {
  TP_TRACE();
  return reduce_qkv_gqa_grad(dWp, d, n_heads, n_kv_heads, head_dim, t, dW, accumulate, S(stream));
}

// ------------------------------------------------------------------ LayerNorm
tp_status tp_sp_layernorm_forward(const tp_bf16* X_sh, int64_t s, int64_t h, int t, const tp_bf16* gamma,
                                  const tp_bf16* beta, float eps, tp_bf16* Y_sh, float* mean, float* rstd,
                                  tp_stream stream) {
  TP_TRACE();
  return run_ln_forward(X_sh, s, h, t, gamma, beta, eps, Y_sh, mean, rstd, S(stream));
}

tp_status tp_sp_layernorm_forward_f16(const tp_bf16* X_sh, int64_t s, int64_t h, int t, const tp_bf16* gamma,
                                      const tp_bf16* beta, float eps, uint16_t* Y_sh, float* mean, float* rstd,
                                      tp_stream stream) {
  TP_TRACE();
  return run_ln_forward(X_sh, s, h, t, gamma, beta, eps, Y_sh, mean, rstd, S(stream), 1);
}

tp_status tp_convert_bf16_to_f16(const tp_bf16* src, int64_t n, uint16_t* dst, tp_stream stream) {
  TP_TRACE();
  return run_bf16_to_f16(src, n, dst, S(stream));
}

tp_status tp_sp_layernorm_backward(const tp_bf16* dY_sh, const tp_bf16* X_sh, const tp_bf16* gamma,
                                   const float* mean, const float* rstd, const tp_bf16* dres, int64_t s, int64_t h,
                                   int t, tp_bf16* dX_sh, float* dgamma_part, float* dbeta_part, float* dgamma,
                                   float* dbeta, tp_stream stream) {
  TP_TRACE();
  return run_ln_backward(dY_sh, X_sh, gamma, mean, rstd, dres, s, h, t, dX_sh, dgamma_part, dbeta_part, dgamma,
                         dbeta, S(stream));
}

// ------------------------------------------------------------------ utilities
tp_status tp_shard_reduce(const float* P, int64_t rows, int64_t cols, int t, const tp_bf16* bias,
                          const tp_bf16* residual, tp_bf16* out_bf16, float* out_f32, tp_stream stream) {
  TP_TRACE();
  return run_shard_reduce(P, rows, cols, t, bias, residual, out_bf16, out_f32, S(stream));
}

size_t tp_colsum_workspace_size(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0) return 0;
  return colsum_ws_floats(rows, cols) * sizeof(float);
}

tp_status tp_colsum(const tp_bf16* G, int64_t rows, int64_t cols, float* out, int accumulate, void* ws,
                    size_t ws_bytes, tp_stream stream) {
  TP_TRACE();
  return run_colsum(G, rows, cols, cols, out, accumulate, static_cast<float*>(ws), ws_bytes / sizeof(float),
                    S(stream));
}

}  // extern "C"
