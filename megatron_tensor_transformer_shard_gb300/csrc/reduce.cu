// HBM-bound reductions of the TP block:
//   shard_reduce  out = sum_{i=0..t-1} P_i + bias (once) + residual -- the
//                 unfused stand-in for the g / f all-reduce ("Tensor and sequence
//                 parallelism", f/g table), summing the t partial buffers in
//                 shard order;
//   colsum        fixed-order column sums (bias gradients db = sum over rows).
#include <cuda_runtime.h>

#include "devmath.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace tp {
namespace {

constexpr int COLSUM_ROWS_PER_CHUNK = 64;
constexpr int COLSUM_THREADS = 128;  // x 2 columns each = 256 columns per CTA

// Phase 1: ws[batch][chunk][col] = sum of rows [chunk*64, chunk*64+64) of batch b, in row order.
// blockIdx.x = chunk * cblocks + column block (the chunk count can exceed gridDim.y's 65535),
// blockIdx.y = batch.
__global__ void colsum_partial_kernel(const uint16_t* __restrict__ G, int64_t rows, int64_t cols, int64_t ld,
                                      int64_t batch_stride, int nchunks, int cblocks, float* __restrict__ ws) {
  const int cb = static_cast<int>(blockIdx.x % static_cast<unsigned>(cblocks));
  const int chunk = static_cast<int>(blockIdx.x / static_cast<unsigned>(cblocks));
  const int64_t c = (static_cast<int64_t>(cb) * COLSUM_THREADS + threadIdx.x) * 2;
  const int b = blockIdx.y;
  if (c >= cols) return;
  const int64_t r0 = static_cast<int64_t>(chunk) * COLSUM_ROWS_PER_CHUNK;
  const int64_t r1 = r0 + COLSUM_ROWS_PER_CHUNK < rows ? r0 + COLSUM_ROWS_PER_CHUNK : rows;
  const uint16_t* g = G + b * batch_stride + c;
  float s0 = 0.0f, s1 = 0.0f;
  if (c + 1 < cols) {
    for (int64_t r = r0; r < r1; ++r) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(g + r * ld);
      float a, bb;
      unpack_bf16x2(w, a, bb);
      s0 += a;
      s1 += bb;
    }
  } else {
    for (int64_t r = r0; r < r1; ++r) s0 += bf16_bits_to_float(g[r * ld]);
  }
  float* o = ws + (static_cast<int64_t>(b) * nchunks + chunk) * cols + c;
  o[0] = s0;
  if (c + 1 < cols) o[1] = s1;
}

// Phase 2: out[b*cols + c] (+)= sum_{chunk} ws[b][chunk][c], chunks in order.
__global__ void colsum_final_kernel(const float* __restrict__ ws, int64_t cols, int nchunks, int nbatch,
                                    float* __restrict__ out, int accumulate) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= cols * nbatch) return;
  const int64_t b = idx / cols, c = idx - b * cols;
  const float* w = ws + b * nchunks * cols + c;
  float s = 0.0f;
  for (int k = 0; k < nchunks; ++k) s += w[static_cast<int64_t>(k) * cols];
  out[idx] = accumulate ? out[idx] + s : s;
}

__global__ void shard_reduce_kernel(const float* __restrict__ P, int64_t rows, int64_t cols, int t,
                                    const uint16_t* __restrict__ bias, const uint16_t* __restrict__ res,
                                    uint16_t* __restrict__ out_bf16, float* __restrict__ out_f32) {
  const int64_t n4 = rows * cols / 4;
  const int64_t shard = rows * cols;
  for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < n4;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = q * 4;
    float4 acc = reinterpret_cast<const float4*>(P + e)[0];
    for (int i = 1; i < t; ++i) {  // fixed shard order
      const float4 v = reinterpret_cast<const float4*>(P + i * shard + e)[0];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    const int64_t c = e % cols;
    if (bias) {
      acc.x += bf16_bits_to_float(bias[c]);
      acc.y += bf16_bits_to_float(bias[c + 1]);
      acc.z += bf16_bits_to_float(bias[c + 2]);
      acc.w += bf16_bits_to_float(bias[c + 3]);
    }
    if (res) {
      acc.x += bf16_bits_to_float(res[e]);
      acc.y += bf16_bits_to_float(res[e + 1]);
      acc.z += bf16_bits_to_float(res[e + 2]);
      acc.w += bf16_bits_to_float(res[e + 3]);
    }
    if (out_f32) reinterpret_cast<float4*>(out_f32 + e)[0] = acc;
    if (out_bf16) {
      uint2 w;
      w.x = pack_bf16x2(acc.x, acc.y);
      w.y = pack_bf16x2(acc.z, acc.w);
      reinterpret_cast<uint2*>(out_bf16 + e)[0] = w;
    }
  }
}

// ---- fused column sums of two matrices (e.g. db_down from dY and every
// shard's db_up from dZ) in two launches: a partial pass with 16-byte loads,
// 64-row chunks (a warp's 8 rows all in flight), 8 warps per CTA combined in warp
// order, and a final pass in which 8 warps take consecutive runs of a column's
// chunks, each run summed in order, and the runs are added in order.  Deterministic.
constexpr int CS2_ROWS = 64;
constexpr int CS2_THREADS = 256;  // 8 warps x 32 lanes x 8 columns: 256 columns per CTA

__device__ __forceinline__ const ColsumJob& pick(const ColsumJob& a, const ColsumJob& b, bool first) {
  return first ? a : b;
}

// Two 16-bit values of a job's matrix (bf16, or IEEE fp16 when f16) as floats.
__device__ __forceinline__ void unpack2(uint32_t w, bool f16, float& a, float& b) {
  if (f16) unpack_f16x2(w, a, b);
  else unpack_bf16x2(w, a, b);
}

// Both colsum2 kernels are launched with programmatic dependent launch: they wait
// for the previous kernel's results before reading anything and let the next
// kernel on the stream set up while they run.
__global__ void __launch_bounds__(CS2_THREADS) colsum2_partial_kernel(ColsumJob j0, ColsumJob j1, int64_t n0) {
  __shared__ float red[8][256];
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const bool first = blockIdx.x < n0;
  const ColsumJob& j = pick(j0, j1, first);
  const int64_t local = first ? blockIdx.x : blockIdx.x - n0;
  const int64_t cb = local % j.cblocks;
  const int64_t rest = local / j.cblocks;
  const int chunk = static_cast<int>(rest % j.nchunks);
  const int b = static_cast<int>(rest / j.nchunks);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t c0 = cb * 256 + lane * 8;
  const int64_t r0 = static_cast<int64_t>(chunk) * CS2_ROWS;
  const int64_t r1 = r0 + CS2_ROWS < j.rows ? r0 + CS2_ROWS : j.rows;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const uint16_t* g = j.G + b * j.bs;
  const bool f16 = j.f16 != 0;
  if (c0 + 8 <= j.cols) {
    int64_t r = r0 + warp;
    for (; r + 56 < r1; r += 64) {  // eight rows in flight per thread
      uint4 w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) w[u] = *reinterpret_cast<const uint4*>(g + (r + 8 * u) * j.ld + c0);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float a0, a1;
        unpack2(w[u].x, f16, a0, a1); acc[0] += a0; acc[1] += a1;
        unpack2(w[u].y, f16, a0, a1); acc[2] += a0; acc[3] += a1;
        unpack2(w[u].z, f16, a0, a1); acc[4] += a0; acc[5] += a1;
        unpack2(w[u].w, f16, a0, a1); acc[6] += a0; acc[7] += a1;
      }
    }
    for (; r < r1; r += 8) {
      const uint4 w = *reinterpret_cast<const uint4*>(g + r * j.ld + c0);
      float a0, a1;
      unpack2(w.x, f16, a0, a1); acc[0] += a0; acc[1] += a1;
      unpack2(w.y, f16, a0, a1); acc[2] += a0; acc[3] += a1;
      unpack2(w.z, f16, a0, a1); acc[4] += a0; acc[5] += a1;
      unpack2(w.w, f16, a0, a1); acc[6] += a0; acc[7] += a1;
    }
  } else {
    for (int64_t r = r0 + warp; r < r1; r += 8)
      for (int e = 0; e < 8; ++e)
        if (c0 + e < j.cols) {
          const uint16_t x = g[r * j.ld + c0 + e];
          acc[e] += f16 ? __half2float(*reinterpret_cast<const __half*>(&x)) : bf16_bits_to_float(x);
        }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) red[warp][lane * 8 + e] = acc[e];
  __syncthreads();
  const int64_t c = cb * 256 + threadIdx.x;
  if (c < j.cols) {
    float s2 = 0.0f;
#pragma unroll
    for (int w2 = 0; w2 < 8; ++w2) s2 += red[w2][threadIdx.x];
    j.ws[(static_cast<int64_t>(b) * j.nchunks + chunk) * j.cols + c] = s2;
  }
}

constexpr int CS2F_WARPS = 8;  // final pass: 32 columns per CTA, a run of chunks per warp

__global__ void __launch_bounds__(CS2F_WARPS * 32) colsum2_final_kernel(ColsumJob j0, ColsumJob j1, int64_t n0,
                                                                        int64_t n) {
  __shared__ float red[CS2F_WARPS][32];
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const bool first = idx < n0;
  const ColsumJob& j = pick(j0, j1, first);
  const int64_t local = first ? idx : idx - n0;
  float s = 0.0f;
  if (idx < n) {
    const int64_t b = local / j.cols, c = local - b * j.cols;
    const float* w = j.ws + b * j.nchunks * j.cols + c;
    // warp `warp` sums chunks [k0, k1) in order, up to 16 loads in flight
    const int k0 = static_cast<int>(static_cast<int64_t>(j.nchunks) * warp / CS2F_WARPS);
    const int k1 = static_cast<int>(static_cast<int64_t>(j.nchunks) * (warp + 1) / CS2F_WARPS);
#pragma unroll 16
    for (int k = k0; k < k1; ++k) s += w[static_cast<int64_t>(k) * j.cols];
  }
  red[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && idx < n) {
    float t = 0.0f;
#pragma unroll
    for (int w2 = 0; w2 < CS2F_WARPS; ++w2) t += red[w2][lane];  // the runs in order
    j.out[local] = j.accumulate ? j.out[local] + t : t;
  }
}

}  // namespace

size_t colsum2_ws_floats(int64_t rows, int64_t cols, int nbatch) {
  const int64_t nchunks = (rows + CS2_ROWS - 1) / CS2_ROWS;
  return static_cast<size_t>(nchunks > 0 ? nchunks : 1) * static_cast<size_t>(cols) * static_cast<size_t>(nbatch);
}

// Column sums of two jobs ([nbatch][rows][cols], row stride ld, batch stride bs)
// into job.out[nbatch][cols]; job.ws must hold colsum2_ws_floats() floats.
tp_status run_colsum2(ColsumJob a, ColsumJob b, cudaStream_t s) {
  ColsumJob* js[2] = {&a, &b};
  int64_t ctas[2] = {0, 0}, outs[2] = {0, 0};
  for (int k = 0; k < 2; ++k) {
    ColsumJob& j = *js[k];
    if (j.rows < 0 || j.cols < 0 || j.nbatch < 1) return TP_ERR_INVALID_ARG;
    if (j.cols == 0) continue;
    if (j.partials_ready) {  // the partials are in ws already: only the final sum
      if (!j.out || !j.ws || j.nchunks < 1) return TP_ERR_INVALID_ARG;
      outs[k] = j.cols * j.nbatch;
      continue;
    }
    if (!j.G || !j.out || !j.ws || (j.cols & 7) || (j.ld & 7) || (j.bs & 7) || !aligned16(j.G))
      return TP_ERR_ALIGN;
    j.nchunks = static_cast<int>((j.rows + CS2_ROWS - 1) / CS2_ROWS);
    j.cblocks = (j.cols + 255) / 256;
    if (j.nchunks == 0) {
      j.nchunks = 1;  // no rows: the partial pass writes zeros
    }
    ctas[k] = j.cblocks * j.nchunks * j.nbatch;
    outs[k] = j.cols * j.nbatch;
  }
  const int64_t n = outs[0] + outs[1];
  if (n == 0) return TP_OK;
  TP_RETURN_IF(ready());
  if (ctas[0] + ctas[1] > 0) {
    TP_CUDA_CHECK(launch_pdl(colsum2_partial_kernel, dim3(static_cast<unsigned>(ctas[0] + ctas[1])),
                             dim3(CS2_THREADS), 0, s, a, b, ctas[0]));
    count_launch();
  }
  TP_CUDA_CHECK(launch_pdl(colsum2_final_kernel, dim3(static_cast<unsigned>((n + 31) / 32)), dim3(CS2F_WARPS * 32), 0,
                           s, a, b, outs[0], n));
  count_launch();
  return TP_OK;
}

size_t colsum_ws_floats(int64_t rows, int64_t cols) {
  const int64_t nchunks = (rows + COLSUM_ROWS_PER_CHUNK - 1) / COLSUM_ROWS_PER_CHUNK;
  return static_cast<size_t>(nchunks > 0 ? nchunks : 1) * static_cast<size_t>(cols);
}

// Column sums of `nbatch` matrices [rows][cols] (row stride ld, batch stride
// rows*ld) -> out[nbatch][cols].  ws must hold nbatch * colsum_ws_floats(rows, cols).
tp_status run_colsum_batched(const uint16_t* G, int64_t rows, int64_t cols, int64_t ld, int nbatch,
                             int64_t batch_stride, float* out, int accumulate, float* ws, size_t ws_floats,
                             cudaStream_t s) {
  if (rows < 0 || cols < 0 || nbatch < 1) return TP_ERR_INVALID_ARG;
  if (cols == 0) return TP_OK;
  if (!G || !out || !ws) return TP_ERR_INVALID_ARG;
  if ((cols & 1) || (ld & 1) || (batch_stride & 1) || (reinterpret_cast<uintptr_t>(G) & 3)) return TP_ERR_ALIGN;
  const int64_t nchunks64 = (rows + COLSUM_ROWS_PER_CHUNK - 1) / COLSUM_ROWS_PER_CHUNK;
  if (nchunks64 > 0x7fffffffLL) return TP_ERR_SHAPE;
  const int nchunks = static_cast<int>(nchunks64);
  if (ws_floats < colsum_ws_floats(rows, cols) * static_cast<size_t>(nbatch)) return TP_ERR_WORKSPACE;
  // Grid: (chunks x column blocks, batches); both within CUDA's grid limits, else refused.
  const int64_t cblocks = (cols / 2 + COLSUM_THREADS - 1) / COLSUM_THREADS;
  if (static_cast<int64_t>(nchunks) * cblocks > 0x7fffffffLL || nbatch > 65535) return TP_ERR_SHAPE;
  TP_RETURN_IF(ready());
  if (nchunks == 0) {
    if (!accumulate) TP_CUDA_CHECK(cudaMemsetAsync(out, 0, sizeof(float) * cols * nbatch, s));
    return TP_OK;
  }
  dim3 g1(static_cast<unsigned>(static_cast<int64_t>(nchunks) * cblocks), static_cast<unsigned>(nbatch));
  colsum_partial_kernel<<<g1, COLSUM_THREADS, 0, s>>>(G, rows, cols, ld, batch_stride, nchunks,
                                                      static_cast<int>(cblocks), ws);
  TP_LAUNCHED();
  const int64_t n = cols * nbatch;
  colsum_final_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(ws, cols, nchunks, nbatch, out,
                                                                             accumulate);
  TP_LAUNCHED();
  return TP_OK;
}

tp_status run_colsum(const uint16_t* G, int64_t rows, int64_t cols, int64_t ld, float* out, int accumulate,
                     float* ws, size_t ws_floats, cudaStream_t s) {
  return run_colsum_batched(G, rows, cols, ld, 1, rows * ld, out, accumulate, ws, ws_floats, s);
}

tp_status run_shard_reduce(const float* P, int64_t rows, int64_t cols, int t, const uint16_t* bias,
                           const uint16_t* residual, uint16_t* out_bf16, float* out_f32, cudaStream_t s) {
  if (rows < 0 || cols < 0 || t < 1) return TP_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return TP_OK;
  if (!P || (!out_bf16 && !out_f32)) return TP_ERR_INVALID_ARG;
  if (cols % 8 != 0 || !aligned16(P) || (out_f32 && !aligned16(out_f32)) || (out_bf16 && !aligned16(out_bf16)) ||
      (residual && !aligned16(residual)) || (bias && !aligned16(bias)))
    return TP_ERR_ALIGN;
  TP_RETURN_IF(ready());
  const int64_t n4 = rows * cols / 4;
  int64_t blocks = (n4 + 255) / 256;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  shard_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(P, rows, cols, t, bias, residual, out_bf16,
                                                                     out_f32);
  TP_LAUNCHED();
  return TP_OK;
}

}  // namespace tp
