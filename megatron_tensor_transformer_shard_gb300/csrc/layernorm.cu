// Sequence-parallel LayerNorm ("Tensor and sequence parallelism", section
// "Sequence parallelism"; "02 — Tensor Parallelism", "Sequence parallelism
// (Megatron-3)").  X_sh [t][s/t][h] is the same bytes as [s][h]: the
// all-gather that enters the TP region and the reduce-scatter that leaves it
// are layouts, not copies.  What sequence parallelism adds is the weight
// gradient: each shard j only sees its own rows, so it produces a partial
// (dgamma_j, dbeta_j) and the partials are summed over j -- the extra
// all-reduce -- in a fixed shard order.
//
//   row kernels     one CTA per row, the row held in registers as packed bf16
//                   words (8-element chunks, up to 4 per thread), block
//                   reductions for the statistics (two-pass mean and variance);
//                   HBM-bound: read x (+ dy, dres), write y / dx.
//   column kernel   one CTA per (64-column block, shard), 16-byte loads, eight
//                   warps of four rows each striding the shard's rows, combined
//                   in a fixed order; then one launch sums the shard partials in
//                   shard order.
#include <cuda_runtime.h>

#include "devmath.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace tp {
namespace {

constexpr int LN_CHUNKS = 4;  // 8-element chunks per thread -> h <= 1024*32

__device__ __forceinline__ void load8(const uint16_t* p, float (&v)[8]) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  unpack_bf16x2(w.x, v[0], v[1]);
  unpack_bf16x2(w.y, v[2], v[3]);
  unpack_bf16x2(w.z, v[4], v[5]);
  unpack_bf16x2(w.w, v[6], v[7]);
}

__device__ __forceinline__ void store8(uint16_t* p, const float (&v)[8]) {
  uint4 w;
  w.x = pack_bf16x2(v[0], v[1]);
  w.y = pack_bf16x2(v[2], v[3]);
  w.z = pack_bf16x2(v[4], v[5]);
  w.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = w;
}

__device__ __forceinline__ void store8_f16(uint16_t* p, const float (&v)[8]) {
  *reinterpret_cast<uint4*>(p) =
      make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]), pack_f16x2(v[4], v[5]), pack_f16x2(v[6], v[7]));
}

// Fixed-order block sum of two values (warp butterfly, then warps in order).
__device__ __forceinline__ float2 block_sum2(float a, float b, float2* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = make_float2(a, b);
  __syncthreads();
  float2 s = make_float2(0.0f, 0.0f);
  const int nw = blockDim.x >> 5;
  for (int w = 0; w < nw; ++w) {
    s.x += red[w].x;
    s.y += red[w].y;
  }
  __syncthreads();
  return s;
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&v)[8]) {
  unpack_bf16x2(w.x, v[0], v[1]);
  unpack_bf16x2(w.y, v[2], v[3]);
  unpack_bf16x2(w.z, v[4], v[5]);
  unpack_bf16x2(w.w, v[6], v[7]);
}

// The row stays in registers as packed bf16 words (4 registers per 8 elements) and is
// unpacked in each pass: half the registers of an fp32 copy, so more rows are in flight.
// OUT_F16: Y is written as IEEE fp16 (the attention block's input, whose rounding sets the
// precision of Q and K), else bf16.
template <bool OUT_F16>
__global__ void ln_fwd_kernel(const uint16_t* __restrict__ X, int64_t h, const uint16_t* __restrict__ gamma,
                              const uint16_t* __restrict__ beta, float eps, uint16_t* __restrict__ Y,
                              float* __restrict__ mean_out, float* __restrict__ rstd_out) {
  ptx::griddep_wait();  // inputs come from the previous kernel on the stream
  ptx::griddep_launch_dependents();
  __shared__ float2 red[32];
  const int64_t row = blockIdx.x;
  const uint16_t* x = X + row * h;
  const int64_t nch = h / 8;
  uint4 xw[LN_CHUNKS];
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < LN_CHUNKS; ++k) {
    const int64_t c = threadIdx.x + static_cast<int64_t>(k) * blockDim.x;
    if (c < nch) xw[k] = *reinterpret_cast<const uint4*>(x + c * 8);
  }
#pragma unroll
  for (int k = 0; k < LN_CHUNKS; ++k) {
    const int64_t c = threadIdx.x + static_cast<int64_t>(k) * blockDim.x;
    if (c < nch) {
      float v[8];
      unpack8(xw[k], v);
#pragma unroll
      for (int e = 0; e < 8; ++e) s += v[e];
    }
  }
  const float mean = block_sum2(s, 0.0f, red).x / static_cast<float>(h);
  float q = 0.0f;
#pragma unroll
  for (int k = 0; k < LN_CHUNKS; ++k) {
    const int64_t c = threadIdx.x + static_cast<int64_t>(k) * blockDim.x;
    if (c < nch) {
      float v[8];
      unpack8(xw[k], v);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float d = v[e] - mean;
        q += d * d;
      }
    }
  }
  const float var = block_sum2(q, 0.0f, red).x / static_cast<float>(h);
  const float rstd = rsqrtf(var + eps);
#pragma unroll
  for (int k = 0; k < LN_CHUNKS; ++k) {
    const int64_t c = threadIdx.x + static_cast<int64_t>(k) * blockDim.x;
    if (c < nch) {
      float v[8], g[8], b[8], o[8];
      unpack8(xw[k], v);
      load8(gamma + c * 8, g);
      load8(beta + c * 8, b);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = (v[e] - mean) * rstd * g[e] + b[e];
      if (OUT_F16) store8_f16(Y + row * h + c * 8, o);
      else store8(Y + row * h + c * 8, o);
    }
  }
  if (threadIdx.x == 0) {
    mean_out[row] = mean;
    rstd_out[row] = rstd;
  }
}

// dx = rstd * (g - mean(g) - xhat * mean(g * xhat)) (+ dres),  g = dy * gamma.
__global__ void ln_bwd_rows_kernel(const uint16_t* __restrict__ dY, const uint16_t* __restrict__ X,
                                   const uint16_t* __restrict__ gamma, const float* __restrict__ mean_in,
                                   const float* __restrict__ rstd_in, const uint16_t* __restrict__ dres, int64_t h,
                                   uint16_t* __restrict__ dX) {
  ptx::griddep_wait();  // inputs come from the previous kernel on the stream
  ptx::griddep_launch_dependents();
  __shared__ float2 red[32];
  const int64_t row = blockIdx.x;
  const float mean = mean_in[row], rstd = rstd_in[row];
  const int64_t nch = h / 8;
  // Packed bf16 words of x and dy stay in registers; gamma (the same for every row,
  // so an L1 / L2 hit) is re-read in each pass instead of taking registers.
  uint4 xw[LN_CHUNKS], dw[LN_CHUNKS];
#pragma unroll
  for (int k = 0; k < LN_CHUNKS; ++k) {
    const int64_t c = threadIdx.x + static_cast<int64_t>(k) * blockDim.x;
    if (c < nch) {
      xw[k] = *reinterpret_cast<const uint4*>(X + row * h + c * 8);
      dw[k] = *reinterpret_cast<const uint4*>(dY + row * h + c * 8);
    }
  }
  float sg = 0.0f, sgx = 0.0f;
#pragma unroll
  for (int k = 0; k < LN_CHUNKS; ++k) {
    const int64_t c = threadIdx.x + static_cast<int64_t>(k) * blockDim.x;
    if (c < nch) {
      float xv[8], dy[8], gm[8];
      unpack8(xw[k], xv);
      unpack8(dw[k], dy);
      unpack8(__ldg(reinterpret_cast<const uint4*>(gamma + c * 8)), gm);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float g = dy[e] * gm[e];
        sg += g;
        sgx += g * ((xv[e] - mean) * rstd);
      }
    }
  }
  const float2 tot = block_sum2(sg, sgx, red);
  const float inv_h = 1.0f / static_cast<float>(h);
  const float mg = tot.x * inv_h, mgx = tot.y * inv_h;
#pragma unroll
  for (int k = 0; k < LN_CHUNKS; ++k) {
    const int64_t c = threadIdx.x + static_cast<int64_t>(k) * blockDim.x;
    if (c < nch) {
      float xv[8], dy[8], gm[8], o[8];
      unpack8(xw[k], xv);
      unpack8(dw[k], dy);
      unpack8(__ldg(reinterpret_cast<const uint4*>(gamma + c * 8)), gm);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = rstd * (dy[e] * gm[e] - mg - ((xv[e] - mean) * rstd) * mgx);
      if (dres) {
        float r[8];
        load8(dres + row * h + c * 8, r);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] += r[e];
      }
      store8(dX + row * h + c * 8, o);
    }
  }
}

// Partial weight grads of shard j over its rows [j*rows_per, (j+1)*rows_per): one CTA
// per (64-column block, shard), 1024 CTAs at the sequence-parallel layer shape so that
// the SMs get an even share.  A lane owns 8 columns (16-byte loads) of one of the 4
// rows a warp covers per step (lane / 8 = row, lane % 8 = column group); the 8 warps
// step through the shard's rows 32 at a time, 8 rows in flight per lane.  Sums are
// combined in a fixed order: rows in sequence, then the 4 row lanes, then warps.
constexpr int COLS_THREADS = 256;
constexpr int COLS_BLOCK = 64;

__device__ __forceinline__ void cols_accum(const uint4& xv, const uint4& dv, float mu, float rs, float (&dg)[8],
                                           float (&db)[8]) {
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
  const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float x0, x1, d0, d1;
    unpack_bf16x2(xw[q], x0, x1);
    unpack_bf16x2(dw[q], d0, d1);
    dg[2 * q] += d0 * (x0 - mu) * rs;
    dg[2 * q + 1] += d1 * (x1 - mu) * rs;
    db[2 * q] += d0;
    db[2 * q + 1] += d1;
  }
}

__global__ void __launch_bounds__(COLS_THREADS)
    ln_bwd_cols_kernel(const uint16_t* __restrict__ dY, const uint16_t* __restrict__ X,
                       const float* __restrict__ mean_in, const float* __restrict__ rstd_in, int64_t h,
                       int64_t rows_per, float* __restrict__ dg_part, float* __restrict__ db_part) {
  ptx::griddep_wait();  // inputs come from the previous kernel on the stream
  ptx::griddep_launch_dependents();
  __shared__ float red[2][COLS_THREADS / 32][COLS_BLOCK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane >> 3, cg = lane & 7;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * COLS_BLOCK + cg * 8;
  const int j = blockIdx.y;
  float dg[8] = {0, 0, 0, 0, 0, 0, 0, 0}, db[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (c0 < h) {
    const int64_t r1 = static_cast<int64_t>(j + 1) * rows_per;
    int64_t r = static_cast<int64_t>(j) * rows_per + warp * 4 + sub;
    for (; r + 7 * 32 < r1; r += 8 * 32) {
      uint4 xv[8], dv[8];
      float mu[8], rs[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t rr = r + 32 * u;
        xv[u] = *reinterpret_cast<const uint4*>(X + rr * h + c0);
        dv[u] = *reinterpret_cast<const uint4*>(dY + rr * h + c0);
        mu[u] = mean_in[rr];
        rs[u] = rstd_in[rr];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) cols_accum(xv[u], dv[u], mu[u], rs[u], dg, db);
    }
    for (; r < r1; r += 32)
      cols_accum(*reinterpret_cast<const uint4*>(X + r * h + c0), *reinterpret_cast<const uint4*>(dY + r * h + c0),
                 mean_in[r], rstd_in[r], dg, db);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    dg[e] += __shfl_xor_sync(0xffffffffu, dg[e], 8);
    dg[e] += __shfl_xor_sync(0xffffffffu, dg[e], 16);
    db[e] += __shfl_xor_sync(0xffffffffu, db[e], 8);
    db[e] += __shfl_xor_sync(0xffffffffu, db[e], 16);
  }
  if (sub == 0) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      red[0][warp][cg * 8 + e] = dg[e];
      red[1][warp][cg * 8 + e] = db[e];
    }
  }
  __syncthreads();
  if (threadIdx.x < 2 * COLS_BLOCK) {
    const int which = threadIdx.x / COLS_BLOCK, col = threadIdx.x % COLS_BLOCK;
    const int64_t c = static_cast<int64_t>(blockIdx.x) * COLS_BLOCK + col;
    if (c < h) {
      float acc = 0.0f;
#pragma unroll
      for (int w = 0; w < COLS_THREADS / 32; ++w) acc += red[which][w][col];
      (which ? db_part : dg_part)[static_cast<int64_t>(j) * h + c] = acc;
    }
  }
}

// The LayerNorm weight-gradient all-reduce: sum of the t shard partials, shard order.
__global__ void ln_bwd_shard_sum_kernel(const float* __restrict__ dg_part, const float* __restrict__ db_part,
                                        int64_t h, int t, float* __restrict__ dgamma, float* __restrict__ dbeta) {
  ptx::griddep_wait();  // inputs come from the previous kernel on the stream
  ptx::griddep_launch_dependents();
  const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= h) return;
  float sg = 0.0f, sb = 0.0f;
  for (int j = 0; j < t; ++j) {
    sg += dg_part[static_cast<int64_t>(j) * h + c];
    sb += db_part[static_cast<int64_t>(j) * h + c];
  }
  dgamma[c] = sg;
  dbeta[c] = sb;
}

int row_threads(int64_t h) {
  const int64_t nch = h / 8;
  int64_t th = (nch + LN_CHUNKS - 1) / LN_CHUNKS;
  th = (th + 31) / 32 * 32;
  return static_cast<int>(th < 32 ? 32 : th);
}

tp_status check(int64_t s, int64_t h, int t) {
  if (s < 0 || h < 1 || t < 1) return TP_ERR_INVALID_ARG;
  if (s % t != 0 || h > 1024LL * 8 * LN_CHUNKS) return TP_ERR_SHAPE;
  if (h % 8 != 0) return TP_ERR_ALIGN;
  return TP_OK;
}

}  // namespace

tp_status run_ln_forward(const uint16_t* X, int64_t s, int64_t h, int t, const uint16_t* gamma,
                         const uint16_t* beta, float eps, uint16_t* Y, float* mean, float* rstd, cudaStream_t st,
                         int out_f16) {
  TP_RETURN_IF(check(s, h, t));
  if (s == 0) return TP_OK;
  if (!X || !gamma || !beta || !Y || !mean || !rstd || !(eps >= 0.0f)) return TP_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(gamma) || !aligned16(beta) || !aligned16(Y)) return TP_ERR_ALIGN;
  if (s > 0x7fffffffLL) return TP_ERR_SHAPE;
  TP_RETURN_IF(ready());
  if (out_f16)
    TP_CUDA_CHECK(launch_pdl(ln_fwd_kernel<true>, dim3(static_cast<unsigned>(s)), dim3(row_threads(h)), 0, st, X, h,
                             gamma, beta, eps, Y, mean, rstd));
  else
    TP_CUDA_CHECK(launch_pdl(ln_fwd_kernel<false>, dim3(static_cast<unsigned>(s)), dim3(row_threads(h)), 0, st, X,
                             h, gamma, beta, eps, Y, mean, rstd));
  count_launch();
  return TP_OK;
}

tp_status run_ln_backward(const uint16_t* dY, const uint16_t* X, const uint16_t* gamma, const float* mean,
                          const float* rstd, const uint16_t* dres, int64_t s, int64_t h, int t, uint16_t* dX,
                          float* dg_part, float* db_part, float* dgamma, float* dbeta, cudaStream_t st) {
  TP_RETURN_IF(check(s, h, t));
  if (!dg_part || !db_part || !dgamma || !dbeta) return TP_ERR_INVALID_ARG;
  if (s > 0 && (!dY || !X || !gamma || !mean || !rstd || !dX)) return TP_ERR_INVALID_ARG;
  if ((s > 0 && (!aligned16(dY) || !aligned16(X) || !aligned16(gamma) || !aligned16(dX))) ||
      (dres && !aligned16(dres)) || !aligned16(dg_part) || !aligned16(db_part) || !aligned16(dgamma) ||
      !aligned16(dbeta))
    return TP_ERR_ALIGN;
  if (s > 0x7fffffffLL) return TP_ERR_SHAPE;
  TP_RETURN_IF(ready());
  if (s == 0) {
    TP_CUDA_CHECK(cudaMemsetAsync(dg_part, 0, sizeof(float) * t * h, st));
    TP_CUDA_CHECK(cudaMemsetAsync(db_part, 0, sizeof(float) * t * h, st));
    TP_CUDA_CHECK(cudaMemsetAsync(dgamma, 0, sizeof(float) * h, st));
    TP_CUDA_CHECK(cudaMemsetAsync(dbeta, 0, sizeof(float) * h, st));
    return TP_OK;
  }
  TP_CUDA_CHECK(launch_pdl(ln_bwd_rows_kernel, dim3(static_cast<unsigned>(s)), dim3(row_threads(h)), 0, st, dY, X, gamma,
                           mean, rstd, dres, h, dX));
  count_launch();
  dim3 g(static_cast<unsigned>((h + COLS_BLOCK - 1) / COLS_BLOCK), static_cast<unsigned>(t));
  TP_CUDA_CHECK(launch_pdl(ln_bwd_cols_kernel, g, dim3(COLS_THREADS), 0, st, dY, X, mean, rstd, h, s / t, dg_part,
                           db_part));
  count_launch();
  // The LayerNorm weight-gradient all-reduce over the sequence shards, fixed order.
  TP_CUDA_CHECK(launch_pdl(ln_bwd_shard_sum_kernel, dim3(static_cast<unsigned>((h + 255) / 256)), dim3(256), 0, st,
                           dg_part, db_part, h, t, dgamma, dbeta));
  count_launch();
  return TP_OK;
}

}  // namespace tp
