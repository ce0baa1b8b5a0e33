// Decode-time SwiGLU MLP on t logical shards: a memory-bound weight stream.
// ("02 — Tensor Parallelism": the up-projection is doubled for SwiGLU in "The
// core observation", and decode is bandwidth-bound, which is what TP splits
// across HBMs, in "When to use TP".)
//
//   kernel 1 (column-parallel):  a[m][n] = silu(x[m] . Wg[:, n]) * (x[m] . Wu[:, n])
//   kernel 2 (row-parallel + g): y[m][c] = sum_{i=0..t-1} ( a[m][C_i] . W_down,i[c][:] )
//
// Weights are read exactly once, 16 bytes per load, through the non-coherent
// path without L1 allocation; the small activation vectors are read through
// L1.  One CTA of 128 threads owns one output unit at a time (a hidden unit in
// kernel 1, an output column in kernel 2): every thread streams an equal
// slice of that unit's weight rows, and the partial dot products are combined
// in a fixed order (warp butterfly, then warps 0..3, then shards 0..t-1), so
// the result is deterministic.  Several CTAs per SM keep enough loads in
// flight to cover HBM latency while one CTA is in its reduction.
#include <cuda_runtime.h>

#include "devmath.cuh"
#include "internal.h"

namespace tp {
namespace {

constexpr int GEMV_THREADS = 128;
constexpr int GEMV_WARPS = GEMV_THREADS / 32;
constexpr int MAX_T = 8;

__device__ __forceinline__ uint4 ld_stream(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float dot8(const uint4 w, const uint4 x) {
  float a0, a1, b0, b1, s = 0.0f;
  unpack_bf16x2(w.x, a0, a1); unpack_bf16x2(x.x, b0, b1); s = fmaf(a0, b0, s); s = fmaf(a1, b1, s);
  unpack_bf16x2(w.y, a0, a1); unpack_bf16x2(x.y, b0, b1); s = fmaf(a0, b0, s); s = fmaf(a1, b1, s);
  unpack_bf16x2(w.z, a0, a1); unpack_bf16x2(x.z, b0, b1); s = fmaf(a0, b0, s); s = fmaf(a1, b1, s);
  unpack_bf16x2(w.w, a0, a1); unpack_bf16x2(x.w, b0, b1); s = fmaf(a0, b0, s); s = fmaf(a1, b1, s);
  return s;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Block-wide fixed-order sum of NV values per thread; result valid in red[v] after the call.
template <int NV>
__device__ __forceinline__ void block_sum(float (&v)[NV], float (*red)[NV], float* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const float s = warp_sum(v[k]);
    if (lane == 0) red[warp][k] = s;
  }
  __syncthreads();
  if (threadIdx.x < NV) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < GEMV_WARPS; ++w) s += red[w][threadIdx.x];
    out[threadIdx.x] = s;
  }
  __syncthreads();
}

// Kernel 1: one hidden unit n per CTA iteration.  Wgu is [t][Ft/128][2][128][h]:
// gate row of unit n sits at packed row 2n - (n % 128), its up row 128 rows later.
template <int M>
__global__ void __launch_bounds__(GEMV_THREADS)
    swiglu_gate_up_kernel(const uint16_t* __restrict__ x, int64_t h, int64_t F,
                          const uint16_t* __restrict__ Wgu, uint16_t* __restrict__ a) {
  __shared__ float red[GEMV_WARPS][2 * M];
  __shared__ float tot[2 * M];
  const int64_t chunks = h / 8;
  for (int64_t n = blockIdx.x; n < F; n += gridDim.x) {
    const int64_t e = n & 127;
    const uint16_t* g_row = Wgu + (2 * n - e) * h;
    const uint16_t* u_row = g_row + 128 * h;
    float acc[2 * M];
#pragma unroll
    for (int k = 0; k < 2 * M; ++k) acc[k] = 0.0f;
    for (int64_t c = threadIdx.x; c < chunks; c += GEMV_THREADS * 4) {
      uint4 wg[4], wu[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t cc = c + j * GEMV_THREADS;
        if (cc < chunks) {
          wg[j] = ld_stream(g_row + cc * 8);
          wu[j] = ld_stream(u_row + cc * 8);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t cc = c + j * GEMV_THREADS;
        if (cc < chunks) {
#pragma unroll
          for (int m = 0; m < M; ++m) {
            const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + m * h) + cc);
            acc[2 * m] += dot8(wg[j], xv);
            acc[2 * m + 1] += dot8(wu[j], xv);
          }
        }
      }
    }
    block_sum<2 * M>(acc, red, tot);
    if (threadIdx.x < M) {
      const int m = threadIdx.x;
      a[m * F + n] = float_to_bf16_bits(silu(tot[2 * m]) * tot[2 * m + 1]);
    }
  }
}

// Kernel 2: one output column c per CTA iteration; shards summed in order.
// Wd is [t][h][Ft]: row c of shard i is contiguous.
template <int M>
__global__ void __launch_bounds__(GEMV_THREADS)
    down_reduce_kernel(const uint16_t* __restrict__ a, int64_t lda, int64_t h, int64_t F, int t,
                       const uint16_t* __restrict__ Wd, const uint16_t* __restrict__ bias,
                       uint16_t* __restrict__ y) {
  __shared__ float red[GEMV_WARPS][MAX_T * M];
  __shared__ float tot[MAX_T * M];
  const int64_t Ft = F / t;
  const int64_t chunks = Ft / 8;
  for (int64_t col = blockIdx.x; col < h; col += gridDim.x) {
    float acc[MAX_T * M];
#pragma unroll
    for (int k = 0; k < MAX_T * M; ++k) acc[k] = 0.0f;
#pragma unroll
    for (int i = 0; i < MAX_T; ++i) {
      if (i < t) {
        const uint16_t* row = Wd + (static_cast<int64_t>(i) * h + col) * Ft;
        const uint16_t* ai = a + i * Ft;
        for (int64_t c = threadIdx.x; c < chunks; c += GEMV_THREADS * 4) {
          uint4 w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int64_t cc = c + j * GEMV_THREADS;
            if (cc < chunks) w[j] = ld_stream(row + cc * 8);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int64_t cc = c + j * GEMV_THREADS;
            if (cc < chunks) {
#pragma unroll
              for (int m = 0; m < M; ++m) {
                const uint4 av = __ldg(reinterpret_cast<const uint4*>(ai + m * lda) + cc);
                acc[i * M + m] += dot8(w[j], av);
              }
            }
          }
        }
      }
    }
    block_sum<MAX_T * M>(acc, red, tot);
    if (threadIdx.x < M) {
      const int m = threadIdx.x;
      float s = 0.0f;
      for (int i = 0; i < t; ++i) s += tot[i * M + m];  // g: fixed shard order
      if (bias) s += bf16_bits_to_float(bias[col]);      // once, after the sum
      y[m * h + col] = float_to_bf16_bits(s);
    }
  }
}

template <int M>
tp_status launch_decode(const uint16_t* x, int64_t h, int64_t F, int t, const uint16_t* Wgu, const uint16_t* Wd,
                        uint16_t* y, uint16_t* a, cudaStream_t s) {
  int per_sm1 = 0, per_sm2 = 0;
  TP_CUDA_CHECK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm1, swiglu_gate_up_kernel<M>, GEMV_THREADS, 0));
  TP_CUDA_CHECK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm2, down_reduce_kernel<M>, GEMV_THREADS, 0));
  const int64_t sms = device_sm_count();
  int64_t g1 = sms * (per_sm1 > 0 ? per_sm1 : 1), g2 = sms * (per_sm2 > 0 ? per_sm2 : 1);
  if (g1 > F) g1 = F;
  if (g2 > h) g2 = h;
  swiglu_gate_up_kernel<M><<<static_cast<unsigned>(g1), GEMV_THREADS, 0, s>>>(x, h, F, Wgu, a);
  TP_LAUNCHED();
  down_reduce_kernel<M><<<static_cast<unsigned>(g2), GEMV_THREADS, 0, s>>>(a, F, h, F, t, Wd, nullptr, y);
  TP_LAUNCHED();
  return TP_OK;
}

template <int M>
tp_status launch_row(const uint16_t* a, int64_t K, int64_t h, int t, const uint16_t* Wd, const uint16_t* bias,
                     uint16_t* y, cudaStream_t s) {
  int per_sm = 0;
  TP_CUDA_CHECK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, down_reduce_kernel<M>, GEMV_THREADS, 0));
  int64_t g = static_cast<int64_t>(device_sm_count()) * (per_sm > 0 ? per_sm : 1);
  if (g > h) g = h;
  down_reduce_kernel<M><<<static_cast<unsigned>(g), GEMV_THREADS, 0, s>>>(a, K, h, K, t, Wd, bias, y);
  TP_LAUNCHED();
  return TP_OK;
}

}  // namespace

// Row-parallel GEMV followed by g: y[m] = sum_{i<t} a[m][C_i] W_i^T + bias (once),
// a [M][K], W [t][h][K/t].  Rows are taken 8 at a time (each group re-streams W).
tp_status run_row_gemv(const uint16_t* a, int64_t M, int64_t K, int64_t h, int t, const uint16_t* Wd,
                       const uint16_t* bias, uint16_t* y, cudaStream_t s) {
  if (M < 0 || K < 1 || h < 1 || t < 1) return TP_ERR_INVALID_ARG;
  if (t > MAX_T || K % t != 0 || (K / t) % 8 != 0) return TP_ERR_SHAPE;
  if (M == 0) return TP_OK;
  for (int64_t m0 = 0; m0 < M; m0 += 8) {
    const int mg = static_cast<int>(M - m0 < 8 ? M - m0 : 8);
    const uint16_t* am = a + m0 * K;
    uint16_t* ym = y + m0 * h;
    tp_status st;
    switch (mg) {
      case 1: st = launch_row<1>(am, K, h, t, Wd, bias, ym, s); break;
      case 2: st = launch_row<2>(am, K, h, t, Wd, bias, ym, s); break;
      case 3: st = launch_row<3>(am, K, h, t, Wd, bias, ym, s); break;
      case 4: st = launch_row<4>(am, K, h, t, Wd, bias, ym, s); break;
      case 5: st = launch_row<5>(am, K, h, t, Wd, bias, ym, s); break;
      case 6: st = launch_row<6>(am, K, h, t, Wd, bias, ym, s); break;
      case 7: st = launch_row<7>(am, K, h, t, Wd, bias, ym, s); break;
      default: st = launch_row<8>(am, K, h, t, Wd, bias, ym, s); break;
    }
    TP_RETURN_IF(st);
  }
  return TP_OK;
}

tp_status run_decode_swiglu(const uint16_t* x, int64_t M, int64_t h, int64_t F, int t, const uint16_t* Wgu,
                            const uint16_t* Wd, uint16_t* y, uint16_t* a, cudaStream_t s) {
  if (M < 0 || h < 1 || F < 1 || t < 1) return TP_ERR_INVALID_ARG;
  if (t > MAX_T || M > 8 || F % t != 0 || (F / t) % 128 != 0) return TP_ERR_SHAPE;
  if (h % 8 != 0) return TP_ERR_ALIGN;
  if (M == 0) return TP_OK;
  if (!x || !Wgu || !Wd || !y || !a) return TP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wgu) || !aligned16(Wd) || !aligned16(a)) return TP_ERR_ALIGN;
  TP_RETURN_IF(ready());
  switch (M) {
    case 1: return launch_decode<1>(x, h, F, t, Wgu, Wd, y, a, s);
    case 2: return launch_decode<2>(x, h, F, t, Wgu, Wd, y, a, s);
    case 3: return launch_decode<3>(x, h, F, t, Wgu, Wd, y, a, s);
    case 4: return launch_decode<4>(x, h, F, t, Wgu, Wd, y, a, s);
    case 5: return launch_decode<5>(x, h, F, t, Wgu, Wd, y, a, s);
    case 6: return launch_decode<6>(x, h, F, t, Wgu, Wd, y, a, s);
    case 7: return launch_decode<7>(x, h, F, t, Wgu, Wd, y, a, s);
    default: return launch_decode<8>(x, h, F, t, Wgu, Wd, y, a, s);
  }
}

}  // namespace tp
