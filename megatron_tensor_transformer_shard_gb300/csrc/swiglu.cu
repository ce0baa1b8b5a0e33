// SwiGLU for the token-parallel (prefill / training) MLP ("02 — Tensor
// Parallelism", section "The core observation": with SwiGLU the up-projection is
// twice as wide; gate and up are both split by the same hidden columns C_i, so
// silu(gate) * up stays local to the shard and the row-parallel half is unchanged).
//
// Z [rows][2 Ft] is the column-parallel GEMM's output over the interleaved packed
// weights of tp_pack_swiglu: for hidden columns [128 k, 128 k + 128) of a shard,
// columns [256 k, 256 k + 128) of Z are the gate pre-activations g and the next
// 128 the up pre-activations u.  rows = t M (the shards' Z blocks one after another).
//   forward:  A[r][c]  = silu(g) u
//   backward: dg = dA u silu'(g),  du = dA silu(g),  silu'(g) = s (1 + g (1 - s)),  s = sigmoid(g)
// One thread per 8 consecutive hidden columns (16-byte loads and stores).
#include <cuda_runtime.h>

#include "devmath.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace tp {
namespace {

constexpr int SWIGLU_GROUP = 128;  // gate / up interleaving of tp_pack_swiglu

__device__ __forceinline__ void unpack8(const uint4& w, float (&v)[8]) {
  unpack_bf16x2(w.x, v[0], v[1]);
  unpack_bf16x2(w.y, v[2], v[3]);
  unpack_bf16x2(w.z, v[4], v[5]);
  unpack_bf16x2(w.w, v[6], v[7]);
}

__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

// Offset in a Z row of the gate value of hidden column c (the up value is SWIGLU_GROUP further).
__device__ __forceinline__ int64_t gate_col(int64_t c) {
  return (c / SWIGLU_GROUP) * (2 * SWIGLU_GROUP) + (c % SWIGLU_GROUP);
}

__global__ void swiglu_act_kernel(const uint16_t* __restrict__ Z, int64_t rows, int64_t Ft, uint16_t* __restrict__ A) {
  ptx::griddep_wait();  // Z comes from the previous kernel
  ptx::griddep_launch_dependents();
  const int64_t per_row = Ft / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= rows * per_row) return;
  const int64_t r = idx / per_row, c = (idx - r * per_row) * 8;
  const uint16_t* zr = Z + r * 2 * Ft + gate_col(c);
  float g[8], u[8], a[8];
  unpack8(*reinterpret_cast<const uint4*>(zr), g);
  unpack8(*reinterpret_cast<const uint4*>(zr + SWIGLU_GROUP), u);
#pragma unroll
  for (int e = 0; e < 8; ++e) a[e] = silu(g[e]) * u[e];
  *reinterpret_cast<uint4*>(A + r * Ft + c) = pack8(a);
}

__global__ void dswiglu_kernel(const uint16_t* __restrict__ dA, const uint16_t* __restrict__ Z, int64_t rows,
                               int64_t Ft, uint16_t* __restrict__ dZ) {
  ptx::griddep_wait();  // dA comes from the previous kernel
  ptx::griddep_launch_dependents();
  const int64_t per_row = Ft / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= rows * per_row) return;
  const int64_t r = idx / per_row, c = (idx - r * per_row) * 8;
  const int64_t zc = r * 2 * Ft + gate_col(c);
  float g[8], u[8], da[8], dg[8], du[8];
  unpack8(*reinterpret_cast<const uint4*>(Z + zc), g);
  unpack8(*reinterpret_cast<const uint4*>(Z + zc + SWIGLU_GROUP), u);
  unpack8(*reinterpret_cast<const uint4*>(dA + r * Ft + c), da);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float s = 1.0f / (1.0f + expf(-g[e]));
    dg[e] = da[e] * u[e] * (s * (1.0f + g[e] * (1.0f - s)));
    du[e] = da[e] * (g[e] * s);
  }
  *reinterpret_cast<uint4*>(dZ + zc) = pack8(dg);
  *reinterpret_cast<uint4*>(dZ + zc + SWIGLU_GROUP) = pack8(du);
}

unsigned grid_for(int64_t threads) { return static_cast<unsigned>((threads + 255) / 256); }

}  // namespace

tp_status run_swiglu_act(const uint16_t* Z, int64_t rows, int64_t Ft, uint16_t* A, cudaStream_t s) {
  if (rows < 0 || Ft < 1 || Ft % SWIGLU_GROUP != 0) return TP_ERR_SHAPE;
  if (rows == 0) return TP_OK;
  if (!Z || !A) return TP_ERR_INVALID_ARG;
  if (!aligned16(Z) || !aligned16(A)) return TP_ERR_ALIGN;
  TP_RETURN_IF(ready());
  TP_CUDA_CHECK(launch_pdl(swiglu_act_kernel, dim3(grid_for(rows * (Ft / 8))), dim3(256), 0, s, Z, rows, Ft, A));
  count_launch();
  return TP_OK;
}

tp_status run_dswiglu(const uint16_t* dA, const uint16_t* Z, int64_t rows, int64_t Ft, uint16_t* dZ, cudaStream_t s) {
  if (rows < 0 || Ft < 1 || Ft % SWIGLU_GROUP != 0) return TP_ERR_SHAPE;
  if (rows == 0) return TP_OK;
  if (!dA || !Z || !dZ) return TP_ERR_INVALID_ARG;
  if (!aligned16(dA) || !aligned16(Z) || !aligned16(dZ)) return TP_ERR_ALIGN;
  TP_RETURN_IF(ready());
  TP_CUDA_CHECK(launch_pdl(dswiglu_kernel, dim3(grid_for(rows * (Ft / 8))), dim3(256), 0, s, dA, Z, rows, Ft, dZ));
  count_launch();
  return TP_OK;
}

}  // namespace tp
