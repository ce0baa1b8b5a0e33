// Tile plan of decode attention over a sharded KV cache: stream
// s = (i * kv_t + jl) * B + b (shard i, its local KV head jl, sequence b) owns
// ceil(len_b / 128) tiles of 128 keys, len_b = pos[b] + 1; its first tile in
// the flattened list of all streams' tiles is (s / B) * TB + pre[b], with
// pre the exclusive prefix of the sequences' tile counts and TB their total.
#pragma once

#include <cstdint>

namespace tp {

constexpr int kDecodeTileKeys = 128;
constexpr int kDecodeErrPos = 0x201;

// Called by every thread of one CTA: a position outside [0, L_max) is
// recorded as a device-side argument error (the kernels clamp it).
__device__ __forceinline__ void decode_check_positions(const int32_t* pos, int B, int64_t L_max, int* err) {
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int64_t p = pos[b];
    if (p < 0 || p >= L_max) atomicCAS(err, 0, kDecodeErrPos);
  }
}

// Exclusive prefix of the sequences' tile counts into shared memory:
// pre[b] = sum_{b' < b} ceil(len_b' / 128), pre[B] = the total.  Called by
// every thread of the CTA (contains __syncthreads).
__device__ __forceinline__ void decode_tile_prefix(const int32_t* pos, int B, int64_t L_max, int* pre) {
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    int64_t p = pos[b];
    if (p < 0) p = 0;
    if (p >= L_max) p = L_max - 1;
    pre[b] = static_cast<int>((p + 1 + kDecodeTileKeys - 1) / kDecodeTileKeys);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int b = 0; b < B; ++b) {
      const int n = pre[b];
      pre[b] = run;
      run += n;
    }
    pre[B] = run;
  }
  __syncthreads();
}

}  // namespace tp
