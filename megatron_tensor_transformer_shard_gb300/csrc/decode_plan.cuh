// Tile plan of decode attention over a sharded KV cache: stream
// s = (i * kv_t + jl) * B + b (shard i, its local KV head jl, sequence b) owns
// ceil(len_b / 128) tiles of 128 keys, len_b = pos[b] + 1, and
// tile_start[s] is its first tile in the flattened list of all streams'
// tiles (tile_start[S] = the total).  Written by one CTA of a kernel that runs
// before the attention kernel; a position outside [0, L_max) is clamped and
// recorded as a device-side argument error.
#pragma once

#include <cstdint>

namespace tp {

constexpr int kDecodeTileKeys = 128;
constexpr int kDecodeErrPos = 0x201;

// Called by every thread of one CTA (blockDim.x threads); `scratch` holds at
// least B + 1 ints of shared memory.
// `done` (S ints, nullable) is zeroed: per-stream counts of finished pieces.
__device__ __forceinline__ void decode_tile_plan(const int32_t* pos, int B, int64_t L_max, int groups,
                                                 int* tile_start, int* done, int* err, int* scratch) {
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int64_t p = pos[b];
    int64_t len = p + 1;
    if (p < 0 || p >= L_max) {
      atomicCAS(err, 0, kDecodeErrPos);
      len = p < 0 ? 1 : L_max;
    }
    scratch[b] = static_cast<int>((len + kDecodeTileKeys - 1) / kDecodeTileKeys);
  }
  __syncthreads();
  if (threadIdx.x == 0) {  // exclusive prefix over the sequences, in place
    int run = 0;
    for (int b = 0; b < B; ++b) {
      const int n = scratch[b];
      scratch[b] = run;
      run += n;
    }
    scratch[B] = run;
  }
  __syncthreads();
  const int per_group = scratch[B];
  const int S = groups * B;
  for (int s = threadIdx.x; s <= S; s += blockDim.x) {
    const int c = s / B, b = s - c * B;
    tile_start[s] = c * per_group + scratch[b];
    if (done && s < S) done[s] = 0;
  }
}

}  // namespace tp
