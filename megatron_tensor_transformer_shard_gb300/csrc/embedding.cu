// Vocab-parallel embedding ("Megatron-LM: Tensor Parallelism" (vanos001),
// "Common Pitfalls", item 5: the embedding lookup is sharded by vocabulary).
//
// Shard i owns the contiguous vocabulary rows [i V/t, (i+1) V/t) of E; the
// packed table [t][V/t][h] is E's own row-major layout.  Forward: shard i
// contributes E_i[id - i V/t] for the ids it owns and zeros for the rest, and
// g sums the t partials; exactly one partial of every token is non-zero, so
// the fused sum is a gather from the owning shard.  Backward: every shard gets
// dY (g backward is the identity) and adds dY[n] into its own row for each
// token it owns.
//
// The backward is deterministic: within a chunk of up to 8192 tokens the keys
// (id << 13 | n) are sorted in shared memory (bitonic; the keys are distinct,
// so the order is unique) and cut into segments of equal ids; each
// (segment, 256-column chunk) item sums the segment's dY rows in a fixed order
// (a warp in token order for short segments; 8 warps over contiguous token
// ranges, then the warps in order, for long ones) into dE.
// Chunks run one after another on the stream.
#include <cuda_runtime.h>

#include "devmath.cuh"
#include "internal.h"

namespace tp {
namespace {

constexpr int EMB_THREADS = 128;
constexpr int SORT_THREADS = 1024;
constexpr int SORT_MAX = 8192;  // tokens per chunk: 13 bits of token index in a key
constexpr int ERR_EMB_ID = 0x202;  // a token id outside [0, V): argument error found on the device

__device__ __forceinline__ uint4 ld_nc16(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// One CTA per token (grid-stride): Y[n] = E_shard(id)[id - shard * Vt], 16 bytes per access.
__global__ void __launch_bounds__(EMB_THREADS)
    emb_fwd_kernel(const int32_t* __restrict__ ids, int64_t N, int64_t V, int64_t Vt, int64_t h,
                   const uint16_t* __restrict__ E, uint16_t* __restrict__ Y, int* err) {
  const int64_t chunks = h / 8;
  for (int64_t n = blockIdx.x; n < N; n += gridDim.x) {
    const int64_t id = ids[n];
    uint16_t* yrow = Y + n * h;
    if (id < 0 || id >= V) {
      if (threadIdx.x == 0) atomicCAS(err, 0, ERR_EMB_ID);
      for (int64_t c = threadIdx.x; c < chunks; c += EMB_THREADS)
        *reinterpret_cast<uint4*>(yrow + c * 8) = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const int64_t shard = id / Vt, local = id - shard * Vt;  // the owning shard's partial
    const uint16_t* erow = E + (shard * Vt + local) * h;
    for (int64_t c = threadIdx.x; c < chunks; c += EMB_THREADS * 4) {
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (c + j * EMB_THREADS < chunks) v[j] = ld_nc16(erow + (c + j * EMB_THREADS) * 8);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (c + j * EMB_THREADS < chunks) *reinterpret_cast<uint4*>(yrow + (c + j * EMB_THREADS) * 8) = v[j];
    }
  }
}

constexpr int LONG_SEG = 8;  // longer segments of equal ids are summed by a whole CTA

// Exclusive scan of one int per thread over the CTA (SORT_THREADS threads);
// *total gets the sum.  wsum: SORT_THREADS / 32 ints of shared memory.
__device__ __forceinline__ int block_exclusive_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  __syncthreads();  // wsum may still be read by a previous scan
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < SORT_THREADS / 32 ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    if (lane < SORT_THREADS / 32) wsum[lane] = w;
  }
  __syncthreads();
  *total = wsum[SORT_THREADS / 32 - 1];
  return incl - v + (warp > 0 ? wsum[warp - 1] : 0);
}

// Bitonic sorting network over key[0, P), all stages from size `size0` on, in shared
// memory: every compare-exchange step is followed by a block barrier.  A stage
// starts at stride size / 2; stride_min stops the stage early (smaller strides are
// left to the caller).
__device__ __forceinline__ void bitonic_smem_steps(uint32_t* key, int P, int size, int stride_hi, int stride_lo) {
  for (int stride = stride_hi; stride >= stride_lo; stride >>= 1) {
    for (int i = threadIdx.x; i < P / 2; i += SORT_THREADS) {
      const int lo = 2 * i - (i & (stride - 1));  // first element of the i-th compared pair
      const int hi = lo + stride;
      const bool up = (lo & size) == 0;
      const uint32_t a = key[lo], b = key[hi];
      if ((a > b) == up) {
        key[lo] = b;
        key[hi] = a;
      }
    }
    __syncthreads();
  }
}

__device__ __forceinline__ void bitonic_smem(uint32_t* key, int P, int size0, int stride_lo) {
  for (int size = size0; size <= P; size <<= 1) bitonic_smem_steps(key, P, size, size >> 1, stride_lo);
}

// The same network with E consecutive keys per thread (P = E * SORT_THREADS): strides
// below E are compare-exchanges in registers, strides below 32 E are exchanges with the
// lane (stride / E) away, and only larger strides go through shared memory.  On exit the
// sorted keys are back in key[].
template <int E>
__device__ __forceinline__ void bitonic_regs(uint32_t* key) {
  constexpr int P = E * SORT_THREADS;
  uint32_t v[E];
  const int t = threadIdx.x;
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = key[t * E + e];
  for (int size = 2; size <= P; size <<= 1) {
    int stride = size >> 1;
    if (stride >= 32 * E) {  // partner in another warp: shared memory
#pragma unroll
      for (int e = 0; e < E; ++e) key[t * E + e] = v[e];
      __syncthreads();
      bitonic_smem_steps(key, P, size, stride, 32 * E);
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = key[t * E + e];
      __syncthreads();  // key[] is rewritten by the next shared-memory step
      stride = 16 * E;
    }
    for (; stride >= E; stride >>= 1) {  // partner lane (stride / E) away in this warp
      const int dl = stride / E;
      const bool lower = (t & dl) == 0;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int i = t * E + e;
        const bool up = (i & size) == 0;
        const uint32_t o = __shfl_xor_sync(0xffffffffu, v[e], dl);
        v[e] = (lower == up) ? min(v[e], o) : max(v[e], o);
      }
    }
    for (; stride > 0; stride >>= 1) {  // partner in this thread's registers
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if ((e & stride) == 0) {
          const int i = t * E + e;
          const bool up = (i & size) == 0;
          const uint32_t a = v[e], b = v[e | stride];
          if ((a > b) == up) {
            v[e] = b;
            v[e | stride] = a;
          }
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) key[t * E + e] = v[e];
  __syncthreads();
}

// Sorts the chunk's keys (id << 13 | n) ascending in shared memory and writes
// them, plus the segments of equal ids in two lists: seg[0] / seg[1] = number
// of short / long segments, seg[4 + 2j], seg[5 + 2j] = first sorted position and length
// of short segment j, and the long list at seg + 4 + 2 SORT_MAX likewise.
// Invalid ids sort to the end (key 0xFFFFFFFF), belong to no segment and are
// reported.  Dynamic shared memory: 2 * SORT_MAX ints (keys, segment starts).
__global__ void __launch_bounds__(SORT_THREADS)
    emb_sort_kernel(const int32_t* __restrict__ ids, int64_t n0, int n, int64_t V, uint32_t* __restrict__ keys_out,
                    int* __restrict__ seg, int* err) {
  extern __shared__ uint32_t sm[];
  uint32_t* key = sm;
  int* starts = reinterpret_cast<int*>(sm + SORT_MAX);
  __shared__ int wsum[SORT_THREADS / 32];
  __shared__ int nv_s;
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = threadIdx.x; i < P; i += SORT_THREADS) {
    uint32_t k = 0xFFFFFFFFu;
    if (i < n) {
      const int64_t id = ids[n0 + i];
      if (id >= 0 && id < V) k = (static_cast<uint32_t>(id) << 13) | static_cast<uint32_t>(i);
      else atomicCAS(err, 0, ERR_EMB_ID);
    }
    key[i] = k;
  }
  if (threadIdx.x == 0) nv_s = 0;
  __syncthreads();
  if (P <= SORT_THREADS) bitonic_smem(key, P, 2, 1);
  else if (P == 2 * SORT_THREADS) bitonic_regs<2>(key);
  else if (P == 4 * SORT_THREADS) bitonic_regs<4>(key);
  else bitonic_regs<8>(key);
  // valid keys: up to the first sentinel (one thread sees the boundary)
  for (int i = threadIdx.x; i < P; i += SORT_THREADS)
    if (key[i] != 0xFFFFFFFFu && (i + 1 == P || key[i + 1] == 0xFFFFFFFFu)) nv_s = i + 1;
  for (int i = threadIdx.x; i < n; i += SORT_THREADS) keys_out[i] = key[i];
  __syncthreads();
  const int nv = nv_s;
  // 1. compact the segment starts (thread = PER consecutive positions)
  constexpr int PER = SORT_MAX / SORT_THREADS;
  const int base = threadIdx.x * PER;
  auto is_start = [&](int i) { return i < nv && (i == 0 || (key[i] >> 13) != (key[i - 1] >> 13)); };
  int cnt = 0;
#pragma unroll
  for (int e = 0; e < PER; ++e) cnt += is_start(base + e) ? 1 : 0;
  int nseg;
  int j = block_exclusive_scan(cnt, wsum, &nseg);
#pragma unroll
  for (int e = 0; e < PER; ++e)
    if (is_start(base + e)) starts[j++] = base + e;
  __syncthreads();
  // 2. lengths from consecutive starts; split into the short and long lists
  auto seg_len = [&](int q) { return (q + 1 < nseg ? starts[q + 1] : nv) - starts[q]; };
  const int q0 = threadIdx.x * PER;
  int cs = 0, cl = 0;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int q = q0 + e;
    if (q < nseg) {
      if (seg_len(q) > LONG_SEG) ++cl; else ++cs;
    }
  }
  int tot_s, tot_l;
  int js = block_exclusive_scan(cs, wsum, &tot_s);
  int jl = block_exclusive_scan(cl, wsum, &tot_l);
  int* seg_s = seg + 4;
  int* seg_l = seg + 4 + 2 * SORT_MAX;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int q = q0 + e;
    if (q < nseg) {
      const int len = seg_len(q);
      int* dst = len > LONG_SEG ? seg_l + 2 * jl++ : seg_s + 2 * js++;
      dst[0] = starts[q];
      dst[1] = len;
    }
  }
  if (threadIdx.x == 0) {
    seg[0] = tot_s;
    seg[1] = tot_l;
  }
}

// Persistent: first every long (segment,
// 256-column chunk) item is summed by a whole CTA (8 warps over contiguous
// token ranges, then the warps in order), then every short (segment,
// 1024-column group) item by one warp in token order.  Either order is fixed,
// so the result is deterministic; each item adds into its dE row (fp32) once.
constexpr int BWD_WARPS = 8;

// acc[w][8] += sum over sorted positions q in [q0, q1) of dY[token(q)][col + 256 w .. + 8], w < W.
template <int W, int DEPTH>
__device__ __forceinline__ void accum_rows(const uint32_t* __restrict__ keys, int q0, int q1, int64_t n0, int64_t h,
                                           int64_t col, const uint16_t* __restrict__ dY, int lane,
                                           float (&acc)[W][8]) {
  for (int qb = q0; qb < q1; qb += 32) {
    const int nq = q1 - qb < 32 ? q1 - qb : 32;
    const uint32_t mykey = lane < nq ? keys[qb + lane] : 0u;  // 32 token indices, one coalesced load
    for (int u = 0; u < nq; u += DEPTH) {
      uint4 v[DEPTH][W];
#pragma unroll
      for (int r = 0; r < DEPTH; ++r) {
        const uint32_t kq = __shfl_sync(0xffffffffu, mykey, (u + r) & 31);
        const uint16_t* row = dY + (n0 + (kq & 8191u)) * h;
#pragma unroll
        for (int w = 0; w < W; ++w) {
          const int64_t c = col + 256 * w;
          v[r][w] = make_uint4(0u, 0u, 0u, 0u);
          if (u + r < nq && c < h) v[r][w] = *reinterpret_cast<const uint4*>(row + c);
        }
      }
#pragma unroll
      for (int r = 0; r < DEPTH; ++r) {
        if (u + r < nq) {
#pragma unroll
          for (int w = 0; w < W; ++w) {
            float a, b;
            unpack_bf16x2(v[r][w].x, a, b); acc[w][0] += a; acc[w][1] += b;
            unpack_bf16x2(v[r][w].y, a, b); acc[w][2] += a; acc[w][3] += b;
            unpack_bf16x2(v[r][w].z, a, b); acc[w][4] += a; acc[w][5] += b;
            unpack_bf16x2(v[r][w].w, a, b); acc[w][6] += a; acc[w][7] += b;
          }
        }
      }
    }
  }
}

__global__ void __launch_bounds__(BWD_WARPS * 32)
    emb_bwd_kernel(const uint32_t* __restrict__ keys, int* __restrict__ seg, int64_t n0, int64_t h,
                   const uint16_t* __restrict__ dY, float* __restrict__ dE) {
  __shared__ float part[BWD_WARPS][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nshort = seg[0], nlong = seg[1];
  const int* seg_s = seg + 4;
  const int* seg_l = seg + 4 + 2 * SORT_MAX;
  // long items: one CTA each, round-robin over the CTAs
  const int64_t ncl = (h + 255) / 256;
  for (int64_t it = blockIdx.x; it < static_cast<int64_t>(nlong) * ncl; it += gridDim.x) {
    const int j = static_cast<int>(it / ncl);
    const int64_t col0 = (it - static_cast<int64_t>(j) * ncl) * 256;
    const int start = seg_l[2 * j], len = seg_l[2 * j + 1];
    float acc[1][8] = {{0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}};
    accum_rows<1, 8>(keys, start + (len * warp) / BWD_WARPS, start + (len * (warp + 1)) / BWD_WARPS, n0, h,
                     col0 + lane * 8, dY, lane, acc);
#pragma unroll
    for (int e = 0; e < 8; ++e) part[warp][lane * 8 + e] = acc[0][e];
    __syncthreads();
    const int c = threadIdx.x;
    if (col0 + c < h) {
      float sum = 0.0f;
#pragma unroll
      for (int w = 0; w < BWD_WARPS; ++w) sum += part[w][c];
      dE[static_cast<int64_t>(keys[start] >> 13) * h + col0 + c] += sum;
    }
    __syncthreads();  // part is rewritten by the next item
  }
  // short items: one warp each, 1024 columns (4 x 8 per lane), assigned
  // round-robin starting from the last CTAs (the first ones took the long items)
  const int64_t ncs = (h + 1023) / 1024;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * BWD_WARPS;
  const int64_t gw = static_cast<int64_t>(gridDim.x - 1 - blockIdx.x) * BWD_WARPS + warp;
  for (int64_t it = gw; it < static_cast<int64_t>(nshort) * ncs; it += nwarps) {
    const int j = static_cast<int>(it / ncs);
    const int64_t col = (it - static_cast<int64_t>(j) * ncs) * 1024 + lane * 8;
    const int start = seg_s[2 * j], len = seg_s[2 * j + 1];
    float acc[4][8];
#pragma unroll
    for (int w = 0; w < 4; ++w)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[w][e] = 0.0f;
    accum_rows<4, 2>(keys, start, start + len, n0, h, col, dY, lane, acc);
    float* drow = dE + static_cast<int64_t>(keys[start] >> 13) * h;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int64_t c = col + 256 * w;
      if (c < h) {
        float4* d4 = reinterpret_cast<float4*>(drow + c);
        float4 d0 = d4[0], d1 = d4[1];
        d0.x += acc[w][0]; d0.y += acc[w][1]; d0.z += acc[w][2]; d0.w += acc[w][3];
        d1.x += acc[w][4]; d1.y += acc[w][5]; d1.z += acc[w][6]; d1.w += acc[w][7];
        d4[0] = d0;
        d4[1] = d1;
      }
    }
  }
}

}  // namespace

size_t emb_bwd_ws_bytes(int64_t N) {
  const int64_t c = N < SORT_MAX ? N : SORT_MAX;
  const size_t n = static_cast<size_t>(c > 0 ? c : 1);
  return ((n * 4 + 255) & ~static_cast<size_t>(255)) + (4 + 4 * SORT_MAX) * 4;  // sorted keys, two segment lists
}

tp_status run_emb_forward(const int32_t* ids, int64_t N, int64_t V, int64_t h, int t, const uint16_t* E, uint16_t* Y,
                          cudaStream_t s) {
  if (N < 0 || V < 1 || h < 1 || t < 1) return TP_ERR_INVALID_ARG;
  if (V % t != 0 || V >= (1LL << 19)) return TP_ERR_SHAPE;  // keys: 19 bits of id, 13 of token
  if (h % 8 != 0) return TP_ERR_ALIGN;
  if (N == 0) return TP_OK;
  if (!ids || !E || !Y) return TP_ERR_INVALID_ARG;
  if (!aligned16(E) || !aligned16(Y)) return TP_ERR_ALIGN;
  TP_RETURN_IF(ready());
  int64_t grid = static_cast<int64_t>(device_sm_count()) * 8;
  if (grid > N) grid = N;
  emb_fwd_kernel<<<static_cast<unsigned>(grid), EMB_THREADS, 0, s>>>(ids, N, V, V / t, h, E, Y, device_error_word());
  TP_LAUNCHED();
  return TP_OK;
}

tp_status run_emb_backward(const int32_t* ids, const uint16_t* dY, int64_t N, int64_t V, int64_t h, int t, float* dE,
                           int accumulate, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (N < 0 || V < 1 || h < 1 || t < 1) return TP_ERR_INVALID_ARG;
  if (V % t != 0 || V >= (1LL << 19)) return TP_ERR_SHAPE;  // keys: 19 bits of id, 13 of token
  if (h % 8 != 0) return TP_ERR_ALIGN;
  if (!dE) return TP_ERR_INVALID_ARG;
  if (N > 0 && (!ids || !dY || !ws)) return TP_ERR_INVALID_ARG;
  if (!aligned16(dE) || (N > 0 && (!aligned16(dY) || !aligned16(ws)))) return TP_ERR_ALIGN;
  if (N > 0 && ws_bytes < emb_bwd_ws_bytes(N)) return TP_ERR_WORKSPACE;
  TP_RETURN_IF(ready());
  if (!accumulate) TP_CUDA_CHECK(cudaMemsetAsync(dE, 0, static_cast<size_t>(V) * h * sizeof(float), s));
  static bool configured[64] = {};
  int dev = 0;
  TP_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return TP_ERR_CUDA;
  if (!configured[dev]) {
    TP_CUDA_CHECK(cudaFuncSetAttribute(emb_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * SORT_MAX * 4));
    configured[dev] = true;
  }
  uint32_t* keys = static_cast<uint32_t*>(ws);
  const int64_t cmax = N < SORT_MAX ? N : SORT_MAX;
  int* seg = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + ((static_cast<size_t>(cmax) * 4 + 255) & ~static_cast<size_t>(255)));
  for (int64_t n0 = 0; n0 < N; n0 += SORT_MAX) {
    const int n = static_cast<int>(N - n0 < SORT_MAX ? N - n0 : SORT_MAX);
    emb_sort_kernel<<<1, SORT_THREADS, 2 * SORT_MAX * 4, s>>>(ids, n0, n, V, keys, seg, device_error_word());
    TP_LAUNCHED();
    emb_bwd_kernel<<<static_cast<unsigned>(device_sm_count() * 2), BWD_WARPS * 32, 0, s>>>(keys, seg, n0, h, dY, dE);
    TP_LAUNCHED();
  }
  return TP_OK;
}

}  // namespace tp
