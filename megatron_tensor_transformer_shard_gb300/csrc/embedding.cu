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
// The backward is deterministic: within a chunk of up to 8192 tokens the tokens are
// grouped by id -- each token's rank among its id's tokens, the id's count and first
// token counted by brute force over the chunk's ids, on every SM -- and placed in the
// order (first token of the id, token), which cuts them into segments of equal ids;
// each segment's dY rows are summed in a fixed order (a warp in token order for short
// segments; 8 warps over contiguous token ranges, then the warps in order, for long
// ones) into dE.  The rows are prefetched into L2 while the grouping runs.  Chunks
// run one after another on the stream.
#include <cuda_runtime.h>

#include "devmath.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace tp {
namespace {

constexpr int EMB_THREADS = 128;
constexpr int SORT_MAX = 8192;  // tokens per chunk: 13 bits of token index in a key
constexpr int ERR_EMB_ID = 0x202;  // a token id outside [0, V): argument error found on the device

__device__ __forceinline__ uint4 ld_nc16(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// acc[0..7] += the 8 bf16 values of w, in order.
__device__ __forceinline__ void add_bf16x8(const uint4& w, float (&acc)[8]) {
  float a, b;
  unpack_bf16x2(w.x, a, b); acc[0] += a; acc[1] += b;
  unpack_bf16x2(w.y, a, b); acc[2] += a; acc[3] += b;
  unpack_bf16x2(w.z, a, b); acc[4] += a; acc[5] += b;
  unpack_bf16x2(w.w, a, b); acc[6] += a; acc[7] += b;
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

constexpr int LONG_SEG = 8;     // longer segments of equal ids are summed by a whole CTA
constexpr int SHORT_DESC = 12;  // ints per short-segment descriptor: id, length, 8 tokens, 2 unused

// The rows the backward of tokens [n0, n0 + n) reads and adds into -- dY[n] and
// dE[id(n)] -- pulled into L2 by bulk prefetches, one 16 KB piece per thread of the
// grid (pieces q, q + stride, ...).  The kernel runs on a side stream beside the
// grouping, so the rows stream in meanwhile and nothing waits for it.  Only a cache
// hint; the sums do not depend on it.
__device__ __forceinline__ void emb_prefetch_rows(const int32_t* __restrict__ ids, int64_t n0, int n, int64_t V,
                                                  int64_t h, const uint16_t* __restrict__ dY,
                                                  const float* __restrict__ dE, int64_t q0, int64_t stride) {
  const int64_t py = (h * 2 + 16383) / 16384, pe = (h * 4 + 16383) / 16384;  // 16 KB pieces per row
  const int64_t per = py + pe;
  for (int64_t q = q0; q < n * per; q += stride) {
    const int64_t i = q / per, k = q - i * per;
    const uint8_t* p;
    int64_t off, bytes;
    if (k < py) {
      p = reinterpret_cast<const uint8_t*>(dY + (n0 + i) * h);
      off = k * 16384;
      bytes = h * 2;
    } else {
      const int64_t id = ids[n0 + i];
      if (id < 0 || id >= V) continue;
      p = reinterpret_cast<const uint8_t*>(dE + id * h);
      off = (k - py) * 16384;
      bytes = h * 4;
    }
    const uint32_t sz = static_cast<uint32_t>(bytes - off < 16384 ? bytes - off : 16384);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p + off), "r"(sz) : "memory");
  }
}

constexpr int PREFETCH_THREADS = 128;
__global__ void __launch_bounds__(PREFETCH_THREADS)
    emb_prefetch_kernel(const int32_t* __restrict__ ids, int64_t n0, int n, int64_t V, int64_t h,
                        const uint16_t* __restrict__ dY, const float* __restrict__ dE) {
  emb_prefetch_rows(ids, n0, n, V, h, dY, dE, static_cast<int64_t>(blockIdx.x) * PREFETCH_THREADS + threadIdx.x,
                    static_cast<int64_t>(gridDim.x) * PREFETCH_THREADS);
}

// Grouping of a chunk's tokens by id without a sort, spread over the GPU.
// Pass 1 (a warp per token, the chunk's ids in every CTA's shared memory, four ids a
// lane load) counts per token i: `before`, the tokens of its id before it; `total`,
// the tokens of its id; `first`, its id's first token.  An id outside [0, V) is
// reported and gets first = INT_MAX, total = 0: it joins no segment.
// Pass 2 (1024 tokens per CTA) places the tokens in the order (first token of the id,
// token): every CTA scans the chunk's per-token flags itself (n <= 8192) for each id's
// offset and short-list index, then writes its tokens: keys[offset(first) + before] =
// id << 13 | i; a short id's descriptor (id, length, tokens) with every token filling
// its own slot; a long id's (start, length) at its rank, longest first (ties by first
// token).  seg[0], seg[1] = the numbers of short and long segments.
constexpr int COUNT_WARPS = 16;   // tokens per CTA in pass 1
constexpr int PLACE_THREADS = 1024;  // short serial runs in the scans (the pass is latency-bound)
constexpr int kPlaceSmem = (5 * (SORT_MAX + SORT_MAX / 32 + 2) + SORT_MAX) * 4;

__global__ void __launch_bounds__(COUNT_WARPS * 32)
    emb_count_kernel(const int32_t* __restrict__ ids, int64_t n0, int n, int64_t V, int* __restrict__ before,
                     int* __restrict__ total, int* __restrict__ first, int* err) {
  __shared__ __align__(16) int sid[SORT_MAX];
  const int npad = (n + 127) & ~127;
  {
    constexpr int K = SORT_MAX / (COUNT_WARPS * 32);
    int v[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {  // every load in flight before the first store
      const int m = threadIdx.x + k * COUNT_WARPS * 32;
      v[k] = -1 - m;  // padding and invalid ids match nothing
      if (m < n) {
        const int64_t id = ids[n0 + m];
        if (id >= 0 && id < V) v[k] = static_cast<int>(id);
      }
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int m = threadIdx.x + k * COUNT_WARPS * 32;
      if (m < npad) sid[m] = v[k];
    }
  }
  __syncthreads();
  ptx::griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * COUNT_WARPS + warp;
  if (i >= n) return;
  const int me = sid[i];
  int b = 0, tt = 0, f = 0x7fffffff;
  const int4* s4 = reinterpret_cast<const int4*>(sid);
  // Nearly every group of four holds no match: one combined test, the counts only on a hit
  // (the loop was issue-bound at about 11 instructions an id).
#pragma unroll 4
  for (int q = lane; q < npad / 4; q += 32) {
    const int4 v = s4[q];
    if ((v.x == me) | (v.y == me) | (v.z == me) | (v.w == me)) {
      const int m = 4 * q;
      if (v.x == me) { ++tt; b += m < i; f = min(f, m); }
      if (v.y == me) { ++tt; b += m + 1 < i; f = min(f, m + 1); }
      if (v.z == me) { ++tt; b += m + 2 < i; f = min(f, m + 2); }
      if (v.w == me) { ++tt; b += m + 3 < i; f = min(f, m + 3); }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    b += __shfl_xor_sync(0xffffffffu, b, o);
    tt += __shfl_xor_sync(0xffffffffu, tt, o);
    f = min(f, __shfl_xor_sync(0xffffffffu, f, o));
  }
  if (lane == 0) {
    const bool ok = me >= 0;
    if (!ok) atomicCAS(err, 0, ERR_EMB_ID);
    before[i] = ok ? b : 0;
    total[i] = ok ? tt : 0;
    first[i] = ok ? f : 0x7fffffff;
  }
}

// Exclusive prefix sums over m < n of three per-entry counts f(m) = (a, b, c) into
// p0[m], p1[m], p2[m] (p*[n] = the totals).  Thread t takes the PLACE_RUN consecutive
// entries [t R, t R + R) in registers (entry m is read from shared memory at m + m / 32,
// the padding that keeps these strided reads free of bank conflicts), one block scan of
// the run sums, then the run's prefixes.  wsum: 3 * 32 ints.
constexpr int PLACE_RUN = SORT_MAX / PLACE_THREADS;
__device__ __forceinline__ int pad32(int m) { return m + (m >> 5); }

template <typename F>
__device__ __forceinline__ void place_scan3(int n, F f, int* p0, int* p1, int* p2, int* wsum) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  constexpr int NW = PLACE_THREADS / 32;
  int3 v[PLACE_RUN];
  int3 run = make_int3(0, 0, 0);
#pragma unroll
  for (int k = 0; k < PLACE_RUN; ++k) {
    const int m = t * PLACE_RUN + k;
    v[k] = m < n ? f(m) : make_int3(0, 0, 0);
    run.x += v[k].x;
    run.y += v[k].y;
    run.z += v[k].z;
  }
  int3 inc = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ux = __shfl_up_sync(0xffffffffu, inc.x, o), uy = __shfl_up_sync(0xffffffffu, inc.y, o),
              uz = __shfl_up_sync(0xffffffffu, inc.z, o);
    if (lane >= o) {
      inc.x += ux;
      inc.y += uy;
      inc.z += uz;
    }
  }
  if (lane == 31) {
    wsum[warp] = inc.x;
    wsum[32 + warp] = inc.y;
    wsum[64 + warp] = inc.z;
  }
  __syncthreads();
  int3 e = make_int3(inc.x - run.x, inc.y - run.y, inc.z - run.z), tot = make_int3(0, 0, 0);
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const int x = wsum[w], y = wsum[32 + w], z = wsum[64 + w];
    if (w < warp) {
      e.x += x;
      e.y += y;
      e.z += z;
    }
    tot.x += x;
    tot.y += y;
    tot.z += z;
  }
#pragma unroll
  for (int k = 0; k < PLACE_RUN; ++k) {
    const int m = t * PLACE_RUN + k;
    if (m < n) {
      p0[pad32(m)] = e.x;
      p1[pad32(m)] = e.y;
      p2[pad32(m)] = e.z;
    }
    e.x += v[k].x;
    e.y += v[k].y;
    e.z += v[k].z;
  }
  if (t == 0) {
    p0[pad32(n)] = tot.x;
    p1[pad32(n)] = tot.y;
    p2[pad32(n)] = tot.z;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(PLACE_THREADS)
    emb_place_kernel(const int32_t* __restrict__ ids, int64_t n0, int n, const int* __restrict__ before,
                     const int* __restrict__ total, const int* __restrict__ first, uint32_t* __restrict__ keys,
                     int* __restrict__ seg) {
  extern __shared__ int place_sm[];  // first, total; offsets, short indices, long indices (padded); long reps
  constexpr int PADN = SORT_MAX + SORT_MAX / 32 + 2;
  int* sf = place_sm;
  int* st = sf + PADN;
  int* poff = st + PADN;
  int* pshort = poff + PADN;
  int* plong = pshort + PADN;
  int* lrep = plong + PADN;  // long ids' first tokens, in first-token order
  __shared__ int wsum[96];
  ptx::griddep_wait();  // pass 1's counts
  {
    constexpr int K = SORT_MAX / PLACE_THREADS;
    int vf[K], vt[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {  // every load in flight before the first store
      const int m = threadIdx.x + k * PLACE_THREADS;
      vf[k] = m < n ? first[m] : 0;
      vt[k] = m < n ? total[m] : 0;
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int m = threadIdx.x + k * PLACE_THREADS;
      if (m < n) {
        sf[pad32(m)] = vf[k];
        st[pad32(m)] = vt[k];
      }
    }
  }
  __syncthreads();
  // per entry: tokens of a first occurrence, short first occurrences, long first occurrences
  place_scan3(
      n,
      [&](int m) {
        const int fm = sf[pad32(m)], tm = st[pad32(m)];
        const bool rep = fm == m;
        return make_int3(rep ? tm : 0, (rep && tm <= LONG_SEG) ? 1 : 0, (rep && tm > LONG_SEG) ? 1 : 0);
      },
      poff, pshort, plong, wsum);
  const int nl = plong[pad32(n)];
  for (int m = threadIdx.x; m < n; m += PLACE_THREADS)
    if (sf[pad32(m)] == m && st[pad32(m)] > LONG_SEG) lrep[plong[pad32(m)]] = m;
  __syncthreads();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    seg[0] = pshort[pad32(n)];
    seg[1] = nl;
  }
  const int i = blockIdx.x * PLACE_THREADS + threadIdx.x;
  if (i >= n) return;
  const int r = sf[pad32(i)];
  if (r == 0x7fffffff) return;  // invalid id
  const int len = st[pad32(i)];
  const int b = before[i];
  const int id = static_cast<int>(ids[n0 + i]);
  const int off = poff[pad32(r)];
  keys[off + b] = (static_cast<uint32_t>(id) << 13) | static_cast<uint32_t>(i);
  if (len <= LONG_SEG) {
    int* d = seg + 4 + SHORT_DESC * pshort[pad32(r)];
    d[2 + b] = i;
    if (b == 0) {
      d[0] = id;
      d[1] = len;
      for (int k = len; k < SHORT_DESC - 2; ++k) d[2 + k] = 0;
    }
  } else if (b == 0) {
    int rank = 0;  // longest first, ties by first token
    for (int k = 0; k < nl; ++k) {
      const int mk = lrep[k], tk = st[pad32(mk)];
      rank += (tk > len || (tk == len && mk < r)) ? 1 : 0;
    }
    int* d = seg + 4 + SHORT_DESC * SORT_MAX + 2 * rank;
    d[0] = off;
    d[1] = len;
  }
}

// Persistent: first every long (segment, 256-column chunk) item is summed by a
// whole CTA (8 warps over contiguous token ranges, then the warps in order), then
// every short (segment, 512-column group) item by one warp in token order.  Either
// order is fixed, so the result is deterministic; each item adds into its dE row
// (fp32) once.  The dE values an item adds to are loaded with its dY rows, and a
// warp loads its next short descriptor while the current item's rows are in flight.
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
          for (int w = 0; w < W; ++w) add_bf16x8(v[r][w], acc[w]);
        }
      }
    }
  }
}

__device__ __forceinline__ void load_desc(const int* __restrict__ d, int4 (&q)[SHORT_DESC / 4]) {
#pragma unroll
  for (int k = 0; k < SHORT_DESC / 4; ++k) q[k] = __ldcg(reinterpret_cast<const int4*>(d) + k);
}

__device__ __forceinline__ int desc_word(const int4 (&q)[SHORT_DESC / 4], int i) {
  const int4 x = q[i / 4];
  return (i & 3) == 0 ? x.x : (i & 3) == 1 ? x.y : (i & 3) == 2 ? x.z : x.w;
}

__global__ void __launch_bounds__(BWD_WARPS * 32)
    emb_bwd_kernel(const uint32_t* __restrict__ keys, int* __restrict__ seg, int64_t n0, int64_t h,
                   const uint16_t* __restrict__ dY, float* __restrict__ dE) {
  __shared__ float part[BWD_WARPS][256];
  ptx::griddep_wait();  // the grouping's keys and lists
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nshort = seg[0], nlong = seg[1];
  const int* seg_s = seg + 4;
  const int* seg_l = seg + 4 + SHORT_DESC * SORT_MAX;
  // long items: one CTA each, round-robin over the CTAs, longest segments first
  const int64_t ncl = (h + 255) / 256;
  for (int64_t it = blockIdx.x; it < static_cast<int64_t>(nlong) * ncl; it += gridDim.x) {
    const int j = static_cast<int>(it / ncl);
    const int64_t col0 = (it - static_cast<int64_t>(j) * ncl) * 256;
    const int start = seg_l[2 * j], len = seg_l[2 * j + 1];
    const int64_t row = keys[start] >> 13;
    const int c = threadIdx.x;  // column col0 + c of the final sum
    const float d0 = (col0 + c < h) ? dE[row * h + col0 + c] : 0.0f;
    float acc[1][8] = {{0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}};
    accum_rows<1, 16>(keys, start + (len * warp) / BWD_WARPS, start + (len * (warp + 1)) / BWD_WARPS, n0, h,
                      col0 + lane * 8, dY, lane, acc);
#pragma unroll
    for (int e = 0; e < 8; ++e) part[warp][lane * 8 + e] = acc[0][e];
    __syncthreads();
    float s0 = 0.0f;
#pragma unroll
    for (int w = 0; w < BWD_WARPS; ++w) s0 += part[w][c];
    if (col0 + c < h) dE[row * h + col0 + c] = d0 + s0;
    __syncthreads();  // part is rewritten by the next item
  }
  // short items: one warp each, 512 columns (2 x 8 per lane), assigned round-robin
  // starting from the last CTAs (the first ones took the long items)
  const int64_t ncs = (h + 511) / 512;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * BWD_WARPS;
  const int64_t gw = static_cast<int64_t>(gridDim.x - 1 - blockIdx.x) * BWD_WARPS + warp;
  const int64_t nitems = static_cast<int64_t>(nshort) * ncs;
  int4 dq[SHORT_DESC / 4];
  if (gw < nitems) load_desc(seg_s + SHORT_DESC * (gw / ncs), dq);
  for (int64_t it = gw; it < nitems; it += nwarps) {
    const int j = static_cast<int>(it / ncs);
    const int64_t col = (it - static_cast<int64_t>(j) * ncs) * 512 + lane * 8;
    const int64_t row = desc_word(dq, 0);
    const int len = desc_word(dq, 1);
    // this item's dE values and all its dY rows at once
    float4 e4[2][2];
    uint4 v[LONG_SEG][2];
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const int64_t c = col + 256 * w;
      e4[w][0] = e4[w][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < h) {
        const float4* d4 = reinterpret_cast<const float4*>(dE + row * h + c);
        e4[w][0] = d4[0];
        e4[w][1] = d4[1];
      }
    }
#pragma unroll
    for (int r = 0; r < LONG_SEG; ++r) {
      const int64_t tok = desc_word(dq, 2 + r);
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const int64_t c = col + 256 * w;
        v[r][w] = make_uint4(0u, 0u, 0u, 0u);
        if (r < len && c < h) v[r][w] = *reinterpret_cast<const uint4*>(dY + (n0 + tok) * h + c);
      }
    }
    const int64_t nx = it + nwarps;  // the next item's descriptor, while the rows arrive
    if (nx < nitems && nx / ncs != j) load_desc(seg_s + SHORT_DESC * (nx / ncs), dq);
    float acc[2][8];
#pragma unroll
    for (int w = 0; w < 2; ++w)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[w][e] = 0.0f;
#pragma unroll
    for (int r = 0; r < LONG_SEG; ++r) {
      if (r < len) {
#pragma unroll
        for (int w = 0; w < 2; ++w) add_bf16x8(v[r][w], acc[w]);
      }
    }
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const int64_t c = col + 256 * w;
      if (c < h) {
        float4* d4 = reinterpret_cast<float4*>(dE + row * h + c);
        d4[0] = make_float4(e4[w][0].x + acc[w][0], e4[w][0].y + acc[w][1], e4[w][0].z + acc[w][2],
                            e4[w][0].w + acc[w][3]);
        d4[1] = make_float4(e4[w][1].x + acc[w][4], e4[w][1].y + acc[w][5], e4[w][1].z + acc[w][6],
                            e4[w][1].w + acc[w][7]);
      }
    }
  }
}

}  // namespace

size_t emb_bwd_ws_bytes(int64_t N) {
  const int64_t c = N < SORT_MAX ? N : SORT_MAX;
  const size_t n = static_cast<size_t>(c > 0 ? c : 1);
  // keys; the two segment lists; the grouping's three per-token counts
  return ((n * 4 + 255) & ~static_cast<size_t>(255)) + (4 + (SHORT_DESC + 2 + 3) * SORT_MAX) * 4;
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
    TP_CUDA_CHECK(cudaFuncSetAttribute(emb_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPlaceSmem));
    configured[dev] = true;
  }
  // side stream and events of the prefetch (per device; events per call, released when done)
  static cudaStream_t sides[64] = {};
  if (!sides[dev]) TP_CUDA_CHECK(cudaStreamCreateWithFlags(&sides[dev], cudaStreamNonBlocking));
  cudaStream_t side = sides[dev];
  cudaEvent_t fork = nullptr, join = nullptr;
  TP_CUDA_CHECK(cudaEventCreateWithFlags(&fork, cudaEventDisableTiming));
  TP_CUDA_CHECK(cudaEventCreateWithFlags(&join, cudaEventDisableTiming));
  struct EvGuard {
    cudaEvent_t a, b;
    ~EvGuard() {
      cudaEventDestroy(a);
      cudaEventDestroy(b);
    }
  } ev_guard{fork, join};
  uint32_t* keys = static_cast<uint32_t*>(ws);
  const int64_t cmax = N < SORT_MAX ? N : SORT_MAX;
  int* seg = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + ((static_cast<size_t>(cmax) * 4 + 255) & ~static_cast<size_t>(255)));
  int* cnt_before = seg + 4 + (SHORT_DESC + 2) * SORT_MAX;  // the grouping's per-token counts
  int* cnt_total = cnt_before + SORT_MAX;
  int* cnt_first = cnt_total + SORT_MAX;
  for (int64_t n0 = 0; n0 < N; n0 += SORT_MAX) {
    const int n = static_cast<int>(N - n0 < SORT_MAX ? N - n0 : SORT_MAX);
    // the rows' prefetch on the side stream, beside the grouping; then the sums
    TP_CUDA_CHECK(cudaEventRecord(fork, s));
    TP_CUDA_CHECK(cudaStreamWaitEvent(side, fork, 0));
    emb_prefetch_kernel<<<static_cast<unsigned>(device_sm_count()), PREFETCH_THREADS, 0, side>>>(ids, n0, n, V, h,
                                                                                                dY, dE);
    TP_LAUNCHED();
    TP_CUDA_CHECK(cudaEventRecord(join, side));
    emb_count_kernel<<<static_cast<unsigned>((n + COUNT_WARPS - 1) / COUNT_WARPS), COUNT_WARPS * 32, 0, s>>>(
        ids, n0, n, V, cnt_before, cnt_total, cnt_first, device_error_word());
    TP_LAUNCHED();
    TP_CUDA_CHECK(launch_pdl(emb_place_kernel, dim3(static_cast<unsigned>((n + PLACE_THREADS - 1) / PLACE_THREADS)),
                             dim3(PLACE_THREADS), kPlaceSmem, s, ids, n0, n,
                             static_cast<const int*>(cnt_before), static_cast<const int*>(cnt_total),
                             static_cast<const int*>(cnt_first), keys, seg));
    TP_CUDA_CHECK(launch_pdl(emb_bwd_kernel, dim3(static_cast<unsigned>(device_sm_count() * 2)),
                             dim3(BWD_WARPS * 32), 0, s, static_cast<const uint32_t*>(keys), seg, n0, h, dY, dE));
    count_launch(2);
    TP_CUDA_CHECK(cudaStreamWaitEvent(s, join, 0));  // the side stream rejoins (its work is long done)
  }
  return TP_OK;
}

}  // namespace tp
