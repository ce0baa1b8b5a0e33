// Persistent, warp-specialised bf16 GEMM on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory) fed by TMA, for sm_103a.
//
// This one kernel carries every dense contraction of the TP block:
//   column-parallel  Z_i = X W_up,i + b, A_i = act(Z_i)        (output batch = shard)
//   row-parallel     Y = sum_i A_i W_down,i + b (+ residual)    (shards summed in the accumulator)
//   dgrad            dZ_i = (dY W_down,i^T) * act'(Z_i)
//   f backward       dX = sum_i dZ_i W_up,i^T
//   wgrad            dW_down,i = A_i^T dY, dW_up,i = dZ_i^T X    (MN-major operands)
//   SwiGLU           Z_i = X [W_gate | W_up]_i, A_i = silu(gate) up in the epilogue; its
//                    dgrad epilogue turns dA into d gate / d up (gate / up interleaved in
//                    groups of 128 columns, so one 256-column tile holds both halves)
// ("02 — Tensor Parallelism", "Column-parallel vs row-parallel — the
// derivation" and "The MLP pairing"; "Parallelism Strategies #1 - Tensor
// Parallelism", sharded backward.)
//
// The g all-reduce of the row-parallel GEMM needs no buffer on one GPU: shard
// i's K range is accumulated into the same TMEM accumulator right after shard
// i-1's, so the accumulator ends holding P_0 + P_1 + ... + P_{t-1} in shard
// order, and the output bias is added once in the epilogue.
//
// CTA layout (192 threads, one CTA per SM, persistent over output tiles):
//   warp 0     TMA producer: fills a STAGES-deep ring of A/B tiles (128B swizzle)
//   warp 1     allocates 512 TMEM columns; lane 0 issues tcgen05.mma 128x256x16
//              into one of two 256-column accumulators (double-buffered so the
//              epilogue of tile n overlaps the main loop of tile n+1)
//   warps 2-5  epilogue: tcgen05.ld rows of the accumulator (warp w reads TMEM
//              lanes 32*(w%4)..+31), apply bias / activation / residual, store.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <type_traits>
#include <atomic>
#include <ctime>
#include <mutex>

#include "devmath.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace tp {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // one 128-byte swizzle row of bf16
constexpr int STAGES = 4;
constexpr int A_TILE_BYTES = BM * BK * 2;
constexpr int B_TILE_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_TILE_BYTES + B_TILE_BYTES;
constexpr int MN_CHUNK_BYTES = 64 * BK * 2;  // one 64-wide MN-major TMA box
constexpr int TMEM_COLS = 2 * BN;
constexpr int NUM_THREADS = 192;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;

enum : int { ERR_WAIT_PRODUCER = 0x101, ERR_WAIT_MMA = 0x102, ERR_WAIT_EPI = 0x103, ERR_WAIT_DRAIN = 0x104,
              ERR_WAIT_OVL = 0x105, ERR_WAIT_SK = 0x106 };

struct GemmArgs {
  int M, N;
  int nbatch, nsum;
  int a_sharded, b_sharded;
  // Operand viewed through a 4-D map, one copy per stage: MN-major (64 columns, K, 64-column
  // chunks, shard) when its row count is a multiple of 64; K-major in the pair kernel's
  // two-k-block stages (64 K, rows, k-blocks, shard) when K is a multiple of 64.
  int a_4d, b_4d;
  int mt, nt, kt;
  int epi, act;
  int f16ab;  // A and B are IEEE fp16 (else bf16)
  void* d;
  int64_t ldd, d_bs;
  void* d2;
  int64_t ldd2, d2_bs;  // EPI_GLU: the activation output's strides
  const uint16_t* bias;
  int64_t bias_bs;
  const uint16_t* aux;
  int64_t ld_aux, aux_bs;
  float* cs;      // EPI_DACT: per 32-row block column sums [nbatch][cs_chunks][N] (nullable)
  int cs_chunks;
  const uint16_t* res;
  int64_t ld_res;
  int accumulate;
  int out_f16;
  int tma_store;  // pair kernel: outputs staged in shared memory and written by TMA bulk stores
  // K ranges per output tile: 1, except in gemm_splitc_kernel, where the nsum * kt k-steps of
  // a tile are cut into ksplit nearly equal ranges, one per CTA of a cluster.
  int ksplit;
  // Split K across CTA pairs (pair kernel).  The first sp_rounds * nclusters tiles are
  // whole; the next sp_tiles tiles are cut into sp_split K ranges at the same k-stages (range
  // j covers [j U / S, (j + 1) U / S) of the sp_units stages).  Every range writes its fp32
  // partial to a slot, then counts itself in the tile's counter for its CTA and warp; the
  // range that completes the count adds the partials in range order and applies the
  // epilogue.  sp_split = 0: every tile whole.
  // Overlapped shard reduction (sp_seq, EPI_BF16): every tile is cut at its sp_split shard
  // boundaries, each shard an item; shard j's fp32 partial goes to the caller's [S][M][N]
  // buffer (sp_user = 1) and, by TMA, into the tile's fp32 running sum (stored for shard 0,
  // added in L2 for the next ones, each after the previous shard's flag sp_cnt = epoch << 32
  // | j says its add is complete); the last shard adds its accumulator to the running sum
  // and applies the epilogue.
  // Chained ranges (sp_chain, EPI_BF16): the ranges of a split tile add into the tile's fp32
  // running sum in range order, as the shards do in the overlapped reduction, and no range
  // writes a partial of its own: range 0 stores, the middle ranges add in L2, the last range
  // loads the sum, adds its accumulator and applies the epilogue.  The overlapped reduction
  // is the chained form with sp_seq and sp_user set.
  // Chained ranges are dealt range-major (every split tile's range 0, then every tile's range
  // 1, ...), so the pairs working side by side mostly share one K slice of the panels.
  int sp_rounds, sp_tiles, sp_split, sp_units, sp_seq, sp_chain;
  int sp_user;              // partials in the caller's [S][M][N] buffer, else 256 x 256 slots
  float* sp_part;           // slots [split tiles * S][256][256], or the caller's buffer (unused when chained)
  int64_t sp_ld, sp_bs;     // sp_user: row and range strides in floats
  unsigned long long* sp_cnt;  // [split tiles][2 CTAs][4 warps]
  uint32_t sp_epoch;
  int* err;
  uint64_t timeout_ns;
};

// Pair kernel tile numbering: row blocks fastest (neighbouring clusters share the weight
// panel), then column blocks, then the batch.
__device__ __forceinline__ void pair_tile(int tile, int mt2, int nt2, int& mb, int& nb, int& b) {
  mb = tile % mt2;
  const int rest = tile / mt2;
  nb = rest % nt2;
  b = rest / nt2;
}

__device__ __forceinline__ void decode_tile(int tile, const GemmArgs& p, int& b, int& mb, int& nb, int& j) {
  mb = tile % p.mt;
  int rest = tile / p.mt;
  nb = rest % p.nt;
  rest /= p.nt;
  b = rest % p.nbatch;
  j = rest / p.nbatch;  // K range (0 unless split)
}

// K steps [lo, hi) of range j when `ksteps` are cut into `ksplit` nearly equal ranges.
__device__ __forceinline__ void split_range(int ksteps, int ksplit, int j, int& lo, int& hi) {
  lo = static_cast<int>((static_cast<int64_t>(j) * ksteps) / ksplit);
  hi = static_cast<int>((static_cast<int64_t>(j + 1) * ksteps) / ksplit);
}

__device__ __forceinline__ void load_bf16x32(const uint16_t* src, float (&v)[32]) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = s4[q];
    unpack_bf16x2(w.x, v[8 * q + 0], v[8 * q + 1]);
    unpack_bf16x2(w.y, v[8 * q + 2], v[8 * q + 3]);
    unpack_bf16x2(w.z, v[8 * q + 4], v[8 * q + 5]);
    unpack_bf16x2(w.w, v[8 * q + 6], v[8 * q + 7]);
  }
}

__device__ __forceinline__ void store_f16x32(uint16_t* dst, const float (&v)[32]) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_f16x2(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_f16x2(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_f16x2(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_f16x2(v[8 * q + 6], v[8 * q + 7]);
    d4[q] = w;
  }
}

__device__ __forceinline__ uint16_t float_to_f16_bits(float f) {
  __half h = __float2half_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const float (&v)[32]) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    d4[q] = w;
  }
}

// Epilogue for 32 consecutive columns n0..n0+31 of row m of output batch b.
// `full` = all 32 columns are inside N (vector path); else column-by-column.
template <int EPI, int ACT>
__device__ __forceinline__ void epilogue_chunk(const GemmArgs& p, int b, int m, int n0, const uint32_t (&r)[32]) {
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
  const bool full = (n0 + 32 <= p.N);
  const int ncols = full ? 32 : (p.N - n0);

  if constexpr (EPI == EPI_F32) {
    float* dst = static_cast<float*>(p.d) + b * p.d_bs + static_cast<int64_t>(m) * p.ldd + n0;
    if (full) {
      float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 w = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        if (p.accumulate) {
          const float4 o = d4[q];
          w.x += o.x; w.y += o.y; w.z += o.z; w.w += o.w;
        }
        d4[q] = w;
      }
    } else {
      _Pragma("unroll") for (int j = 0; j < 32; ++j) if (j < ncols) dst[j] = v[j] + (p.accumulate ? dst[j] : 0.0f);
    }
    return;
  }

  if constexpr (EPI == EPI_BF16) {
    if (p.bias) {
      if (full) {
        float bb[32];
        load_bf16x32(p.bias + n0, bb);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += bb[j];
      } else {
        _Pragma("unroll") for (int j = 0; j < 32; ++j) if (j < ncols) v[j] += bf16_bits_to_float(p.bias[n0 + j]);
      }
    }
    if (p.res) {
      const uint16_t* rp = p.res + static_cast<int64_t>(m) * p.ld_res + n0;
      if (full) {
        float rr[32];
        load_bf16x32(rp, rr);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += rr[j];
      } else {
        _Pragma("unroll") for (int j = 0; j < 32; ++j) if (j < ncols) v[j] += bf16_bits_to_float(rp[j]);
      }
    }
  } else if constexpr (EPI == EPI_ACT) {
    if (p.bias) {
      const uint16_t* bp = p.bias + b * p.bias_bs + n0;
      if (full) {
        float bb[32];
        load_bf16x32(bp, bb);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += bb[j];
      } else {
        _Pragma("unroll") for (int j = 0; j < 32; ++j) if (j < ncols) v[j] += bf16_bits_to_float(bp[j]);
      }
    }
    if (p.d) {  // save Z for the backward pass
      uint16_t* zp = static_cast<uint16_t*>(p.d) + b * p.d_bs + static_cast<int64_t>(m) * p.ldd + n0;
      if (full) {
        if (p.out_f16) store_f16x32(zp, v);
        else store_bf16x32(zp, v);
      } else {
        _Pragma("unroll") for (int j = 0; j < 32; ++j) if (j < ncols) zp[j] =
            p.out_f16 ? float_to_f16_bits(v[j]) : float_to_bf16_bits(v[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = act_apply_t<ACT>(v[j]);
    uint16_t* ap = static_cast<uint16_t*>(p.d2) + b * p.d_bs + static_cast<int64_t>(m) * p.ldd + n0;
    if (full) {
      if (p.out_f16) store_f16x32(ap, v);
      else store_bf16x32(ap, v);
    } else {
      _Pragma("unroll") for (int j = 0; j < 32; ++j) if (j < ncols) ap[j] =
          p.out_f16 ? float_to_f16_bits(v[j]) : float_to_bf16_bits(v[j]);
    }
    return;
  } else {  // EPI_DACT
    const uint16_t* zp = p.aux + b * p.aux_bs + static_cast<int64_t>(m) * p.ld_aux + n0;
    if (full) {
      float z[32];
      load_bf16x32(zp, z);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= act_grad_t<ACT>(z[j]);
    } else {
      _Pragma("unroll") for (int j = 0; j < 32; ++j) if (j < ncols) v[j] *= act_grad_t<ACT>(bf16_bits_to_float(zp[j]));
    }
  }
  uint16_t* dst = static_cast<uint16_t*>(p.d) + b * p.d_bs + static_cast<int64_t>(m) * p.ldd + n0;
  if (full) store_bf16x32(dst, v);
  else _Pragma("unroll") for (int j = 0; j < 32; ++j) if (j < ncols) dst[j] = float_to_bf16_bits(v[j]);
}

// Epilogue math for 32 columns n0..n0+31 of row m, without storing: v receives
// D's values, v2 the activation output (EPI_ACT only).  Loads past M or N are
// skipped (their outputs are clipped by the TMA store).
template <int EPI, int ACT>
__device__ __forceinline__ void epilogue_values(const GemmArgs& p, int b, int m, int n0, const uint32_t (&r)[32],
                                                float (&v)[32], float (&v2)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
  if constexpr (EPI == EPI_F32) return;
  const bool row_ok = m < p.M;
  const bool full = (n0 + 32 <= p.N);
  const int ncols = full ? 32 : (p.N - n0);
  if constexpr (EPI == EPI_BF16 || EPI == EPI_ACT) {
    if (p.bias) {
      const uint16_t* bp = p.bias + (EPI == EPI_ACT ? b * p.bias_bs : 0) + n0;
      if (full) {
        float bb[32];
        load_bf16x32(bp, bb);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += bb[j];
      } else {
        _Pragma("unroll") for (int j = 0; j < 32; ++j) if (j < ncols) v[j] += bf16_bits_to_float(bp[j]);
      }
    }
    if (EPI == EPI_BF16 && p.res && row_ok) {
      const uint16_t* rp = p.res + static_cast<int64_t>(m) * p.ld_res + n0;
      if (full) {
        float rr[32];
        load_bf16x32(rp, rr);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += rr[j];
      } else {
        _Pragma("unroll") for (int j = 0; j < 32; ++j) if (j < ncols) v[j] += bf16_bits_to_float(rp[j]);
      }
    }
    if constexpr (EPI == EPI_ACT) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v2[j] = act_apply_t<ACT>(v[j]);
    }
    return;
  }
  // EPI_DACT
  if (!row_ok) return;
  const uint16_t* zp = p.aux + b * p.aux_bs + static_cast<int64_t>(m) * p.ld_aux + n0;
  if (full) {
    float z[32];
    load_bf16x32(zp, z);
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= act_grad_t<ACT>(z[j]);
  } else {
    _Pragma("unroll") for (int j = 0; j < 32; ++j) if (j < ncols) v[j] *= act_grad_t<ACT>(bf16_bits_to_float(zp[j]));
  }
}

// SwiGLU: columns [256 k, 256 k + 128) of Z hold the gate pre-activations of hidden
// columns [128 k, 128 k + 128), the next 128 the up ones.
constexpr int GLU_GROUP = 128;
__device__ __forceinline__ int glu_gate_col(int c) { return (c / GLU_GROUP) * (2 * GLU_GROUP) + c % GLU_GROUP; }

// EPI_GLU, per-thread stores: gate chunk rg (Z columns zg..zg+31 of row m) and the up chunk
// 128 columns further -> Z (if kept) and A = silu(g) u at hidden columns glu_col(zg).
__device__ __forceinline__ void glu_chunk(const GemmArgs& p, int b, int m, int zg, const uint32_t (&rg)[32],
                                          const uint32_t (&ru)[32]) {
  float g[32], u[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    g[j] = __uint_as_float(rg[j]);
    u[j] = __uint_as_float(ru[j]);
  }
  if (p.d) {
    uint16_t* zp = static_cast<uint16_t*>(p.d) + b * p.d_bs + static_cast<int64_t>(m) * p.ldd + zg;
    store_bf16x32(zp, g);
    store_bf16x32(zp + GLU_GROUP, u);
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) g[j] = silu(g[j]) * u[j];
  const int ac = (zg / (2 * GLU_GROUP)) * GLU_GROUP + zg % (2 * GLU_GROUP);
  store_bf16x32(static_cast<uint16_t*>(p.d2) + b * p.d2_bs + static_cast<int64_t>(m) * p.ldd2 + ac, g);
}

// EPI_DGLU for 32 hidden columns n0..n0+31 of row m (N is a multiple of 128, so a chunk is
// whole): v = dA; reads gate / up from Z (aux), returns d gate in v and d up in v2.
__device__ __forceinline__ void dglu_values(const GemmArgs& p, int b, int m, int n0, float (&v)[32],
                                            float (&v2)[32]) {
  const uint16_t* zp = p.aux + b * p.aux_bs + static_cast<int64_t>(m) * p.ld_aux + glu_gate_col(n0);
  float g[32], u[32];
  load_bf16x32(zp, g);
  load_bf16x32(zp + GLU_GROUP, u);
#pragma unroll
  for (int j = 0; j < 32; ++j) swiglu_grad(g[j], u[j], v[j], v[j], v2[j]);
}

__device__ __forceinline__ void dglu_chunk(const GemmArgs& p, int b, int m, int n0, const uint32_t (&r)[32]) {
  float v[32], v2[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
  dglu_values(p, b, m, n0, v, v2);
  uint16_t* dst = static_cast<uint16_t*>(p.d) + b * p.d_bs + static_cast<int64_t>(m) * p.ldd + glu_gate_col(n0);
  store_bf16x32(dst, v);
  store_bf16x32(dst + GLU_GROUP, v2);
}

// One thread's 32 values into 64 bytes (half of a 128-byte staging row), 2-byte format.
__device__ __forceinline__ void stage_half_row16(uint8_t* buf, int row, int half, const float (&v)[32], bool f16) {
  uint8_t* rowp = buf + row * 128;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint4 w;
    if (f16) {
      w = make_uint4(pack_f16x2(v[8 * k + 0], v[8 * k + 1]), pack_f16x2(v[8 * k + 2], v[8 * k + 3]),
                     pack_f16x2(v[8 * k + 4], v[8 * k + 5]), pack_f16x2(v[8 * k + 6], v[8 * k + 7]));
    } else {
      w = make_uint4(pack_bf16x2(v[8 * k + 0], v[8 * k + 1]), pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                     pack_bf16x2(v[8 * k + 4], v[8 * k + 5]), pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
    }
    const int c = half * 4 + k;
    *reinterpret_cast<uint4*>(rowp + ((c ^ (row & 7)) << 4)) = w;
  }
}

// One thread's 32 fp32 values: a full 128-byte staging row.
__device__ __forceinline__ void stage_row32(uint8_t* buf, int row, const float (&v)[32]) {
  uint8_t* rowp = buf + row * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<float4*>(rowp + ((c ^ (row & 7)) << 4)) =
        make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

// Column sums of a warp's 32 rows (one row per lane, 32 columns each): a fixed butterfly of
// 31 shuffles after which lane j holds the sum of column j (v is consumed).
__device__ __forceinline__ float warp_column_sum32(float (&v)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float keep = upper ? v[i + off] : v[i];
      const float send = upper ? v[i] : v[i + off];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

// The fused bias-gradient pass of EPI_DACT: the warp's rows m0..m0+31 (lanes past M count
// as zero) and columns n0..n0+31 -> cs[b][m0 / 32][n0 + lane].  Callers pass only m0 < M,
// so m0 / 32 < cs_chunks.
__device__ __forceinline__ void dact_colsum_chunk(const GemmArgs& p, int b, int m0, int n0, int lane,
                                                  float (&v)[32]) {
  if (m0 + lane >= p.M) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = 0.0f;
  }
  const float s = warp_column_sum32(v, lane);
  if (n0 + lane < p.N)
    p.cs[(static_cast<int64_t>(b) * p.cs_chunks + m0 / 32) * p.N + n0 + lane] = s;
}

// One k-step of the single-CTA kernels: the TMA copies of A's and B's tiles for k-step ks
// of output tile (b, mb, nb) into stage buffers a_dst / b_dst, completing on `bar`.
template <bool A_MN, bool B_MN, int NB = BN>
__device__ __forceinline__ void load_stage(const GemmArgs& p, const CUtensorMap* tmA, const CUtensorMap* tmB,
                                           uint8_t* a_dst, uint8_t* b_dst, uint64_t* bar, int ks, int b, int mb,
                                           int nb) {
  const int s = ks / p.kt;
  const int kb = ks - s * p.kt;
  ptx::mbar_arrive_expect_tx(bar, A_TILE_BYTES + NB * BK * 2);
  const int ash = p.a_sharded ? (p.nsum > 1 ? s : b) : 0;
  const int bsh = p.b_sharded ? (p.nsum > 1 ? s : b) : 0;
  if (!A_MN) {
    ptx::tma_load_3d(a_dst, tmA, bar, kb * BK, mb * BM, ash);
  } else if (p.a_4d) {
    ptx::tma_load_4d(a_dst, tmA, bar, 0, kb * BK, mb * (BM / 64), ash);
  } else {
#pragma unroll
    for (int j = 0; j < BM / 64; ++j)
      ptx::tma_load_3d(a_dst + j * MN_CHUNK_BYTES, tmA, bar, mb * BM + j * 64, kb * BK, ash);
  }
  if (!B_MN) {
    ptx::tma_load_3d(b_dst, tmB, bar, kb * BK, nb * NB, bsh);
  } else if (p.b_4d) {
    ptx::tma_load_4d(b_dst, tmB, bar, 0, kb * BK, nb * (NB / 64), bsh);
  } else {
#pragma unroll
    for (int j = 0; j < NB / 64; ++j)
      ptx::tma_load_3d(b_dst + j * MN_CHUNK_BYTES, tmB, bar, nb * NB + j * 64, kb * BK, bsh);
  }
}

// Instruction descriptor of the 128 x NB MMA for this launch's operand format.
template <bool A_MN, bool B_MN, int NB = BN>
__device__ __forceinline__ uint32_t single_idesc(const GemmArgs& p) {
  return p.f16ab ? ptx::idesc_f16_f32(BM, NB, A_MN, B_MN) : ptx::idesc_bf16_f32(BM, NB, A_MN, B_MN);
}

// The MMAs of one stage (BK deep) into the accumulator at d_tmem; `first` starts it afresh.
template <bool A_MN, bool B_MN>
__device__ __forceinline__ void mma_stage(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr, bool first,
                                          uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < BK / 16; ++kk) {
    // K-major: 16 K-elements = 32 bytes inside the 128-byte swizzle row; 8-row groups 1024 B apart.
    // MN-major: 16 K-rows = two 1024-byte groups; 64-wide MN chunks MN_CHUNK_BYTES apart.
    const uint64_t ad = A_MN ? ptx::sdesc_at(ptx::sdesc_sw128(a_addr, MN_CHUNK_BYTES, 1024), kk * 2048)
                             : ptx::sdesc_at(ptx::sdesc_sw128(a_addr, 16, 1024), kk * 32);
    const uint64_t bd = B_MN ? ptx::sdesc_at(ptx::sdesc_sw128(b_addr, MN_CHUNK_BYTES, 1024), kk * 2048)
                             : ptx::sdesc_at(ptx::sdesc_sw128(b_addr, 16, 1024), kk * 32);
    ptx::mma_bf16(d_tmem, ad, bd, idesc, (!first || kk > 0) ? 1u : 0u);
  }
}

template <bool A_MN, bool B_MN, int EPI, int ACT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmArgs p) {
  extern __shared__ uint8_t dsmem[];
  const uint32_t pad = (1024u - (ptx::smem_addr(dsmem) & 1023u)) & 1023u;
  uint8_t* base = dsmem + pad;
  uint8_t* sA = base;
  uint8_t* sB = base + STAGES * A_TILE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 128);
    }
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncwarp();  // lane-0 roles rejoin their warp: bar.sync needs converged warps
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total = p.nbatch * p.mt * p.nt;
  const int ksteps = p.nsum * p.kt;
  // Programmatic dependent launch: the next kernel on the stream may be scheduled
  // now (its CTAs take SMs as ours leave).  Everything this kernel reads from or
  // writes to global memory comes after the producer's griddepcontrol.wait (the
  // MMAs and the epilogue follow its loads through the barriers), so the previous
  // kernel has completed and its writes are visible by then.
  ptx::griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      ptx::griddep_wait();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int b, mb, nb, j;
        decode_tile(tile, p, b, mb, nb, j);
        for (int ks = 0; ks < ksteps; ++ks) {
          if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err, ERR_WAIT_PRODUCER, p.timeout_ns)) {
            ok = false;
            break;
          }
          load_stage<A_MN, B_MN>(p, &tmA, &tmB, sA + stage * A_TILE_BYTES, sB + stage * B_TILE_BYTES,
                                 &full[stage], ks, b, mb, nb);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every copy issued must land before the CTA may exit, also after an abort.
      volatile int never = 0;
      for (int s = 0; s < STAGES && s < issued; ++s) {
        const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
        ptx::mbar_wait(&full[s], par, &never, p.err, ERR_WAIT_DRAIN, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        if (!ptx::mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.err, ERR_WAIT_MMA, p.timeout_ns)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int ks = 0; ks < ksteps; ++ks) {
          if (!ptx::mbar_wait(&full[stage], phase, abort_flag, p.err, ERR_WAIT_MMA, p.timeout_ns)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          mma_stage<A_MN, B_MN>(d_tmem, ptx::smem_addr(sA + stage * A_TILE_BYTES),
                                ptx::smem_addr(sB + stage * B_TILE_BYTES), ks == 0, single_idesc<A_MN, B_MN>(p));
          ptx::mma_commit(&empty[stage]);  // frees this smem stage once its MMAs are done
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(&tfull[acc]);  // accumulator ready for the epilogue
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // No MMA may still be running when TMEM is released.
      ptx::mma_commit(mma_done);
      volatile int never = 0;
      ptx::mbar_wait(mma_done, 0, &never, p.err, ERR_WAIT_DRAIN, p.timeout_ns);
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int b, mb, nb, j;
      decode_tile(tile, p, b, mb, nb, j);
      if (!ptx::mbar_wait(&tfull[acc], acc_phase, abort_flag, p.err, ERR_WAIT_EPI, p.timeout_ns)) break;
      ptx::tc_fence_after();
      const int m = mb * BM + row;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if constexpr (EPI == EPI_GLU) {
        // N is a multiple of 256: the tile is one whole gate / up group
#pragma unroll 1
        for (int c = 0; c < GLU_GROUP / 32; ++c) {
          uint32_t rg[32], ru[32];
          ptx::tmem_ld32(t_row + c * 32, rg);
          ptx::tmem_ld32(t_row + GLU_GROUP + c * 32, ru);
          ptx::tmem_ld_wait();
          if (m < p.M) glu_chunk(p, b, m, nb * BN + c * 32, rg, ru);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int n0 = nb * BN + c * 32;
          if (n0 >= p.N) break;  // warp-uniform
          uint32_t r[32];
          ptx::tmem_ld32(t_row + c * 32, r);
          ptx::tmem_ld_wait();
          if (m < p.M) {
            if constexpr (EPI == EPI_DGLU) dglu_chunk(p, b, m, n0, r);
            else epilogue_chunk<EPI, ACT>(p, b, m, n0, r);
          }
          if constexpr (EPI == EPI_DACT) {
            // Warp-uniform.  A warp whose 32 rows all lie past M owns no 32-row block of the
            // partials (block m0 / 32 would index the next shard's first block, or past the
            // buffer for the last shard), so it writes nothing.  This kernel serves M <= 128,
            // so act'(Z) is simply recomputed.
            const int m0 = mb * BM + quad * 32;
            if (p.cs && m0 < p.M) {
              float v[32], v2[32];
              epilogue_values<EPI, ACT>(p, b, m, n0, r, v, v2);
              dact_colsum_chunk(p, b, m0, n0, lane, v);
            }
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  ptx::tc_fence_before();
  __syncwarp();  // lane-0 roles rejoin their warp: bar.sync needs converged warps
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}


// ------------------------------------------------- split K inside a cluster
// For problems with too few output tiles to occupy the GPU (M <= 128, one 128-row tile of
// tokens): the S = ksplit CTAs of a cluster compute the same 128 x 256 output tile, CTA j
// (its cluster rank) over K range j -- for a row-parallel GEMM the t shards' K ranges laid
// end to end.  The partial sums never leave the chip: once every CTA's MMAs are complete
// (cluster barrier), each epilogue thread reads its accumulator row from TMEM and writes it
// into the shared memory of the CTA that owns that row (R = 128 / S rows per CTA), in the
// slot of its K range; the operand stages, idle by then, hold what arrives.  After a second
// cluster barrier each CTA sums its R rows over the S ranges in range order -- the result
// does not depend on timing -- and applies the epilogue with coalesced stores.
template <int SBN>
constexpr int splitc_rowf() { return SBN + 4; }  // floats per received row (16 bytes of padding spread the banks)
// Per epilogue warp, a 32 x 32 block of its partial on its way out: written row per lane,
// read back as 128-byte row segments so that every remote store moves whole segments.
constexpr int SPLITC_XF = 32 + 4;  // floats per staged row
constexpr int SPLITC_RECV_BYTES = BM * splitc_rowf<BN>() * 4;  // room for the widest tile
constexpr int SPLITC_XBYTES = 32 * SPLITC_XF * 4;
static_assert(SPLITC_RECV_BYTES + 4 * SPLITC_XBYTES <= STAGES * STAGE_BYTES,
              "received partials and the staging blocks must fit the operand stages");

// Epilogue of two adjacent columns n, n + 1 (n even, N even) of row m after the split sum;
// (b0, b1) is the bias of the two columns (zeros without one).
template <int EPI, int ACT>
__device__ __forceinline__ void splitc_store2(const GemmArgs& p, int b, int m, int n, float v0, float v1, float b0,
                                              float b1) {
  const int64_t off = b * p.d_bs + static_cast<int64_t>(m) * p.ldd + n;
  if constexpr (EPI == EPI_F32) {
    float2* d = reinterpret_cast<float2*>(static_cast<float*>(p.d) + off);
    if (p.accumulate) {
      const float2 o = *d;
      v0 += o.x;
      v1 += o.y;
    }
    *d = make_float2(v0, v1);
    return;
  }
  v0 += b0;
  v1 += b1;
  if constexpr (EPI == EPI_BF16) {
    if (p.res) {
      float r0, r1;
      unpack_bf16x2(*reinterpret_cast<const uint32_t*>(p.res + static_cast<int64_t>(m) * p.ld_res + n), r0, r1);
      v0 += r0;
      v1 += r1;
    }
    *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.d) + off) = pack_bf16x2(v0, v1);
  } else {  // EPI_ACT
    if (p.d)
      *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.d) + off) =
          p.out_f16 ? pack_f16x2(v0, v1) : pack_bf16x2(v0, v1);
    v0 = act_apply_t<ACT>(v0);
    v1 = act_apply_t<ACT>(v1);
    *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.d2) + off) =
        p.out_f16 ? pack_f16x2(v0, v1) : pack_bf16x2(v0, v1);
  }
}

template <bool A_MN, bool B_MN, int EPI, int ACT, int SBN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_splitc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const GemmArgs p) {
  static_assert(SBN == BN || SBN == BN / 2, "tile width of the split kernel");
  constexpr int ROWF = splitc_rowf<SBN>();
  extern __shared__ uint8_t dsmem[];
  const uint32_t pad = (1024u - (ptx::smem_addr(dsmem) & 1023u)) & 1023u;
  uint8_t* base = dsmem + pad;
  uint8_t* sA = base;
  uint8_t* sB = base + STAGES * A_TILE_BYTES;
  float* recv = reinterpret_cast<float*>(base);  // after the main loop: [S][R][SPLITC_ROWF]
  uint64_t* full = reinterpret_cast<uint64_t*>(base + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.ksplit;
  const int R = BM / S;
  const int j = static_cast<int>(ptx::cluster_ctarank());
  int b, mb, nb, unused;
  decode_tile(static_cast<int>(blockIdx.x) / S, p, b, mb, nb, unused);
  int klo, khi;
  split_range(p.nsum * p.kt, S, j, klo, khi);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(tfull, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, SBN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncwarp();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Programmatic dependent launch, as in gemm_kernel: every global access follows the
  // producer's griddepcontrol.wait through the barriers.
  ptx::griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      ptx::griddep_wait();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      for (int ks = klo; ks < khi; ++ks) {
        if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err, ERR_WAIT_PRODUCER, p.timeout_ns)) break;
        load_stage<A_MN, B_MN, SBN>(p, &tmA, &tmB, sA + stage * A_TILE_BYTES, sB + stage * B_TILE_BYTES, &full[stage],
                               ks, b, mb, nb);
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      volatile int never = 0;  // every copy issued lands before the stages are reused
      for (int s = 0; s < STAGES && s < issued; ++s) {
        const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
        ptx::mbar_wait(&full[s], par, &never, p.err, ERR_WAIT_DRAIN, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      for (int ks = klo; ks < khi; ++ks) {
        if (!ptx::mbar_wait(&full[stage], phase, abort_flag, p.err, ERR_WAIT_MMA, p.timeout_ns)) break;
        ptx::tc_fence_after();
        mma_stage<A_MN, B_MN>(tmem_base, ptx::smem_addr(sA + stage * A_TILE_BYTES),
                              ptx::smem_addr(sB + stage * B_TILE_BYTES), ks == klo,
                              single_idesc<A_MN, B_MN, SBN>(p));
        ptx::mma_commit(&empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // Always committed, also after an abort: once it completes no MMA is running.
      ptx::mma_commit(tfull);
      volatile int never = 0;
      ptx::mbar_wait(tfull, 0, &never, p.err, ERR_WAIT_DRAIN, p.timeout_ns);
    }
  } else {
    ptx::mbar_wait(tfull, 0, abort_flag, p.err, ERR_WAIT_EPI, p.timeout_ns);
  }

  // Barrier 1: every CTA's MMAs are complete, so every CTA's operand stages are free.
  ptx::tc_fence_before();
  __syncwarp();
  ptx::cluster_sync();
  if (warp >= 2) {
    ptx::tc_fence_after();
    const int quad = warp & 3;  // TMEM lanes 32 * (warp % 4) .. + 31
    const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    float* xs = reinterpret_cast<float*>(base + SPLITC_RECV_BYTES + quad * SPLITC_XBYTES);
    // After the transpose through xs, lane l carries columns 4 (l % 8) .. + 3 of rows
    // 4 i + l / 8 (i = 0..7) of the warp's 32: eight lanes cover a row's 128 bytes.
    const int seg = lane & 7;
#pragma unroll 1
    for (int c = 0; c < SBN / 32; ++c) {
      if (nb * SBN + c * 32 >= p.N) break;  // warp-uniform: columns past N are never summed
      uint32_t r[32];
      ptx::tmem_ld32(t_row + c * 32, r);
      ptx::tmem_ld_wait();
      float* mine = xs + lane * SPLITC_XF;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<uint4*>(mine + 4 * q) = make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rl = 4 * i + (lane >> 3);  // row within the warp's 32
        const int row = quad * 32 + rl;
        const uint4 v = *reinterpret_cast<const uint4*>(xs + rl * SPLITC_XF + 4 * seg);
        const uint32_t dst = ptx::mapa_shared(
            ptx::smem_addr(recv + (static_cast<int64_t>(j) * R + row % R) * ROWF + c * 32 + 4 * seg),
            static_cast<uint32_t>(row / R));
        ptx::st_cluster_v4(dst, v.x, v.y, v.z, v.w);
      }
      __syncwarp();  // xs is rewritten by the next chunk
    }
  }
  // Barrier 2: every partial row has arrived where it is summed.
  ptx::tc_fence_before();
  __syncwarp();
  ptx::cluster_sync();
  // The sums: 256-column tiles on the four epilogue warps, thread e taking columns 2 e,
  // 2 e + 1 of every owned row; 128-column tiles on all six warps, thread e taking columns
  // 2 cp, 2 cp + 1 of the owned rows rg, rg + 3, ...
  constexpr int SUM_T = SBN == BN ? 128 : NUM_THREADS;
  if (SUM_T == NUM_THREADS || warp >= 2) {
    constexpr int CP = SBN / 2, RG = SUM_T / CP;
    const int e = static_cast<int>(threadIdx.x) - (NUM_THREADS - SUM_T);
    const int cp = e % CP, rg = e / CP;
    const int n = nb * SBN + 2 * cp;
    if (n < p.N) {
      float b0 = 0.0f, b1 = 0.0f;
      if (EPI != EPI_F32 && p.bias)
        unpack_bf16x2(*reinterpret_cast<const uint32_t*>(p.bias + (EPI == EPI_ACT ? b * p.bias_bs : 0) + n), b0, b1);
      const int rows = min(R, p.M - (mb * BM + j * R));
      // Eight rows at a time: every load of the batch is issued before the first store, so
      // the shared-memory latency is paid once per batch rather than once per row.
      const float* __restrict__ rbase = recv + 2 * cp;
#pragma unroll 1
      for (int r0 = rg; r0 < rows; r0 += 8 * RG) {
        float2 acc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          acc[u] = *reinterpret_cast<const float2*>(rbase + min(r0 + u * RG, R - 1) * ROWF);
        for (int k = 1; k < S; ++k) {  // K ranges in order
          const float* __restrict__ src = rbase + static_cast<int64_t>(k) * R * ROWF;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float2 x = *reinterpret_cast<const float2*>(src + min(r0 + u * RG, R - 1) * ROWF);
            acc[u].x += x.x;
            acc[u].y += x.y;
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (r0 + u * RG < rows)
            splitc_store2<EPI, ACT>(p, b, mb * BM + j * R + r0 + u * RG, n, acc[u].x, acc[u].y, b0, b1);
      }
    }
  }

  ptx::tc_fence_before();
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, SBN);
  }
}

// ---------------------------------------------------- split-K items (pair kernel)
enum : int { ITEM_WHOLE = 0, ITEM_RANGE = 1 };
struct PairItem {
  int tile, klo, khi, kind;
  int range;  // ITEM_RANGE: which of the tile's sp_split K ranges
  int st;     // ITEM_RANGE: index of the tile among those that are split (counters, partial slots)
};

__device__ __forceinline__ void sp_cut(const GemmArgs& p, int j, PairItem& it) {
  it.kind = ITEM_RANGE;
  it.range = j;
  it.klo = static_cast<int>(static_cast<int64_t>(j) * p.sp_units / p.sp_split);
  it.khi = static_cast<int>(static_cast<int64_t>(j + 1) * p.sp_units / p.sp_split);
}

// Work item idx of cluster c (nclusters launched); false past the cluster's last item.
// Without split K: the whole tiles c, c + nclusters, ...  Overlapped shard reduction
// (sp_seq): every tile's shard ranges as items, shard-major (all tiles' shard 0, then shard
// 1, ...), dealt round-robin, so a tile's shard j comes `total` items after its shard j - 1.  Split K:
// first the sp_rounds whole rounds, then items u = c, c + nclusters, ... of the sp_tiles
// remaining tiles: counted ranges u = S i + j (range j of remaining tile i; a tile's ranges
// run side by side on neighbouring clusters), chained ranges u = sp_tiles j + i (range-major:
// a tile's range j comes sp_tiles items after its range j - 1, the item it waits for).  Every
// role of the kernel enumerates the same items.
__device__ __forceinline__ bool pair_item(const GemmArgs& p, int c, int nclusters, int total, int ksteps, int idx,
                                          PairItem& it) {
  it.range = 0;
  it.st = 0;
  if (p.sp_seq) {  // shard-major: item u = c + idx nclusters is shard u / total of tile u % total
    const int64_t u = c + static_cast<int64_t>(idx) * nclusters;
    if (u >= static_cast<int64_t>(total) * p.sp_split) return false;
    const int j = static_cast<int>(u / total);
    it.tile = static_cast<int>(u - static_cast<int64_t>(j) * total);
    it.st = it.tile;
    sp_cut(p, j, it);
    return true;
  }
  if (p.sp_split > 0) {
    const int S = p.sp_split;
    if (idx < p.sp_rounds) {
      it.tile = c + idx * nclusters;
      it.klo = 0;
      it.khi = ksteps;
      it.kind = ITEM_WHOLE;
      return true;
    }
    const int64_t u = c + static_cast<int64_t>(idx - p.sp_rounds) * nclusters;
    if (u >= static_cast<int64_t>(p.sp_tiles) * S) return false;
    // chained: range-major (range u / tiles of tile u % tiles); counted: a tile's ranges side by side
    const int i = static_cast<int>(p.sp_chain ? u % p.sp_tiles : u / S);
    const int j = static_cast<int>(p.sp_chain ? u / p.sp_tiles : u - static_cast<int64_t>(i) * S);
    it.tile = p.sp_rounds * nclusters + i;
    it.st = i;
    sp_cut(p, j, it);
    return true;
  }
  const int tile = c + idx * nclusters;
  if (tile >= total) return false;
  it.tile = tile;
  it.klo = 0;
  it.khi = ksteps;
  it.kind = ITEM_WHOLE;
  return true;
}

// Counts one finished range of a split tile in its (tile, CTA, warp) counter: a 64-bit word
// (launch epoch << 32 | ranges counted); a word left by another launch counts as zero.
// Returns true for the range that completes the count, which then owns the sum and resets
// the word (so a graph replay, which repeats the epoch, starts from zero).  The partial
// must be globally visible before the call.
__device__ __forceinline__ bool sp_arrive(const GemmArgs& p, unsigned long long* w, volatile int* abort_flag) {
  const unsigned long long ep = static_cast<unsigned long long>(p.sp_epoch) << 32;
  unsigned long long old = atomicAdd(w, 0ull);
  for (int tries = 0; tries < (1 << 20); ++tries) {
    const unsigned long long n = ((old & 0xffffffff00000000ull) == ep) ? (old & 0xffffffffull) : 0ull;
    const unsigned long long prev = atomicCAS(w, old, ep | (n + 1));
    if (prev == old) {
      if (n + 1 < static_cast<unsigned long long>(p.sp_split)) return false;
      atomicExch(w, 0ull);
      __threadfence();  // the other ranges' partials are read after their counts
      return true;
    }
    old = prev;
  }
  *abort_flag = 1;
  if (p.err) atomicCAS(p.err, 0, ERR_WAIT_SK);
  return false;
}

// Epilogues whose pair-kernel launches may split K (TMA-store outputs).
constexpr bool sk_epi(int epi) { return epi == EPI_BF16 || epi == EPI_ACT || epi == EPI_F32 || epi == EPI_DACT; }

// ------------------------------------------------------------ CTA-pair GEMM
// Same contract as gemm_kernel, computed by clusters of two CTAs on two SMs
// sharing one 256 x 256 output tile through tcgen05.mma.cta_group::2 (M = 256):
// CTA rank r of the pair loads rows [128 r, 128 r + 128) of the tile's A and
// rows [128 r, 128 r + 128) of its B (N) into its own shared memory, so each
// SM streams 32 KB per 64-deep k-block instead of 48 KB for the same work, and
// six stages fit.  The leader (rank 0) issues every MMA; its "full" barrier
// counts both CTAs' TMA bytes; MMA completion is multicast to both CTAs'
// "empty" and "accumulator full" barriers; both epilogues arrive on the
// leader's "accumulator empty" barrier.  Each CTA's TMEM holds its own 128
// rows of the 256-column accumulator (two buffers, 512 columns).
constexpr int P_BN = 256;                       // tile N (pair)
constexpr int P_HALF = 128;                     // rows of A and of B per CTA
constexpr int P_A_BYTES = P_HALF * BK * 2;      // 16 KB
constexpr int P_B_BYTES = P_HALF * BK * 2;      // 16 KB
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
constexpr int STG_BOX_BYTES = 32 * 128;         // one 32-row x 128-byte output box
// 64-wide k-blocks per pipeline stage of the pair kernel.  One-output epilogues take two:
// each operand then arrives in one 32 KB copy per stage (three stages of 64 KB), which halves
// the copies and barrier round trips per MMA and ran 1.5-3 % faster at K = 2048 (no gain
// for the GeLU epilogue, which keeps six single-block stages).
constexpr int pair_kb(int epi) { return (epi == EPI_F32 || epi == EPI_BF16 || epi == EPI_DACT) ? 2 : 1; }

template <int EPI>
struct PairCfg {
  static constexpr int outputs = (EPI == EPI_GLU) ? 3 : (EPI == EPI_ACT || EPI == EPI_DGLU) ? 2 : 1;
  static constexpr int kb = pair_kb(EPI);
  static constexpr int stages = (kb == 2) ? 3 : (EPI == EPI_GLU || EPI == EPI_DGLU) ? 5 : 6;
  // Staging once instead of twice leaves room for one more operand stage: the epilogue then
  // waits for the previous box's stores to finish reading shared memory, which costs less
  // than the stage (SwiGLU forward: 5 stages instead of 4, ~7 % faster at K = 8192; GeLU:
  // 6 instead of 5, 2-4 % faster).
  static constexpr int buffers = (EPI == EPI_GLU || EPI == EPI_ACT) ? 1 : 2;
  static constexpr int stg_warp_bytes = buffers * outputs * STG_BOX_BYTES;
  static constexpr int stg_bytes = 4 * stg_warp_bytes;                 // 4 epilogue warps
  static constexpr int smem_bytes = 1024 + stages * kb * P_STAGE_BYTES + stg_bytes + BAR_BYTES;
};

// Bounded wait until *f == want (acquire).  False (abort flag raised, error recorded) when
// the limit passes or the CTA is aborting.
__device__ __forceinline__ bool sp_wait_flag(const unsigned long long* f, unsigned long long want,
                                             volatile int* abort_flag, const GemmArgs& p) {
  const uint64_t* q = reinterpret_cast<const uint64_t*>(f);
  if (ptx::ld_acquire_u64(q) == want) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (ptx::ld_acquire_u64(q) != want) {
    if (*abort_flag || ptx::globaltimer_ns() - t0 > p.timeout_ns) {
      *abort_flag = 1;
      if (p.err) atomicCAS(p.err, 0, ERR_WAIT_OVL);
      return false;
    }
    __nanosleep(128);
  }
  return true;
}

// Start of row r of range j's partial, at this lane's 8 columns: row trow of slot (st S + j)
// (tile column tc), or row m of range j in the caller's [S][M][N] buffer (column n).
__device__ __forceinline__ const float4* sp_row(const GemmArgs& p, int st, int j, int trow, int m, int n, int tc) {
  if (p.sp_user) return reinterpret_cast<const float4*>(p.sp_part + j * p.sp_bs + static_cast<int64_t>(m) * p.sp_ld + n);
  return reinterpret_cast<const float4*>(p.sp_part + (static_cast<int64_t>(st * p.sp_split + j) * 256 + trow) * 256 + tc);
}

__device__ __forceinline__ void unpack8_bf16(const uint4& w, float (&v)[8]) {
  unpack_bf16x2(w.x, v[0], v[1]);
  unpack_bf16x2(w.y, v[2], v[3]);
  unpack_bf16x2(w.z, v[4], v[5]);
  unpack_bf16x2(w.w, v[6], v[7]);
}

// (row, range) partial loads in flight per lane while a completed tile is summed.
constexpr int SP_PAIRS = 8;

// A split tile whose ranges are all counted: this warp's 32 rows (from mrow0; tile rows from
// trow0) are summed over the S partials in range order and run through the epilogue.  The
// accumulator is already handed back, so the tensor cores go on with the next item meanwhile.
// Lane l holds tile columns 8 l .. 8 l + 7 of one row at a time (a warp reads a 1 KB row
// segment per partial: coalesced), SP_PAIRS (row, range) loads are in flight, and outputs go
// out as direct 16-byte stores.  The epilogue arithmetic is epilogue_values' (bias, then the
// residual; act / act'); the DACT column sums add the warp's rows in row order.
template <int EPI, int ACT>
__device__ __forceinline__ void sp_reduce_rows(const GemmArgs& p, const PairItem& it, int b, int mrow0, int trow0,
                                               int nb, int lane) {
  const int S = p.sp_split;
  const int tc = lane * 8;
  const int n = nb * P_BN + tc;
  if (n >= p.N) return;  // N % 8 == 0: a lane's 8 columns are all inside or all outside
  const int nrows = min(32, p.M - mrow0);
  float bv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if constexpr (EPI == EPI_BF16 || EPI == EPI_ACT) {
    if (p.bias)
      unpack8_bf16(*reinterpret_cast<const uint4*>(p.bias + (EPI == EPI_ACT ? b * p.bias_bs : 0) + n), bv);
  }
  float cs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float acc[8];
  const int pairs = nrows * S;
#pragma unroll 1
  for (int base = 0; base < pairs; base += SP_PAIRS) {
    float4 x[SP_PAIRS][2];
    uint4 y[SP_PAIRS];  // the row's residual (BF16) or Z (DACT), loaded with its last range
#pragma unroll
    for (int q = 0; q < SP_PAIRS; ++q) {
      const int pq = min(base + q, pairs - 1);  // past the end: reload the last pair (unused)
      const int r = pq / S, j = pq - r * S;
      const int m = mrow0 + r;
      const float4* src = sp_row(p, it.st, j, trow0 + r, m, n, tc);
      x[q][0] = __ldcg(src);
      x[q][1] = __ldcg(src + 1);
      y[q] = make_uint4(0u, 0u, 0u, 0u);
      if (EPI == EPI_BF16 && p.res && j == S - 1)
        y[q] = *reinterpret_cast<const uint4*>(p.res + static_cast<int64_t>(m) * p.ld_res + n);
      if (EPI == EPI_DACT && j == S - 1)
        y[q] = *reinterpret_cast<const uint4*>(p.aux + b * p.aux_bs + static_cast<int64_t>(m) * p.ld_aux + n);
    }
#pragma unroll
    for (int q = 0; q < SP_PAIRS; ++q) {
      const int pq = base + q;
      if (pq < pairs) {
        const int r = pq / S, j = pq - r * S;
        const float xv[8] = {x[q][0].x, x[q][0].y, x[q][0].z, x[q][0].w, x[q][1].x, x[q][1].y, x[q][1].z, x[q][1].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = (j == 0) ? xv[e] : acc[e] + xv[e];
        if (j == S - 1) {
          const int m = mrow0 + r;
          const int64_t off = b * p.d_bs + static_cast<int64_t>(m) * p.ldd + n;
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = acc[e];
          if constexpr (EPI == EPI_F32) {
            float4* d = reinterpret_cast<float4*>(static_cast<float*>(p.d) + off);
            d[0] = make_float4(v[0], v[1], v[2], v[3]);
            d[1] = make_float4(v[4], v[5], v[6], v[7]);
          } else if constexpr (EPI == EPI_BF16) {
            if (p.bias) {
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] += bv[e];
            }
            if (p.res) {
              float rv[8];
              unpack8_bf16(y[q], rv);
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] += rv[e];
            }
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.d) + off) =
                make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                           pack_bf16x2(v[6], v[7]));
          } else if constexpr (EPI == EPI_ACT) {
            if (p.bias) {
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] += bv[e];
            }
            const bool f16 = p.out_f16 != 0;
            auto pk = [f16](float a0, float a1) { return f16 ? pack_f16x2(a0, a1) : pack_bf16x2(a0, a1); };
            if (p.d)
              *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.d) + off) =
                  make_uint4(pk(v[0], v[1]), pk(v[2], v[3]), pk(v[4], v[5]), pk(v[6], v[7]));
            float a[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) a[e] = act_apply_t<ACT>(v[e]);
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.d2) + off) =
                make_uint4(pk(a[0], a[1]), pk(a[2], a[3]), pk(a[4], a[5]), pk(a[6], a[7]));
          } else if constexpr (EPI == EPI_DACT) {
            float z[8];
            unpack8_bf16(y[q], z);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              v[e] *= act_grad_t<ACT>(z[e]);
              cs[e] += v[e];
            }
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.d) + off) =
                make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                           pack_bf16x2(v[6], v[7]));
          }
        }
      }
    }
  }
  if constexpr (EPI == EPI_DACT) {
    if (p.cs) {
      float4* c = reinterpret_cast<float4*>(p.cs + (static_cast<int64_t>(b) * p.cs_chunks + mrow0 / 32) * p.N + n);
      c[0] = make_float4(cs[0], cs[1], cs[2], cs[3]);
      c[1] = make_float4(cs[4], cs[5], cs[6], cs[7]);
    }
  }
}

template <int EPI>
constexpr int pair_smem_bytes() {
  return PairCfg<EPI>::smem_bytes;
}

template <bool A_MN, bool B_MN, int EPI, int ACT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD2,
                     const __grid_constant__ CUtensorMap tmP, const GemmArgs p) {
  constexpr int P_STAGES = PairCfg<EPI>::stages;
  static_assert((2 * P_STAGES + 14) * 8 <= BAR_BYTES, "barriers, TMEM slot and abort flag fit their region");
  constexpr int STG_BYTES = PairCfg<EPI>::stg_bytes;
  constexpr int STG_WARP_BYTES = PairCfg<EPI>::stg_warp_bytes;
  constexpr int NOUT = PairCfg<EPI>::outputs;
  constexpr int KB = PairCfg<EPI>::kb;
  constexpr int SA_BYTES = KB * P_A_BYTES;  // one stage of A (B: the same)
  extern __shared__ uint8_t dsmem[];
  const uint32_t pad = (1024u - (ptx::smem_addr(dsmem) & 1023u)) & 1023u;
  uint8_t* base = dsmem + pad;
  uint8_t* sA = base;
  uint8_t* sB = base + P_STAGES * SA_BYTES;
  uint8_t* sStage = base + P_STAGES * 2 * SA_BYTES;  // epilogue output staging (1024-byte aligned boxes)
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + STG_BYTES);
  uint64_t* empty = full + P_STAGES;
  uint64_t* tfull = empty + P_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* ebar = mma_done + 2;  // two per epilogue warp: its running-sum loads (overlapped form)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = (rank == 0);
  const int cluster = static_cast<int>(blockIdx.x >> 1);
  const int nclusters = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 256);  // both CTAs' epilogue threads (used in the leader)
    }
    ptx::mbar_init(mma_done, 1);
    for (int q = 0; q < 8; ++q) ptx::mbar_init(&ebar[q], 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_slot, TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncwarp();  // lane-0 roles rejoin their warp before the cluster barrier
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int mt2 = (p.M + 2 * P_HALF - 1) / (2 * P_HALF);
  const int nt2 = (p.N + P_BN - 1) / P_BN;
  const int total = p.nbatch * mt2 * nt2;
  const int kt2 = (p.kt + KB - 1) / KB;  // stages per shard of K
  const int ksteps = p.nsum * kt2;
  // Programmatic dependent launch: as in gemm_kernel, every global access follows the
  // producers' griddepcontrol.wait.
  ptx::griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer (both CTAs)
      ptx::tma_prefetch_desc(&tmA);
      ptx::tma_prefetch_desc(&tmB);
      ptx::griddep_wait();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      PairItem it;
      for (int idx = 0; ok && pair_item(p, cluster, nclusters, total, ksteps, idx, it); ++idx) {
        int mb, nb, b;
        pair_tile(it.tile, mt2, nt2, mb, nb, b);
        const int m0 = mb * 2 * P_HALF + static_cast<int>(rank) * P_HALF;
        const int n0 = nb * P_BN + static_cast<int>(rank) * P_HALF;
        for (int ks = it.klo; ks < it.khi; ++ks) {
          const int s = ks / kt2;
          const int kb = (ks - s * kt2) * KB;  // first 64-wide k-block of this stage
          if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err, ERR_WAIT_PRODUCER, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t bar = ptx::mapa_shared(ptx::smem_addr(&full[stage]), 0);
          if (leader) ptx::mbar_arrive_expect_tx(&full[stage], 2 * 2 * SA_BYTES);
          const int ash = p.a_sharded ? (p.nsum > 1 ? s : b) : 0;
          const int bsh = p.b_sharded ? (p.nsum > 1 ? s : b) : 0;
          uint8_t* a_dst = sA + stage * SA_BYTES;
          uint8_t* b_dst = sB + stage * SA_BYTES;
          // One copy per operand where the 4-D view applies; else one copy per k-block
          // (K-major, 16 KB panels) or per 64-column chunk (MN-major, 64 * KB K-rows deep).
          // k-blocks past K arrive zero-filled.
          if (!A_MN) {
            if (KB == 2 && p.a_4d) {
              ptx::tma_load_4d_pair(a_dst, &tmA, bar, 0, m0, kb, ash);
            } else {
#pragma unroll
              for (int j = 0; j < KB; ++j) ptx::tma_load_3d_pair(a_dst + j * P_A_BYTES, &tmA, bar, (kb + j) * BK, m0, ash);
            }
          } else if (p.a_4d) {
            ptx::tma_load_4d_pair(a_dst, &tmA, bar, 0, kb * BK, m0 / 64, ash);
          } else {
#pragma unroll
            for (int j = 0; j < P_HALF / 64; ++j)
              ptx::tma_load_3d_pair(a_dst + j * KB * MN_CHUNK_BYTES, &tmA, bar, m0 + j * 64, kb * BK, ash);
          }
          if (!B_MN) {
            if (KB == 2 && p.b_4d) {
              ptx::tma_load_4d_pair(b_dst, &tmB, bar, 0, n0, kb, bsh);
            } else {
#pragma unroll
              for (int j = 0; j < KB; ++j) ptx::tma_load_3d_pair(b_dst + j * P_B_BYTES, &tmB, bar, (kb + j) * BK, n0, bsh);
            }
          } else if (p.b_4d) {
            ptx::tma_load_4d_pair(b_dst, &tmB, bar, 0, kb * BK, n0 / 64, bsh);
          } else {
#pragma unroll
            for (int j = 0; j < P_HALF / 64; ++j)
              ptx::tma_load_3d_pair(b_dst + j * KB * MN_CHUNK_BYTES, &tmB, bar, n0 + j * 64, kb * BK, bsh);
          }
          ++issued;
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (leader) {  // both CTAs' copies land on the leader's barriers
        volatile int never = 0;
        for (int s = 0; s < P_STAGES && s < issued; ++s) {
          const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
          ptx::mbar_wait_cluster(&full[s], par, &never, p.err, ERR_WAIT_DRAIN, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------- MMA issuer (leader only)
      const uint32_t idesc = p.f16ab ? ptx::idesc_f16_f32(2 * P_HALF, P_BN, A_MN, B_MN)
                                     : ptx::idesc_bf16_f32(2 * P_HALF, P_BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      PairItem it;
      for (int idx = 0; ok && pair_item(p, cluster, nclusters, total, ksteps, idx, it); ++idx) {
        if (!ptx::mbar_wait_cluster(&tempty[acc], acc_phase ^ 1u, abort_flag, p.err, ERR_WAIT_MMA, p.timeout_ns))
          break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * P_BN);
        for (int ks = it.klo; ks < it.khi; ++ks) {
          if (!ptx::mbar_wait_cluster(&full[stage], phase, abort_flag, p.err, ERR_WAIT_MMA, p.timeout_ns)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_addr(sA + stage * SA_BYTES);
          const uint32_t b_addr = ptx::smem_addr(sB + stage * SA_BYTES);
#pragma unroll
          for (int kk = 0; kk < KB * BK / 16; ++kk) {
            // K-major: a 16 KB panel per 64-wide k-block, 32 bytes per K = 16 inside it.
            // MN-major: 64 * KB K-rows per 64-column chunk, chunks KB * 8 KB apart.
            const uint64_t ad =
                A_MN ? ptx::sdesc_at(ptx::sdesc_sw128(a_addr, KB * MN_CHUNK_BYTES, 1024), kk * 2048)
                     : ptx::sdesc_at(ptx::sdesc_sw128(a_addr, 16, 1024), (kk >> 2) * P_A_BYTES + (kk & 3) * 32);
            const uint64_t bd =
                B_MN ? ptx::sdesc_at(ptx::sdesc_sw128(b_addr, KB * MN_CHUNK_BYTES, 1024), kk * 2048)
                     : ptx::sdesc_at(ptx::sdesc_sw128(b_addr, 16, 1024), (kk >> 2) * P_B_BYTES + (kk & 3) * 32);
            ptx::mma_bf16_pair(d_tmem, ad, bd, idesc, (ks > it.klo || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit_pair_mc(&empty[stage], 0x3);  // frees this stage in both CTAs
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair_mc(&tfull[acc], 0x3);  // accumulator ready in both CTAs
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      ptx::mma_commit_pair_mc(mma_done, 0x1);
      volatile int never = 0;
      ptx::mbar_wait(mma_done, 0, &never, p.err, ERR_WAIT_DRAIN, p.timeout_ns);
    }
  } else {
    // ----------------------------------------------------------- epilogue (both CTAs)
    const int quad = warp & 3;
    const uint32_t tempty_leader0 = ptx::mapa_shared(ptx::smem_addr(&tempty[0]), 0);
    uint8_t* stg = sStage + quad * STG_WARP_BYTES;  // [buffer][output] boxes of this warp
    const bool two_out = (EPI == EPI_ACT || EPI == EPI_GLU) && p.d != nullptr;
    const bool wide = (EPI == EPI_F32);           // fp32 boxes hold 32 columns, 2-byte boxes 64
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t step = 0;
    constexpr bool SK_OK = sk_epi(EPI);
    static_assert(!SK_OK || STG_WARP_BYTES >= 2 * STG_BOX_BYTES, "split-K partials need two fp32 staging boxes");
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmD);
      ptx::tma_prefetch_desc(&tmD2);
      if (SK_OK && p.sp_split > 0 && !p.sp_chain) ptx::tma_prefetch_desc(&tmP);
    }
    uint32_t ephase = 0;  // phases of this warp's two running-sum load barriers (bits 0, 1)
    PairItem it;
    for (int idx = 0; pair_item(p, cluster, nclusters, total, ksteps, idx, it); ++idx) {
      int mb, nb, b;
      pair_tile(it.tile, mt2, nt2, mb, nb, b);
      if (!ptx::mbar_wait_cluster(&tfull[acc], acc_phase, abort_flag, p.err, ERR_WAIT_EPI, p.timeout_ns)) break;
      ptx::tc_fence_after();
      const int mrow0 = mb * 2 * P_HALF + static_cast<int>(rank) * P_HALF + quad * 32;
      const int m = mrow0 + lane;
      const int trow = static_cast<int>(rank) * P_HALF + quad * 32 + lane;  // row within the tile
      const uint32_t t_row =
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * P_BN);
      // A K range of a split tile: its fp32 partial of this warp's 32 rows goes out through two
      // alternating 32 x 32 staging boxes (to slot st S + j, or to range j of the caller's
      // buffer), then the range counts itself; the range that completes the count goes on to
      // the epilogue below with the sum of all ranges, the others are done with the tile.
      bool sp_last = false;
      bool ovl_item = false;
      unsigned long long* ovl_flag = nullptr;  // set (to ovl_set) once this shard's adds are complete
      unsigned long long ovl_set = 0;
      if constexpr (EPI == EPI_BF16) {
        if (p.sp_chain && it.kind == ITEM_RANGE) {
          // Overlapped shard reduction: shard j = it.range of tile it.tile (the chained split
          // K: range j of split tile it.st, with no partial of its own written).  Its fp32 partial is
          // staged 32 columns at a time in two alternating boxes; from a box it goes to the
          // caller's buffer with coalesced stores (a warp store covers four 128-byte rows; TMA
          // stores of these scattered rows held up the operand loads) and, by TMA, into the
          // tile's running sum (stored for shard 0, added in L2 for the next shards).  Shard j
          // adds only after shard j - 1's flag (epoch << 32 | j) says its adds are complete, so
          // the sum runs in shard order; that shard was dealt a whole pass of the tiles earlier,
          // so the flag is normally set long before.  The last shard loads the running sum one
          // box ahead, adds its accumulator, and writes its own partial and Y (bias once, then
          // the residual) with coalesced stores.
          ovl_item = true;
          if (mrow0 < p.M) {
            const int S = p.sp_split, j = it.range;
            const int rrow = static_cast<int>(rank) * P_HALF + quad * 32;  // rows in the running sum
            float* part = p.sp_user ? p.sp_part + j * p.sp_bs : nullptr;
            const unsigned long long ep = static_cast<unsigned long long>(p.sp_epoch) << 32;
            unsigned long long* flag = p.sp_cnt + (static_cast<int64_t>(it.st) * 2 + rank) * 4 + quad;
            if (lane == 0) ptx::bulk_wait_group<0>();
            int use_sum = 1;  // this shard touches the running sum (0 after a failed wait: result void)
            if (j > 0 && lane == 0) use_sum = sp_wait_flag(flag, ep | static_cast<unsigned long long>(j), abort_flag, p);
            use_sum = __shfl_sync(0xffffffffu, use_sum, 0);
            int nch = 0;  // 32-column chunks inside N
            while (nch < P_BN / 32 && nb * P_BN + nch * 32 < p.N) ++nch;
            const bool load_sum = (j == S - 1) && S > 1 && use_sum;
            if (load_sum) {
              ptx::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                asm volatile("fence.proxy.async.global;" ::: "memory");
                for (int c = 0; c < 2 && c < nch; ++c) {
                  ptx::mbar_arrive_expect_tx(&ebar[quad * 2 + c], STG_BOX_BYTES);
                  ptx::tma_load_3d(stg + c * STG_BOX_BYTES, &tmD2, &ebar[quad * 2 + c], c * 32, rrow, it.st);
                }
              }
            }
#pragma unroll 1
            for (int c = 0; c < nch; ++c) {
              const int n0 = nb * P_BN + c * 32;
              uint8_t* buf = stg + (c & 1) * STG_BOX_BYTES;
              if (j < S - 1 && c >= 2) {
                if (lane == 0) ptx::bulk_wait_group_read<1>();  // the box's running-sum copy read it
              }
              __syncwarp();
              uint32_t r[32];
              ptx::tmem_ld32(t_row + c * 32, r);
              ptx::tmem_ld_wait();
              float v[32], sum[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = sum[e] = __uint_as_float(r[e]);
              if (load_sum) {
                const int eb = quad * 2 + (c & 1);
                if (!ptx::mbar_wait(&ebar[eb], (ephase >> (c & 1)) & 1u, abort_flag, p.err, ERR_WAIT_EPI,
                                    p.timeout_ns)) {
                  volatile int never = 0;  // the copy may still land: wait for it (bounded) first
                  ptx::mbar_wait(&ebar[eb], (ephase >> (c & 1)) & 1u, &never, nullptr, 0, p.timeout_ns);
                }
                ephase ^= 1u << (c & 1);
                const uint8_t* rowp = buf + lane * 128;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const float4 x = *reinterpret_cast<const float4*>(rowp + ((k ^ (lane & 7)) << 4));
                  sum[4 * k] = x.x + v[4 * k];
                  sum[4 * k + 1] = x.y + v[4 * k + 1];
                  sum[4 * k + 2] = x.z + v[4 * k + 2];
                  sum[4 * k + 3] = x.w + v[4 * k + 3];
                }
              }
              if (part || j < S - 1) {  // the last chained range has nothing to stage
                stage_row32(buf, lane, v);  // a lane overwrites only the row it read
                ptx::fence_proxy_async_smem();
                __syncwarp();
              }
              if (part) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {  // rows 4 i .. 4 i + 3, 16 bytes a lane
                  const int row = 4 * i + (lane >> 3), k = lane & 7;
                  const float4 x = *reinterpret_cast<const float4*>(buf + row * 128 + ((k ^ (row & 7)) << 4));
                  if (mrow0 + row < p.M && n0 + 4 * k < p.N)
                    *reinterpret_cast<float4*>(part + static_cast<int64_t>(mrow0 + row) * p.sp_ld + n0 + 4 * k) = x;
                }
              }
              if (j < S - 1) {
                if (lane == 0 && use_sum) {
                  if (j == 0)
                    ptx::tma_store_3d(&tmD2, buf, c * 32, rrow, it.st);
                  else
                    ptx::tma_reduce_add_3d(&tmD2, buf, c * 32, rrow, it.st);
                  ptx::bulk_commit_group();
                }
                continue;
              }
              // last shard: Y = running sum + own accumulator, + bias, + residual
              uint32_t sb[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) sb[e] = __float_as_uint(sum[e]);
              float y[32], y2[32];
              epilogue_values<EPI, ACT>(p, b, m, n0, sb, y, y2);
              __syncwarp();  // the partial's rows are read out of the box
              {
                uint8_t* rowp = buf + lane * 64;  // 64-byte rows, 16-byte chunks rotated by (row / 2) % 4
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  *reinterpret_cast<uint4*>(rowp + ((k ^ ((lane >> 1) & 3)) << 4)) =
                      make_uint4(pack_bf16x2(y[8 * k], y[8 * k + 1]), pack_bf16x2(y[8 * k + 2], y[8 * k + 3]),
                                 pack_bf16x2(y[8 * k + 4], y[8 * k + 5]), pack_bf16x2(y[8 * k + 6], y[8 * k + 7]));
              }
              __syncwarp();
              uint16_t* Y = static_cast<uint16_t*>(p.d);
#pragma unroll
              for (int i = 0; i < 4; ++i) {  // rows 8 i .. 8 i + 7, 16 bytes a lane
                const int row = 8 * i + (lane >> 2), k = lane & 3;
                const uint4 x = *reinterpret_cast<const uint4*>(buf + row * 64 + ((k ^ ((row >> 1) & 3)) << 4));
                if (mrow0 + row < p.M && n0 + 8 * k < p.N)
                  *reinterpret_cast<uint4*>(Y + static_cast<int64_t>(mrow0 + row) * p.ldd + n0 + 8 * k) = x;
              }
              if (load_sum && c + 2 < nch) {  // the box takes the running sum two chunks on
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                  ptx::mbar_arrive_expect_tx(&ebar[quad * 2 + (c & 1)], STG_BOX_BYTES);
                  ptx::tma_load_3d(buf, &tmD2, &ebar[quad * 2 + (c & 1)], (c + 2) * 32, rrow, it.st);
                }
              }
            }
            if (use_sum) {
              ovl_flag = flag;  // next shard may add (or, after the last, reset for the next launch)
              ovl_set = (j < S - 1) ? (ep | static_cast<unsigned long long>(j + 1)) : 0ull;
            }
          }
        }
      }
      if (!ovl_item && SK_OK && it.kind == ITEM_RANGE && mrow0 < p.M) {
        if (lane == 0) ptx::bulk_wait_group_read<0>();  // the staging boxes are free
        __syncwarp();
#pragma unroll 1
        for (int c = 0; c < P_BN / 32; ++c) {
          if (nb * P_BN + c * 32 >= p.N) break;  // warp-uniform
          uint8_t* buf = stg + (c & 1) * STG_BOX_BYTES;
          if (c >= 2) {
            if (lane == 0) ptx::bulk_wait_group_read<1>();
            __syncwarp();
          }
          uint32_t r[32];
          ptx::tmem_ld32(t_row + c * 32, r);
          ptx::tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
          stage_row32(buf, lane, v);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (p.sp_user)
              ptx::tma_store_3d(&tmP, buf, nb * P_BN + c * 32, mrow0, it.range);
            else
              ptx::tma_store_3d(&tmP, buf, c * 32, static_cast<int>(rank) * P_HALF + quad * 32,
                                it.st * p.sp_split + it.range);
            ptx::bulk_commit_group();
          }
        }
        int last = 0;
        if (lane == 0) {
          ptx::bulk_wait_group<0>();  // the partial is in global memory
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __threadfence();
          last = sp_arrive(p, p.sp_cnt + (static_cast<int64_t>(it.st) * 2 + rank) * 4 + quad, abort_flag) ? 1 : 0;
        }
        sp_last = __shfl_sync(0xffffffffu, last, 0) != 0;
        if (sp_last) __threadfence();  // every lane reads the ranges' partials after the count
      }
      if (ovl_item || it.kind == ITEM_RANGE) {
        // partial written (or rows past M); a completing range sums the tile below, after the
        // accumulator is handed back
      } else if constexpr (EPI == EPI_GLU) {
        // The tile is one gate / up group (N is a multiple of 256).  Per 64 hidden columns:
        // Z's gate box, Z's up box (when Z is kept) and the activation box, three TMA stores.
        if (mrow0 < p.M) {
#pragma unroll 1
          for (int g0 = 0; g0 < GLU_GROUP; g0 += 64) {
            uint8_t* bufG = stg;  // one staging set: the previous step's stores must have read it
            uint8_t* bufU = bufG + STG_BOX_BYTES;
            uint8_t* bufA = bufU + STG_BOX_BYTES;
            if (lane == 0) ptx::bulk_wait_group_read<0>();
            __syncwarp();
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
              uint32_t rg[32], ru[32];
              ptx::tmem_ld32(t_row + g0 + h * 32, rg);
              ptx::tmem_ld32(t_row + GLU_GROUP + g0 + h * 32, ru);
              ptx::tmem_ld_wait();
              float g[32], u[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                g[j] = __uint_as_float(rg[j]);
                u[j] = __uint_as_float(ru[j]);
              }
              if (two_out) {
                stage_half_row16(bufG, lane, h, g, false);
                stage_half_row16(bufU, lane, h, u, false);
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) g[j] = silu(g[j]) * u[j];
              stage_half_row16(bufA, lane, h, g, false);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int zg = nb * P_BN + g0;
              if (two_out) {
                ptx::tma_store_3d(&tmD, bufG, zg, mrow0, b);
                ptx::tma_store_3d(&tmD, bufU, zg + GLU_GROUP, mrow0, b);
              }
              ptx::tma_store_3d(&tmD2, bufA, nb * GLU_GROUP + g0, mrow0, b);
              ptx::bulk_commit_group();
            }
            ++step;
          }
        }
      } else if constexpr (EPI == EPI_DGLU) {
        // dA columns n0.. of the tile -> d gate / d up boxes at their interleaved Z columns.
        if (mrow0 < p.M) {
#pragma unroll 1
          for (int g0 = 0; g0 < P_BN; g0 += 64) {
            const int n0 = nb * P_BN + g0;
            if (n0 >= p.N) break;  // warp-uniform; N is a multiple of 128
            uint8_t* bufG = stg + (step & 1) * (NOUT * STG_BOX_BYTES);
            uint8_t* bufU = bufG + STG_BOX_BYTES;
            if (lane == 0) ptx::bulk_wait_group_read<1>();
            __syncwarp();
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
              uint32_t r[32];
              ptx::tmem_ld32(t_row + g0 + h * 32, r);
              ptx::tmem_ld_wait();
              float v[32], v2[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                v[j] = __uint_as_float(r[j]);
                v2[j] = 0.0f;
              }
              if (m < p.M) dglu_values(p, b, m, n0 + h * 32, v, v2);  // rows past M: clipped by the store
              stage_half_row16(bufG, lane, h, v, false);
              stage_half_row16(bufU, lane, h, v2, false);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int zg = glu_gate_col(n0);
              ptx::tma_store_3d(&tmD, bufG, zg, mrow0, b);
              ptx::tma_store_3d(&tmD, bufU, zg + GLU_GROUP, mrow0, b);
              ptx::bulk_commit_group();
            }
            ++step;
          }
        }
      } else if (!p.tma_store) {
#pragma unroll 1
        for (int c = 0; c < P_BN / 32; ++c) {
          const int n0 = nb * P_BN + c * 32;
          if (n0 >= p.N) break;  // warp-uniform
          uint32_t r[32];
          ptx::tmem_ld32(t_row + c * 32, r);
          ptx::tmem_ld_wait();
          if (m < p.M) epilogue_chunk<EPI, ACT>(p, b, m, n0, r);
        }
      } else if (mrow0 < p.M) {  // warps whose 32 rows are all past M store nothing
        const int box_cols = wide ? 32 : 64;
#pragma unroll 1
        for (int g0 = 0; g0 < P_BN; g0 += box_cols) {
          const int n0 = nb * P_BN + g0;
          if (n0 >= p.N) break;  // warp-uniform
          constexpr int NBUF = PairCfg<EPI>::buffers;
          uint8_t* bufD = stg + (NBUF == 2 ? (step & 1) : 0) * (NOUT * STG_BOX_BYTES);
          uint8_t* bufD2 = bufD + (NOUT - 1) * STG_BOX_BYTES;  // second output (EPI_ACT only)
          // a buffer is reused NBUF steps after it was handed to TMA: it must have been read
          if (lane == 0) ptx::bulk_wait_group_read<NBUF - 1>();
          __syncwarp();
#pragma unroll 1
          for (int h = 0; h < box_cols / 32; ++h) {
            uint32_t r[32];
            ptx::tmem_ld32(t_row + g0 + h * 32, r);
            ptx::tmem_ld_wait();
            float v[32], v2[32];
            epilogue_values<EPI, ACT>(p, b, m, n0 + h * 32, r, v, v2);
            if (wide) {
              stage_row32(bufD, lane, v);
            } else if (EPI == EPI_ACT) {
              if (two_out) stage_half_row16(bufD, lane, h, v, p.out_f16 != 0);
              stage_half_row16(bufD2, lane, h, v2, p.out_f16 != 0);
            } else {
              stage_half_row16(bufD, lane, h, v, false);
            }
            if constexpr (EPI == EPI_DACT) {
              if (p.cs) dact_colsum_chunk(p, b, mrow0, n0 + h * 32, lane, v);  // v is staged: consume it
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (EPI == EPI_ACT) {
              if (two_out) ptx::tma_store_3d(&tmD, bufD, n0, mrow0, b);
              ptx::tma_store_3d(&tmD2, bufD2, n0, mrow0, b);
            } else {
              ptx::tma_store_3d(&tmD, bufD, n0, mrow0, b);
            }
            ptx::bulk_commit_group();
          }
          ++step;
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive_cluster(tempty_leader0 + static_cast<uint32_t>(acc * sizeof(uint64_t)));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
      if (ovl_flag && lane == 0) {  // with the accumulator handed back: the adds complete, then the flag
        ptx::bulk_wait_group<0>();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __threadfence();
        ptx::st_release_u64(reinterpret_cast<uint64_t*>(ovl_flag), ovl_set);
      }
      if constexpr (SK_OK) {
        if (sp_last) sp_reduce_rows<EPI, ACT>(p, it, b, mrow0, trow - lane, nb, lane);
      }
    }
    if (lane == 0) ptx::bulk_wait_group<0>();  // every output written before the CTA exits
  }

  __syncwarp();
  ptx::tc_fence_before();
  ptx::cluster_sync();  // the peer's shared memory and TMEM stay alive until the pair is done
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D map (inner, outer, shard) over a bf16 operand with a 128-byte swizzle.
// K-major: inner = K, outer = rows, box = 64 x box_rows (4-D: two k-blocks per box when kb = 2).
// MN-major: inner = rows (MN), outer = K, box = 64 x 64 kb (4-D: every 64-column chunk of the
// box_rows in one box).  kb = 64-wide k-blocks per pipeline stage.
bool make_operand_map(CUtensorMap* map, const GemmOperand& op, int64_t rows, int64_t K, int nshards,
                      int box_rows, int kb, int* four_d) {
  auto enc = encode_fn();
  if (!enc) return false;
  *four_d = 0;
  if (!op.mn_major && kb == 2 && K % 64 == 0) {
    // K-major [shard][rows][K] as (64 K, rows, K / 64 blocks, shard): one box of two k-blocks
    // lands as two [rows][64] panels.  K not a multiple of 64 keeps one box per k-block (a
    // 4-D box would read the next row's first columns past K instead of zeros).
    const int64_t ss = (op.sharded && nshards > 1) ? op.shard_stride : op.ld * rows;
    cuuint64_t d4[4] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(K / 64),
                        static_cast<cuuint64_t>(nshards)};
    cuuint64_t s4[3] = {static_cast<cuuint64_t>(op.ld) * 2, 128, static_cast<cuuint64_t>(ss) * 2};
    cuuint32_t b4[4] = {64, static_cast<cuuint32_t>(box_rows), 2, 1};
    cuuint32_t e4[4] = {1, 1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(op.ptr), d4, s4, b4, e4,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      char buf[200];
      std::snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled (4-D K-major)=%d ptr=%p rows=%lld K=%lld ld=%lld",
                    static_cast<int>(r), static_cast<const void*>(op.ptr), static_cast<long long>(rows),
                    static_cast<long long>(K), static_cast<long long>(op.ld));
      set_error_detail(__FILE__, __LINE__, buf);
      return false;
    }
    *four_d = 1;
    return true;
  }
  if (op.mn_major && rows % 64 == 0) {
    // MN-major [shard][K][rows] as (64 columns, K, rows / 64 chunks, shard): the chunk stride
    // (128 bytes) is below the K stride, so one box of box_rows / 64 chunks lands in shared
    // memory as [chunk][K][64], the layout of the 64-column boxes it replaces.  A row count
    // that is not a multiple of 64 keeps the per-chunk boxes (a 4-D box would read past it).
    const int64_t ss = (op.sharded && nshards > 1) ? op.shard_stride : op.ld * K;
    cuuint64_t d4[4] = {64, static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows / 64),
                        static_cast<cuuint64_t>(nshards)};
    cuuint64_t s4[3] = {static_cast<cuuint64_t>(op.ld) * 2, 128, static_cast<cuuint64_t>(ss) * 2};
    cuuint32_t b4[4] = {64, static_cast<cuuint32_t>(BK * kb), static_cast<cuuint32_t>(box_rows / 64), 1};
    cuuint32_t e4[4] = {1, 1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(op.ptr), d4, s4, b4, e4,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      char buf[200];
      std::snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled (4-D MN-major)=%d ptr=%p rows=%lld K=%lld ld=%lld",
                    static_cast<int>(r), static_cast<const void*>(op.ptr), static_cast<long long>(rows),
                    static_cast<long long>(K), static_cast<long long>(op.ld));
      set_error_detail(__FILE__, __LINE__, buf);
      return false;
    }
    *four_d = 1;
    return true;
  }
  cuuint64_t dims[3];
  cuuint64_t strides[2];
  cuuint32_t box[3];
  cuuint32_t estr[3] = {1, 1, 1};
  const int64_t outer = op.mn_major ? K : rows;
  if (!op.mn_major) {
    dims[0] = static_cast<cuuint64_t>(K);
    dims[1] = static_cast<cuuint64_t>(rows);
    box[0] = BK;
    box[1] = static_cast<cuuint32_t>(box_rows);
  } else {
    dims[0] = static_cast<cuuint64_t>(rows);
    dims[1] = static_cast<cuuint64_t>(K);
    box[0] = 64;
    box[1] = static_cast<cuuint32_t>(BK * kb);
  }
  dims[2] = static_cast<cuuint64_t>(nshards);
  box[2] = 1;
  strides[0] = static_cast<cuuint64_t>(op.ld) * 2;
  const int64_t ss = (op.sharded && nshards > 1) ? op.shard_stride : op.ld * outer;
  strides[1] = static_cast<cuuint64_t>(ss) * 2;
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(op.ptr), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[200];
    std::snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled=%d ptr=%p dims=%llu,%llu,%llu strides=%llu,%llu box=%u,%u",
                  static_cast<int>(r), static_cast<const void*>(op.ptr), (unsigned long long)dims[0],
                  (unsigned long long)dims[1], (unsigned long long)dims[2], (unsigned long long)strides[0],
                  (unsigned long long)strides[1], box[0], box[1]);
    set_error_detail(__FILE__, __LINE__, buf);
  }
  return r == CUDA_SUCCESS;
}

}  // namespace

bool make_map_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
                      uint64_t s2_bytes, uint32_t b0, uint32_t b1) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <bool A_MN, bool B_MN, int EPI, int ACT>
tp_status launch(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a, int grid, cudaStream_t s) {
  static bool configured[64] = {};
  int dev = 0;
  TP_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return TP_ERR_CUDA;
  if (!configured[dev]) {
    TP_CUDA_CHECK(cudaFuncSetAttribute(gemm_kernel<A_MN, B_MN, EPI, ACT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES));
    configured[dev] = true;
  }
  TP_CUDA_CHECK(launch_pdl(gemm_kernel<A_MN, B_MN, EPI, ACT>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, s, ta, tb, a));
  count_launch();
  return TP_OK;
}

// Clusters of the pair kernel that can be resident at once on this device.
template <bool A_MN, bool B_MN, int EPI, int ACT>
int pair_clusters(int dev) {
  static int cached[64] = {};
  if (cached[dev] > 0) return cached[dev];
  if (cudaFuncSetAttribute(gemm_pair_kernel<A_MN, B_MN, EPI, ACT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           pair_smem_bytes<EPI>()) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 256, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = pair_smem_bytes<EPI>();
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<A_MN, B_MN, EPI, ACT>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = device_sm_count() / 2;
  }
  cached[dev] = n;
  return n;
}

// Split-K plan of a pair-kernel launch: T tiles of U k-stages on nc resident clusters.  The
// data-parallel schedule takes ceil(T / nc) rounds of whole tiles, the last one with only
// T mod nc clusters busy.  Here the full rounds stay whole and the remaining tiles are cut
// into S equal k-ranges (the same cut points for every tile), dealt to all the clusters:
// ceil(rem S / nc) items of U / S stages instead of one more round of U, plus the completing
// range's sum of the S partials.  That sum reads about 16 GB/s per SM (generic loads, with
// the stages holding nearly all shared memory: 8 us per 128 KB partial of a CTA, measured),
// about kSkSumStages k-stages per range.  S is the cut that finishes first by this count;
// ties keep fewer partials; a cut that saves less than kSkMinGain is not taken.  Ranges keep
// at least kSkMinUnits k-stages, and the workspace bounds the partial slots.  (Contiguous
// stream-K ranges were measured first and lost: ranges that start at staggered k break the
// clusters' lockstep -- the 2048 x 4096 x 16384 row-parallel GEMM, 128 tiles on 76 clusters,
// read 575 MB from DRAM against 276 MB and ran 185 us against 167 us, and a 32-tile one ran
// 109 us against 87 us.)  TP_STREAMK=0 turns the split off.
//
// Chained ranges (EPI_BF16) sum through a running sum in L2 instead: each range's TMA store
// or add runs while its cluster's MMAs go on with the next item, so only the last round's
// chain of S adds is exposed, about 2.2 us a link (a 4-tile, 19-range tail of the 2048 x
// 12288 x 49152 row-parallel GEMM).  Charged kChainLinkStages per range, and taken from a
// gain of kChainMinGain.  The chained ranges are dealt range-major, so the pairs that run side
// by side work on one or two K slices of the panels (dealt tile by tile, a tile's S ranges on
// neighbouring pairs, the 2048 x 4096 x 16384 GEMM's split -- 52 tiles past a round of 76, four
// ranges each -- read four K slices at once and ran 178.8 us against 172.7 us whole; range-major,
// 168.6 against 170.7 us).  Chains are planned only for at most half a round of split tiles: a
// partial round that keeps more than half the pairs busy runs each tile faster than a full round
// does, and against it the split gained 1 % (and lost 1 % at K = 12288).
constexpr int kSkMinUnits = 8;
constexpr int kSkSumStages = 10;
constexpr double kSkMinGain = 0.1;
constexpr int kChainLinkStages = 4;
constexpr double kChainMinGain = 0.03;
bool make_output_map(CUtensorMap* map, void* d, CUtensorMapDataType dt, int esz, int64_t N, int64_t M, int nbatch,
                     int64_t ldd, int64_t dbs);
struct SpPlan {
  int rounds = 0, tiles = 0, split = 0, clusters = 0;
};
SpPlan sp_plan(int64_t T, int U, int nc, int64_t max_slots, bool chain) {
  SpPlan pl;
  const char* e = std::getenv("TP_STREAMK");
  if ((e && e[0] == '0') || T <= 0 || U <= 0 || nc <= 0) return pl;
  const int64_t R = T / nc, rem = T - R * nc;
  if (rem == 0) return pl;
  if (chain && (rem > max_slots || 2 * rem > nc)) return pl;  // one running sum per split tile
  const double whole = static_cast<double>((R + 1) * U);
  double best = whole;
  int bestS = 0;
  for (int S = 2; U / S >= kSkMinUnits && (chain || rem * S <= max_slots); ++S) {
    const double tm = static_cast<double>(R * U) + static_cast<double>((rem * S + nc - 1) / nc) * U / S +
                      static_cast<double>(S) * (chain ? kChainLinkStages : kSkSumStages);
    if (tm < best - 1e-9) {
      best = tm;
      bestS = S;
    }
  }
  if (bestS == 0 || best > whole * (1.0 - (chain ? kChainMinGain : kSkMinGain))) return pl;
  pl.rounds = static_cast<int>(R);
  pl.tiles = static_cast<int>(rem);
  pl.split = bestS;
  pl.clusters = R > 0 ? nc : static_cast<int>(rem * bestS < nc ? rem * bestS : nc);
  return pl;
}

// Launch tag of the split-K counters: a value no recent launch used (counters are reset by
// the range that completes them, and a fresh workspace would have to hold this exact value
// in a counter's upper half by chance).
uint32_t next_sp_epoch() {
  static std::atomic<uint32_t> ctr{static_cast<uint32_t>(std::time(nullptr)) ^
                                   static_cast<uint32_t>(reinterpret_cast<uintptr_t>(&ctr) >> 4)};
  uint32_t v;
  do {
    v = ctr.fetch_add(0x9E3779B9u);  // odd step: every 32-bit value once per 2^32 launches
  } while (v == 0);
  return v;
}

// The completing range of a split tile writes its outputs with 16-byte accesses of 8 columns.
bool sp_layout_ok(const GemmArgs& a) {
  auto al = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  if (a.N % 8 != 0 || !al(a.d) || !al(a.d2) || !al(a.bias) || !al(a.res) || !al(a.aux) || !al(a.cs)) return false;
  return a.ldd % 8 == 0 && a.d_bs % 8 == 0 && a.ld_res % 8 == 0 && a.ld_aux % 8 == 0 && a.aux_bs % 8 == 0 &&
         a.bias_bs % 8 == 0;
}

// Overlapped shard reduction (ovl_part != NULL): the tiles' K ranges are the t shards, every
// shard's fp32 partial goes to ovl_part [t][M][N], and ovl_run holds a 256 x 256 fp32 running
// sum per output tile followed by 8 flags per tile (gemm_overlap_scratch_bytes).
template <bool A_MN, bool B_MN, int EPI, int ACT>
tp_status launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td, const CUtensorMap& td2,
                      const GemmArgs& a0, int64_t tiles, cudaStream_t s, void* sk_ws = nullptr,
                      size_t sk_ws_bytes = 0, float* ovl_part = nullptr, float* ovl_run = nullptr) {
  int dev = 0;
  TP_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return TP_ERR_CUDA;
  const int nc = pair_clusters<A_MN, B_MN, EPI, ACT>(dev);
  if (nc <= 0) return TP_FAIL_DETAIL("no co-resident CTA pairs");
  int clusters = static_cast<int>(tiles < nc ? tiles : nc);
  GemmArgs a = a0;
  CUtensorMap tp_map, run_map;
  std::memset(&tp_map, 0, sizeof(tp_map));
  std::memset(&run_map, 0, sizeof(run_map));
  const int U = a.nsum * ((a.kt + PairCfg<EPI>::kb - 1) / PairCfg<EPI>::kb);
  if constexpr (sk_epi(EPI)) {
    if (ovl_part) {
      // every tile cut at its shard boundaries, one cluster walking a tile's shards in turn
      if constexpr (EPI != EPI_BF16) return TP_ERR_UNSUPPORTED;
      if (!sp_layout_ok(a)) return TP_ERR_ALIGN;
      clusters = static_cast<int>(tiles * a.nsum < nc ? tiles * a.nsum : nc);
      a.sp_split = a.nsum;
      a.sp_units = U;
      a.sp_seq = 1;
      a.sp_chain = 1;
      a.sp_user = 1;
      a.sp_part = ovl_part;
      a.sp_ld = a.N;
      a.sp_bs = static_cast<int64_t>(a.M) * a.N;
      if (!make_output_map(&tp_map, ovl_part, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.N, a.M, a.nsum, a.N, a.sp_bs))
        return TP_FAIL_DETAIL("tensor map of the shard partials");
      if (!make_output_map(&run_map, ovl_run, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 256, 256, static_cast<int>(tiles),
                           256, 256 * 256))
        return TP_FAIL_DETAIL("tensor map of the running sums");
      a.sp_cnt = reinterpret_cast<unsigned long long*>(ovl_run + static_cast<size_t>(tiles) * 256 * 256);
      a.sp_epoch = next_sp_epoch();
    } else if (sk_ws && sp_layout_ok(a)) {
      int64_t slots = static_cast<int64_t>(sk_ws_bytes / (kSkSlotBytes + kSkCounterBytes));
      if (slots > kSkMaxSlots) slots = kSkMaxSlots;
      const char* ec = std::getenv("TP_SPLIT_CHAIN");
      bool chain = EPI == EPI_BF16 && !(ec && ec[0] == '0');
      SpPlan pl = sp_plan(tiles, U, nc, slots, chain);
      if (chain && pl.split == 0) {  // no chain planned: the counted form may still pay
        chain = false;
        pl = sp_plan(tiles, U, nc, slots, false);
      }
      if (pl.split > 0 && chain) {
        // a running sum (slot) and 8 flags per split tile: [tiles][256][256] fp32, then flags
        a.sp_rounds = pl.rounds;
        a.sp_tiles = pl.tiles;
        a.sp_split = pl.split;
        a.sp_units = U;
        a.sp_chain = 1;
        a.sp_cnt = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(sk_ws) +
                                                         static_cast<size_t>(pl.tiles) * kSkSlotBytes);
        a.sp_epoch = next_sp_epoch();
        if (!make_output_map(&run_map, sk_ws, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 256, 256, pl.tiles, 256,
                             256 * 256))
          return TP_FAIL_DETAIL("tensor map of the split-K running sums");
        clusters = pl.clusters;
      } else if (pl.split > 0) {
        const int used = pl.tiles * pl.split;  // partial slots
        a.sp_rounds = pl.rounds;
        a.sp_tiles = pl.tiles;
        a.sp_split = pl.split;
        a.sp_units = U;
        a.sp_part = static_cast<float*>(sk_ws);
        a.sp_cnt = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(sk_ws) +
                                                         static_cast<size_t>(used) * kSkSlotBytes);
        a.sp_epoch = next_sp_epoch();
        if (!make_output_map(&tp_map, a.sp_part, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 256, 256, used, 256, 256 * 256))
          return TP_FAIL_DETAIL("tensor map of the split-K partials");
        clusters = pl.clusters;
      }
    }
  } else if (ovl_part) {
    return TP_ERR_UNSUPPORTED;
  }
  TP_CUDA_CHECK(launch_pdl(gemm_pair_kernel<A_MN, B_MN, EPI, ACT>, dim3(2 * clusters), dim3(NUM_THREADS),
                           pair_smem_bytes<EPI>(), s, ta, tb, td, a.sp_chain ? run_map : td2, tp_map, a));
  count_launch();
  return TP_OK;
}

// The CTA-pair kernel is used when a 256-row output tile is not mostly
// padding; TP_GEMM_PAIR=0 forces the single-CTA kernel (tests cover both).
bool use_pair(int64_t M) {
  const char* e = std::getenv("TP_GEMM_PAIR");
  if (e && e[0] == '0') return false;
  return M > 128;
}

// Output map for the TMA-store epilogue: (N, M, batch), 32-row boxes of 128 bytes, 128B swizzle.
bool make_output_map(CUtensorMap* map, void* d, CUtensorMapDataType dt, int esz, int64_t N, int64_t M, int nbatch,
                     int64_t ldd, int64_t dbs) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(nbatch)};
  const int64_t bs = (nbatch > 1) ? dbs : ldd * M;
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldd * esz), static_cast<cuuint64_t>(bs * esz)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esz), 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, dt, 3, d, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The (operand majors, epilogue, activation) combinations the library uses;
// each is its own kernel instantiation.
template <class F>
tp_status dispatch(bool amn, bool bmn, int epi, int act, F&& f) {
  using T = std::true_type;
  using Fl = std::false_type;
  using I0 = std::integral_constant<int, 0>;
  using I1 = std::integral_constant<int, 1>;
  using I2 = std::integral_constant<int, 2>;
  using I3 = std::integral_constant<int, 3>;
  using E_BF16 = std::integral_constant<int, EPI_BF16>;
  using E_ACT = std::integral_constant<int, EPI_ACT>;
  using E_DACT = std::integral_constant<int, EPI_DACT>;
  using E_F32 = std::integral_constant<int, EPI_F32>;
  using E_GLU = std::integral_constant<int, EPI_GLU>;
  using E_DGLU = std::integral_constant<int, EPI_DGLU>;
  if (!amn && !bmn) {  // forward GEMMs
    if (epi == EPI_GLU) return f(Fl{}, Fl{}, E_GLU{}, I0{});
    if (epi == EPI_ACT) {
      switch (act) {
        case 0: return f(Fl{}, Fl{}, E_ACT{}, I0{});
        case 1: return f(Fl{}, Fl{}, E_ACT{}, I1{});
        case 2: return f(Fl{}, Fl{}, E_ACT{}, I2{});
        case 3: return f(Fl{}, Fl{}, E_ACT{}, I3{});
      }
    }
    if (epi == EPI_BF16) return f(Fl{}, Fl{}, E_BF16{}, I0{});
    if (epi == EPI_F32) return f(Fl{}, Fl{}, E_F32{}, I0{});
  } else if (!amn && bmn) {  // dgrad and f-reduced dX
    if (epi == EPI_DGLU) return f(Fl{}, T{}, E_DGLU{}, I0{});
    if (epi == EPI_DACT) {
      switch (act) {
        case 0: return f(Fl{}, T{}, E_DACT{}, I0{});
        case 1: return f(Fl{}, T{}, E_DACT{}, I1{});
        case 2: return f(Fl{}, T{}, E_DACT{}, I2{});
        case 3: return f(Fl{}, T{}, E_DACT{}, I3{});
      }
    }
    if (epi == EPI_ACT && act == 0) return f(Fl{}, T{}, E_ACT{}, I0{});
    if (epi == EPI_BF16) return f(Fl{}, T{}, E_BF16{}, I0{});
    if (epi == EPI_F32) return f(Fl{}, T{}, E_F32{}, I0{});
  } else if (amn && bmn) {  // weight gradients
    if (epi == EPI_F32) return f(T{}, T{}, E_F32{}, I0{});
  }
  return TP_ERR_UNSUPPORTED;
}

// ----------------------------------------------------- split K: launch
// Clusters of S CTAs that can be resident at once for this instance (0 if none).
template <bool A_MN, bool B_MN, int EPI, int ACT, int SBN>
int splitc_clusters(int dev, int S) {
  static int cached[64][5] = {};  // [device][log2 S - 1] + 1
  int li = 0;
  while ((2 << li) < S) ++li;
  if (dev < 0 || dev >= 64 || li > 4) return 0;
  if (cached[dev][li]) return cached[dev][li] - 1;
  auto kern = gemm_splitc_kernel<A_MN, B_MN, EPI, ACT, SBN>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) == cudaSuccess &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S * 16, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = S;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  cached[dev][li] = n + 1;
  return n;
}

template <bool A_MN, bool B_MN, int EPI, int ACT, int SBN>
tp_status launch_splitc(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a, int64_t tiles, int S,
                        cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * S), 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = S;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  TP_CUDA_CHECK(cudaLaunchKernelEx(&cfg, gemm_splitc_kernel<A_MN, B_MN, EPI, ACT, SBN>, ta, tb, a));
  count_launch();
  return TP_OK;
}

// Instances of the cluster-split kernel: the epilogues a small-M problem can have.
template <class F>
tp_status dispatch_splitc(bool amn, bool bmn, int epi, int act, F&& f) {
  using T = std::true_type;
  using Fl = std::false_type;
  using E_BF16 = std::integral_constant<int, EPI_BF16>;
  using E_ACT = std::integral_constant<int, EPI_ACT>;
  using E_F32 = std::integral_constant<int, EPI_F32>;
  using I0 = std::integral_constant<int, 0>;
  if (!amn && !bmn) {
    if (epi == EPI_ACT) {
      switch (act) {
        case 0: return f(Fl{}, Fl{}, E_ACT{}, I0{});
        case 1: return f(Fl{}, Fl{}, E_ACT{}, std::integral_constant<int, 1>{});
        case 2: return f(Fl{}, Fl{}, E_ACT{}, std::integral_constant<int, 2>{});
        case 3: return f(Fl{}, Fl{}, E_ACT{}, std::integral_constant<int, 3>{});
      }
    }
    if (epi == EPI_BF16) return f(Fl{}, Fl{}, E_BF16{}, I0{});
    if (epi == EPI_F32) return f(Fl{}, Fl{}, E_F32{}, I0{});
  } else if (!amn && bmn) {
    if (epi == EPI_ACT && act == 0) return f(Fl{}, T{}, E_ACT{}, I0{});
    if (epi == EPI_BF16) return f(Fl{}, T{}, E_BF16{}, I0{});
    if (epi == EPI_F32) return f(Fl{}, T{}, E_F32{}, I0{});
  }
  return TP_ERR_UNSUPPORTED;
}

// K ranges per tile for a small-M problem: a power of two up to 8 such that the tiles
// times S CTAs about fill the GPU and every range keeps at least kSplitMinSteps k-blocks.
// (On a GB300, the 128-token forward: 8 ranges of the row-parallel GEMM ran 21.9 us against
// 22.2 us for 16, whose exchange through distributed shared memory waits longer for the
// slowest CTA.)  TP_SPLITK=<S> asks for S, up to 16 (rounded down to a power of two;
// 1 disables the split).
constexpr int kSplitMinSteps = 4;
constexpr int kSplitAutoMax = 8;
int splitc_ranges(int64_t tiles, int64_t ksteps) {
  int64_t want;
  const char* e = std::getenv("TP_SPLITK");
  if (e && e[0]) {
    want = std::atol(e);
  } else {
    const int64_t sms = device_sm_count();
    if (tiles * 2 > sms) return 1;
    want = sms / tiles;
    if (want > ksteps / kSplitMinSteps) want = ksteps / kSplitMinSteps;
    if (want > kSplitAutoMax) want = kSplitAutoMax;
  }
  if (want > ksteps) want = ksteps;
  int S = 1;
  while (S * 2 <= want && S < 16) S *= 2;
  return S;
}

bool operand_ok(const GemmOperand& o) {
  return o.ptr && aligned16(o.ptr) && o.ld > 0 && o.ld % 8 == 0 && (!o.sharded || o.shard_stride % 8 == 0);
}

}  // namespace

tp_status run_gemm(const GemmProblem& P, cudaStream_t s) {
  if (P.M < 0 || P.N < 0 || P.K < 0 || P.nbatch < 1 || P.nsum < 1) return TP_ERR_INVALID_ARG;
  if (P.M == 0 || P.N == 0) return TP_OK;
  if (P.nbatch > 1 && P.nsum > 1) return TP_ERR_INVALID_ARG;
  if (!operand_ok(P.a) || !operand_ok(P.b)) return TP_ERR_ALIGN;
  const bool glu = P.epi == EPI_GLU || P.epi == EPI_DGLU;
  if (P.epi == EPI_ACT || P.epi == EPI_GLU) {
    if (!P.d2 || !aligned16(P.d2) || (P.d && !aligned16(P.d))) return TP_ERR_ALIGN;
  } else if (!P.d || !aligned16(P.d)) {
    return TP_ERR_ALIGN;
  }
  if (P.ldd % 8 != 0 || P.d_batch_stride % 8 != 0) return TP_ERR_ALIGN;
  if (P.bias && (!aligned16(P.bias) || P.bias_batch_stride % 8 != 0)) return TP_ERR_ALIGN;
  if ((P.epi == EPI_DACT || P.epi == EPI_DGLU) &&
      (!P.aux || !aligned16(P.aux) || P.ld_aux % 8 != 0 || P.aux_batch_stride % 8 != 0))
    return TP_ERR_ALIGN;
  // SwiGLU epilogues: whole gate / up groups per tile, no bias, no residual, bf16 outputs
  if (glu && (P.N % (P.epi == EPI_GLU ? 2 * GLU_GROUP : GLU_GROUP) != 0)) return TP_ERR_SHAPE;
  if (glu && (P.bias || P.residual || P.out_f16 || P.nsum != 1)) return TP_ERR_UNSUPPORTED;
  if (P.epi == EPI_GLU && (P.ldd2 % 8 != 0 || P.d2_batch_stride % 8 != 0)) return TP_ERR_ALIGN;
  if (P.residual && (!aligned16(P.residual) || P.ld_res % 8 != 0)) return TP_ERR_ALIGN;
  if (P.colsum && P.epi != EPI_DACT) return TP_ERR_UNSUPPORTED;
  if (P.K == 0) return TP_ERR_SHAPE;
  const int64_t mt = (P.M + BM - 1) / BM, nt = (P.N + BN - 1) / BN, kt = (P.K + BK - 1) / BK;
  if (mt * nt * P.nbatch > (1LL << 30) || P.M > (1LL << 30) || P.N > (1LL << 30)) return TP_ERR_SHAPE;
  const int nsh_a = P.a.sharded ? (P.nsum > 1 ? P.nsum : P.nbatch) : 1;
  const int nsh_b = P.b.sharded ? (P.nsum > 1 ? P.nsum : P.nbatch) : 1;

  TP_RETURN_IF(ready());
  const bool pair = use_pair(P.M);
  if (P.ovl_part) {
    // overlapped reduction: pair kernel, the nsum shards' fp32 partials written by TMA
    if (!pair || P.epi != EPI_BF16 || P.accumulate || P.nbatch != 1 || !P.ovl_run) return TP_ERR_UNSUPPORTED;
    if (!aligned16(P.ovl_part) || !aligned16(P.ovl_run)) return TP_ERR_ALIGN;
  }
  CUtensorMap ta, tb;
  int a_4d = 0, b_4d = 0;
  const int kb = pair ? pair_kb(P.epi) : 1;  // k-blocks per stage
  if (!make_operand_map(&ta, P.a, P.M, P.K, nsh_a, BM, kb, &a_4d)) return TP_ERR_CUDA;
  if (!make_operand_map(&tb, P.b, P.N, P.K, nsh_b, pair ? P_HALF : BN, kb, &b_4d)) return TP_ERR_CUDA;

  GemmArgs a{};
  a.M = static_cast<int>(P.M);
  a.N = static_cast<int>(P.N);
  a.nbatch = P.nbatch;
  a.nsum = P.nsum;
  a.a_sharded = P.a.sharded;
  a.b_sharded = P.b.sharded;
  a.a_4d = a_4d;
  a.b_4d = b_4d;
  a.mt = static_cast<int>(mt);
  a.nt = static_cast<int>(nt);
  a.kt = static_cast<int>(kt);
  a.epi = P.epi;
  a.act = P.act;
  a.f16ab = P.f16_ab;
  a.d = P.d;
  a.ldd = P.ldd;
  a.d_bs = P.d_batch_stride;
  a.d2 = P.d2;
  a.ldd2 = P.ldd2;
  a.d2_bs = P.d2_batch_stride;
  a.bias = P.bias;
  a.bias_bs = P.bias_batch_stride;
  a.aux = P.aux;
  a.ld_aux = P.ld_aux;
  a.aux_bs = P.aux_batch_stride;
  a.cs = P.colsum;
  a.cs_chunks = static_cast<int>((P.M + 31) / 32);
  a.res = P.residual;
  a.ld_res = P.ld_res;
  a.accumulate = P.accumulate;
  a.out_f16 = P.out_f16;
  a.ksplit = 1;
  a.err = device_error_word();
  a.timeout_ns = wait_timeout_ns();
  if (!a.err) return TP_ERR_CUDA;

  const bool amn = P.a.mn_major, bmn = P.b.mn_major;
  if (pair) {
    // Outputs go through shared memory and TMA stores, except accumulation into fp32
    // (a read-modify-write), which keeps the per-thread store path.
    CUtensorMap td, td2;
    std::memset(&td, 0, sizeof(td));
    std::memset(&td2, 0, sizeof(td2));
    a.tma_store = !(P.epi == EPI_F32 && P.accumulate);
    if (a.tma_store) {
      const int esz = (P.epi == EPI_F32) ? 4 : 2;
      const CUtensorMapDataType dt = (P.epi == EPI_F32) ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : (P.epi == EPI_ACT && P.out_f16) ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
      if (P.epi == EPI_GLU) {
        // D = Z (N columns; mapped to D2 as a placeholder when Z is not kept), D2 = A (N / 2)
        if (!make_output_map(&td, P.d ? P.d : P.d2, dt, esz, P.d ? P.N : P.N / 2, P.M, P.nbatch,
                             P.d ? P.ldd : P.ldd2, P.d ? P.d_batch_stride : P.d2_batch_stride))
          return TP_FAIL_DETAIL("tensor map of output Z");
        if (!make_output_map(&td2, P.d2, dt, esz, P.N / 2, P.M, P.nbatch, P.ldd2, P.d2_batch_stride))
          return TP_FAIL_DETAIL("tensor map of output A");
      } else {
        void* d_main = (P.epi == EPI_ACT) ? (P.d ? P.d : P.d2) : P.d;
        const int64_t n_out = (P.epi == EPI_DGLU) ? 2 * P.N : P.N;  // dZ is twice as wide as dA
        if (!make_output_map(&td, d_main, dt, esz, n_out, P.M, P.nbatch, P.ldd, P.d_batch_stride))
          return TP_FAIL_DETAIL("tensor map of output D");
        if (P.epi == EPI_ACT &&
            !make_output_map(&td2, P.d2, dt, esz, P.N, P.M, P.nbatch, P.ldd, P.d_batch_stride))
          return TP_FAIL_DETAIL("tensor map of output D2");
      }
    }
    const int64_t ptiles = ((P.M + 255) / 256) * ((P.N + P_BN - 1) / P_BN) * P.nbatch;
    if (P.ovl_part) {
      if (amn || bmn || !a.tma_store) return TP_ERR_UNSUPPORTED;
      return launch_pair<false, false, EPI_BF16, TP_ACT_IDENTITY>(ta, tb, td, td2, a, ptiles, s, nullptr, 0,
                                                                   P.ovl_part, P.ovl_run);
    }
    // Split K needs the TMA-store epilogue and a 256-byte aligned workspace.
    void* sk_ws = (P.sk_ws && a.tma_store && (reinterpret_cast<uintptr_t>(P.sk_ws) & 255u) == 0) ? P.sk_ws : nullptr;
    return dispatch(amn, bmn, P.epi, P.act, [&](auto am, auto bm, auto ep, auto ac) {
      return launch_pair<decltype(am)::value, decltype(bm)::value, decltype(ep)::value, decltype(ac)::value>(
          ta, tb, td, td2, a, ptiles, s, sk_ws, P.sk_ws_bytes);
    });
  }
  const int64_t tiles = mt * nt * P.nbatch;
  // Split K inside a cluster when few output tiles would leave most SMs idle (M <= 128):
  // the S CTAs of a cluster compute one tile's K ranges and sum them on chip, in order.
  if (P.M <= 128 && P.N % 8 == 0 && !P.colsum && (P.epi == EPI_BF16 || P.epi == EPI_ACT || P.epi == EPI_F32)) {
    int dev = 0;
    TP_CUDA_CHECK(cudaGetDevice(&dev));
    // 128-column tiles (K-major operands) where even they leave SMs idle: twice the CTAs,
    // each with half the operand bytes, half the partial to exchange and half the rows'
    // columns to sum.  TP_SPLITC_NARROW=0 keeps 256-column tiles, =1 asks for 128.
    const char* en = std::getenv("TP_SPLITC_NARROW");
    const bool narrow = !amn && !bmn && (en && en[0] ? en[0] == '1' : tiles * 4 <= device_sm_count());
    const int64_t snt = narrow ? (P.N + BN / 2 - 1) / (BN / 2) : nt;
    const int64_t stiles = mt * snt * P.nbatch;
    auto clusters_ok = [&](int S) {
      return dispatch_splitc(amn, bmn, P.epi, P.act, [&](auto am, auto bm, auto ep, auto ac) {
        constexpr bool AM = decltype(am)::value, BM_ = decltype(bm)::value;
        constexpr int EP = decltype(ep)::value, AC = decltype(ac)::value;
        int n = 0;
        if constexpr (!AM && !BM_)
          n = narrow ? splitc_clusters<AM, BM_, EP, AC, BN / 2>(dev, S) : splitc_clusters<AM, BM_, EP, AC, BN>(dev, S);
        else
          n = splitc_clusters<AM, BM_, EP, AC, BN>(dev, S);
        return n > 0 ? TP_OK : TP_ERR_UNSUPPORTED;
      });
    };
    int S = splitc_ranges(stiles, static_cast<int64_t>(P.nsum) * kt);
    while (S > 1 && clusters_ok(S) != TP_OK) S /= 2;  // the largest cluster size this device can schedule
    if (S > 1) {
      a.ksplit = S;
      CUtensorMap tbn = tb;
      if (narrow) {
        int b4 = 0;
        if (!make_operand_map(&tbn, P.b, P.N, P.K, nsh_b, BN / 2, 1, &b4)) return TP_ERR_CUDA;
        a.b_4d = b4;
        a.nt = static_cast<int>(snt);
      }
      return dispatch_splitc(amn, bmn, P.epi, P.act, [&](auto am, auto bm, auto ep, auto ac) {
        constexpr bool AM = decltype(am)::value, BM_ = decltype(bm)::value;
        constexpr int EP = decltype(ep)::value, AC = decltype(ac)::value;
        if constexpr (!AM && !BM_) {
          if (narrow) return launch_splitc<AM, BM_, EP, AC, BN / 2>(ta, tbn, a, stiles, S, s);
        }
        return launch_splitc<AM, BM_, EP, AC, BN>(ta, tbn, a, stiles, S, s);
      });
    }
  }
  const int grid = static_cast<int>(tiles < device_sm_count() ? tiles : device_sm_count());
  return dispatch(amn, bmn, P.epi, P.act, [&](auto am, auto bm, auto ep, auto ac) {
    return launch<decltype(am)::value, decltype(bm)::value, decltype(ep)::value, decltype(ac)::value>(ta, tb, a, grid,
                                                                                                      s);
  });
}

}  // namespace tp
