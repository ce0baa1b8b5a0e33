// Head-local causal softmax attention on tcgen05 ("02 — Tensor Parallelism",
// "The attention pairing": heads don't talk, so each shard runs attention on
// its own heads with no communication; "Megatron-LM: Tensor Parallelism",
// "The Transformer Layer Partitioning": S = Q K^T, P = softmax(S), O = P V).
//
// The QKV buffer is the column-parallel GEMM's output, [t][N][3d/t] with the
// shard's heads laid out [Q_i | K_i | V_i], head jj at columns jj*128 of each.
// Q, K, V, P (and in backward dO, dS) are IEEE fp16: the logits of a wide
// model have a spread of several units, and a 2^-9 relative rounding of Q
// and K (bf16) turns into a ~1% error of P; fp16 keeps 3 more mantissa bits
// at the same cost.  Inputs, weights and O / dQKV stay bf16.
//
// Forward: one CTA per (head, pair of adjacent 128-query tiles), heavy (late)
// pairs first.  The two tiles take turns on the tensor pipe, so one tile's
// softmax runs while the other tile's MMAs do:
//   warp 0      TMA: both Q tiles once, then K_j, V_j through a 5-slot ring
//   warp 1      tcgen05.mma, per key block j: O_0 += P_0 V_j, S_0 = Q_0 K_{j+1}^T,
//               O_1 += P_1 V_j, S_1 = Q_1 K_{j+1}^T (fp32 S and O in TMEM)
//   warps 2-5   softmax of tile 0, warps 6-9 of tile 1, one query row per
//               thread: block max in the log2 domain, a reference max raised
//               only by a jump of more than 2^8 (then O is rescaled in TMEM),
//               P written as fp16 over its own S columns in TMEM, where the
//               P V MMA reads it as the A operand; final O / l and log-sum-exp.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>

#include "devmath.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace tp {

// Shared with gemm.cu's map encoder: 3-D bf16 map with 128-byte swizzle.
bool make_map_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
                      uint64_t s2_bytes, uint32_t b0, uint32_t b1);

namespace {

constexpr int BQ = 128, BKV = 128, HD = 128;
constexpr int PANEL = 128 * 64 * 2;  // 128 rows x 64 bf16 (one 128-byte swizzle row each)
constexpr int TILE = 2 * PANEL;      // 128 x 128 bf16
constexpr int FWD_THREADS = 320;  // TMA warp, MMA warp, two softmax warpgroups
constexpr int KV_SLOTS = 5;       // K and V tiles share one ring
constexpr int FWD_SMEM = 1024 + (2 + KV_SLOTS) * TILE + 256;
constexpr float kLazyRescale = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum : int { ERR_ATT_PRODUCER = 0x111, ERR_ATT_MMA = 0x112, ERR_ATT_SOFTMAX = 0x113, ERR_ATT_DRAIN = 0x114 };

struct AttnFwdArgs {
  int N, H, hpr, causal;
  int nsb, nkb;          // pairs of 128-row query tiles; 128-row key blocks
  int Gs;                // query heads of a shard per KV head (1: multi-head)
  int64_t dt;            // width of one shard's Q block (and of its O)
  int64_t kcol0, vcol0;  // first column of the shard's K and V blocks in a QKV row
  float scale_log2;      // softmax scale * log2(e)
  uint16_t* O;           // [t][N][dt]
  float* lse;            // [t][hpr][N]
  int* err;
  uint64_t timeout_ns;
};

// K-major 128x128 bf16 tile in two 64-column panels: descriptor of MMA k-step kk (16 columns).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk) {
  return ptx::sdesc_sw128(base + (kk >> 2) * PANEL + (kk & 3) * 32, 16, 1024);
}
// Same tile read MN-major (the 64-column panels are the MN chunks): k-step kk = 16 rows.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int kk) {
  return ptx::sdesc_sw128(base + kk * 2048, PANEL, 1024);
}


template <bool NEG>
__global__ void __launch_bounds__(FWD_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_qkv, const AttnFwdArgs p) {
  extern __shared__ uint8_t dsmem[];
  const uint32_t pad = (1024u - (ptx::smem_addr(dsmem) & 1023u)) & 1023u;
  uint8_t* base = dsmem + pad;
  uint8_t* sQ = base;              // two query tiles
  uint8_t* sKV = base + 2 * TILE;  // ring of KV_SLOTS tiles: K_0, V_0, K_1, V_1, ...
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + (2 + KV_SLOTS) * TILE);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;                 // [KV_SLOTS]
  uint64_t* kv_empty = bars + 1 + KV_SLOTS;     // [KV_SLOTS]
  uint64_t* s_full = bars + 1 + 2 * KV_SLOTS;   // [2] S_b ready in TMEM
  uint64_t* p_full = bars + 3 + 2 * KV_SLOTS;   // [2] P_b written over S_b
  uint64_t* o_full = bars + 5 + 2 * KV_SLOTS;   // [2] last P_b V done
  uint64_t* mma_done = bars + 7 + 2 * KV_SLOTS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8 + 2 * KV_SLOTS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x % p.H;
  const int sb = p.nsb - 1 - static_cast<int>(blockIdx.x / p.H);  // heavy (late) query pairs first
  const int shard = head / p.hpr, jj = head - shard * p.hpr;
  int nkv[2];
#pragma unroll
  for (int b = 0; b < 2; ++b) nkv[b] = p.causal ? min(2 * sb + b + 1, p.nkb) : p.nkb;
  const int nkv_max = nkv[1];  // the later tile sees at least as many key blocks
  const int qcol = jj * HD;
  const int kcol = static_cast<int>(p.kcol0) + (jj / p.Gs) * HD;  // the KV head this query head reads
  const int vcol = static_cast<int>(p.vcol0) + (jj / p.Gs) * HD;

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    for (int s = 0; s < KV_SLOTS; ++s) {
      ptx::mbar_init(&kv_full[s], 1);
      ptx::mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&s_full[b], 1);
      ptx::mbar_init(&p_full[b], 128);
      ptx::mbar_init(&o_full[b], 1);
    }
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncwarp();  // lane-0 roles rejoin their warp: bar.sync needs converged warps
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S_0 | S_1 | O_0 | O_1, 128 each.  P_b (fp16 pairs) overwrites the first 64 columns of S_b.
  const uint32_t tS[2] = {tmem, tmem + 128};
  const uint32_t tO[2] = {tmem + 256, tmem + 384};

  if (warp == 0) {
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_qkv);
      ptx::mbar_arrive_expect_tx(q_full, 2 * TILE);
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        ptx::tma_load_3d(sQ + b * TILE, &tm_qkv, q_full, qcol, (2 * sb + b) * BQ, shard);
        ptx::tma_load_3d(sQ + b * TILE + PANEL, &tm_qkv, q_full, qcol + 64, (2 * sb + b) * BQ, shard);
      }
      int issued = 0;
      for (int i = 0; i < 2 * nkv_max; ++i) {
        const int slot = i % KV_SLOTS;
        const uint32_t ph = (i / KV_SLOTS) & 1;
        if (!ptx::mbar_wait(&kv_empty[slot], ph ^ 1u, abort_flag, p.err, ERR_ATT_PRODUCER, p.timeout_ns)) break;
        const int col = (i & 1) ? vcol : kcol;
        uint8_t* dst = sKV + slot * TILE;
        ptx::mbar_arrive_expect_tx(&kv_full[slot], TILE);
        ptx::tma_load_3d(dst, &tm_qkv, &kv_full[slot], col, (i >> 1) * BKV, shard);
        ptx::tma_load_3d(dst + PANEL, &tm_qkv, &kv_full[slot], col + 64, (i >> 1) * BKV, shard);
        ++issued;
      }
      // drain: every issued copy must land before the CTA exits
      volatile int never = 0;
      ptx::mbar_wait(q_full, 0, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
      for (int i = (issued > KV_SLOTS ? issued - KV_SLOTS : 0); i < issued; ++i)
        ptx::mbar_wait(&kv_full[i % KV_SLOTS], (i / KV_SLOTS) & 1, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = ptx::idesc_f16_f32(BQ, BKV, false, false);
      constexpr uint32_t idesc_o = ptx::idesc_f16_f32(BQ, HD, false, true);
      const uint32_t aQ[2] = {ptx::smem_addr(sQ), ptx::smem_addr(sQ + TILE)};
      const uint32_t aKV = ptx::smem_addr(sKV);
      auto item_ready = [&](int i) {
        return ptx::mbar_wait(&kv_full[i % KV_SLOTS], (i / KV_SLOTS) & 1, abort_flag, p.err, ERR_ATT_MMA,
                              p.timeout_ns);
      };
      auto issue_s = [&](int b, uint32_t aK) {
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          ptx::mma_bf16(tS[b], kmajor_desc(aQ[b], kk), kmajor_desc(aK, kk), idesc_s, kk > 0 ? 1u : 0u);
        ptx::mma_commit(&s_full[b]);
      };
      bool ok = ptx::mbar_wait(q_full, 0, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns) && item_ready(0);
      if (ok) {
        ptx::tc_fence_after();
        issue_s(0, aKV);
        issue_s(1, aKV);
        ptx::mma_commit(&kv_empty[0]);
      }
      // Order per key block j: P_0 V_j, S_0 for block j+1, P_1 V_j, S_1 for block j+1.  A tile's next S
      // overwrites the columns its P occupies; tcgen05 MMAs of one thread run in issue order, so the
      // P V that reads them has finished with them first.
      for (int j = 0; ok && j < nkv_max; ++j) {
        const int iv = 2 * j + 1, ik = 2 * j + 2;
        if (!item_ready(iv)) break;
        bool k_next = false;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          if (j >= nkv[b]) continue;
          if (!ptx::mbar_wait(&p_full[b], j & 1, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t aV = aKV + (iv % KV_SLOTS) * TILE;
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)
            ptx::mma_f16_ts(tO[b], tS[b] + kk * 8, mnmajor_desc(aV, kk), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
          if (j + 1 < nkv[b]) {
            if (!k_next) {
              if (!item_ready(ik)) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              k_next = true;
            }
            issue_s(b, aKV + (ik % KV_SLOTS) * TILE);
          } else {
            ptx::mma_commit(&o_full[b]);
          }
        }
        if (!ok) break;
        ptx::mma_commit(&kv_empty[iv % KV_SLOTS]);
        if (k_next) ptx::mma_commit(&kv_empty[ik % KV_SLOTS]);
      }
      ptx::mma_commit(mma_done);
      volatile int never = 0;
      ptx::mbar_wait(mma_done, 0, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------- softmax rows
    // Warps 2-5 own query tile 0, warps 6-9 tile 1; a warp reads the TMEM lanes
    // of its rank within a warpgroup (warp & 3), one query row per thread.
    const int b = (warp - 2) >> 2;
    const uint32_t tSb = tmem + 128 * b, tOb = tmem + 256 + 128 * b;  // scalars: no local-memory arrays
    const int nkv_b = p.causal ? min(2 * sb + b + 1, p.nkb) : p.nkb;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int qb = 2 * sb + b;
    const int q = qb * BQ + row;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = NEG ? -p.scale_log2 : p.scale_log2;  // > = 0 once S is negated under a negative scale
    // m is the row's reference maximum (log2 domain).  It is raised only when a
    // block's maximum exceeds it by more than kLazyRescale, so most blocks skip the
    // O rescale; P is then at most 2^kLazyRescale, well inside fp16.
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nkv_b; ++j) {
      if (!ptx::mbar_wait(&s_full[b], j & 1, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const int kv0 = j * BKV;
      const bool edge = (p.causal && j == qb) || (kv0 + BKV > p.N);
      // columns c <= lim are visible to this row (key index kv0 + c)
      const int lim = (p.causal ? min(q, p.N - 1) : p.N - 1) - kv0;
      // Pass 1: the block's row maximum, 64 columns at a time (S stays in TMEM,
      // so a thread never holds the whole row: no register spills).
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t r[2][32];
        ptx::tmem_ld32(tSb + lane_base + hf * 64, r[0]);
        ptx::tmem_ld32(tSb + lane_base + hf * 64 + 32, r[1]);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const int c = hf * 64 + e;
          float v = __uint_as_float(r[e >> 5][e & 31]);
          if (NEG) v = -v;
          if (edge && c > lim) v = -INFINITY;
          mx4[e & 3] = fmaxf(mx4[e & 3], v);
        }
      }
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2;
      const float m_new = (mx > m + kLazyRescale) ? mx : m;
      const float alpha = ptx::exp2_approx(m - m_new);  // 0 on the first block (m = -inf), 1 when m stays
      if (j > 0 && __any_sync(0xffffffffu, m_new != m)) {
        // O_b is idle: the P V of block j-1 finished before S_b of block j was committed.
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(tOb + lane_base + c * 32, o);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          ptx::tmem_st32(tOb + lane_base + c * 32, o);
        }
      }
      // Pass 2: P = 2^(S scale - m), 32 columns at a time, written as fp16 pairs
      // over S's first 64 columns.  Chunk h's P lands in columns [16h, 16h + 16),
      // which pass 2 has already read (chunks 0 .. h), so nothing is overwritten early.
      const float neg_m = -m_new;
      float rs4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t r[32];
        ptx::tmem_ld32(tSb + lane_base + h * 32, r);
        ptx::tmem_ld_wait();
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = h * 32 + 2 * e;
          float s0 = __uint_as_float(r[2 * e]), s1 = __uint_as_float(r[2 * e + 1]);
          if (NEG) {
            s0 = -s0;
            s1 = -s1;
          }
          float p0 = ptx::exp2_approx(fmaf(s0, sl2, neg_m));
          float p1 = ptx::exp2_approx(fmaf(s1, sl2, neg_m));
          if (edge) {
            p0 = c <= lim ? p0 : 0.0f;
            p1 = c + 1 <= lim ? p1 : 0.0f;
          }
          rs4[e & 3] += p0 + p1;
          w[e] = pack_f16x2(p0, p1);
        }
        ptx::tmem_st16(tSb + lane_base + h * 16, w);
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&p_full[b]);
      l = fmaf(l, alpha, (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]));
      m = m_new;
    }
    if (ok && ptx::mbar_wait(&o_full[b], 0, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
      ptx::tc_fence_after();
      const float inv_l = 1.0f / l;
      uint16_t* orow = p.O + (static_cast<int64_t>(shard) * p.N + q) * p.dt + qcol;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        ptx::tmem_ld32(tOb + lane_base + c * 32, o);
        ptx::tmem_ld_wait();
        if (q < p.N) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[e + 0]) * inv_l, __uint_as_float(o[e + 1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv_l, __uint_as_float(o[e + 3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv_l, __uint_as_float(o[e + 5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv_l, __uint_as_float(o[e + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + c * 32 + e) = v;
          }
        }
      }
      if (q < p.N) p.lse[(static_cast<int64_t>(shard) * p.hpr + jj) * p.N + q] = (m + __log2f(l)) * kLn2;
    }
  }

  ptx::tc_fence_before();
  __syncwarp();  // lane-0 roles rejoin their warp: bar.sync needs converged warps
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ backward
//
// With P = softmax(scale * Q K^T) recomputed from the saved log-sum-exp and
// D = rowsum(dO * O), the head-local gradients are
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
// Two kernels, no atomics (deterministic): one CTA per (head, key block) for
// dK / dV, looping over query blocks; one CTA per (head, query block) for dQ,
// looping over key blocks.  P and dS are written once into 128B-swizzled
// tiles with the query index as the row; the same bytes are the K-major A
// operand of dQ = dS K and the MN-major A operand of dV = P^T dO and
// dK = dS^T Q, so no transpose is ever materialised.

constexpr int BWD_THREADS = 192;
constexpr int DKV_SMEM = 1024 + 6 * TILE + 256;
constexpr int DQ_SMEM = 1024 + 7 * TILE + 256;

struct AttnBwdArgs {
  int N, H, hpr, nqb, causal;
  int Gs, kv_t, Hkv;     // query heads per KV head in a shard, KV heads per shard, KV heads in all
  int64_t dt;            // width of a shard's Q block (= its O and dO)
  int64_t row_w, kcol0, vcol0;  // QKV row width per shard; first K and V columns
  float scale, scale_log2;
  const float* lse;   // [t][hpr][N] natural log
  const float* Dvec;  // [t][hpr][N]
  uint16_t* dQKV;     // [t][N][row_w]
  int* err;
  uint64_t timeout_ns;
};

// Writes 32 consecutive columns (chunk c of 4) of row `row` into a K-major swizzled tile.
__device__ __forceinline__ void store_chunk_swizzled(uint8_t* tile, int row, int c, const uint32_t (&w)[16]) {
  uint8_t* rowp = tile + (c >> 1) * PANEL + row * 128;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int ch = (c & 1) * 4 + k;
    *reinterpret_cast<uint4*>(rowp + ((ch ^ (row & 7)) << 4)) =
        make_uint4(w[4 * k + 0], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
  }
}

// P and dS for 32 columns of one query row; returns them packed as bf16 pairs.
__device__ __forceinline__ void p_ds_chunk(const uint32_t (&s)[32], const uint32_t (&dp)[32], int q, int kv0,
                                           const AttnBwdArgs& p, float lse2, float Dq, uint32_t (&wp)[16],
                                           uint32_t (&wds)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float pv[2], dv[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int kv = kv0 + e + u;
      const bool valid = q < p.N && kv < p.N && (!p.causal || kv <= q);
      const float pr = valid ? ptx::exp2_approx(__uint_as_float(s[e + u]) * p.scale_log2 - lse2) : 0.0f;
      pv[u] = pr;
      dv[u] = pr * (__uint_as_float(dp[e + u]) - Dq);
    }
    wp[e >> 1] = pack_f16x2(pv[0], pv[1]);
    wds[e >> 1] = pack_f16x2(dv[0], dv[1]);
  }
}

__global__ void attn_bwd_dot_kernel(const uint16_t* __restrict__ dO, const uint16_t* __restrict__ O, int N, int hpr,
                                    int64_t dt, int64_t total, float* __restrict__ Dvec) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= total) return;
  const int64_t i = w / (static_cast<int64_t>(N) * hpr);
  const int64_t rem = w - i * N * hpr;
  const int64_t q = rem / hpr, jj = rem - q * hpr;
  const int64_t off = (i * N + q) * dt + jj * HD + lane * 4;
  const uint2 a = *reinterpret_cast<const uint2*>(dO + off);
  const uint2 b = *reinterpret_cast<const uint2*>(O + off);
  float a0, a1, a2, a3, b0, b1, b2, b3;
  unpack_f16x2(a.x, a0, a1);  // dO is fp16, O is bf16
  unpack_f16x2(a.y, a2, a3);
  unpack_bf16x2(b.x, b0, b1);
  unpack_bf16x2(b.y, b2, b3);
  float sum = a0 * b0 + a1 * b1 + a2 * b2 + a3 * b3;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) Dvec[(i * hpr + jj) * N + q] = sum;
}

// Writes row `grow` (< N) of a 128-column TMEM accumulator, times `mul`, as bf16 at dst.
__device__ __forceinline__ void tmem_row_to_bf16(uint32_t taddr, float mul, uint16_t* dst, bool write) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t r[32];
    ptx::tmem_ld32(taddr + c * 32, r);
    ptx::tmem_ld_wait();
    if (write) {
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        uint4 v;
        v.x = pack_bf16x2(__uint_as_float(r[e + 0]) * mul, __uint_as_float(r[e + 1]) * mul);
        v.y = pack_bf16x2(__uint_as_float(r[e + 2]) * mul, __uint_as_float(r[e + 3]) * mul);
        v.z = pack_bf16x2(__uint_as_float(r[e + 4]) * mul, __uint_as_float(r[e + 5]) * mul);
        v.w = pack_bf16x2(__uint_as_float(r[e + 6]) * mul, __uint_as_float(r[e + 7]) * mul);
        *reinterpret_cast<uint4*>(dst + c * 32 + e) = v;
      }
    }
  }
}

__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                        const AttnBwdArgs p) {
  extern __shared__ uint8_t dsmem[];
  const uint32_t pad = (1024u - (ptx::smem_addr(dsmem) & 1023u)) & 1023u;
  uint8_t* base = dsmem + pad;
  uint8_t* sK = base;
  uint8_t* sV = base + TILE;
  uint8_t* sQ = base + 2 * TILE;
  uint8_t* sdO = base + 3 * TILE;
  uint8_t* sP = base + 4 * TILE;
  uint8_t* sdS = base + 5 * TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + 6 * TILE);
  uint64_t* kv_full = bars + 0;
  uint64_t* qdo_full = bars + 1;
  uint64_t* qdo_empty = bars + 2;
  uint64_t* sdp_full = bars + 3;
  uint64_t* sdp_free = bars + 4;
  uint64_t* pds_full = bars + 5;
  uint64_t* pds_free = bars + 6;
  uint64_t* mma_done = bars + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // One CTA per (KV head, key block): dK and dV sum over the query heads of
  // the KV head's group on this shard, so the loop runs over (group head,
  // query block) pairs and the TMEM accumulators carry across all of them.
  const int kvh = blockIdx.x % p.Hkv;
  const int kb = static_cast<int>(blockIdx.x / p.Hkv);  // early key blocks see the most query blocks (causal)
  const int shard = kvh / p.kv_t, jl = kvh - shard * p.kv_t;
  const int q_first = p.causal ? kb : 0;
  const int nq = p.nqb - q_first;
  const int nloop = nq * p.Gs;
  const int kcol = static_cast<int>(p.kcol0) + jl * HD, vcol = static_cast<int>(p.vcol0) + jl * HD;

  if (threadIdx.x == 0) {
    ptx::mbar_init(kv_full, 1);
    ptx::mbar_init(qdo_full, 1);
    ptx::mbar_init(qdo_empty, 1);
    ptx::mbar_init(sdp_full, 1);
    ptx::mbar_init(sdp_free, 128);
    ptx::mbar_init(pds_full, 128);
    ptx::mbar_init(pds_free, 1);
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncwarp();  // lane-0 roles rejoin their warp: bar.sync needs converged warps
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;

  if (warp == 0) {
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_qkv);
      ptx::tma_prefetch_desc(&tm_do);
      ptx::mbar_arrive_expect_tx(kv_full, 2 * TILE);
      ptx::tma_load_3d(sK, &tm_qkv, kv_full, kcol, kb * BKV, shard);
      ptx::tma_load_3d(sK + PANEL, &tm_qkv, kv_full, kcol + 64, kb * BKV, shard);
      ptx::tma_load_3d(sV, &tm_qkv, kv_full, vcol, kb * BKV, shard);
      ptx::tma_load_3d(sV + PANEL, &tm_qkv, kv_full, vcol + 64, kb * BKV, shard);
      int issued = 0;
      for (int n = 0; n < nloop; ++n) {
        const int g = n / nq, qi = q_first + (n - g * nq);
        const int qcol = (jl * p.Gs + g) * HD;
        if (!ptx::mbar_wait(qdo_empty, (n & 1) ^ 1u, abort_flag, p.err, ERR_ATT_PRODUCER, p.timeout_ns)) break;
        ptx::mbar_arrive_expect_tx(qdo_full, 2 * TILE);
        ptx::tma_load_3d(sQ, &tm_qkv, qdo_full, qcol, qi * BQ, shard);
        ptx::tma_load_3d(sQ + PANEL, &tm_qkv, qdo_full, qcol + 64, qi * BQ, shard);
        ptx::tma_load_3d(sdO, &tm_do, qdo_full, qcol, qi * BQ, shard);
        ptx::tma_load_3d(sdO + PANEL, &tm_do, qdo_full, qcol + 64, qi * BQ, shard);
        ++issued;
      }
      volatile int never = 0;
      ptx::mbar_wait(kv_full, 0, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
      if (issued > 0) ptx::mbar_wait(qdo_full, (issued - 1) & 1, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_kk = ptx::idesc_f16_f32(128, 128, false, false);  // S, dP
      constexpr uint32_t idesc_mm = ptx::idesc_f16_f32(128, 128, true, true);    // dV, dK
      const uint32_t aK = ptx::smem_addr(sK), aV = ptx::smem_addr(sV), aQ = ptx::smem_addr(sQ);
      const uint32_t adO = ptx::smem_addr(sdO), aP = ptx::smem_addr(sP), adS = ptx::smem_addr(sdS);
      bool ok = ptx::mbar_wait(kv_full, 0, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns);
      for (int n = 0; ok && n < nloop; ++n) {
        if (!ptx::mbar_wait(qdo_full, n & 1, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns)) break;
        if (n >= 1 && !ptx::mbar_wait(sdp_free, (n - 1) & 1, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns)) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tS, kmajor_desc(aQ, kk), kmajor_desc(aK, kk), idesc_kk, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tdP, kmajor_desc(adO, kk), kmajor_desc(aV, kk), idesc_kk, kk > 0 ? 1u : 0u);
        ptx::mma_commit(sdp_full);
        if (!ptx::mbar_wait(pds_full, n & 1, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns)) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tdV, mnmajor_desc(aP, kk), mnmajor_desc(adO, kk), idesc_mm, (n > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tdK, mnmajor_desc(adS, kk), mnmajor_desc(aQ, kk), idesc_mm, (n > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(pds_free);
        ptx::mma_commit(qdo_empty);
      }
      ptx::mma_commit(mma_done);
      volatile int never = 0;
      ptx::mbar_wait(mma_done, 0, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
    }
  } else {
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    bool ok = true;
    for (int n = 0; n < nloop; ++n) {
      const int g = n / nq;
      const int64_t vec_base = (static_cast<int64_t>(shard) * p.hpr + jl * p.Gs + g) * p.N;
      const int q = (q_first + (n - g * nq)) * BQ + row;
      const float lse2 = q < p.N ? p.lse[vec_base + q] * kLog2e : 0.0f;
      const float Dq = q < p.N ? p.Dvec[vec_base + q] : 0.0f;
      if (!ptx::mbar_wait(sdp_full, n & 1, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
        ok = false;
        break;
      }
      if (n >= 1 && !ptx::mbar_wait(pds_free, (n - 1) & 1, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t s[32], dp[32], wp[16], wds[16];
        ptx::tmem_ld32(tS + lane_base + c * 32, s);
        ptx::tmem_ld32(tdP + lane_base + c * 32, dp);
        ptx::tmem_ld_wait();
        p_ds_chunk(s, dp, q, kb * BKV + c * 32, p, lse2, Dq, wp, wds);
        store_chunk_swizzled(sP, row, c, wp);
        store_chunk_swizzled(sdS, row, c, wds);
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(sdp_free);
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(pds_full);
    }
    if (ok && nloop > 0 &&
        ptx::mbar_wait(pds_free, (nloop - 1) & 1, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
      ptx::tc_fence_after();
      const int kvrow = kb * BKV + row;  // accumulator rows are key rows
      uint16_t* drow = p.dQKV + (static_cast<int64_t>(shard) * p.N + kvrow) * p.row_w;
      tmem_row_to_bf16(tdV + lane_base, 1.0f, drow + vcol, kvrow < p.N);
      tmem_row_to_bf16(tdK + lane_base, p.scale, drow + kcol, kvrow < p.N);
    }
  }

  ptx::tc_fence_before();
  __syncwarp();  // lane-0 roles rejoin their warp: bar.sync needs converged warps
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                       const AttnBwdArgs p) {
  extern __shared__ uint8_t dsmem[];
  const uint32_t pad = (1024u - (ptx::smem_addr(dsmem) & 1023u)) & 1023u;
  uint8_t* base = dsmem + pad;
  uint8_t* sQ = base;
  uint8_t* sdO = base + TILE;
  uint8_t* sK = base + 2 * TILE;  // 2 stages
  uint8_t* sV = base + 4 * TILE;  // 2 stages
  uint8_t* sdS = base + 6 * TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + 7 * TILE);
  uint64_t* qdo_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [2]
  uint64_t* v_full = bars + 3;    // [2]
  uint64_t* kv_empty = bars + 5;  // [2]
  uint64_t* sdp_full = bars + 7;
  uint64_t* sdp_free = bars + 8;
  uint64_t* ds_full = bars + 9;
  uint64_t* ds_free = bars + 10;
  uint64_t* mma_done = bars + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x % p.H;
  const int qb = p.nqb - 1 - static_cast<int>(blockIdx.x / p.H);
  const int shard = head / p.hpr, jj = head - shard * p.hpr;
  const int nkv = p.causal ? qb + 1 : (p.N + BKV - 1) / BKV;
  const int qcol = jj * HD;
  const int kcol = static_cast<int>(p.kcol0) + (jj / p.Gs) * HD, vcol = static_cast<int>(p.vcol0) + (jj / p.Gs) * HD;

  if (threadIdx.x == 0) {
    ptx::mbar_init(qdo_full, 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&k_full[s], 1);
      ptx::mbar_init(&v_full[s], 1);
      ptx::mbar_init(&kv_empty[s], 1);
    }
    ptx::mbar_init(sdp_full, 1);
    ptx::mbar_init(sdp_free, 128);
    ptx::mbar_init(ds_full, 128);
    ptx::mbar_init(ds_free, 1);
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncwarp();  // lane-0 roles rejoin their warp: bar.sync needs converged warps
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tdP = tmem + 128, tdQ = tmem + 256;

  if (warp == 0) {
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_qkv);
      ptx::tma_prefetch_desc(&tm_do);
      ptx::mbar_arrive_expect_tx(qdo_full, 2 * TILE);
      ptx::tma_load_3d(sQ, &tm_qkv, qdo_full, qcol, qb * BQ, shard);
      ptx::tma_load_3d(sQ + PANEL, &tm_qkv, qdo_full, qcol + 64, qb * BQ, shard);
      ptx::tma_load_3d(sdO, &tm_do, qdo_full, jj * HD, qb * BQ, shard);
      ptx::tma_load_3d(sdO + PANEL, &tm_do, qdo_full, jj * HD + 64, qb * BQ, shard);
      int issued = 0;
      for (int j = 0; j < nkv; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!ptx::mbar_wait(&kv_empty[st], ph ^ 1u, abort_flag, p.err, ERR_ATT_PRODUCER, p.timeout_ns)) break;
        ptx::mbar_arrive_expect_tx(&k_full[st], TILE);
        ptx::tma_load_3d(sK + st * TILE, &tm_qkv, &k_full[st], kcol, j * BKV, shard);
        ptx::tma_load_3d(sK + st * TILE + PANEL, &tm_qkv, &k_full[st], kcol + 64, j * BKV, shard);
        ptx::mbar_arrive_expect_tx(&v_full[st], TILE);
        ptx::tma_load_3d(sV + st * TILE, &tm_qkv, &v_full[st], vcol, j * BKV, shard);
        ptx::tma_load_3d(sV + st * TILE + PANEL, &tm_qkv, &v_full[st], vcol + 64, j * BKV, shard);
        ++issued;
      }
      volatile int never = 0;
      ptx::mbar_wait(qdo_full, 0, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
      for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j) {
        const uint32_t ph = (j >> 1) & 1;
        ptx::mbar_wait(&k_full[j & 1], ph, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
        ptx::mbar_wait(&v_full[j & 1], ph, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_kk = ptx::idesc_f16_f32(128, 128, false, false);  // S, dP
      constexpr uint32_t idesc_q = ptx::idesc_f16_f32(128, 128, false, true);    // dQ = dS K
      const uint32_t aQ = ptx::smem_addr(sQ), adO = ptx::smem_addr(sdO), adS = ptx::smem_addr(sdS);
      bool ok = ptx::mbar_wait(qdo_full, 0, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns);
      for (int j = 0; ok && j < nkv; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!ptx::mbar_wait(&k_full[st], ph, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns)) break;
        if (!ptx::mbar_wait(&v_full[st], ph, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns)) break;
        if (j >= 1 && !ptx::mbar_wait(sdp_free, (j - 1) & 1, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns)) break;
        ptx::tc_fence_after();
        const uint32_t aK = ptx::smem_addr(sK + st * TILE), aV = ptx::smem_addr(sV + st * TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tS, kmajor_desc(aQ, kk), kmajor_desc(aK, kk), idesc_kk, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tdP, kmajor_desc(adO, kk), kmajor_desc(aV, kk), idesc_kk, kk > 0 ? 1u : 0u);
        ptx::mma_commit(sdp_full);
        if (!ptx::mbar_wait(ds_full, j & 1, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns)) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tdQ, kmajor_desc(adS, kk), mnmajor_desc(aK, kk), idesc_q, (j > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(ds_free);
        ptx::mma_commit(&kv_empty[st]);
      }
      ptx::mma_commit(mma_done);
      volatile int never = 0;
      ptx::mbar_wait(mma_done, 0, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
    }
  } else {
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int q = qb * BQ + row;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int64_t vec_base = (static_cast<int64_t>(shard) * p.hpr + jj) * p.N;
    const float lse2 = q < p.N ? p.lse[vec_base + q] * kLog2e : 0.0f;
    const float Dq = q < p.N ? p.Dvec[vec_base + q] : 0.0f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      if (!ptx::mbar_wait(sdp_full, j & 1, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
        ok = false;
        break;
      }
      if (j >= 1 && !ptx::mbar_wait(ds_free, (j - 1) & 1, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t s[32], dp[32], wp[16], wds[16];
        ptx::tmem_ld32(tS + lane_base + c * 32, s);
        ptx::tmem_ld32(tdP + lane_base + c * 32, dp);
        ptx::tmem_ld_wait();
        p_ds_chunk(s, dp, q, j * BKV + c * 32, p, lse2, Dq, wp, wds);
        store_chunk_swizzled(sdS, row, c, wds);
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(sdp_free);
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(ds_full);
    }
    if (ok && ptx::mbar_wait(ds_free, (nkv - 1) & 1, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
      ptx::tc_fence_after();
      uint16_t* drow = p.dQKV + (static_cast<int64_t>(shard) * p.N + q) * p.row_w;
      tmem_row_to_bf16(tdQ + lane_base, p.scale, drow + qcol, q < p.N);
    }
  }

  ptx::tc_fence_before();
  __syncwarp();  // lane-0 roles rejoin their warp: bar.sync needs converged warps
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

// Shape of a shard's QKV row under grouped-query sharding (n_kv = n_heads:
// multi-head): q_t query heads, kv_t KV heads, Gs query heads per KV head.
struct AttnShape {
  int q_t, kv_t, Gs;
  int64_t dt, row_w, kcol0, vcol0;
};

bool attn_shape(int64_t d, int n_heads, int n_kv, int head_dim, int t, AttnShape& a) {
  if (head_dim != HD || t < 1 || n_heads < 1 || n_kv < 1) return false;
  if (static_cast<int64_t>(n_heads) * head_dim != d || n_heads % t != 0 || n_heads % n_kv != 0) return false;
  if (n_kv >= t ? (n_kv % t != 0) : (t % n_kv != 0)) return false;
  a.q_t = n_heads / t;
  a.kv_t = n_kv >= t ? n_kv / t : 1;
  const int G = n_heads / n_kv;
  a.Gs = G < a.q_t ? G : a.q_t;
  a.dt = static_cast<int64_t>(a.q_t) * HD;
  a.row_w = static_cast<int64_t>(a.q_t + 2 * a.kv_t) * HD;
  a.kcol0 = a.dt;
  a.vcol0 = a.dt + static_cast<int64_t>(a.kv_t) * HD;
  return true;
}

tp_status run_attention_fwd(const uint16_t* QKV, int64_t N, int64_t d, int n_heads, int n_kv, int head_dim, int t,
                            int causal, float scale, uint16_t* O, float* lse, cudaStream_t s) {
  if (N < 0 || d < 1 || n_heads < 1 || n_kv < 1 || t < 1) return TP_ERR_INVALID_ARG;
  AttnShape sh;
  if (!attn_shape(d, n_heads, n_kv, head_dim, t, sh)) return TP_ERR_SHAPE;
  if (N == 0) return TP_OK;
  if (!QKV || !O || !lse) return TP_ERR_INVALID_ARG;
  if (!aligned16(QKV) || !aligned16(O)) return TP_ERR_ALIGN;
  if (N > (1LL << 30) / 1) return TP_ERR_SHAPE;
  TP_RETURN_IF(ready());
  CUtensorMap map;
  if (!make_map_3d_bf16(&map, QKV, sh.row_w, N, t, sh.row_w * 2, N * sh.row_w * 2, 64, 128)) return TP_ERR_CUDA;
  AttnFwdArgs a{};
  a.N = static_cast<int>(N);
  a.H = n_heads;
  a.hpr = n_heads / t;
  a.nkb = static_cast<int>((N + BKV - 1) / BKV);
  a.nsb = (a.nkb + 1) / 2;
  a.causal = causal ? 1 : 0;
  a.Gs = sh.Gs;
  a.dt = sh.dt;
  a.kcol0 = sh.kcol0;
  a.vcol0 = sh.vcol0;
  a.scale_log2 = scale * kLog2e;
  a.O = O;
  a.lse = lse;
  a.err = device_error_word();
  a.timeout_ns = wait_timeout_ns();
  static bool configured[64] = {};
  int dev = 0;
  TP_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return TP_ERR_CUDA;
  if (!configured[dev]) {
    TP_CUDA_CHECK(
        cudaFuncSetAttribute(attn_fwd_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, FWD_SMEM));
    TP_CUDA_CHECK(
        cudaFuncSetAttribute(attn_fwd_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, FWD_SMEM));
    configured[dev] = true;
  }
  const int64_t grid = static_cast<int64_t>(n_heads) * a.nsb;
  if (grid > 0x7fffffff) return TP_ERR_SHAPE;
  if (a.scale_log2 < 0.0f)
    attn_fwd_kernel<true><<<static_cast<unsigned>(grid), FWD_THREADS, FWD_SMEM, s>>>(map, a);
  else
    attn_fwd_kernel<false><<<static_cast<unsigned>(grid), FWD_THREADS, FWD_SMEM, s>>>(map, a);
  TP_LAUNCHED();
  return TP_OK;
}

}  // namespace tp

namespace tp {

tp_status run_attention_bwd(const uint16_t* QKV, const uint16_t* O, const uint16_t* dO, const float* lse, int64_t N,
                            int64_t d, int n_heads, int n_kv, int head_dim, int t, int causal, float scale, float* Dvec,
                            uint16_t* dQKV, cudaStream_t s) {
  if (N < 0 || d < 1 || n_heads < 1 || n_kv < 1 || t < 1) return TP_ERR_INVALID_ARG;
  AttnShape sh;
  if (!attn_shape(d, n_heads, n_kv, head_dim, t, sh)) return TP_ERR_SHAPE;
  if (N == 0) return TP_OK;
  if (!QKV || !O || !dO || !lse || !Dvec || !dQKV) return TP_ERR_INVALID_ARG;
  if (!aligned16(QKV) || !aligned16(O) || !aligned16(dO) || !aligned16(dQKV)) return TP_ERR_ALIGN;
  TP_RETURN_IF(ready());
  const int64_t dt = sh.dt;
  const int hpr = n_heads / t;
  CUtensorMap m_qkv, m_do;
  if (!make_map_3d_bf16(&m_qkv, QKV, sh.row_w, N, t, sh.row_w * 2, N * sh.row_w * 2, 64, 128)) return TP_ERR_CUDA;
  if (!make_map_3d_bf16(&m_do, dO, dt, N, t, dt * 2, N * dt * 2, 64, 128)) return TP_ERR_CUDA;
  const int64_t rows = static_cast<int64_t>(t) * N * hpr;
  attn_bwd_dot_kernel<<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, s>>>(dO, O, static_cast<int>(N), hpr,
                                                                                     dt, rows, Dvec);
  TP_LAUNCHED();
  AttnBwdArgs a{};
  a.N = static_cast<int>(N);
  a.H = n_heads;
  a.hpr = hpr;
  a.nqb = static_cast<int>((N + BQ - 1) / BQ);
  a.causal = causal ? 1 : 0;
  a.Gs = sh.Gs;
  a.kv_t = sh.kv_t;
  a.Hkv = t * sh.kv_t;
  a.dt = dt;
  a.row_w = sh.row_w;
  a.kcol0 = sh.kcol0;
  a.vcol0 = sh.vcol0;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.lse = lse;
  a.Dvec = Dvec;
  a.dQKV = dQKV;
  a.err = device_error_word();
  a.timeout_ns = wait_timeout_ns();
  static bool configured[64] = {};
  int dev = 0;
  TP_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return TP_ERR_CUDA;
  if (!configured[dev]) {
    TP_CUDA_CHECK(cudaFuncSetAttribute(attn_bwd_dkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DKV_SMEM));
    TP_CUDA_CHECK(cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DQ_SMEM));
    configured[dev] = true;
  }
  const unsigned grid_kv = static_cast<unsigned>(static_cast<int64_t>(a.Hkv) * a.nqb);
  attn_bwd_dkv_kernel<<<grid_kv, BWD_THREADS, DKV_SMEM, s>>>(m_qkv, m_do, a);
  TP_LAUNCHED();
  const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(n_heads) * a.nqb);
  attn_bwd_dq_kernel<<<grid, BWD_THREADS, DQ_SMEM, s>>>(m_qkv, m_do, a);
  TP_LAUNCHED();
  return TP_OK;
}

}  // namespace tp
