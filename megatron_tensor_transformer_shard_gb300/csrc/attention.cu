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
// at the same cost.  O stays bf16; dQKV is bf16, or fp16 for callers whose attention
// input and W_qkv are fp16 (the QKV GEMM's operands set the precision of Q and K).
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

// Packed two-lane fp32 arithmetic (one instruction for two values) and a three-input
// maximum: the softmax of an interior key block is bound by instruction issue, not by the
// exponential unit, so these cut its instruction count per score.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
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
  return ptx::sdesc_at(ptx::sdesc_sw128(base, 16, 1024), (kk >> 2) * PANEL + (kk & 3) * 32);
}
// Same tile read MN-major (the 64-column panels are the MN chunks): k-step kk = 16 rows.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int kk) {
  return ptx::sdesc_at(ptx::sdesc_sw128(base, PANEL, 1024), kk * 2048);
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
  // Programmatic dependent launch: set-up above overlapped the previous kernel's tail;
  // nothing it writes is read before this wait.
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
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
      const bool plain = !NEG && !edge;  // interior block: no negation, no mask
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t r[2][32];
        ptx::tmem_ld32(tSb + lane_base + hf * 64, r[0]);
        ptx::tmem_ld32(tSb + lane_base + hf * 64 + 32, r[1]);
        ptx::tmem_ld_wait();
        if (plain) {
#pragma unroll
          for (int e = 0; e < 64; e += 8) {
            const uint32_t* x = &r[e >> 5][e & 31];
            mx4[0] = max3f(mx4[0], __uint_as_float(x[0]), __uint_as_float(x[1]));
            mx4[1] = max3f(mx4[1], __uint_as_float(x[2]), __uint_as_float(x[3]));
            mx4[2] = max3f(mx4[2], __uint_as_float(x[4]), __uint_as_float(x[5]));
            mx4[3] = max3f(mx4[3], __uint_as_float(x[6]), __uint_as_float(x[7]));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) {
            const int c = hf * 64 + e;
            float v = __uint_as_float(r[e >> 5][e & 31]);
            if (NEG) v = -v;
            if (edge && c > lim) v = -INFINITY;
            mx4[e & 3] = fmaxf(mx4[e & 3], v);
          }
        }
      }
      const float mx = max3f(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3])) * sl2;
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
      if (plain) {
        // two scores per instruction: x = s scale - m and the running row sums, packed
        const uint64_t sl2x2 = f2_pack(sl2, sl2), negm2 = f2_pack(neg_m, neg_m);
        uint64_t rs2[2] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f)};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t r[32];
          ptx::tmem_ld32(tSb + lane_base + h * 32, r);
          ptx::tmem_ld_wait();
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint64_t x2 =
                f2_fma(f2_pack(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1])), sl2x2, negm2);
            float x0, x1;
            f2_unpack(x2, x0, x1);
            const float p0 = ptx::exp2_approx(x0), p1 = ptx::exp2_approx(x1);
            rs2[e & 1] = f2_add(rs2[e & 1], f2_pack(p0, p1));
            w[e] = pack_f16x2(p0, p1);
          }
          ptx::tmem_st16(tSb + lane_base + h * 16, w);
        }
        f2_unpack(rs2[0], rs4[0], rs4[1]);
        f2_unpack(rs2[1], rs4[2], rs4[3]);
      }
#pragma unroll
      for (int h = 0; h < (plain ? 0 : 4); ++h) {
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
// Two kernels, no atomics (deterministic):
//   dK / dV: one CTA per (KV head, 128-key block), looping over 64-row query
//     blocks of the group's query heads.  It forms S^T = K Q^T and dP^T = V dO^T
//     with the keys on the TMEM lanes, so P^T and dS^T (fp16, written over their
//     own S^T / dP^T columns) are the TMEM A operands of dV += P^T dO and
//     dK += dS^T Q.
//   dQ: one CTA per (head, 128-query block), looping over 64-key blocks: S and dP
//     with the queries on the lanes, dS in TMEM as the A operand of dQ += dS K.
// S^T / dP^T (S / dP) are double-buffered in TMEM: the MMAs of block n+1 run
// while eight warps turn block n into P and dS.  Each of those warps reads 32
// of the 64 columns of its lane quarter and writes its fp16 results into the
// first half of the columns it read, so k-step kk (16 elements) of such an A
// operand starts at column 32 (kk / 2) + 8 (kk % 2).

constexpr int BWD_THREADS = 320;       // TMA warp, MMA warp, eight compute warps
constexpr int BWD_STAGES = 4;
constexpr int PANEL64 = 64 * 64 * 2;   // 64 rows x 64 fp16 (one 128-byte swizzle row each)
constexpr int TILE64 = 2 * PANEL64;    // 64 x 128 fp16
constexpr int DKV_SMEM = 1024 + 2 * TILE + BWD_STAGES * (2 * TILE64 + 512) + 256;
constexpr int DQ_SMEM = 1024 + 2 * TILE + BWD_STAGES * 2 * TILE64 + 256;

struct AttnBwdArgs {
  int N, H, hpr, nqb, causal;
  int nb64;              // 64-row blocks of the sequence
  int Gs, kv_t, Hkv;     // query heads per KV head in a shard, KV heads per shard, KV heads in all
  int64_t dt;            // width of a shard's Q block (= its O and dO)
  int64_t row_w, kcol0, vcol0;  // QKV row width per shard; first K and V columns
  float scale, scale_log2;
  const float* lse;   // [t][hpr][N] natural log
  const float* Dvec;  // [t][hpr][N]
  uint16_t* dQKV;     // [t][N][row_w]
  int dqkv_f16;       // dQKV as IEEE fp16 (else bf16)
  int* err;
  uint64_t timeout_ns;
};

// K-major 64-row tile in two 64-column panels: descriptor of MMA k-step kk (16 columns).
__device__ __forceinline__ uint64_t kmajor64_desc(uint32_t base, int kk) {
  return ptx::sdesc_at(ptx::sdesc_sw128(base, 16, 1024), (kk >> 2) * PANEL64 + (kk & 3) * 32);
}
// The same tile read MN-major: k-step kk = rows 16 kk .. 16 kk + 15.
__device__ __forceinline__ uint64_t mnmajor64_desc(uint32_t base, int kk) {
  return ptx::sdesc_at(ptx::sdesc_sw128(base, PANEL64, 1024), kk * 2048);
}
// TMEM column of k-step kk of an fp16 A operand written by the two column halves.
__device__ __forceinline__ uint32_t half_split_col(int kk) { return (kk >> 1) * 32 + (kk & 1) * 8; }

// Loads a 128-row, 128-column fp16 tile as four 64 x 64 boxes (same bytes as one 128-row box).
__device__ __forceinline__ void tma_tile128(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int col, int row,
                                            int shard) {
#pragma unroll
  for (int pnl = 0; pnl < 2; ++pnl)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr)
      ptx::tma_load_3d(dst + pnl * PANEL + hr * PANEL64, map, bar, col + 64 * pnl, row + 64 * hr, shard);
}
// A 64-row, 128-column fp16 tile as two 64 x 64 boxes.
__device__ __forceinline__ void tma_tile64(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int col, int row,
                                           int shard) {
  ptx::tma_load_3d(dst, map, bar, col, row, shard);
  ptx::tma_load_3d(dst + PANEL64, map, bar, col + 64, row, shard);
}

// 64 accumulator columns of this thread's TMEM lane, times `mul`, as bf16 (or IEEE fp16 when
// f16) at dst.
__device__ __forceinline__ void tmem_cols64_to_16(uint32_t taddr, float mul, uint16_t* dst, bool write, bool f16) {
  uint32_t r[2][32];
  ptx::tmem_ld32(taddr, r[0]);
  ptx::tmem_ld32(taddr + 32, r[1]);
  ptx::tmem_ld_wait();
  if (!write) return;
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int e = 0; e < 32; e += 8) {
      float f[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) f[k] = __uint_as_float(r[c][e + k]) * mul;
      uint4 v;
      if (f16) {
        v = make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]), pack_f16x2(f[6], f[7]));
      } else {
        v = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                       pack_bf16x2(f[6], f[7]));
      }
      *reinterpret_cast<uint4*>(dst + c * 32 + e) = v;
    }
}

// D[i][jj][q] = rowsum(dO * O) over head jj's 128 columns.  One warp per (shard, query)
// row: a lane reads 8 consecutive columns (16 bytes of dO and of O), so a pass covers two
// heads and each head's sum is a reduction over 16 lanes.
__global__ void attn_bwd_dot_kernel(const uint16_t* __restrict__ dO, const uint16_t* __restrict__ O, int N, int hpr,
                                    int64_t dt, int64_t rows, float* __restrict__ Dvec) {
  ptx::griddep_wait();  // dO comes from the previous kernel
  ptx::griddep_launch_dependents();
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= rows) return;
  const int64_t i = w / N, q = w - i * N;
  const uint16_t* drow = dO + w * dt;
  const uint16_t* orow = O + w * dt;
  for (int64_t c0 = 0; c0 < dt; c0 += 256) {
    const int64_t c = c0 + lane * 8;
    float sum = 0.0f;
    if (c < dt) {
      const uint4 a = *reinterpret_cast<const uint4*>(drow + c);
      const uint4 b = *reinterpret_cast<const uint4*>(orow + c);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float a0, a1, b0, b1;
        unpack_f16x2(aw[k], a0, a1);  // dO is fp16, O is bf16
        unpack_bf16x2(bw[k], b0, b1);
        sum = fmaf(a0, b0, sum);
        sum = fmaf(a1, b1, sum);
      }
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if ((lane & 15) == 0 && c < dt) {
      const int64_t jj = c / HD;
      Dvec[(i * hpr + jj) * N + q] = sum;
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
  uint8_t* sQd = base + 2 * TILE;  // stage s: Q_n at s * 2 TILE64, dO_n after it
  float* sLD = reinterpret_cast<float*>(base + 2 * TILE + BWD_STAGES * 2 * TILE64);  // stage s: -lse2[64], -D[64]
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + 2 * TILE + BWD_STAGES * (2 * TILE64 + 512));
  uint64_t* kv_full = bars + 0;
  uint64_t* qd_full = bars + 1;                    // [BWD_STAGES] TMA bytes + 32 lse/D writers
  uint64_t* qd_empty = bars + 1 + BWD_STAGES;      // [BWD_STAGES]
  uint64_t* st_full = bars + 1 + 2 * BWD_STAGES;   // [2] S^T, dP^T of a block in TMEM
  uint64_t* pds_full = bars + 3 + 2 * BWD_STAGES;  // [2] P^T, dS^T written
  uint64_t* acc_done = bars + 5 + 2 * BWD_STAGES;
  uint64_t* mma_done = bars + 6 + 2 * BWD_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 7 + 2 * BWD_STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // One CTA per (KV head, key block): dK and dV sum over the query heads of
  // the KV head's group on this shard, so the loop runs over (group head,
  // query block) pairs and the TMEM accumulators carry across all of them.
  const int kvh = blockIdx.x % p.Hkv;
  const int kb = static_cast<int>(blockIdx.x / p.Hkv);  // early key blocks see the most query blocks (causal)
  const int shard = kvh / p.kv_t, jl = kvh - shard * p.kv_t;
  const int q_first = p.causal ? 2 * kb : 0;  // first 64-row query block that sees this key block
  const int nq = p.nb64 - q_first;
  const int nloop = nq * p.Gs;
  const int kcol = static_cast<int>(p.kcol0) + jl * HD, vcol = static_cast<int>(p.vcol0) + jl * HD;

  if (threadIdx.x == 0) {
    ptx::mbar_init(kv_full, 1);
    for (int s = 0; s < BWD_STAGES; ++s) {
      ptx::mbar_init(&qd_full[s], 33);
      ptx::mbar_init(&qd_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&st_full[b], 1);
      ptx::mbar_init(&pds_full[b], 256);
    }
    ptx::mbar_init(acc_done, 1);
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncwarp();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Programmatic dependent launch: set-up above overlapped the previous kernel's tail;
  // nothing it writes is read before this wait.
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  // TMEM columns: S^T_0 | S^T_1 (64 each) | dP^T_0 | dP^T_1 (64 each) | dV (128) | dK (128).
  const uint32_t tdV = tmem + 256, tdK = tmem + 384;

  if (warp == 0) {
    // Producer warp: lane 0 issues the tile copies, all 32 lanes stage lse2 / D.
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_qkv);
      ptx::tma_prefetch_desc(&tm_do);
      ptx::mbar_arrive_expect_tx(kv_full, 2 * TILE);
      tma_tile128(sK, &tm_qkv, kv_full, kcol, kb * BKV, shard);
      tma_tile128(sV, &tm_qkv, kv_full, vcol, kb * BKV, shard);
    }
    int issued = 0;
    for (int n = 0; n < nloop; ++n) {
      const int slot = n % BWD_STAGES;
      bool ok = true;
      if (lane == 0)
        ok = ptx::mbar_wait(&qd_empty[slot], ((n / BWD_STAGES) & 1) ^ 1u, abort_flag, p.err, ERR_ATT_PRODUCER,
                            p.timeout_ns);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      __syncwarp();
      const int g = n / nq, qi = q_first + (n - g * nq);
      const int qh = jl * p.Gs + g;
      const int q0 = qi * 64;
      uint8_t* dst = sQd + slot * 2 * TILE64;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&qd_full[slot], 2 * TILE64);
        tma_tile64(dst, &tm_qkv, &qd_full[slot], qh * HD, q0, shard);
        tma_tile64(dst + TILE64, &tm_do, &qd_full[slot], qh * HD, q0, shard);
      }
      const int64_t vec = (static_cast<int64_t>(shard) * p.hpr + qh) * p.N;
      float* ld = sLD + slot * 128;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int idx = lane + 32 * k, q = q0 + idx;
        // Stored negated (the compute warps add them).  A query row past the end gets
        // lse = +inf: its P and dS are exactly 0.
        ld[idx] = q < p.N ? -(p.lse[vec + q] * kLog2e) : -INFINITY;
        ld[64 + idx] = q < p.N ? -p.Dvec[vec + q] : 0.0f;
      }
      ptx::mbar_arrive(&qd_full[slot]);
      ++issued;
    }
    __syncwarp();
    if (lane == 0) {
      volatile int never = 0;
      ptx::mbar_wait(kv_full, 0, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
      for (int n = (issued > BWD_STAGES ? issued - BWD_STAGES : 0); n < issued; ++n)
        ptx::mbar_wait(&qd_full[n % BWD_STAGES], (n / BWD_STAGES) & 1, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_st = ptx::idesc_f16_f32(128, 64, false, false);   // S^T, dP^T
      constexpr uint32_t idesc_acc = ptx::idesc_f16_f32(128, 128, false, true);  // dV, dK
      const uint32_t aK = ptx::smem_addr(sK), aV = ptx::smem_addr(sV), aQd = ptx::smem_addr(sQd);
      auto issue_st = [&](int n) {
        const int slot = n % BWD_STAGES, b = n & 1;
        if (!ptx::mbar_wait(&qd_full[slot], (n / BWD_STAGES) & 1, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns))
          return false;
        ptx::tc_fence_after();
        const uint32_t aQ = aQd + slot * 2 * TILE64, adO = aQ + TILE64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tmem + 64 * b, kmajor_desc(aK, kk), kmajor64_desc(aQ, kk), idesc_st, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tmem + 128 + 64 * b, kmajor_desc(aV, kk), kmajor64_desc(adO, kk), idesc_st, kk > 0 ? 1u : 0u);
        ptx::mma_commit(&st_full[b]);
        return true;
      };
      bool ok = ptx::mbar_wait(kv_full, 0, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns);
      if (ok && nloop > 0) ok = issue_st(0);
      // Block n+1's S^T / dP^T go in before block n's dV / dK: the tensor pipe works on
      // them while the compute warps form P^T_n and dS^T_n.  Buffer (n+1) & 1 was last
      // read by the dV / dK MMAs of block n-1, issued (and so executed) before.
      for (int n = 0; ok && n < nloop; ++n) {
        if (n + 1 < nloop && !issue_st(n + 1)) break;
        const int b = n & 1, slot = n % BWD_STAGES;
        if (!ptx::mbar_wait(&pds_full[b], (n >> 1) & 1, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns)) break;
        ptx::tc_fence_after();
        const uint32_t aQ = aQd + slot * 2 * TILE64, adO = aQ + TILE64;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_f16_ts(tdV, tmem + 64 * b + half_split_col(kk), mnmajor64_desc(adO, kk), idesc_acc,
                          (n > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_f16_ts(tdK, tmem + 128 + 64 * b + half_split_col(kk), mnmajor64_desc(aQ, kk), idesc_acc,
                          (n > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(&qd_empty[slot]);
      }
      ptx::mma_commit(acc_done);
      ptx::mma_commit(mma_done);
      volatile int never = 0;
      ptx::mbar_wait(mma_done, 0, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
    }
  } else {
    // Compute warps: lane quarter warp & 3 (key rows), column half h of each 64-query block.
    const int quad = warp & 3, h = (warp - 2) >> 2;
    const int row = quad * 32 + lane;
    const int kv = kb * BKV + row;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int n = 0; n < nloop; ++n) {
      const int b = n & 1, slot = n % BWD_STAGES;
      if (!ptx::mbar_wait(&st_full[b], (n >> 1) & 1, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns) ||
          !ptx::mbar_wait(&qd_full[slot], (n / BWD_STAGES) & 1, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tSb = tmem + 64 * b + lane_base + 32 * h, tdPb = tSb + 128;
      uint32_t s[32], dp[32];
      ptx::tmem_ld32(tSb, s);
      ptx::tmem_ld32(tdPb, dp);
      ptx::tmem_ld_wait();
      const int g = n / nq, qi = q_first + (n - g * nq);
      const int c0 = qi * 64 + 32 * h;  // query index of column 0 of this half
      // causal: query c0 + e sees key kv only if kv <= c0 + e
      const bool edge = p.causal && c0 < kv;
      const float4* l2 = reinterpret_cast<const float4*>(sLD + slot * 128 + 32 * h);
      const float4* dd = reinterpret_cast<const float4*>(sLD + slot * 128 + 64 + 32 * h);
      uint32_t wp[16], wds[16];
      if (!edge) {
        // two columns per instruction: x = s scale - L, dP - D, P (dP - D), packed
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 L4 = l2[e4], D4 = dd[e4];
#pragma unroll
          for (int u2 = 0; u2 < 2; ++u2) {
            const int e = 4 * e4 + 2 * u2;
            const uint64_t nl2 = u2 ? f2_pack(L4.z, L4.w) : f2_pack(L4.x, L4.y);
            const uint64_t nd2 = u2 ? f2_pack(D4.z, D4.w) : f2_pack(D4.x, D4.y);
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), sl2x2, nl2), x0, x1);
            const float p0 = ptx::exp2_approx(x0), p1 = ptx::exp2_approx(x1);
            float d0, d1;
            f2_unpack(f2_mul(f2_pack(p0, p1),
                             f2_add(f2_pack(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), nd2)),
                      d0, d1);
            wp[2 * e4 + u2] = pack_f16x2(p0, p1);
            wds[2 * e4 + u2] = pack_f16x2(d0, d1);
          }
        }
      } else {
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 L4 = l2[e4], D4 = dd[e4];
          const float Lv[4] = {L4.x, L4.y, L4.z, L4.w}, Dv[4] = {D4.x, D4.y, D4.z, D4.w};
          float pv[4], dv[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int e = 4 * e4 + u;
            float pr = ptx::exp2_approx(fmaf(__uint_as_float(s[e]), sl2, Lv[u]));
            if (c0 + e < kv) pr = 0.0f;
            pv[u] = pr;
            dv[u] = pr * (__uint_as_float(dp[e]) + Dv[u]);
          }
          wp[2 * e4] = pack_f16x2(pv[0], pv[1]);
          wp[2 * e4 + 1] = pack_f16x2(pv[2], pv[3]);
          wds[2 * e4] = pack_f16x2(dv[0], dv[1]);
          wds[2 * e4 + 1] = pack_f16x2(dv[2], dv[3]);
        }
      }
      ptx::tmem_st16(tSb, wp);
      ptx::tmem_st16(tdPb, wds);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&pds_full[b]);
    }
    if (ok && ptx::mbar_wait(acc_done, 0, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
      ptx::tc_fence_after();
      uint16_t* drow = p.dQKV + (static_cast<int64_t>(shard) * p.N + kv) * p.row_w;
      tmem_cols64_to_16(tdV + lane_base + 64 * h, 1.0f, drow + vcol + 64 * h, kv < p.N, p.dqkv_f16 != 0);
      tmem_cols64_to_16(tdK + lane_base + 64 * h, p.scale, drow + kcol + 64 * h, kv < p.N, p.dqkv_f16 != 0);
    }
  }

  ptx::tc_fence_before();
  __syncwarp();
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
  uint8_t* sKV = base + 2 * TILE;  // stage s: K_j at s * 2 TILE64, V_j after it
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + 2 * TILE + BWD_STAGES * 2 * TILE64);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;                    // [BWD_STAGES]
  uint64_t* kv_empty = bars + 1 + BWD_STAGES;      // [BWD_STAGES]
  uint64_t* s_full = bars + 1 + 2 * BWD_STAGES;    // [2] S, dP of a key block in TMEM
  uint64_t* ds_full = bars + 3 + 2 * BWD_STAGES;   // [2] dS written
  uint64_t* acc_done = bars + 5 + 2 * BWD_STAGES;
  uint64_t* mma_done = bars + 6 + 2 * BWD_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 7 + 2 * BWD_STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x % p.H;
  const int qb = p.nqb - 1 - static_cast<int>(blockIdx.x / p.H);  // heavy (late) query blocks first
  const int shard = head / p.hpr, jj = head - shard * p.hpr;
  const int nkv = p.causal ? min(2 * qb + 2, p.nb64) : p.nb64;   // 64-key blocks this query block sees
  const int qcol = jj * HD;
  const int kcol = static_cast<int>(p.kcol0) + (jj / p.Gs) * HD, vcol = static_cast<int>(p.vcol0) + (jj / p.Gs) * HD;

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    for (int s = 0; s < BWD_STAGES; ++s) {
      ptx::mbar_init(&kv_full[s], 1);
      ptx::mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&s_full[b], 1);
      ptx::mbar_init(&ds_full[b], 256);
    }
    ptx::mbar_init(acc_done, 1);
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncwarp();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Programmatic dependent launch: set-up above overlapped the previous kernel's tail;
  // nothing it writes is read before this wait.
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  // TMEM columns: S_0 | S_1 (64 each) | dP_0 | dP_1 (64 each) | dQ (128).
  const uint32_t tdQ = tmem + 256;

  if (warp == 0) {
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_qkv);
      ptx::tma_prefetch_desc(&tm_do);
      ptx::mbar_arrive_expect_tx(q_full, 2 * TILE);
      tma_tile128(sQ, &tm_qkv, q_full, qcol, qb * BQ, shard);
      tma_tile128(sdO, &tm_do, q_full, jj * HD, qb * BQ, shard);
      int issued = 0;
      for (int j = 0; j < nkv; ++j) {
        const int slot = j % BWD_STAGES;
        if (!ptx::mbar_wait(&kv_empty[slot], ((j / BWD_STAGES) & 1) ^ 1u, abort_flag, p.err, ERR_ATT_PRODUCER,
                            p.timeout_ns))
          break;
        uint8_t* dst = sKV + slot * 2 * TILE64;
        ptx::mbar_arrive_expect_tx(&kv_full[slot], 2 * TILE64);
        tma_tile64(dst, &tm_qkv, &kv_full[slot], kcol, j * 64, shard);
        tma_tile64(dst + TILE64, &tm_qkv, &kv_full[slot], vcol, j * 64, shard);
        ++issued;
      }
      volatile int never = 0;
      ptx::mbar_wait(q_full, 0, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
      for (int j = (issued > BWD_STAGES ? issued - BWD_STAGES : 0); j < issued; ++j)
        ptx::mbar_wait(&kv_full[j % BWD_STAGES], (j / BWD_STAGES) & 1, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = ptx::idesc_f16_f32(128, 64, false, false);  // S, dP
      constexpr uint32_t idesc_q = ptx::idesc_f16_f32(128, 128, false, true);  // dQ = dS K
      const uint32_t aQ = ptx::smem_addr(sQ), adO = ptx::smem_addr(sdO), aKV = ptx::smem_addr(sKV);
      auto issue_s = [&](int j) {
        const int slot = j % BWD_STAGES, b = j & 1;
        if (!ptx::mbar_wait(&kv_full[slot], (j / BWD_STAGES) & 1, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns))
          return false;
        ptx::tc_fence_after();
        const uint32_t aK = aKV + slot * 2 * TILE64, aV = aK + TILE64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tmem + 64 * b, kmajor_desc(aQ, kk), kmajor64_desc(aK, kk), idesc_s, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tmem + 128 + 64 * b, kmajor_desc(adO, kk), kmajor64_desc(aV, kk), idesc_s, kk > 0 ? 1u : 0u);
        ptx::mma_commit(&s_full[b]);
        return true;
      };
      bool ok = ptx::mbar_wait(q_full, 0, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns);
      if (ok && nkv > 0) ok = issue_s(0);
      for (int j = 0; ok && j < nkv; ++j) {
        if (j + 1 < nkv && !issue_s(j + 1)) break;
        const int b = j & 1, slot = j % BWD_STAGES;
        if (!ptx::mbar_wait(&ds_full[b], (j >> 1) & 1, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns)) break;
        ptx::tc_fence_after();
        const uint32_t aK = aKV + slot * 2 * TILE64;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_f16_ts(tdQ, tmem + 64 * b + half_split_col(kk), mnmajor64_desc(aK, kk), idesc_q,
                          (j > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(&kv_empty[slot]);
      }
      ptx::mma_commit(acc_done);
      ptx::mma_commit(mma_done);
      volatile int never = 0;
      ptx::mbar_wait(mma_done, 0, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
    }
  } else {
    // Compute warps: lane quarter warp & 3 (query rows), column half h of each 64-key block.
    const int quad = warp & 3, h = (warp - 2) >> 2;
    const int row = quad * 32 + lane;
    const int q = qb * BQ + row;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int64_t vec = (static_cast<int64_t>(shard) * p.hpr + jj) * p.N;
    // A query row past the end gets lse = +inf: its P and dS are exactly 0.
    const float lse2 = q < p.N ? p.lse[vec + q] * kLog2e : INFINITY;
    const float Dq = q < p.N ? p.Dvec[vec + q] : 0.0f;
    const float sl2 = p.scale_log2;
    const int qlim = p.causal ? min(q, p.N - 1) : p.N - 1;  // last key this row sees
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int b = j & 1;
      if (!ptx::mbar_wait(&s_full[b], (j >> 1) & 1, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tSb = tmem + 64 * b + lane_base + 32 * h, tdPb = tSb + 128;
      uint32_t s[32], dp[32];
      ptx::tmem_ld32(tSb, s);
      ptx::tmem_ld32(tdPb, dp);
      ptx::tmem_ld_wait();
      const int lim = qlim - (j * 64 + 32 * h);  // columns e <= lim are visible keys
      const bool edge = lim < 31;
      uint32_t wds[16];
      if (!edge) {
        // two columns per instruction: x = s scale - lse, dP - D, P (dP - D), packed
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nl2 = f2_pack(-lse2, -lse2), nd2 = f2_pack(-Dq, -Dq);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), sl2x2, nl2), x0, x1);
          const float p0 = ptx::exp2_approx(x0), p1 = ptx::exp2_approx(x1);
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(p0, p1), f2_add(f2_pack(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), nd2)),
                    d0, d1);
          wds[e >> 1] = pack_f16x2(d0, d1);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float d2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            float pr = ptx::exp2_approx(fmaf(__uint_as_float(s[e + u]), sl2, -lse2));
            if (e + u > lim) pr = 0.0f;
            d2[u] = pr * (__uint_as_float(dp[e + u]) - Dq);
          }
          wds[e >> 1] = pack_f16x2(d2[0], d2[1]);
        }
      }
      ptx::tmem_st16(tSb, wds);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ds_full[b]);
    }
    if (ok && ptx::mbar_wait(acc_done, 0, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
      ptx::tc_fence_after();
      uint16_t* drow = p.dQKV + (static_cast<int64_t>(shard) * p.N + q) * p.row_w;
      tmem_cols64_to_16(tdQ + lane_base + 64 * h, p.scale, drow + qcol + 64 * h, q < p.N, p.dqkv_f16 != 0);
    }
  }

  ptx::tc_fence_before();
  __syncwarp();
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
    TP_CUDA_CHECK(launch_pdl(attn_fwd_kernel<true>, dim3(static_cast<unsigned>(grid)), dim3(FWD_THREADS), FWD_SMEM, s,
                             map, a));
  else
    TP_CUDA_CHECK(launch_pdl(attn_fwd_kernel<false>, dim3(static_cast<unsigned>(grid)), dim3(FWD_THREADS), FWD_SMEM,
                             s, map, a));
  count_launch();
  return TP_OK;
}

}  // namespace tp

namespace tp {

tp_status run_attention_bwd(const uint16_t* QKV, const uint16_t* O, const uint16_t* dO, const float* lse, int64_t N,
                            int64_t d, int n_heads, int n_kv, int head_dim, int t, int causal, float scale, float* Dvec,
                            uint16_t* dQKV, cudaStream_t s, int dqkv_f16) {
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
  if (!make_map_3d_bf16(&m_qkv, QKV, sh.row_w, N, t, sh.row_w * 2, N * sh.row_w * 2, 64, 64)) return TP_ERR_CUDA;
  if (!make_map_3d_bf16(&m_do, dO, dt, N, t, dt * 2, N * dt * 2, 64, 64)) return TP_ERR_CUDA;
  const int64_t rows = static_cast<int64_t>(t) * N;
  TP_CUDA_CHECK(launch_pdl(attn_bwd_dot_kernel, dim3(static_cast<unsigned>((rows * 32 + 255) / 256)), dim3(256), 0, s,
                           dO, O, static_cast<int>(N), hpr, dt, rows, Dvec));
  count_launch();
  AttnBwdArgs a{};
  a.N = static_cast<int>(N);
  a.H = n_heads;
  a.hpr = hpr;
  a.nqb = static_cast<int>((N + BQ - 1) / BQ);
  a.nb64 = static_cast<int>((N + 63) / 64);
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
  a.dqkv_f16 = dqkv_f16;
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
  TP_CUDA_CHECK(launch_pdl(attn_bwd_dkv_kernel, dim3(grid_kv), dim3(BWD_THREADS), DKV_SMEM, s, m_qkv, m_do, a));
  count_launch();
  const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(n_heads) * a.nqb);
  TP_CUDA_CHECK(launch_pdl(attn_bwd_dq_kernel, dim3(grid), dim3(BWD_THREADS), DQ_SMEM, s, m_qkv, m_do, a));
  count_launch();
  return TP_OK;
}

}  // namespace tp
