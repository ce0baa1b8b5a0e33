// Head-local causal softmax attention on tcgen05 ("02 — Tensor Parallelism",
// "The attention pairing": heads don't talk, so each shard runs attention on
// its own heads with no communication; "Megatron-LM: Tensor Parallelism",
// "The Transformer Layer Partitioning": S = Q K^T, P = softmax(S), O = P V).
//
// The QKV buffer is the column-parallel GEMM's output, [t][N][3d/t] with the
// shard's heads laid out [Q_i | K_i | V_i], head jj at columns jj*128 of each.
//
// Forward: one CTA per (head, 128-query block), heavy (late) query blocks first.
//   warp 0      TMA: Q once, then K_j / V_j through a 2-stage ring
//   warp 1      tcgen05.mma: S_j = Q K_j^T into one of two TMEM S buffers (so
//               S_{j+1} runs while the softmax works on S_j), then O += P_j V_j
//               (P from shared memory, V read MN-major straight from its tile)
//   warps 2-5   one query row per thread: online softmax in the log2 domain,
//               rescale of the O row in TMEM when the row max moves, P written
//               bf16 into a 128B-swizzled tile, final O / l and log-sum-exp.
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
constexpr int FWD_THREADS = 192;
constexpr int FWD_SMEM = 1024 + 6 * TILE + 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum : int { ERR_ATT_PRODUCER = 0x111, ERR_ATT_MMA = 0x112, ERR_ATT_SOFTMAX = 0x113, ERR_ATT_DRAIN = 0x114 };

struct AttnFwdArgs {
  int N, H, hpr, nqb, causal;
  int64_t dt;            // d / t: width of one shard's Q (or K, or V) block
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

// Thread `row` writes its 128 bf16 values (packed pairs) into a K-major 128x128 swizzled tile.
__device__ __forceinline__ void store_row_swizzled(uint8_t* tile, int row, const uint32_t (&w)[64]) {
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    uint8_t* rowp = tile + p * PANEL + row * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 v = make_uint4(w[p * 32 + c * 4 + 0], w[p * 32 + c * 4 + 1], w[p * 32 + c * 4 + 2],
                           w[p * 32 + c * 4 + 3]);
      *reinterpret_cast<uint4*>(rowp + ((c ^ (row & 7)) << 4)) = v;
    }
  }
}

__global__ void __launch_bounds__(FWD_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_qkv, const AttnFwdArgs p) {
  extern __shared__ uint8_t dsmem[];
  const uint32_t pad = (1024u - (ptx::smem_addr(dsmem) & 1023u)) & 1023u;
  uint8_t* base = dsmem + pad;
  uint8_t* sQ = base;
  uint8_t* sK = base + TILE;      // 2 stages
  uint8_t* sV = base + 3 * TILE;  // 2 stages
  uint8_t* sP = base + 5 * TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + 6 * TILE);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;     // [2]
  uint64_t* v_full = bars + 3;     // [2]
  uint64_t* kv_empty = bars + 5;   // [2]
  uint64_t* s_full = bars + 7;     // [2]
  uint64_t* s_free = bars + 9;     // [2]
  uint64_t* p_full = bars + 11;
  uint64_t* o_done = bars + 12;
  uint64_t* mma_done = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x % p.H;
  const int qb = p.nqb - 1 - static_cast<int>(blockIdx.x / p.H);
  const int shard = head / p.hpr, jj = head - shard * p.hpr;
  const int nkv = p.causal ? qb + 1 : (p.N + BKV - 1) / BKV;
  const int qcol = jj * HD;
  const int kcol = static_cast<int>(p.dt) + jj * HD;
  const int vcol = static_cast<int>(2 * p.dt) + jj * HD;

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&k_full[s], 1);
      ptx::mbar_init(&v_full[s], 1);
      ptx::mbar_init(&kv_empty[s], 1);
      ptx::mbar_init(&s_full[s], 1);
      ptx::mbar_init(&s_free[s], 128);
    }
    ptx::mbar_init(p_full, 128);
    ptx::mbar_init(o_done, 1);
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS[2] = {tmem, tmem + 128};
  const uint32_t tO = tmem + 256;

  if (warp == 0) {
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_qkv);
      ptx::mbar_arrive_expect_tx(q_full, TILE);
      ptx::tma_load_3d(sQ, &tm_qkv, q_full, qcol, qb * BQ, shard);
      ptx::tma_load_3d(sQ + PANEL, &tm_qkv, q_full, qcol + 64, qb * BQ, shard);
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
      // drain: every issued copy must land before the CTA exits
      volatile int never = 0;
      ptx::mbar_wait(q_full, 0, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
      for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j) {
        const uint32_t ph = (j >> 1) & 1;
        ptx::mbar_wait(&k_full[j & 1], ph, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
        ptx::mbar_wait(&v_full[j & 1], ph, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(BQ, BKV, false, false);
      constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(BQ, HD, false, true);
      const uint32_t aQ = ptx::smem_addr(sQ), aP = ptx::smem_addr(sP);
      bool ok = ptx::mbar_wait(q_full, 0, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns);
      for (int j = 0; ok && j <= nkv; ++j) {
        if (j < nkv) {
          const int st = j & 1;
          if (!ptx::mbar_wait(&k_full[st], (j >> 1) & 1, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns)) break;
          if (j >= 2 && !ptx::mbar_wait(&s_free[st], ((j >> 1) - 1) & 1, abort_flag, p.err, ERR_ATT_MMA,
                                        p.timeout_ns))
            break;
          ptx::tc_fence_after();
          const uint32_t aK = ptx::smem_addr(sK + st * TILE);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk)
            ptx::mma_bf16(tS[st], kmajor_desc(aQ, kk), kmajor_desc(aK, kk), idesc_s, kk > 0 ? 1u : 0u);
          ptx::mma_commit(&s_full[st]);
        }
        if (j >= 1) {
          const int jp = j - 1, stp = jp & 1;
          if (!ptx::mbar_wait(p_full, jp & 1, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns)) break;
          if (!ptx::mbar_wait(&v_full[stp], (jp >> 1) & 1, abort_flag, p.err, ERR_ATT_MMA, p.timeout_ns)) break;
          ptx::tc_fence_after();
          const uint32_t aV = ptx::smem_addr(sV + stp * TILE);
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)
            ptx::mma_bf16(tO, kmajor_desc(aP, kk), mnmajor_desc(aV, kk), idesc_o, (jp > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit(&kv_empty[stp]);
          ptx::mma_commit(o_done);
        }
      }
      ptx::mma_commit(mma_done);
      volatile int never = 0;
      ptx::mbar_wait(mma_done, 0, &never, p.err, ERR_ATT_DRAIN, p.timeout_ns);
    }
  } else {
    // ---------------------------------------------------------- softmax rows
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int q = qb * BQ + row;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int sb = j & 1;
      if (!ptx::mbar_wait(&s_full[sb], (j >> 1) & 1, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      float s[BKV];
      {
        uint32_t r[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          ptx::tmem_ld32(tS[sb] + lane_base + c * 32, r);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(r[e]);
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&s_free[sb]);
      const int kv0 = j * BKV;
      const bool edge = (p.causal && j == qb) || (kv0 + BKV > p.N);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BKV; ++c) {
        float v = s[c] * p.scale_log2;
        if (edge) {
          const int kv = kv0 + c;
          if (kv >= p.N || (p.causal && kv > q)) v = -INFINITY;
        }
        s[c] = v;
        mx = fmaxf(mx, v);
      }
      const float m_new = fmaxf(m, mx);
      const float alpha = ptx::exp2_approx(m - m_new);  // 0 on the first block (m = -inf)
      float rs = 0.0f;
      uint32_t w[64];
#pragma unroll
      for (int c = 0; c < BKV; c += 2) {
        const float p0 = ptx::exp2_approx(s[c] - m_new);
        const float p1 = ptx::exp2_approx(s[c + 1] - m_new);
        rs += p0 + p1;
        w[c >> 1] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + rs;
      m = m_new;
      if (j >= 1) {
        // P_{j-1} V_{j-1} must be done before O is rescaled and the P tile is rewritten.
        if (!ptx::mbar_wait(o_done, (j - 1) & 1, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        if (__any_sync(0xffffffffu, alpha < 1.0f)) {
          uint32_t r[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            ptx::tmem_ld32(tO + lane_base + c * 32, r);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            ptx::tmem_st32(tO + lane_base + c * 32, r);
          }
          ptx::tmem_st_wait();
        }
      }
      store_row_swizzled(sP, row, w);
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(p_full);
    }
    if (ok && ptx::mbar_wait(o_done, (nkv - 1) & 1, abort_flag, p.err, ERR_ATT_SOFTMAX, p.timeout_ns)) {
      ptx::tc_fence_after();
      const float inv_l = 1.0f / l;
      uint16_t* orow = p.O + (static_cast<int64_t>(shard) * p.N + q) * p.dt + qcol;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        ptx::tmem_ld32(tO + lane_base + c * 32, r);
        ptx::tmem_ld_wait();
        if (q < p.N) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(r[e + 0]) * inv_l, __uint_as_float(r[e + 1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(r[e + 2]) * inv_l, __uint_as_float(r[e + 3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(r[e + 4]) * inv_l, __uint_as_float(r[e + 5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(r[e + 6]) * inv_l, __uint_as_float(r[e + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + c * 32 + e) = v;
          }
        }
      }
      if (q < p.N) p.lse[(static_cast<int64_t>(shard) * p.hpr + jj) * p.N + q] = (m + __log2f(l)) * kLn2;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

tp_status run_attention_fwd(const uint16_t* QKV, int64_t N, int64_t d, int n_heads, int head_dim, int t, int causal,
                            float scale, uint16_t* O, float* lse, cudaStream_t s) {
  if (N < 0 || d < 1 || n_heads < 1 || t < 1) return TP_ERR_INVALID_ARG;
  if (head_dim != HD || static_cast<int64_t>(n_heads) * head_dim != d || n_heads % t != 0) return TP_ERR_SHAPE;
  if (N == 0) return TP_OK;
  if (!QKV || !O || !lse) return TP_ERR_INVALID_ARG;
  if (!aligned16(QKV) || !aligned16(O)) return TP_ERR_ALIGN;
  if (N > (1LL << 30) / 1) return TP_ERR_SHAPE;
  TP_RETURN_IF(ready());
  const int64_t dt = d / t;
  CUtensorMap map;
  if (!make_map_3d_bf16(&map, QKV, 3 * dt, N, t, 3 * dt * 2, N * 3 * dt * 2, 64, 128)) return TP_ERR_CUDA;
  AttnFwdArgs a{};
  a.N = static_cast<int>(N);
  a.H = n_heads;
  a.hpr = n_heads / t;
  a.nqb = static_cast<int>((N + BQ - 1) / BQ);
  a.causal = causal ? 1 : 0;
  a.dt = dt;
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
    TP_CUDA_CHECK(cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FWD_SMEM));
    configured[dev] = true;
  }
  const int64_t grid = static_cast<int64_t>(n_heads) * a.nqb;
  if (grid > 0x7fffffff) return TP_ERR_SHAPE;
  attn_fwd_kernel<<<static_cast<unsigned>(grid), FWD_THREADS, FWD_SMEM, s>>>(map, a);
  TP_LAUNCHED();
  return TP_OK;
}

}  // namespace tp
