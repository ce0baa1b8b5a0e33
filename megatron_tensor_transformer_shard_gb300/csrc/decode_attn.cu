// Decode attention over a head-sharded KV cache, with grouped-query heads
// sharded by KV group.
//
// "02 — Tensor Parallelism" (project-fortress roadmap), section "The critical
// inference-time subtlety: KV cache also shards": each rank holds the KV heads
// of its own query heads, so the cache splits with the heads; section "The
// attention pairing": GQA/MQA shard by KV group.  "Tensor and sequence
// parallelism" (ai-infra handbooks), exercise 1: with fewer KV heads than
// ranks each KV head is replicated on t/n_kv ranks and the KV weights and cache
// exist in several copies.
//
// One decode step, per shard i (t logical shards on this GPU):
//   qkv_i = x W_qkv,i + b_qkv,i            column-parallel GEMV (packed rows
//                                           [Q heads | K heads | V heads])
//   K_i[.., pos[b]] = k, V_i[.., pos[b]] = v   append to the shard's cache copy
//   o_{b,j} = softmax(scale q_{b,j} K^T) V  over keys 0..pos[b] of its KV head
//   y = sum_i O_i W_o,i + b_o               row-parallel GEMV, g in shard order
//
// The attention is a stream of the cache (bandwidth-bound): every (shard, KV
// head, sequence) is a "stream" of ceil(len/128) tiles of 128 keys.  All
// tiles of all streams form one flattened list; CTA k of G takes the
// contiguous range [k T / G, (k+1) T / G), so every SM streams the same
// number of tiles whatever the length mix.  A CTA that covers a stream only
// partly writes an unnormalised partial (O, running max, sum) for it, and a
// combine kernel merges the partials of each query head.  Partial slots are
// indexed by stream + CTA: along the flattened list either the stream or the
// CTA (or both) advances at each boundary, so the sum is strictly increasing
// and no two (stream, CTA) pieces share a slot.
//
// Tensor cores: the keys are the MMA's M dimension and the query heads of one
// KV group are its N dimension (padded to NG = 16 or 32), so a group of 8
// heads costs one 128 x 16 x 128 MMA chain per tile:
//   S^T[key][head] = K_tile (K-major) * Q^T           (tcgen05, fp16 in, fp32 acc)
//   O^T[dim][head] = V_tile^T (read MN-major) * P^T   (P^T written by the softmax warps)
// Warp roles: warp 0 TMA of Q (per stream) and K tiles, warp 6 TMA of V
// tiles (separate rings: a K stage frees after the S MMA, a V stage only after
// the O MMA), warp 1 issues the MMAs, warps 2-5 own one TMEM lane each (a key
// for S, a head dimension for O): masking, exponentials with a lazily raised
// reference max, P, and the running O in registers.  The CTA that finishes a
// stream's last piece merges the stream's partials (no separate combine pass).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>

#include "decode_plan.cuh"
#include "devmath.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace tp {

bool make_map_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
                      uint64_t s2_bytes, uint32_t b0, uint32_t b1);

namespace {

constexpr int HD = 128;           // head dimension
constexpr int BK = 128;           // keys per tile
constexpr int PANEL = 128 * 128;  // 128 rows x 128 bytes (64 fp16 of one 128-byte swizzle row)
constexpr int KV_TILE = 2 * PANEL;
constexpr int DEC_THREADS = 224;
constexpr int MAX_GRID = 256;     // attention CTAs per launch at most (sizes the partial slots)
constexpr float kLog2e = 1.4426950408889634f;

enum : int {
  ERR_DEC_PRODUCER = 0x121,
  ERR_DEC_MMA = 0x122,
  ERR_DEC_SOFTMAX = 0x123,
  ERR_DEC_DRAIN = 0x124,
};

template <int NG>
struct DecCfg {
  static constexpr int STAGES = NG <= 16 ? 3 : 2;
  static constexpr int QBUF = 2 * NG * 128;  // two 64-column panels of NG rows
  static constexpr int PBUF = 2 * NG * 128;
  static constexpr int OFF_V = STAGES * KV_TILE;
  static constexpr int OFF_Q = 2 * STAGES * KV_TILE;
  static constexpr int OFF_P = OFF_Q + 2 * QBUF;
  static constexpr int OFF_BAR = OFF_P + 2 * PBUF;
  static constexpr int OFF_RED = OFF_BAR + 512;
  static constexpr int OFF_PRE = OFF_RED + (2 * 4 * NG + 4 * NG) * 4;
  static constexpr int SMEM = 1024 + OFF_PRE + 260 * 4 + 64;
  static constexpr uint32_t TMEM_COLS = 4 * NG < 32 ? 32 : 4 * NG;
};

struct DecArgs {
  int S;           // streams = t * kv_t * B
  int B, nh, q_t, kv_t, Gs;
  int64_t L_max;
  float scale_log2;
  const int32_t* pos;
  float* o_part;          // [slots][NG][HD]
  float* m_part;          // [slots][NG]
  float* l_part;          // [slots][NG]
  uint16_t* O;            // [B][nh][HD] bf16, written by the combine kernel
  int* zero_cnt;          // the combine kernel zeroes these counters (the W_o GEMM's row blocks)
  int n_zero;
  int* err;
  uint64_t timeout_ns;
};

__device__ __forceinline__ int stream_len(const int32_t* pos, int b, int64_t L_max) {
  int64_t p = static_cast<int64_t>(__ldg(pos + b));
  if (p < 0) p = 0;
  if (p >= L_max) p = L_max - 1;
  return static_cast<int>(p + 1);
}

// Walks the CTA's contiguous range of the flattened tile list; the current
// stream's first tile and the next stream's first tile stay in registers.
// Stream s starts at tile (s / B) * TB + pre[s % B] (pre in shared memory).
struct TileCursor {
  const int* pre;
  int B, TB;
  int x, x1, s, ts_s, ts_n;
  __device__ int start_of(int st) const { return (st / B) * TB + pre[st % B]; }
  __device__ void init(const int* pre_, int B_, int S, int x0, int x1_) {
    pre = pre_;
    B = B_;
    TB = pre[B];
    x = x0;
    x1 = x1_;
    int lo = 0, hi = S - 1;  // largest s with start_of(s) <= x0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (start_of(mid) <= x0) lo = mid; else hi = mid - 1;
    }
    s = lo;
    ts_s = start_of(s);
    ts_n = start_of(s + 1);
  }
  __device__ bool valid() const { return x < x1; }
  __device__ int local_tile() const { return x - ts_s; }
  __device__ bool first(int x0) const { return x == x0 || x == ts_s; }
  __device__ bool last() const { return x + 1 == x1 || x + 1 == ts_n; }
  __device__ void next() {
    ++x;
    if (x < x1 && x >= ts_n) {
      ++s;
      ts_s = ts_n;
      ts_n = start_of(s + 1);
    }
  }
};

__device__ __forceinline__ int cta_of(int64_t x, int64_t G, int64_t T) { return static_cast<int>(((x + 1) * G - 1) / T); }

// K-major operand of R rows in two 64-column panels (panel stride R*128 bytes): k-step kk of 16 columns.
__device__ __forceinline__ uint64_t kmaj(uint32_t base, int panel_bytes, int kk) {
  return ptx::sdesc_sw128(base + (kk >> 2) * panel_bytes + (kk & 3) * 32, 16, 1024);
}
// 128 x 128 tile read MN-major (64-element MN chunks = the panels): k-step kk of 16 rows.
__device__ __forceinline__ uint64_t mnmaj(uint32_t base, int kk) {
  return ptx::sdesc_sw128(base + kk * 2048, PANEL, 1024);
}

template <int NG>
__device__ __forceinline__ void tmem_ld_ng(uint32_t taddr, float (&v)[NG]);

template <>
__device__ __forceinline__ void tmem_ld_ng<16>(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  ptx::tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

template <>
__device__ __forceinline__ void tmem_ld_ng<32>(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  ptx::tmem_ld32(taddr, r);
  ptx::tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Barrier over the 128 softmax threads that also ORs a predicate across them
// (a uniform decision to stop after a failed wait).
__device__ __forceinline__ bool softmax_bar_or(bool pred) {
  __syncwarp();  // the barrier needs converged warps
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(pred))
      : "memory");
  return out != 0;
}

__device__ __forceinline__ void softmax_bar() {
  __syncwarp();
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

template <int NG, int GSZ>
__global__ void __launch_bounds__(DEC_THREADS, 1)
    decode_attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_q, const DecArgs p) {
  using C = DecCfg<NG>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t dsmem[];
  const uint32_t pad = (1024u - (ptx::smem_addr(dsmem) & 1023u)) & 1023u;
  uint8_t* base = dsmem + pad;
  uint8_t* sK = base;
  uint8_t* sV = base + C::OFF_V;
  uint8_t* sQ = base + C::OFF_Q;
  uint8_t* sP = base + C::OFF_P;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::OFF_BAR);
  uint64_t* k_full = bars;            // [ST]
  uint64_t* v_full = bars + ST;       // [ST]
  uint64_t* k_empty = bars + 2 * ST;  // [ST] freed by the S MMA
  uint64_t* v_empty = bars + 3 * ST;  // [ST] freed by the O MMA
  uint64_t* q_full = bars + 4 * ST;   // [2]
  uint64_t* q_empty = q_full + 2;     // [2]
  uint64_t* s_full = q_full + 4;      // [2]
  uint64_t* s_free = q_full + 6;      // [2]
  uint64_t* p_full = q_full + 8;      // [2]
  uint64_t* o_full = q_full + 10;     // [2]
  uint64_t* o_free = q_full + 12;     // [2]
  uint64_t* mma_done = q_full + 14;
  uint64_t* all_done = q_full + 15;   // teardown: every thread arrives before TMEM is freed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_full + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(base + C::OFF_RED);  // [2][4][NG] tile maxima
  float* red2 = red + 2 * 4 * NG;                             // [4][NG] final sums

  int* pre = reinterpret_cast<int*>(base + C::OFF_PRE);     // [B + 1] tile prefix of the sequences

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ptx::griddep_launch_dependents();
  // The plan comes from pos (an input of the call, complete before the first
  // kernel of the call started), so it may be read before griddepcontrol.wait.
  decode_tile_prefix(p.pos, p.B, p.L_max, pre);
  const int T = (p.S / p.B) * pre[p.B];
  const int G = gridDim.x;
  const int k = blockIdx.x;
  const int x0 = static_cast<int>((static_cast<int64_t>(k) * T) / G);
  const int x1 = static_cast<int>((static_cast<int64_t>(k + 1) * T) / G);
  if (x0 >= x1) return;  // uniform for the whole CTA, before any barrier or TMEM use

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      ptx::mbar_init(&k_full[s], 1);
      ptx::mbar_init(&v_full[s], 1);
      ptx::mbar_init(&k_empty[s], 1);
      ptx::mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&q_full[b], 1);
      ptx::mbar_init(&q_empty[b], 1);
      ptx::mbar_init(&s_full[b], 1);
      ptx::mbar_init(&s_free[b], 128);
      ptx::mbar_init(&p_full[b], 128);
      ptx::mbar_init(&o_full[b], 1);
      ptx::mbar_init(&o_free[b], 128);
    }
    ptx::mbar_init(mma_done, 1);
    ptx::mbar_init(all_done, DEC_THREADS);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncwarp();  // lane-0 roles rejoin their warp: bar.sync needs converged warps
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  TileCursor cur;
  cur.init(pre, p.B, p.S, x0, x1);

  if (warp == 0) {
    // ------------------------------------------------- producer of Q and K
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_k);
      ptx::tma_prefetch_desc(&tm_q);
      ptx::griddep_wait();  // Q and the newest cache entries come from the previous kernel
      int u = 0, seg = 0;
      bool ok = true;
      for (; ok && cur.valid(); cur.next()) {
        const int s = cur.s;
        if (cur.first(x0)) {
          const int qb = seg & 1;
          if (!ptx::mbar_wait(&q_empty[qb], ((seg >> 1) & 1) ^ 1u, abort_flag, p.err, ERR_DEC_PRODUCER,
                              p.timeout_ns)) {
            ok = false;
            break;
          }
          const int b = s % p.B, c = s / p.B;
          const int i = c / p.kv_t, jl = c - i * p.kv_t;
          const int qrow = b * p.nh + i * p.q_t + jl * p.Gs;
          uint8_t* dq = sQ + qb * C::QBUF;
          ptx::mbar_arrive_expect_tx(&q_full[qb], C::QBUF);
          ptx::tma_load_3d(dq, &tm_q, &q_full[qb], 0, qrow, 0);
          ptx::tma_load_3d(dq + NG * 128, &tm_q, &q_full[qb], 64, qrow, 0);
          ++seg;
        }
        const int st = u % ST;
        if (!ptx::mbar_wait(&k_empty[st], ((u / ST) & 1) ^ 1u, abort_flag, p.err, ERR_DEC_PRODUCER,
                            p.timeout_ns)) {
          ok = false;
          break;
        }
        const int key0 = cur.local_tile() * BK;
        ptx::mbar_arrive_expect_tx(&k_full[st], KV_TILE);
        ptx::tma_load_3d(sK + st * KV_TILE, &tm_k, &k_full[st], 0, key0, s);
        ptx::tma_load_3d(sK + st * KV_TILE + PANEL, &tm_k, &k_full[st], 64, key0, s);
        ++u;
      }
      // drain: every issued copy lands before the CTA exits
      volatile int never = 0;
      for (int w = (u > ST ? u - ST : 0); w < u; ++w)
        ptx::mbar_wait(&k_full[w % ST], (w / ST) & 1, &never, p.err, ERR_DEC_DRAIN, p.timeout_ns);
      for (int sg = (seg > 2 ? seg - 2 : 0); sg < seg; ++sg)
        ptx::mbar_wait(&q_full[sg & 1], (sg >> 1) & 1, &never, p.err, ERR_DEC_DRAIN, p.timeout_ns);
    }
  } else if (warp == 6) {
    // --------------------------------------------------------- producer of V
    // V tiles have their own ring: a V stage frees only after the O MMA,
    // while a K stage frees right after the S MMA, so K can run further ahead.
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_v);
      ptx::griddep_wait();
      int u = 0;
      for (; cur.valid(); cur.next()) {
        const int st = u % ST;
        if (!ptx::mbar_wait(&v_empty[st], ((u / ST) & 1) ^ 1u, abort_flag, p.err, ERR_DEC_PRODUCER, p.timeout_ns))
          break;
        const int key0 = cur.local_tile() * BK;
        ptx::mbar_arrive_expect_tx(&v_full[st], KV_TILE);
        ptx::tma_load_3d(sV + st * KV_TILE, &tm_v, &v_full[st], 0, key0, cur.s);
        ptx::tma_load_3d(sV + st * KV_TILE + PANEL, &tm_v, &v_full[st], 64, key0, cur.s);
        ++u;
      }
      volatile int never = 0;
      for (int w = (u > ST ? u - ST : 0); w < u; ++w)
        ptx::mbar_wait(&v_full[w % ST], (w / ST) & 1, &never, p.err, ERR_DEC_DRAIN, p.timeout_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc_s = ptx::idesc_f16_f32(128, NG, false, false);
      constexpr uint32_t idesc_o = ptx::idesc_f16_f32(128, NG, true, false);
      const uint32_t aK = ptx::smem_addr(sK), aV = ptx::smem_addr(sV);
      const uint32_t aQ = ptx::smem_addr(sQ), aP = ptx::smem_addr(sP);
      int u = 0, seg = 0, qb = 0;
      bool ok = true;
      auto mma2 = [&](int w) -> bool {
        const int pb = w & 1, stw = w % ST;
        if (!ptx::mbar_wait(&p_full[pb], (w >> 1) & 1, abort_flag, p.err, ERR_DEC_MMA, p.timeout_ns)) return false;
        if (!ptx::mbar_wait(&v_full[stw], (w / ST) & 1, abort_flag, p.err, ERR_DEC_MMA, p.timeout_ns)) return false;
        if (w >= 2 && !ptx::mbar_wait(&o_free[pb], ((w >> 1) - 1) & 1, abort_flag, p.err, ERR_DEC_MMA, p.timeout_ns))
          return false;
        ptx::tc_fence_after();
        const uint32_t v_base = aV + stw * KV_TILE, p_base = aP + pb * C::PBUF;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          ptx::mma_bf16(tmem + (2 + pb) * NG, mnmaj(v_base, kk), kmaj(p_base, NG * 128, kk), idesc_o,
                        kk > 0 ? 1u : 0u);
        ptx::mma_commit(&v_empty[stw]);
        ptx::mma_commit(&o_full[pb]);
        return true;
      };
      for (; cur.valid(); cur.next()) {
        if (cur.first(x0)) {
          qb = seg & 1;
          if (!ptx::mbar_wait(&q_full[qb], (seg >> 1) & 1, abort_flag, p.err, ERR_DEC_MMA, p.timeout_ns)) {
            ok = false;
            break;
          }
          ++seg;
        }
        const int st = u % ST, sb = u & 1;
        if (!ptx::mbar_wait(&k_full[st], (u / ST) & 1, abort_flag, p.err, ERR_DEC_MMA, p.timeout_ns)) {
          ok = false;
          break;
        }
        if (u >= 2 && !ptx::mbar_wait(&s_free[sb], ((u >> 1) - 1) & 1, abort_flag, p.err, ERR_DEC_MMA,
                                      p.timeout_ns)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t k_base = aK + st * KV_TILE, q_base = aQ + qb * C::QBUF;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          ptx::mma_bf16(tmem + sb * NG, kmaj(k_base, PANEL, kk), kmaj(q_base, NG * 128, kk), idesc_s,
                        kk > 0 ? 1u : 0u);
        ptx::mma_commit(&s_full[sb]);
        ptx::mma_commit(&k_empty[st]);
        if (cur.last()) ptx::mma_commit(&q_empty[qb]);
        if (u >= 1 && !mma2(u - 1)) {
          ok = false;
          break;
        }
        ++u;
      }
      if (ok && u >= 1) mma2(u - 1);
      ptx::mma_commit(mma_done);
      volatile int never = 0;
      ptx::mbar_wait(mma_done, 0, &never, p.err, ERR_DEC_DRAIN, p.timeout_ns);
    }
  } else if (warp <= 5) {
    // ---------------------------------------------------- softmax / O rows
    // Lazy rescaling: every head keeps a reference max m_ref; P = 2^(s - m_ref)
    // is used as long as no score of the tile exceeds m_ref + kSlack (then P <=
    // 2^kSlack, exact in fp16's range and precision class), which one vote
    // barrier decides.  Only when some score does (always on a segment's first
    // tile) is the tile max exchanged through shared memory and m_ref raised.
    constexpr float kSlack = 8.0f;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // TMEM lane: a key of S^T, a head dimension of O^T
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int Gs = p.Gs;
    float m_ref[GSZ], l_run[GSZ], o_acc[GSZ], alpha_prev[GSZ], m_fin[GSZ], l_fin[GSZ];
#pragma unroll
    for (int h = 0; h < GSZ; ++h) {
      m_ref[h] = -INFINITY;
      l_run[h] = 0.0f;
      o_acc[h] = 0.0f;
      alpha_prev[h] = 1.0f;
      m_fin[h] = -INFINITY;
      l_fin[h] = 0.0f;
    }
    int u = 0, s_prev = 0, s_cur = -1, len = 1;
    bool last_prev = false, ok = true, stopped = false;

    // A finished piece's partial (unnormalised O, reference max, sum) goes to
    // its slot; the combine kernel merges each stream's pieces afterwards.
    auto write_piece = [&](int s, const float (&mf)[GSZ], const float (&lf)[GSZ]) {
#pragma unroll
      for (int h = 0; h < GSZ; ++h) {
        float v = lf[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red2[quad * NG + h] = v;
      }
      softmax_bar();
      const int64_t slot = static_cast<int64_t>(s) + k;
      if (r < Gs) {
        float tot = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) tot += red2[q * NG + r];
        float mv = mf[0];
#pragma unroll
        for (int h = 1; h < GSZ; ++h)
          if (h == r) mv = mf[h];
        p.l_part[slot * NG + r] = tot;
        p.m_part[slot * NG + r] = mv;
      }
#pragma unroll
      for (int h = 0; h < GSZ; ++h)
        if (h < Gs) p.o_part[(slot * NG + h) * HD + r] = o_acc[h];
      softmax_bar();  // red2 is reused by the next piece
    };

    auto accumulate = [&](int w) -> bool {
      const int ob = w & 1;
      const bool got = ptx::mbar_wait(&o_full[ob], (w >> 1) & 1, abort_flag, p.err, ERR_DEC_SOFTMAX, p.timeout_ns);
      ptx::tc_fence_after();
      float ov[NG];
      tmem_ld_ng<NG>(tmem + (2 + ob) * NG + lane_base, ov);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&o_free[ob]);
#pragma unroll
      for (int h = 0; h < GSZ; ++h) o_acc[h] = fmaf(o_acc[h], alpha_prev[h], ov[h]);
      return got;
    };

    for (; cur.valid(); cur.next()) {
      const int s = cur.s, sb = u & 1;
      if (s != s_cur) {
        s_cur = s;
        len = stream_len(p.pos, s % p.B, p.L_max);
      }
      const int nvalid = len - cur.local_tile() * BK;  // >= 1
      const bool first = cur.first(x0), last = cur.last();
      ok = ptx::mbar_wait(&s_full[sb], (u >> 1) & 1, abort_flag, p.err, ERR_DEC_SOFTMAX, p.timeout_ns) && ok;
      ptx::tc_fence_after();
      float v[NG];
      tmem_ld_ng<NG>(tmem + sb * NG + lane_base, v);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&s_free[sb]);
      if (first && u > 0) {
#pragma unroll
        for (int h = 0; h < GSZ; ++h) {
          m_fin[h] = m_ref[h];
          l_fin[h] = l_run[h];
          m_ref[h] = -INFINITY;
          l_run[h] = 0.0f;
        }
      }
      const bool key_ok = r < nvalid;
      bool need = false;
#pragma unroll
      for (int h = 0; h < GSZ; ++h) {
        v[h] = key_ok ? v[h] * p.scale_log2 : -INFINITY;
        need |= (h < Gs) && (v[h] > m_ref[h] + kSlack);
      }
      const bool stop_now = !ok || *abort_flag;
      float alpha[GSZ];
#pragma unroll
      for (int h = 0; h < GSZ; ++h) alpha[h] = 1.0f;
      if (softmax_bar_or(need || stop_now)) {
        // rare path: exchange the tile max of every head and raise m_ref
        float* rb = red + (u & 1) * 4 * NG;
#pragma unroll
        for (int h = 0; h < GSZ; ++h) {
          float mx = v[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (lane == 0) rb[quad * NG + h] = mx;
        }
        if (softmax_bar_or(stop_now)) {
          stopped = true;
          break;
        }
#pragma unroll
        for (int h = 0; h < GSZ; ++h) {
          const float tmax = fmaxf(fmaxf(rb[h], rb[NG + h]), fmaxf(rb[2 * NG + h], rb[3 * NG + h]));
          const float m_new = fmaxf(m_ref[h], tmax);
          alpha[h] = ptx::exp2_approx(m_ref[h] - m_new);  // 0 on a segment's first tile
          m_ref[h] = m_new;
        }
      }
      float pv[GSZ];
#pragma unroll
      for (int h = 0; h < GSZ; ++h) {
        pv[h] = ptx::exp2_approx(v[h] - m_ref[h]);  // 0 for masked keys
        l_run[h] = fmaf(l_run[h], alpha[h], pv[h]);
      }
      const int st = u % ST;
      if (nvalid < BK) {
        // Keys past the sequence end have P = 0, but 0 * (stale, possibly
        // non-finite cache bytes) would poison O: zero those V rows.
        ok = ptx::mbar_wait(&v_full[st], (u / ST) & 1, abort_flag, p.err, ERR_DEC_SOFTMAX, p.timeout_ns) && ok;
        if (!key_ok) {
          uint4 z = make_uint4(0u, 0u, 0u, 0u);
          uint8_t* vrow = sV + st * KV_TILE + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(vrow + c * 16) = z;
            *reinterpret_cast<uint4*>(vrow + PANEL + c * 16) = z;
          }
        }
      }
      {
        uint8_t* pbuf = sP + sb * C::PBUF + (r >> 6) * (NG * 128);
        const int chunk = (r & 63) >> 3, within = (r & 7) * 2;
#pragma unroll
        for (int h = 0; h < GSZ; ++h) {
          const __half hv = __float2half_rn(pv[h]);
          *reinterpret_cast<__half*>(pbuf + h * 128 + ((chunk ^ (h & 7)) << 4) + within) = hv;
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&p_full[sb]);
      if (u >= 1) {
        ok = accumulate(u - 1) && ok;
        if (last_prev) write_piece(s_prev, m_fin, l_fin);
      }
#pragma unroll
      for (int h = 0; h < GSZ; ++h) alpha_prev[h] = alpha[h];
      s_prev = s;
      last_prev = last;
      ++u;
    }
    if (!stopped && u >= 1) {
      ok = accumulate(u - 1) && ok;
      write_piece(s_prev, m_ref, l_run);
    }
  }

  // Teardown through an mbarrier rather than bar.sync 0: after the softmax
  // group's named-barrier traffic a CTA-wide bar.sync was measured to release
  // before all warps had arrived, which would free TMEM under a reader.
  ptx::tc_fence_before();
  __syncwarp();
  {
    ptx::mbar_arrive(all_done);
    volatile int never = 0;
    ptx::mbar_wait(all_done, 0, &never, p.err, ERR_DEC_DRAIN, p.timeout_ns);
  }
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------ combine
// One warp per (sequence, query head): merge the pieces of the head's stream,
// o = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k (M = max_k m_k), in CTA
// order, and write O [B][n_heads][HD] bf16 -- the W_o projection's input.
// Each lane owns 4 of the 128 dimensions; the loads of up to 4 pieces are in
// flight together.
constexpr int CMB_WARPS = 4;

template <int NG>
__global__ void __launch_bounds__(CMB_WARPS * 32) decode_combine_kernel(const DecArgs p, int G) {
  __shared__ int pre[260];
  ptx::griddep_launch_dependents();
  decode_tile_prefix(p.pos, p.B, p.L_max, pre);  // from pos: no dependency on the previous kernel
  if (blockIdx.x == 0)
    for (int z = threadIdx.x; z < p.n_zero; z += blockDim.x) p.zero_cnt[z] = 0;  // the next kernel's counters
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x * CMB_WARPS + warp;
  if (pair >= p.B * p.nh) return;
  const int qh = pair % p.nh, b = pair / p.nh;
  const int i = qh / p.q_t, w = qh - i * p.q_t;
  const int jl = w / p.Gs, g = w - jl * p.Gs;
  const int s = (i * p.kv_t + jl) * p.B + b;
  const int TB = pre[p.B];
  const uint32_t T = static_cast<uint32_t>((p.S / p.B) * TB), uG = static_cast<uint32_t>(G);
  const uint32_t ts = static_cast<uint32_t>((s / p.B) * TB + pre[s % p.B]);
  const uint32_t te = static_cast<uint32_t>(((s + 1) / p.B) * TB + pre[(s + 1) % p.B]);
  auto cta_of32 = [&](uint32_t x) { return ((x + 1) * uG - 1) / T; };
  auto owns = [&](uint32_t kk) { return (kk * T) / uG != ((kk + 1) * T) / uG; };
  const uint32_t k0 = cta_of32(ts), k1 = cta_of32(te - 1);
  ptx::griddep_wait();  // the partials come from the attention kernel
  float M = -INFINITY, num[4] = {0.f, 0.f, 0.f, 0.f}, den = 0.0f;
  uint32_t kk = k0;
  while (kk <= k1) {
    uint32_t ks[4];
    int n = 0;
    for (; kk <= k1 && n < 4; ++kk)
      if (owns(kk)) ks[n++] = kk;
    float mv[4], lv[4];
    float4 ov[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q < n) {
        const int64_t sl = static_cast<int64_t>(s) + ks[q];
        mv[q] = __ldcg(p.m_part + sl * NG + g);
        lv[q] = __ldcg(p.l_part + sl * NG + g);
        ov[q] = __ldcg(reinterpret_cast<const float4*>(p.o_part + (sl * NG + g) * HD) + lane);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q < n) {
        const float Mn = fmaxf(M, mv[q]);
        const float sc = ptx::exp2_approx(M - Mn), wk = ptx::exp2_approx(mv[q] - Mn);
        num[0] = fmaf(num[0], sc, wk * ov[q].x);
        num[1] = fmaf(num[1], sc, wk * ov[q].y);
        num[2] = fmaf(num[2], sc, wk * ov[q].z);
        num[3] = fmaf(num[3], sc, wk * ov[q].w);
        den = fmaf(den, sc, wk * lv[q]);
        M = Mn;
      }
    }
  }
  const float inv = 1.0f / den;
  uint2 out;
  out.x = pack_bf16x2(num[0] * inv, num[1] * inv);
  out.y = pack_bf16x2(num[2] * inv, num[3] * inv);
  *reinterpret_cast<uint2*>(p.O + (static_cast<int64_t>(b) * p.nh + qh) * HD + lane * 4) = out;
}

// ------------------------------------------------ QKV GEMV + cache append
// Column-parallel projection of the new tokens, one packed row per CTA
// iteration (row r of shard i is one output unit: a Q, K or V coordinate of one
// of its heads), weights streamed once with 16-byte loads; the result goes to
// the fp16 Q buffer or straight into the shard's cache copy at pos[b].
// Block 0 of the first launch also checks the positions.
constexpr int GEMV_T = 128;

__device__ __forceinline__ uint4 ld_stream(const uint16_t* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
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

struct QkvArgs {
  const uint16_t* x;  // [B][d] bf16 (whole batch)
  int64_t d, R_t, L_max;
  const uint16_t* W;     // [t][R_t][d]
  const uint16_t* bias;  // [t][R_t] or null
  int t, q_t, kv_t, nh, B, m0;
  const int32_t* pos;
  uint16_t* q;   // [B][nh][HD] fp16
  uint16_t* Kc;  // [t][kv_t][B][L_max][HD] fp16
  uint16_t* Vc;
  int check_pos;  // block 0 records positions outside [0, L_max)
  int* err;
};

template <int M>
__global__ void __launch_bounds__(GEMV_T) decode_qkv_kernel(const QkvArgs a) {
  __shared__ float red[GEMV_T / 32][M];
  __shared__ float tot[M];
  if (a.check_pos && blockIdx.x == 0) decode_check_positions(a.pos, a.B, a.L_max, a.err);
  const int64_t chunks = a.d / 8;
  const int64_t R = a.R_t * a.t;
  const int64_t qw = static_cast<int64_t>(a.q_t) * HD, kvw = static_cast<int64_t>(a.kv_t) * HD;
  for (int64_t r = blockIdx.x; r < R; r += gridDim.x) {
    const uint16_t* row = a.W + r * a.d;
    float acc[M];
#pragma unroll
    for (int m = 0; m < M; ++m) acc[m] = 0.0f;
    for (int64_t c = threadIdx.x; c < chunks; c += GEMV_T * 8) {
      uint4 w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t cc = c + j * GEMV_T;
        if (cc < chunks) w[j] = ld_stream(row + cc * 8);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t cc = c + j * GEMV_T;
        if (cc < chunks) {
#pragma unroll
          for (int m = 0; m < M; ++m) {
            const uint4 xv = __ldg(reinterpret_cast<const uint4*>(a.x + (a.m0 + m) * a.d) + cc);
            acc[m] += dot8(w[j], xv);
          }
        }
      }
    }
    const int wp = threadIdx.x >> 5, ln = threadIdx.x & 31;
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float v = acc[m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (ln == 0) red[wp][m] = v;
    }
    __syncthreads();
    if (threadIdx.x < M) {
      const int m = threadIdx.x;
      float v = 0.0f;
#pragma unroll
      for (int q = 0; q < GEMV_T / 32; ++q) v += red[q][m];
      if (a.bias) v += bf16_bits_to_float(a.bias[r]);
      tot[m] = v;
    }
    __syncthreads();
    if (threadIdx.x < M) {
      const int m = threadIdx.x, b = a.m0 + m;
      const __half hv = __float2half_rn(tot[m]);
      const uint16_t bits = *reinterpret_cast<const uint16_t*>(&hv);
      const int64_t i = r / a.R_t, lr = r - i * a.R_t;
      if (lr < qw) {
        a.q[(static_cast<int64_t>(b) * a.nh + i * a.q_t) * HD + lr] = bits;
      } else {
        const int64_t p = __ldg(a.pos + b);
        if (p >= 0 && p < a.L_max) {
          const int64_t w2 = lr - qw;
          const int part = w2 >= kvw ? 1 : 0;
          const int64_t w3 = w2 - part * kvw;
          const int64_t jl = w3 / HD, e = w3 - jl * HD;
          uint16_t* cache = part ? a.Vc : a.Kc;
          cache[(((i * a.kv_t + jl) * a.B + b) * a.L_max + p) * HD + e] = bits;
        }
      }
    }
  }
}

template <int M>
tp_status launch_qkv(const QkvArgs& a, cudaStream_t s) {
  int per_sm = 0;
  TP_CUDA_CHECK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_qkv_kernel<M>, GEMV_T, 0));
  int64_t g = static_cast<int64_t>(device_sm_count()) * (per_sm > 0 ? per_sm : 1);
  const int64_t R = a.R_t * a.t;
  if (g > R) g = R;
  decode_qkv_kernel<M><<<static_cast<unsigned>(g), GEMV_T, 0, s>>>(a);
  TP_LAUNCHED();
  return TP_OK;
}

tp_status qkv_dispatch(int M, const QkvArgs& a, cudaStream_t s) {
  switch (M) {
    case 1: return launch_qkv<1>(a, s);
    case 2: return launch_qkv<2>(a, s);
    case 3: return launch_qkv<3>(a, s);
    case 4: return launch_qkv<4>(a, s);
    case 5: return launch_qkv<5>(a, s);
    case 6: return launch_qkv<6>(a, s);
    case 7: return launch_qkv<7>(a, s);
    default: return launch_qkv<8>(a, s);
  }
}

template <int NG, int GSZ>
tp_status launch_attn(const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mq, const DecArgs& a, int grid,
                      cudaStream_t s) {
  static bool configured[64] = {};
  int dev = 0;
  TP_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return TP_ERR_CUDA;
  if (!configured[dev]) {
    TP_CUDA_CHECK(cudaFuncSetAttribute(decode_attn_kernel<NG, GSZ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       DecCfg<NG>::SMEM));
    configured[dev] = true;
  }
  TP_CUDA_CHECK(launch_pdl(decode_attn_kernel<NG, GSZ>, dim3(grid), dim3(DEC_THREADS), DecCfg<NG>::SMEM, s, mk, mv,
                           mq, a));
  count_launch();
  const unsigned cgrid = static_cast<unsigned>((a.B * a.nh + CMB_WARPS - 1) / CMB_WARPS);
  TP_CUDA_CHECK(launch_pdl(decode_combine_kernel<NG>, dim3(cgrid), dim3(CMB_WARPS * 32), 0, s, a, grid));
  count_launch();
  return TP_OK;
}

struct DecShape {
  int q_t, kv_t, Gs, NG, S;
  int64_t R_t;
};

bool decode_shape(int64_t B, int n_heads, int n_kv, int head_dim, int t, DecShape& sh) {
  if (head_dim != HD || t < 1 || t > 8 || n_heads < 1 || n_kv < 1) return false;
  if (n_heads % t != 0 || n_heads % n_kv != 0) return false;
  if (n_kv >= t ? (n_kv % t != 0) : (t % n_kv != 0)) return false;
  sh.q_t = n_heads / t;
  sh.kv_t = n_kv >= t ? n_kv / t : 1;
  const int G = n_heads / n_kv;
  sh.Gs = G < sh.q_t ? G : sh.q_t;
  sh.NG = sh.Gs <= 16 ? 16 : 32;
  if (sh.Gs > 32 || B > 256) return false;
  const int64_t S = static_cast<int64_t>(t) * sh.kv_t * B;
  if (S > (1 << 20)) return false;
  sh.S = static_cast<int>(S);
  sh.R_t = static_cast<int64_t>(sh.q_t + 2 * sh.kv_t) * HD;
  return true;
}

inline size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct DecWs {
  uint16_t* q;
  float *o_part, *m_part, *l_part;
  uint16_t* O;
  float* sk_part;  // skinny-GEMM partials (QKV, then W_o)
  int* sk_cnt;     // W_o row-block counters
  size_t bytes;
};

DecWs decode_ws_layout(void* ws, int64_t B, int64_t d, int n_heads, int t, const DecShape& sh) {
  DecWs w{};
  uint8_t* p = static_cast<uint8_t*>(ws);
  size_t off = 0;
  const size_t slots = static_cast<size_t>(sh.S) + MAX_GRID;
  w.q = reinterpret_cast<uint16_t*>(p + off); off += up256(static_cast<size_t>(B) * n_heads * HD * 2);
  w.o_part = reinterpret_cast<float*>(p + off); off += up256(slots * sh.NG * HD * 4);
  w.m_part = reinterpret_cast<float*>(p + off); off += up256(slots * sh.NG * 4);
  w.l_part = reinterpret_cast<float*>(p + off); off += up256(slots * sh.NG * 4);
  w.O = reinterpret_cast<uint16_t*>(p + off); off += up256(static_cast<size_t>(B) * n_heads * HD * 2);
  const int bq = B > 32 ? 32 : static_cast<int>(B);
  const size_t skq = skinny_part_floats(sh.R_t * t, bq), sko = skinny_part_floats(d, bq);
  w.sk_part = reinterpret_cast<float*>(p + off); off += up256((skq > sko ? skq : sko) * 4);
  w.sk_cnt = reinterpret_cast<int*>(p + off); off += up256(static_cast<size_t>(d / 128 + 1) * 4);
  w.bytes = off;
  return w;
}

}  // namespace

size_t decode_attn_ws_bytes(int64_t B, int64_t d, int n_heads, int n_kv, int head_dim, int t, int64_t L_max) {
  (void)d;
  (void)L_max;
  DecShape sh;
  if (B < 0 || !decode_shape(B, n_heads, n_kv, head_dim, t, sh)) return 0;
  return decode_ws_layout(nullptr, B, d, n_heads, t, sh).bytes;
}

tp_status run_decode_attn(const uint16_t* x, int64_t B, int64_t d, int n_heads, int n_kv, int head_dim, int t,
                          float scale, const uint16_t* Wqkv_p, const uint16_t* bqkv_p, const uint16_t* Wo_p,
                          const uint16_t* bo, uint16_t* Kc, uint16_t* Vc, int64_t L_max, const int32_t* pos,
                          uint16_t* y, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (B < 0 || d < 1 || L_max < 1) return TP_ERR_INVALID_ARG;
  DecShape sh;
  if (!decode_shape(B, n_heads, n_kv, head_dim, t, sh)) return TP_ERR_SHAPE;
  if (d % 8 != 0) return TP_ERR_ALIGN;
  if (L_max > (1LL << 30)) return TP_ERR_SHAPE;
  if (B == 0) return TP_OK;
  if (!x || !Wqkv_p || !Wo_p || !Kc || !Vc || !pos || !y || !ws) return TP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wqkv_p) || !aligned16(Wo_p) || !aligned16(Kc) || !aligned16(Vc) ||
      (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return TP_ERR_ALIGN;
  const DecWs w = decode_ws_layout(ws, B, d, n_heads, t, sh);
  if (ws_bytes < w.bytes) return TP_ERR_WORKSPACE;
  TP_RETURN_IF(ready());

  // Batches of 2..32 run the two projections on the tensor cores (skinny
  // GEMM); a single sequence streams them through the CUDA-core GEMVs.
  const int64_t nq = static_cast<int64_t>(n_heads) * HD;
  const bool skinny = B >= 2 && B <= 32 && skinny_ok(sh.R_t * t, d, static_cast<int>(B)) &&
                      skinny_ok(d, nq, static_cast<int>(B));

  // 1. column-parallel QKV projection; K/V appended to each shard's cache copy.
  if (skinny) {
    SkGemmJob j;
    j.W = Wqkv_p; j.slabs = 1; j.R = sh.R_t * t; j.ku_per_slab = static_cast<int>(d / 128);
    j.x = x; j.ldx = d; j.B = static_cast<int>(B); j.part = w.sk_part;
    j.epi = SK_EPI_QKV; j.bias = bqkv_p;
    j.R_t = sh.R_t; j.L_max = L_max; j.q_t = sh.q_t; j.kv_t = sh.kv_t; j.nh = n_heads;
    j.pos = pos; j.q = w.q; j.Kc = Kc; j.Vc = Vc;
    j.err = device_error_word();
    TP_RETURN_IF(run_skinny_gemm(j, s));
  } else {
    QkvArgs qa{};
    qa.x = x; qa.d = d; qa.R_t = sh.R_t; qa.L_max = L_max; qa.W = Wqkv_p; qa.bias = bqkv_p;
    qa.t = t; qa.q_t = sh.q_t; qa.kv_t = sh.kv_t; qa.nh = n_heads; qa.B = static_cast<int>(B);
    qa.pos = pos; qa.q = w.q; qa.Kc = Kc; qa.Vc = Vc; qa.err = device_error_word();
    for (int64_t m0 = 0; m0 < B; m0 += 8) {
      qa.m0 = static_cast<int>(m0);
      qa.check_pos = m0 == 0 ? 1 : 0;
      TP_RETURN_IF(qkv_dispatch(static_cast<int>(B - m0 < 8 ? B - m0 : 8), qa, s));
    }
  }

  // 2. split-KV attention over the flattened tile list, then the combine.
  CUtensorMap mk, mv, mq;
  const uint64_t S = static_cast<uint64_t>(sh.S);
  if (!make_map_3d_bf16(&mk, Kc, HD, L_max, S, HD * 2, L_max * HD * 2, 64, BK) ||
      !make_map_3d_bf16(&mv, Vc, HD, L_max, S, HD * 2, L_max * HD * 2, 64, BK) ||
      !make_map_3d_bf16(&mq, w.q, HD, static_cast<uint64_t>(B) * n_heads, 1, HD * 2,
                        static_cast<uint64_t>(B) * n_heads * HD * 2, 64, sh.NG))
    return TP_FAIL_DETAIL("cuTensorMapEncodeTiled failed for the KV cache or Q");
  DecArgs a{};
  a.S = sh.S; a.B = static_cast<int>(B); a.nh = n_heads; a.q_t = sh.q_t; a.kv_t = sh.kv_t; a.Gs = sh.Gs;
  a.L_max = L_max; a.scale_log2 = scale * kLog2e; a.pos = pos;
  a.o_part = w.o_part; a.m_part = w.m_part; a.l_part = w.l_part; a.O = w.O;
  a.zero_cnt = w.sk_cnt; a.n_zero = skinny ? static_cast<int>(d / 128) : 0;
  a.err = device_error_word(); a.timeout_ns = wait_timeout_ns();
  int64_t grid = device_sm_count();
  const int64_t max_tiles = S * ((L_max + BK - 1) / BK);
  if (grid > MAX_GRID) grid = MAX_GRID;
  if (grid > max_tiles) grid = max_tiles;
  // compile-time head-group size: the group rounded up to 4, 8, 16 or 32
  if (sh.Gs <= 4) {
    TP_RETURN_IF((launch_attn<16, 4>(mk, mv, mq, a, static_cast<int>(grid), s)));
  } else if (sh.Gs <= 8) {
    TP_RETURN_IF((launch_attn<16, 8>(mk, mv, mq, a, static_cast<int>(grid), s)));
  } else if (sh.Gs <= 16) {
    TP_RETURN_IF((launch_attn<16, 16>(mk, mv, mq, a, static_cast<int>(grid), s)));
  } else {
    TP_RETURN_IF((launch_attn<32, 32>(mk, mv, mq, a, static_cast<int>(grid), s)));
  }

  // 3. row-parallel W_o with g: y = sum_i O_i W_o,i + b_o, bias once.
  if (skinny) {
    SkGemmJob j;
    j.W = Wo_p; j.slabs = t; j.R = d; j.ku_per_slab = static_cast<int>(nq / t / 128);
    j.x = w.O; j.ldx = nq; j.B = static_cast<int>(B); j.part = w.sk_part;
    j.epi = SK_EPI_BF16; j.bias = bo; j.y = y; j.ldy = d; j.err = device_error_word();
    j.cnt = w.sk_cnt;  // zeroed by the combine kernel
    return run_skinny_gemm(j, s);
  }
  return run_row_gemv(w.O, B, nq, d, t, Wo_p, bo, y, s);
}

}  // namespace tp
