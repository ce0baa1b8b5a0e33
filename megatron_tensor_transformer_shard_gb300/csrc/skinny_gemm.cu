// Skinny GEMM for decode batches: y[b][r] = sum_k W[r][k] x[b][k] for a few
// rows b of x (1..32 sequences) against a large weight W (HBM-bound).
//
// On CUDA cores a batch of 8 costs 8 dot products per weight load, which
// makes the GEMV ALU-bound far below HBM speed; the tensor cores do it for
// free.  So the weight is the MMA's M = 128 operand (128 rows per tile) and
// the batch, padded to NB = 16 or 32, is N ("swap AB"):
//   D[row][b] (TMEM, fp32) += W_tile[128 x 16] * X_tile[NB x 16]^T    (tcgen05, bf16)
// K is spread over all SMs stream-K style: the (row block, 128-wide K unit)
// pairs form one list in row-block-major order and CTA k of G takes the
// contiguous range [k U / G, (k+1) U / G); a CTA writes one fp32 partial per
// row block it touches (slot = row block + CTA: along the list either index
// advances at every boundary, so slots never collide), and a second kernel
// sums each row block's partials in K order -- deterministic -- and applies the
// epilogue.  For a row-parallel weight the K order is the shard order, so that
// sum is the g all-reduce ("02 — Tensor Parallelism", "Row-parallel"; "Tensor
// and sequence parallelism", f/g table), with the bias added once after it.
//
// The weight is addressed as [slabs][R][Kt] (slab = shard for row-parallel
// weights, 1 slab otherwise) and K = slabs * Kt runs slab after slab.
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

constexpr int SK_THREADS = 192;
constexpr int SK_PANEL = 128 * 128;     // 128 rows x 128 bytes
constexpr int SK_WTILE = 2 * SK_PANEL;  // 128 rows x 128 K bf16
constexpr int SK_MAX_GRID = 256;

enum : int { ERR_SK_PRODUCER = 0x131, ERR_SK_MMA = 0x132, ERR_SK_EPI = 0x133, ERR_SK_DRAIN = 0x134 };

template <int NB>
struct SkCfg {
  static constexpr int XTILE = 2 * NB * 128;  // NB rows x 128 K bf16, two 64-column panels
  static constexpr int STAGE = SK_WTILE + XTILE;
  static constexpr int STAGES = NB <= 16 ? 6 : 5;
  static constexpr int OFF_BAR = STAGES * STAGE;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
  static constexpr uint32_t TMEM_COLS = 2 * NB < 32 ? 32 : 2 * NB;
};

struct SkArgs {
  int nrb, nku, ku_per_slab;  // row blocks, K units (128 wide) in all, per slab
  float* part;                // [slots][NB][128]
  // fused reduction (cnt non-null): the CTA that writes a row block's last
  // piece sums its pieces in K order and writes y[b][r] = bf16(sum + bias[r])
  int* cnt;                   // [nrb], zero on entry
  const uint16_t* bias;
  uint16_t* y;
  int64_t ldy;
  int B;
  int* err;
  uint64_t timeout_ns;
};

__device__ __forceinline__ uint64_t kdesc(uint32_t base, int panel_bytes, int kk) {
  return ptx::sdesc_sw128(base + (kk >> 2) * panel_bytes + (kk & 3) * 32, 16, 1024);
}

template <int NB>
__device__ __forceinline__ void tmem_ld_nb(uint32_t taddr, float (&v)[NB]);

template <>
__device__ __forceinline__ void tmem_ld_nb<16>(uint32_t taddr, float (&v)[16]) {
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
__device__ __forceinline__ void tmem_ld_nb<32>(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  ptx::tmem_ld32(taddr, r);
  ptx::tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <int NB>
__global__ void __launch_bounds__(SK_THREADS, 1)
    skinny_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                       const SkArgs p) {
  using C = SkCfg<NB>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t dsmem[];
  const uint32_t pad = (1024u - (ptx::smem_addr(dsmem) & 1023u)) & 1023u;
  uint8_t* base = dsmem + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::OFF_BAR);
  uint64_t* full = bars;                // [ST]
  uint64_t* empty = bars + ST;          // [ST]
  uint64_t* acc_full = bars + 2 * ST;   // [2]
  uint64_t* acc_empty = acc_full + 2;   // [2]
  uint64_t* mma_done = acc_full + 4;
  uint64_t* all_done = acc_full + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 6);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ptx::griddep_launch_dependents();
  const int64_t U = static_cast<int64_t>(p.nrb) * p.nku;
  const int G = gridDim.x, k = blockIdx.x;
  const int u0 = static_cast<int>((static_cast<int64_t>(k) * U) / G);
  const int u1 = static_cast<int>((static_cast<int64_t>(k + 1) * U) / G);
  if (u0 >= u1) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&acc_full[b], 1);
      ptx::mbar_init(&acc_empty[b], 128);
    }
    ptx::mbar_init(mma_done, 1);
    ptx::mbar_init(all_done, SK_THREADS);
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

  if (warp == 0) {
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_w);
      ptx::tma_prefetch_desc(&tm_x);
      // The weight tiles of the first ST units do not depend on the previous
      // kernels: stream them while those finish, then wait and add x.
      const int npre = (u1 - u0) < ST ? (u1 - u0) : ST;
      for (int n = 0; n < npre; ++n) {
        const int u = u0 + n;
        const int rb = u / p.nku, ku = u - rb * p.nku;
        const int slab = ku / p.ku_per_slab, kin = (ku - slab * p.ku_per_slab) * 128;
        uint8_t* sw = base + n * C::STAGE;
        ptx::mbar_arrive_expect_tx(&full[n], C::STAGE);
        ptx::tma_load_3d(sw, &tm_w, &full[n], kin, rb * 128, slab);
        ptx::tma_load_3d(sw + SK_PANEL, &tm_w, &full[n], kin + 64, rb * 128, slab);
      }
      ptx::griddep_wait();  // x (and the partial slots) belong to the previous kernels
      for (int n = 0; n < npre; ++n) {
        const int ku = (u0 + n) % p.nku;
        uint8_t* sx = base + n * C::STAGE + SK_WTILE;
        ptx::tma_load_3d(sx, &tm_x, &full[n], ku * 128, 0, 0);
        ptx::tma_load_3d(sx + NB * 128, &tm_x, &full[n], ku * 128 + 64, 0, 0);
      }
      int n = npre;
      for (int u = u0 + npre; u < u1; ++u, ++n) {
        const int st = n % ST;
        if (!ptx::mbar_wait(&empty[st], ((n / ST) & 1) ^ 1u, abort_flag, p.err, ERR_SK_PRODUCER, p.timeout_ns)) break;
        const int rb = u / p.nku, ku = u - rb * p.nku;
        const int slab = ku / p.ku_per_slab, kin = (ku - slab * p.ku_per_slab) * 128;
        uint8_t* sw = base + st * C::STAGE;
        uint8_t* sx = sw + SK_WTILE;
        ptx::mbar_arrive_expect_tx(&full[st], C::STAGE);
        ptx::tma_load_3d(sw, &tm_w, &full[st], kin, rb * 128, slab);
        ptx::tma_load_3d(sw + SK_PANEL, &tm_w, &full[st], kin + 64, rb * 128, slab);
        ptx::tma_load_3d(sx, &tm_x, &full[st], ku * 128, 0, 0);
        ptx::tma_load_3d(sx + NB * 128, &tm_x, &full[st], ku * 128 + 64, 0, 0);
      }
      volatile int never = 0;
      for (int w = (n > ST ? n - ST : 0); w < n; ++w)
        ptx::mbar_wait(&full[w % ST], (w / ST) & 1, &never, p.err, ERR_SK_DRAIN, p.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, NB, false, false);
      const uint32_t a0 = ptx::smem_addr(base);
      int n = 0, piece = 0;
      bool ok = true;
      for (int u = u0; ok && u < u1; ++u, ++n) {
        const int rb = u / p.nku;
        const bool first = (u == u0) || (u - rb * p.nku == 0);
        const bool last = (u + 1 == u1) || ((u + 1) % p.nku == 0);
        const int ab = piece & 1;
        if (first && piece >= 2 &&
            !ptx::mbar_wait(&acc_empty[ab], ((piece >> 1) - 1) & 1, abort_flag, p.err, ERR_SK_MMA, p.timeout_ns)) {
          ok = false;
          break;
        }
        const int st = n % ST;
        if (!ptx::mbar_wait(&full[st], (n / ST) & 1, abort_flag, p.err, ERR_SK_MMA, p.timeout_ns)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sw = a0 + st * C::STAGE, sx = sw + SK_WTILE;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tmem + ab * NB, kdesc(sw, SK_PANEL, kk), kdesc(sx, NB * 128, kk), idesc,
                        (first && kk == 0) ? 0u : 1u);
        ptx::mma_commit(&empty[st]);
        if (last) {
          ptx::mma_commit(&acc_full[ab]);
          ++piece;
        }
      }
      ptx::mma_commit(mma_done);
      volatile int never = 0;
      ptx::mbar_wait(mma_done, 0, &never, p.err, ERR_SK_DRAIN, p.timeout_ns);
    }
  } else {
    // epilogue: TMEM lane = row of the 128-row block, one column per batch row
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    int piece = 0;
    for (int u = u0; u < u1; ++u) {
      const int rb = u / p.nku;
      const bool last = (u + 1 == u1) || ((u + 1) % p.nku == 0);
      if (!last) continue;
      const int ab = piece & 1;
      // no early exit on a failed (bounded) wait: every epilogue thread must
      // reach the same named barriers; the error is already recorded
      ptx::mbar_wait(&acc_full[ab], (piece >> 1) & 1, abort_flag, p.err, ERR_SK_EPI, p.timeout_ns);
      ptx::tc_fence_after();
      float v[NB];
      tmem_ld_nb<NB>(tmem + ab * NB + lane_base, v);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&acc_empty[ab]);
      const int64_t slot = static_cast<int64_t>(rb) + k;
      float* dst = p.part + slot * NB * 128 + row;
#pragma unroll
      for (int b = 0; b < NB; ++b) dst[b * 128] = v[b];
      ++piece;
      if (p.cnt) {
        // pieces of row block rb: CTAs k0..k1 that own units
        const uint32_t uU = static_cast<uint32_t>(U), uG = static_cast<uint32_t>(G);
        auto cta_of = [&](uint32_t x) { return ((x + 1) * uG - 1) / uU; };
        auto owns = [&](uint32_t kk) { return (kk * uU) / uG != ((kk + 1) * uU) / uG; };
        const uint32_t ua = static_cast<uint32_t>(rb) * p.nku;
        const uint32_t k0 = cta_of(ua), k1 = cta_of(ua + p.nku - 1);
        __threadfence();
        __syncwarp();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (row == 0) {
          int npieces = 0;
          for (uint32_t kk = k0; kk <= k1; ++kk) npieces += owns(kk) ? 1 : 0;
          *last_flag = (atomicAdd(p.cnt + rb, 1) == npieces - 1) ? 1 : 0;
        }
        __syncwarp();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (*last_flag) {
          __threadfence();
          float acc[NB];
#pragma unroll
          for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
          for (uint32_t kk = k0; kk <= k1; ++kk) {
            if (!owns(kk)) continue;
            const float* src = p.part + (static_cast<int64_t>(rb) + kk) * NB * 128 + row;
            float t[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) t[b] = b < p.B ? __ldcg(src + b * 128) : 0.0f;
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[b] += t[b];
          }
          const int64_t r = static_cast<int64_t>(rb) * 128 + row;
          const float bv = p.bias ? bf16_bits_to_float(p.bias[r]) : 0.0f;
#pragma unroll
          for (int b = 0; b < NB; ++b)
            if (b < p.B) p.y[b * p.ldy + r] = float_to_bf16_bits(acc[b] + bv);
        }
        __syncwarp();
        asm volatile("bar.sync 1, 128;" ::: "memory");  // last_flag is rewritten by the next piece
      }
    }
  }

  // Teardown through an mbarrier (every thread arrives, then waits) rather
  // than a CTA-wide bar.sync, which the epilogue's named barrier must not
  // disturb; TMEM is freed only after every reader is done.
  ptx::tc_fence_before();
  __syncwarp();
  {
    ptx::mbar_arrive(all_done);
    volatile int never = 0;
    ptx::mbar_wait(all_done, 0, &never, p.err, ERR_SK_DRAIN, p.timeout_ns);
  }
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// CTA whose range holds unit u (32-bit: the host keeps U * G below 2^32).
__device__ __forceinline__ uint32_t sk_cta_of(uint32_t u, uint32_t G, uint32_t U) { return ((u + 1) * G - 1) / U; }

// Sum of row r's partials for batch row b, in K order (CTA order); the loads
// of up to 4 pieces are issued together.
template <int NB>
__device__ __forceinline__ float sk_sum(const SkGemmJob& j, uint32_t G, uint32_t r, int b) {
  const uint32_t nku = static_cast<uint32_t>(j.nku);
  const uint32_t U = static_cast<uint32_t>(j.nrb) * nku;
  const uint32_t rb = r >> 7, row = r & 127u;
  const uint32_t ua = rb * nku;
  const uint32_t k0 = sk_cta_of(ua, G, U), k1 = sk_cta_of(ua + nku - 1, G, U);
  auto owns = [&](uint32_t kk) { return (kk * U) / G != ((kk + 1) * U) / G; };  // else it wrote nothing
  float s = 0.0f;
  uint32_t kk = k0;
  while (kk <= k1) {
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      while (kk <= k1 && !owns(kk)) ++kk;
      v[q] = 0.0f;
      if (kk <= k1) {
        v[q] = __ldcg(j.part + ((static_cast<size_t>(rb) + kk) * NB + b) * 128 + row);
        ++kk;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) s += v[q];
  }
  return s;
}

template <int NB>
__global__ void __launch_bounds__(256) skinny_reduce_kernel(const SkGemmJob j, int G) {
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  if (j.epi == SK_EPI_QKV && blockIdx.x == 0) decode_check_positions(j.pos, j.B, j.L_max, j.err);
  const int64_t n = static_cast<int64_t>(j.R) * j.B;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(idx / j.R);
    const int64_t r = idx - static_cast<int64_t>(b) * j.R;
    float v = sk_sum<NB>(j, static_cast<uint32_t>(G), static_cast<uint32_t>(r), b);
    if (j.bias) v += bf16_bits_to_float(j.bias[r]);
    if (j.epi == SK_EPI_BF16) {
      j.y[static_cast<int64_t>(b) * j.ldy + r] = float_to_bf16_bits(v);
    } else {  // SK_EPI_QKV: route the coordinate to Q or to the shard's cache copy (fp16)
      const __half hv = __float2half_rn(v);
      const uint16_t bits = *reinterpret_cast<const uint16_t*>(&hv);
      const int64_t i = r / j.R_t, lr = r - i * j.R_t;
      const int64_t qw = static_cast<int64_t>(j.q_t) * 128, kvw = static_cast<int64_t>(j.kv_t) * 128;
      if (lr < qw) {
        j.q[(static_cast<int64_t>(b) * j.nh + i * j.q_t) * 128 + lr] = bits;
      } else {
        const int64_t p = j.pos[b];
        if (p >= 0 && p < j.L_max) {
          const int64_t w2 = lr - qw;
          const int part = w2 >= kvw ? 1 : 0;
          const int64_t w3 = w2 - part * kvw;
          const int64_t jl = w3 >> 7, e = w3 & 127;
          uint16_t* cache = part ? j.Vc : j.Kc;
          cache[(((i * j.kv_t + jl) * j.B + b) * j.L_max + p) * 128 + e] = bits;
        }
      }
    }
  }
}

template <int NB>
tp_status launch_skinny(const SkGemmJob& j, cudaStream_t s) {
  CUtensorMap mw, mx;
  const uint64_t Kt = static_cast<uint64_t>(j.ku_per_slab) * 128;
  const uint64_t K = Kt * j.slabs;
  if (!make_map_3d_bf16(&mw, j.W, Kt, j.R, j.slabs, Kt * 2, Kt * j.R * 2, 64, 128) ||
      !make_map_3d_bf16(&mx, j.x, K, j.B, 1, j.ldx * 2, j.ldx * j.B * 2, 64, NB))
    return TP_FAIL_DETAIL("cuTensorMapEncodeTiled failed for the skinny GEMM");
  static bool configured[64] = {};
  int dev = 0;
  TP_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return TP_ERR_CUDA;
  if (!configured[dev]) {
    TP_CUDA_CHECK(cudaFuncSetAttribute(skinny_gemm_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SkCfg<NB>::SMEM));
    configured[dev] = true;
  }
  SkArgs a{};
  a.nrb = j.nrb;
  a.nku = j.nku;
  a.ku_per_slab = j.ku_per_slab;
  a.part = j.part;
  a.cnt = j.cnt;
  a.bias = j.bias;
  a.y = j.y;
  a.ldy = j.ldy;
  a.B = j.B;
  a.err = device_error_word();
  a.timeout_ns = wait_timeout_ns();
  const int64_t U = static_cast<int64_t>(j.nrb) * j.nku;
  int64_t G = device_sm_count();
  if (G > SK_MAX_GRID) G = SK_MAX_GRID;
  if (G > U) G = U;
  TP_CUDA_CHECK(launch_pdl(skinny_gemm_kernel<NB>, dim3(static_cast<unsigned>(G)), dim3(SK_THREADS),
                           SkCfg<NB>::SMEM, s, mw, mx, a));
  count_launch();
  if (j.cnt) return TP_OK;  // reduced in the GEMM kernel
  const int64_t n = static_cast<int64_t>(j.R) * j.B;
  int64_t rg = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  if (rg > cap) rg = cap;
  TP_CUDA_CHECK(launch_pdl(skinny_reduce_kernel<NB>, dim3(static_cast<unsigned>(rg)), dim3(256), 0, s, j,
                           static_cast<int>(G)));
  count_launch();
  return TP_OK;
}

}  // namespace

size_t skinny_part_floats(int64_t R, int B) {
  const int NB = B <= 16 ? 16 : 32;
  return static_cast<size_t>(R / 128 + SK_MAX_GRID) * NB * 128;
}

bool skinny_ok(int64_t R, int64_t Kt, int B) {
  // (R/128) * (K/128) units times up to SK_MAX_GRID + 1 CTAs must stay below 2^32
  return B >= 1 && B <= 32 && R > 0 && R % 128 == 0 && Kt % 128 == 0 && R <= (1LL << 31) &&
         (R / 128) * (Kt / 128) * 8 <= (1LL << 23);
}

tp_status run_skinny_gemm(SkGemmJob j, cudaStream_t s) {
  if (!skinny_ok(j.R, static_cast<int64_t>(j.ku_per_slab) * 128 * j.slabs, j.B) || j.slabs < 1) return TP_ERR_SHAPE;
  if (j.cnt && j.epi != SK_EPI_BF16) return TP_ERR_UNSUPPORTED;
  if (!aligned16(j.W) || !aligned16(j.x) || !aligned16(j.part) || j.ldx % 8 != 0) return TP_ERR_ALIGN;
  j.nrb = static_cast<int>(j.R / 128);
  j.nku = j.ku_per_slab * j.slabs;
  return j.B <= 16 ? launch_skinny<16>(j, s) : launch_skinny<32>(j, s);
}

}  // namespace tp
