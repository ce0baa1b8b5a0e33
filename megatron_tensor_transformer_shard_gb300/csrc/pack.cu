// Shard-layout packing: bit-exact permutations of bf16 weights into the
// per-shard slices each logical rank owns ("Tensor and sequence parallelism",
// section "The implementation": rank r keeps w1[cols] and w2[:, cols];
// "02 — Tensor Parallelism", section "The attention pairing": each rank owns
// n_heads/t heads of Q, K and V).
//
// Every packed layout is a set of output rows, each row r being one column of
// an unpacked matrix read down a contiguous run of its rows:
//     packed[r][k] = src_r[(rowbase(r) + k) * ld + col(r)],   0 <= k < row_len
// so all of them run through one 32x32 shared-memory transpose kernel; the
// unpack direction is the same map with reads and writes swapped.
#include <cuda_runtime.h>

#include "devmath.cuh"
#include "internal.h"

namespace tp {
namespace {

enum PackKind : int { PK_COL = 0, PK_ROW = 1, PK_SWIGLU = 2, PK_QKV = 3, PK_QKV_GQA = 4 };

struct PackMap {
  int kind;
  int64_t R;        // packed rows
  int64_t row_len;  // packed row length
  int64_t ld;       // row stride of the unpacked source
  int64_t Ft;       // F/t (COL, ROW, SWIGLU)
  int64_t h;        // ROW: columns of W_down; SWIGLU: rows of W_gate
  int64_t d;        // QKV model dim
  int64_t dt;       // QKV d/t
  int head_dim;
  int heads_per_shard;
  int group;
  int n_heads, n_kv, kv_t;  // QKV_GQA
  int64_t R_t;              // QKV_GQA rows per shard
};

// Source column and row base for packed row r; `part` selects the source matrix.
__device__ __forceinline__ void map_row(const PackMap& m, int64_t r, int64_t& col, int64_t& rowbase, int& part) {
  part = 0;
  rowbase = 0;
  switch (m.kind) {
    case PK_COL:  // [t][F/t][h] == W^T : packed row r is column r of W (h, F)
      col = r;
      break;
    case PK_ROW: {  // [t][h][F/t] : row (i, c) holds W[i*Ft + k][c]
      const int64_t i = r / m.h;
      col = r - i * m.h;
      rowbase = i * m.Ft;
      break;
    }
    case PK_SWIGLU: {  // [t][Ft/g][2][g][h]
      const int64_t per_shard = 2 * m.Ft;
      const int64_t i = r / per_shard;
      const int64_t rem = r - i * per_shard;
      const int64_t q = rem / (2 * m.group);
      const int64_t w = rem - q * 2 * m.group;
      part = static_cast<int>(w / m.group);
      col = i * m.Ft + q * m.group + (w - part * m.group);
      break;
    }
    case PK_QKV_GQA: {  // [t][R_t][d], rows [Q heads of shard i | its K heads | its V heads]
      const int64_t i = r / m.R_t;
      const int64_t rr = r - i * m.R_t;
      const int64_t qw = static_cast<int64_t>(m.heads_per_shard) * m.head_dim;
      if (rr < qw) {
        col = i * qw + rr;
      } else {
        const int64_t kvw = static_cast<int64_t>(m.kv_t) * m.head_dim;
        const int64_t w2 = rr - qw;
        const int64_t pt = w2 / kvw;  // 0: K, 1: V
        const int64_t w3 = w2 - pt * kvw;
        const int64_t jl = w3 / m.head_dim, e = w3 - jl * m.head_dim;
        // KV heads of shard i: the groups of its query heads; one replicated head when n_kv < t
        const int64_t t = m.R / m.R_t;
        const int64_t first = m.n_kv >= t ? i * m.kv_t : (i * m.n_kv) / t;
        col = static_cast<int64_t>(m.n_heads) * m.head_dim + pt * m.n_kv * m.head_dim + (first + jl) * m.head_dim + e;
      }
      break;
    }
    default: {  // PK_QKV: [t][3d/t][d], rows [Q_i | K_i | V_i]
      const int64_t per_shard = 3 * m.dt;
      const int64_t i = r / per_shard;
      const int64_t rr = r - i * per_shard;
      const int64_t p = rr / m.dt;
      const int64_t w = rr - p * m.dt;
      const int64_t jj = w / m.head_dim;
      const int64_t e = w - jj * m.head_dim;
      col = p * m.d + (i * m.heads_per_shard + jj) * m.head_dim + e;
      break;
    }
  }
}

constexpr int TILE = 32;

// dir 0: pack (unpacked -> packed); dir 1: unpack.
__global__ void pack_kernel(PackMap m, int dir, const uint16_t* __restrict__ u0, const uint16_t* __restrict__ u1,
                            uint16_t* __restrict__ w0, uint16_t* __restrict__ w1, const uint16_t* __restrict__ p_in,
                            uint16_t* __restrict__ p_out) {
  __shared__ uint16_t tile[TILE][TILE + 1];
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * TILE;
  const int64_t k0 = static_cast<int64_t>(blockIdx.y) * TILE;
  const int tx = threadIdx.x, ty = threadIdx.y;
  if (dir == 0) {
    // read the unpacked source: consecutive tx -> consecutive packed rows -> (mostly) consecutive columns
    const int64_t r = r0 + tx;
    if (r < m.R) {
      int64_t col, rowbase;
      int part;
      map_row(m, r, col, rowbase, part);
      const uint16_t* src = part ? u1 : u0;
      for (int k = ty; k < TILE; k += blockDim.y) {
        const int64_t kk = k0 + k;
        if (kk < m.row_len) tile[k][tx] = src[(rowbase + kk) * m.ld + col];
      }
    }
    __syncthreads();
    for (int rr = ty; rr < TILE; rr += blockDim.y) {
      const int64_t r2 = r0 + rr;
      const int64_t kk = k0 + tx;
      if (r2 < m.R && kk < m.row_len) p_out[r2 * m.row_len + kk] = tile[tx][rr];
    }
  } else {
    for (int rr = ty; rr < TILE; rr += blockDim.y) {
      const int64_t r2 = r0 + rr;
      const int64_t kk = k0 + tx;
      if (r2 < m.R && kk < m.row_len) tile[tx][rr] = p_in[r2 * m.row_len + kk];
    }
    __syncthreads();
    const int64_t r = r0 + tx;
    if (r < m.R) {
      int64_t col, rowbase;
      int part;
      map_row(m, r, col, rowbase, part);
      uint16_t* dst = part ? w1 : w0;
      for (int k = ty; k < TILE; k += blockDim.y) {
        const int64_t kk = k0 + k;
        if (kk < m.row_len) dst[(rowbase + kk) * m.ld + col] = tile[k][tx];
      }
    }
  }
}

__global__ void gather_bias_kernel(PackMap m, const uint16_t* __restrict__ b, uint16_t* __restrict__ out) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= m.R) return;
  int64_t col, rowbase;
  int part;
  map_row(m, r, col, rowbase, part);
  out[r] = b[col];
}

tp_status launch_pack(const PackMap& m, int dir, const uint16_t* u0, const uint16_t* u1, uint16_t* w0,
                      uint16_t* w1, const uint16_t* p_in, uint16_t* p_out, cudaStream_t s) {
  if (m.R == 0 || m.row_len == 0) return TP_OK;
  dim3 grid(static_cast<unsigned>((m.R + TILE - 1) / TILE), static_cast<unsigned>((m.row_len + TILE - 1) / TILE));
  if (grid.y > 65535u) return TP_ERR_SHAPE;
  TP_RETURN_IF(ready());
  pack_kernel<<<grid, dim3(TILE, 8), 0, s>>>(m, dir, u0, u1, w0, w1, p_in, p_out);
  TP_LAUNCHED();
  return TP_OK;
}

bool bad_t(int64_t n, int t) { return t < 1 || n % t != 0; }

}  // namespace

// dir 0: src = unpacked W, dst = packed; dir 1: src = packed, dst = unpacked W.
tp_status pack_col(const uint16_t* src, int64_t h, int64_t F, int t, uint16_t* dst, int dir, cudaStream_t s) {
  if (!src || !dst || h < 0 || F < 0 || t < 1) return TP_ERR_INVALID_ARG;
  if (bad_t(F, t)) return TP_ERR_SHAPE;
  PackMap m{};
  m.kind = PK_COL;
  m.R = F;
  m.row_len = h;
  m.ld = F;
  m.Ft = F / t;
  return dir == 0 ? launch_pack(m, 0, src, nullptr, nullptr, nullptr, nullptr, dst, s)
                  : launch_pack(m, 1, nullptr, nullptr, dst, nullptr, src, nullptr, s);
}

tp_status pack_row(const uint16_t* src, int64_t F, int64_t h, int t, uint16_t* dst, int dir, cudaStream_t s) {
  if (!src || !dst || h < 0 || F < 0 || t < 1) return TP_ERR_INVALID_ARG;
  if (bad_t(F, t)) return TP_ERR_SHAPE;
  PackMap m{};
  m.kind = PK_ROW;
  m.R = static_cast<int64_t>(t) * h;
  m.row_len = F / t;
  m.ld = h;
  m.Ft = F / t;
  m.h = h;
  return dir == 0 ? launch_pack(m, 0, src, nullptr, nullptr, nullptr, nullptr, dst, s)
                  : launch_pack(m, 1, nullptr, nullptr, dst, nullptr, src, nullptr, s);
}

tp_status pack_swiglu(const uint16_t* Wg, const uint16_t* Wu, int64_t h, int64_t F, int t, uint16_t* Wp,
                      cudaStream_t s) {
  if (!Wg || !Wu || !Wp || h < 0 || F < 0 || t < 1) return TP_ERR_INVALID_ARG;
  if (bad_t(F, t) || (F / t) % 128 != 0) return TP_ERR_SHAPE;
  PackMap m{};
  m.kind = PK_SWIGLU;
  m.R = 2 * F;
  m.row_len = h;
  m.ld = F;
  m.Ft = F / t;
  m.h = h;
  m.group = 128;
  return launch_pack(m, 0, Wg, Wu, nullptr, nullptr, nullptr, Wp, s);
}

static bool qkv_map(PackMap& m, int64_t d, int n_heads, int head_dim, int t) {
  if (t < 1 || n_heads < 1 || head_dim < 1 || n_heads % t != 0 || static_cast<int64_t>(n_heads) * head_dim != d)
    return false;
  m = PackMap{};
  m.kind = PK_QKV;
  m.R = 3 * d;
  m.row_len = d;
  m.ld = 3 * d;
  m.d = d;
  m.dt = d / t;
  m.head_dim = head_dim;
  m.heads_per_shard = n_heads / t;
  return true;
}

static bool qkv_gqa_map(PackMap& m, int64_t d, int n_heads, int n_kv, int head_dim, int t) {
  if (t < 1 || n_heads < 1 || n_kv < 1 || head_dim < 1 || d < 0) return false;
  if (n_heads % t != 0 || n_heads % n_kv != 0) return false;
  if (n_kv >= t ? (n_kv % t != 0) : (t % n_kv != 0)) return false;
  m = PackMap{};
  m.kind = PK_QKV_GQA;
  m.n_heads = n_heads;
  m.n_kv = n_kv;
  m.kv_t = n_kv >= t ? n_kv / t : 1;
  m.heads_per_shard = n_heads / t;
  m.head_dim = head_dim;
  m.R_t = static_cast<int64_t>(m.heads_per_shard + 2 * m.kv_t) * head_dim;
  m.R = m.R_t * t;
  m.row_len = d;
  m.ld = static_cast<int64_t>(n_heads + 2 * n_kv) * head_dim;
  return true;
}

// dir 1 (unpack) writes a replicated KV column once per copy, the same bits each time.
tp_status pack_qkv_gqa(const uint16_t* src, int64_t d, int n_heads, int n_kv, int head_dim, int t, uint16_t* dst,
                       int dir, cudaStream_t s) {
  if (!src || !dst || d < 0) return TP_ERR_INVALID_ARG;
  PackMap m;
  if (!qkv_gqa_map(m, d, n_heads, n_kv, head_dim, t)) return TP_ERR_SHAPE;
  return dir == 0 ? launch_pack(m, 0, src, nullptr, nullptr, nullptr, nullptr, dst, s)
                  : launch_pack(m, 1, nullptr, nullptr, dst, nullptr, src, nullptr, s);
}

tp_status pack_qkv_gqa_bias(const uint16_t* b, int n_heads, int n_kv, int head_dim, int t, uint16_t* bp,
                            cudaStream_t s) {
  if (!b || !bp) return TP_ERR_INVALID_ARG;
  PackMap m;
  if (!qkv_gqa_map(m, 0, n_heads, n_kv, head_dim, t)) return TP_ERR_SHAPE;
  if (m.R == 0) return TP_OK;
  TP_RETURN_IF(ready());
  gather_bias_kernel<<<static_cast<unsigned>((m.R + 255) / 256), 256, 0, s>>>(m, b, bp);
  TP_LAUNCHED();
  return TP_OK;
}

// Gradient of the unsplit W_qkv from the shards' packed gradients: column c
// of (d, (n_heads + 2 n_kv) head_dim) sums the packed rows of every shard copy
// that holds it, in shard order.  32x32 tiles: reads run along d (coalesced in
// the packed layout), writes along the columns.
struct GqaGradMap {
  int n_heads, n_kv, head_dim, t, q_t, kv_t, copies;
  int64_t d, C, R_t;
};

// Shard and packed row of copy `cp` of unsplit column c.
__device__ __forceinline__ void gqa_owner(const GqaGradMap& m, int64_t c, int cp, int& shard, int64_t& row) {
  const int64_t nq = static_cast<int64_t>(m.n_heads) * m.head_dim;
  const int64_t nk = static_cast<int64_t>(m.n_kv) * m.head_dim;
  if (c < nq) {
    const int64_t qh = c / m.head_dim, e = c - qh * m.head_dim;
    shard = static_cast<int>(qh / m.q_t);
    row = (qh - static_cast<int64_t>(shard) * m.q_t) * m.head_dim + e;
    return;
  }
  const int part = c < nq + nk ? 0 : 1;  // K or V
  const int64_t w = c - nq - part * nk;
  const int64_t j = w / m.head_dim, e = w - j * m.head_dim;
  const int64_t base = (static_cast<int64_t>(m.q_t) + part * m.kv_t) * m.head_dim;
  if (m.n_kv >= m.t) {
    shard = static_cast<int>(j / m.kv_t);
    row = base + (j - static_cast<int64_t>(shard) * m.kv_t) * m.head_dim + e;
  } else {
    shard = static_cast<int>(j * (m.t / m.n_kv) + cp);
    row = base + e;
  }
}

__global__ void gqa_grad_kernel(GqaGradMap m, const float* __restrict__ dWp, float* __restrict__ dW, int accumulate) {
  __shared__ float tile[TILE][TILE + 1];
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * TILE, k0 = static_cast<int64_t>(blockIdx.y) * TILE;
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (int cc = ty; cc < TILE; cc += blockDim.y) {
    const int64_t c = c0 + cc, k = k0 + tx;
    if (c < m.C && k < m.d) {
      const int64_t nq = static_cast<int64_t>(m.n_heads) * m.head_dim;
      const int ncopy = c < nq ? 1 : m.copies;
      float acc = 0.0f;
      for (int cp = 0; cp < ncopy; ++cp) {
        int shard;
        int64_t row;
        gqa_owner(m, c, cp, shard, row);
        acc += dWp[(static_cast<int64_t>(shard) * m.R_t + row) * m.d + k];
      }
      tile[cc][tx] = acc;
    }
  }
  __syncthreads();
  for (int kk = ty; kk < TILE; kk += blockDim.y) {
    const int64_t k = k0 + kk, c = c0 + tx;
    if (c < m.C && k < m.d) {
      float* o = dW + k * m.C + c;
      *o = accumulate ? *o + tile[tx][kk] : tile[tx][kk];
    }
  }
}

tp_status reduce_qkv_gqa_grad(const float* dWp, int64_t d, int n_heads, int n_kv, int head_dim, int t, float* dW,
                              int accumulate, cudaStream_t s) {
  if (!dWp || !dW || d < 0 || head_dim < 1 || t < 1 || n_heads < 1 || n_kv < 1) return TP_ERR_INVALID_ARG;
  if (n_heads % t != 0 || n_heads % n_kv != 0 || (n_kv >= t ? n_kv % t != 0 : t % n_kv != 0)) return TP_ERR_SHAPE;
  GqaGradMap m{};
  m.n_heads = n_heads;
  m.n_kv = n_kv;
  m.head_dim = head_dim;
  m.t = t;
  m.q_t = n_heads / t;
  m.kv_t = n_kv >= t ? n_kv / t : 1;
  m.copies = n_kv >= t ? 1 : t / n_kv;
  m.d = d;
  m.C = static_cast<int64_t>(n_heads + 2 * n_kv) * head_dim;
  m.R_t = static_cast<int64_t>(m.q_t + 2 * m.kv_t) * head_dim;
  if (d == 0) return TP_OK;
  dim3 grid(static_cast<unsigned>((m.C + TILE - 1) / TILE), static_cast<unsigned>((d + TILE - 1) / TILE));
  if (grid.y > 65535u) return TP_ERR_SHAPE;
  TP_RETURN_IF(ready());
  gqa_grad_kernel<<<grid, dim3(TILE, 8), 0, s>>>(m, dWp, dW, accumulate);
  TP_LAUNCHED();
  return TP_OK;
}

tp_status pack_qkv(const uint16_t* src, int64_t d, int n_heads, int head_dim, int t, uint16_t* dst, int dir,
                   cudaStream_t s) {
  if (!src || !dst || d < 0) return TP_ERR_INVALID_ARG;
  PackMap m;
  if (!qkv_map(m, d, n_heads, head_dim, t)) return TP_ERR_SHAPE;
  return dir == 0 ? launch_pack(m, 0, src, nullptr, nullptr, nullptr, nullptr, dst, s)
                  : launch_pack(m, 1, nullptr, nullptr, dst, nullptr, src, nullptr, s);
}

tp_status pack_qkv_bias(const uint16_t* b, int64_t d, int n_heads, int head_dim, int t, uint16_t* bp,
                        cudaStream_t s) {
  if (!b || !bp || d < 0) return TP_ERR_INVALID_ARG;
  PackMap m;
  if (!qkv_map(m, d, n_heads, head_dim, t)) return TP_ERR_SHAPE;
  if (m.R == 0) return TP_OK;
  TP_RETURN_IF(ready());
  gather_bias_kernel<<<static_cast<unsigned>((m.R + 255) / 256), 256, 0, s>>>(m, b, bp);
  TP_LAUNCHED();
  return TP_OK;
}

namespace {
// bf16 -> IEEE fp16, 8 values per thread (n % 8 == 0 handled by the host; a tail loop
// takes the rest).  Round to nearest even; bf16 values below fp16's normal range become
// fp16 subnormals (or zero under 2^-25), values above 65504 become infinity.
__global__ void bf16_to_f16_kernel(const uint16_t* __restrict__ src, int64_t n, uint16_t* __restrict__ dst) {
  const int64_t n8 = n / 8;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 w = reinterpret_cast<const uint4*>(src)[i];
    float a0, a1, b0, b1, c0, c1, d0, d1;
    unpack_bf16x2(w.x, a0, a1);
    unpack_bf16x2(w.y, b0, b1);
    unpack_bf16x2(w.z, c0, c1);
    unpack_bf16x2(w.w, d0, d1);
    reinterpret_cast<uint4*>(dst)[i] =
        make_uint4(pack_f16x2(a0, a1), pack_f16x2(b0, b1), pack_f16x2(c0, c1), pack_f16x2(d0, d1));
  }
  if (blockIdx.x == 0 && threadIdx.x < n - n8 * 8) {
    const int64_t i = n8 * 8 + threadIdx.x;
    const __half h = __float2half_rn(bf16_bits_to_float(src[i]));
    dst[i] = *reinterpret_cast<const uint16_t*>(&h);
  }
}
}  // namespace

tp_status run_bf16_to_f16(const uint16_t* src, int64_t n, uint16_t* dst, cudaStream_t s) {
  if (n < 0) return TP_ERR_INVALID_ARG;
  if (n == 0) return TP_OK;
  if (!src || !dst) return TP_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return TP_ERR_ALIGN;
  TP_RETURN_IF(ready());
  int64_t blocks = (n / 8 + 255) / 256;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  bf16_to_f16_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(src, n, dst);
  TP_LAUNCHED();
  return TP_OK;
}

}  // namespace tp
