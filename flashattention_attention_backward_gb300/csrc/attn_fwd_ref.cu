// attn_fwd_ref: a plain fp32 attention forward that produces what the
// backward consumes: O (bf16) and the natural-log row statistic LSE (fp32)
// ("反向传播算法详解" §1.3; "解析 FlashAttention（3）" §1.1, §3.2 eq. 9 with
// LSE = m + ln l).
//
// One CTA computes 64 query rows of one head against 64-key tiles of its KV
// head, with the running (max, sum) rescaling over key tiles. Scores and the
// P.V products are fp32 SIMT arithmetic with accurate expf/logf/tanhf; the
// per-row running sum is kept in double so that LSE stays within a few ulp.
// This kernel is a reference-quality producer of the saved tensors, not the
// tuned path.
#include <cstdint>
#include <cuda_bf16.h>
#include <math_constants.h>

#include "attn_common.cuh"
#include "philox.cuh"

namespace attn {
namespace fwd {

constexpr int kBM = 64;
constexpr int kBN = 64;
constexpr int kThreads = 256;
constexpr int kPStride = kBN + 4;

template <int D>
struct Smem {
  static constexpr int kQt = 0;                   // [D][64] fp32, Q transposed
  static constexpr int kKt = kQt + D * kBM * 4;   // [D][64] fp32, K transposed
  static constexpr int kV = kKt + D * kBN * 4;    // [64][D] fp32
  static constexpr int kP = kV + kBN * D * 4;     // [64][68] fp32
  static constexpr int kBytes = kP + kBM * kPStride * 4;
};

struct Params {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* o;
  float* lse;
  int B, H, H_kv, N;
  int q_blocks;
  float scale;
  float softcap;  // <= 0: disabled
  // visibility band: key j is visible to query i iff
  // i - win_left <= j <= i + win_right (causal: win_right = 0; an unbounded
  // side holds N)
  int win_left, win_right;
  int dropout;    // 0: off; else the keep mask of philox.cuh scales P in O = P V
  Dropout drop;
};

__device__ __forceinline__ void load8(const __nv_bfloat16* src, bool ok, float (&f)[8]) {
  if (ok) {
    const uint4 u = *reinterpret_cast<const uint4*>(src);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] = __uint_as_float(w[e] << 16);
      f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = 0.f;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) attn_fwd_ref_kernel(const Params p) {
  using S = Smem<D>;
  extern __shared__ __align__(16) uint8_t smem[];
  float* sQt = reinterpret_cast<float*>(smem + S::kQt);
  float* sKt = reinterpret_cast<float*>(smem + S::kKt);
  float* sV = reinterpret_cast<float*>(smem + S::kV);
  float* sP = reinterpret_cast<float*>(smem + S::kP);

  const int qb = blockIdx.x % p.q_blocks;
  const long long bh = blockIdx.x / p.q_blocks;
  const int b = static_cast<int>(bh / p.H);
  const int h = static_cast<int>(bh % p.H);
  const long long kvh = static_cast<long long>(b) * p.H_kv + h / (p.H / p.H_kv);
  const int m0 = qb * kBM;
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  constexpr int kOC = D / 16;  // output columns per thread

  const __nv_bfloat16* qg = p.q + bh * p.N * D;
  const __nv_bfloat16* kg = p.k + kvh * p.N * D;
  const __nv_bfloat16* vg = p.v + kvh * p.N * D;

  for (int idx = tid; idx < kBM * (D / 8); idx += kThreads) {
    const int row = idx % kBM, kc = idx / kBM;
    float f[8];
    load8(qg + static_cast<long long>(m0 + row) * D + kc * 8, m0 + row < p.N, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) sQt[(kc * 8 + e) * kBM + row] = f[e];
  }

  float m_run[4], o[4][kOC];
  double l_run[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m_run[i] = -CUDART_INF_F;
    l_run[i] = 0.0;
#pragma unroll
    for (int c = 0; c < kOC; ++c) o[i][c] = 0.f;
  }

  const int n_tiles = (p.N + kBN - 1) / kBN;
  const int first_tile = max(0, m0 - p.win_left) / kBN;
  const int last_tile = min(n_tiles - 1, (m0 + kBM - 1 + p.win_right) / kBN);
  for (int kt = first_tile; kt <= last_tile; ++kt) {
    const int n0 = kt * kBN;
    __syncthreads();  // previous tile's sKt / sV / sP reads are done
    for (int idx = tid; idx < kBN * (D / 8); idx += kThreads) {
      const int row = idx % kBN, kc = idx / kBN;
      float f[8];
      load8(kg + static_cast<long long>(n0 + row) * D + kc * 8, n0 + row < p.N, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) sKt[(kc * 8 + e) * kBN + row] = f[e];
    }
    for (int idx = tid; idx < kBN * (D / 8); idx += kThreads) {
      const int row = idx / (D / 8), kc = idx % (D / 8);
      float f[8];
      load8(vg + static_cast<long long>(n0 + row) * D + kc * 8, n0 + row < p.N, f);
      float4* dst = reinterpret_cast<float4*>(sV + row * D + kc * 8);
      dst[0] = make_float4(f[0], f[1], f[2], f[3]);
      dst[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    __syncthreads();

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 8
    for (int kk = 0; kk < D; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(sQt + kk * kBM + ty * 4);
      const float4 bb = *reinterpret_cast<const float4*>(sKt + kk * kBN + tx * 4);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }

    // dropout keep bits: bit i of keep[j] for rows m0 + 4 ty + i, key
    // n0 + 4 tx + j (one Philox call covers the four rows of a key)
    uint32_t keep[4] = {0xFu, 0xFu, 0xFu, 0xFu};
    if (p.dropout) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const PhiloxOut r = philox4x32_10(static_cast<uint32_t>((m0 + ty * 4) >> 2),
                                          static_cast<uint32_t>(n0 + tx * 4 + j),
                                          static_cast<uint32_t>(bh), 0u, p.drop.seed_lo,
                                          p.drop.seed_hi);
        keep[j] = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) keep[j] |= (r.w[i] >= p.drop.threshold ? 1u : 0u) << i;
      }
    }
    float alpha[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int qrow = m0 + ty * 4 + i;
      float z[4];
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = n0 + tx * 4 + j;
        float s = acc[i][j] * p.scale;
        if (p.softcap > 0.f) s = p.softcap * tanhf(s / p.softcap);
        const bool ok = key < p.N && key - qrow <= p.win_right && qrow - key <= p.win_left;
        z[j] = ok ? s : -CUDART_INF_F;
        mx = fmaxf(mx, z[j]);
      }
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m_run[i], mx);
      const float shift = m_new == -CUDART_INF_F ? 0.f : m_new;
      alpha[i] = expf(m_run[i] - shift);
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float pv = expf(z[j] - shift);
        // the row sum (hence LSE) is that of P; O takes the dropped P
        sP[(ty * 4 + i) * kPStride + tx * 4 + j] =
            p.dropout ? ((keep[j] >> i) & 1u ? pv * p.drop.inv_keep : 0.f) : pv;
        rs += pv;
      }
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
      l_run[i] = l_run[i] * static_cast<double>(alpha[i]) + static_cast<double>(rs);
      m_run[i] = m_new;
    }
    __syncthreads();

#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < kOC; ++c) o[i][c] *= alpha[i];
    for (int key = 0; key < kBN; ++key) {
      float pv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pv[i] = sP[(ty * 4 + i) * kPStride + key];
#pragma unroll
      for (int cg = 0; cg < kOC / 4; ++cg) {
        const float4 vv = *reinterpret_cast<const float4*>(sV + key * D + cg * 64 + tx * 4);
        const float vv4[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[i][cg * 4 + e] = fmaf(pv[i], vv4[e], o[i][cg * 4 + e]);
      }
    }
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int qrow = m0 + ty * 4 + i;
    if (qrow >= p.N) continue;
    const double l = l_run[i];
    const float inv = l > 0.0 ? static_cast<float>(1.0 / l) : 0.f;
    __nv_bfloat16* orow = p.o + (bh * p.N + qrow) * D;
#pragma unroll
    for (int cg = 0; cg < kOC / 4; ++cg) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(o[i][cg * 4 + 0] * inv, o[i][cg * 4 + 1] * inv);
      __nv_bfloat162 hi = __floats2bfloat162_rn(o[i][cg * 4 + 2] * inv, o[i][cg * 4 + 3] * inv);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(orow + cg * 64 + tx * 4) = u;
    }
    if (tx == 0)
      p.lse[bh * p.N + qrow] =
          l > 0.0 ? static_cast<float>(static_cast<double>(m_run[i]) + log(l)) : -CUDART_INF_F;
  }
}

template <int D>
int launch(const Params& p, cudaStream_t s) {
  static std::atomic<bool> configured[kMaxTrackedDevices];
  if (!set_smem_limit_once(attn_fwd_ref_kernel<D>, Smem<D>::kBytes, configured))
    return ATTN_ERR_LAUNCH;
  const long long grid = static_cast<long long>(p.q_blocks) * p.B * p.H;
  if (grid > 0x7fffffffLL) return ATTN_ERR_TOO_LARGE;
  attn_fwd_ref_kernel<D><<<static_cast<unsigned>(grid), kThreads, Smem<D>::kBytes, s>>>(p);
  return launch_status();
}

}  // namespace fwd
}  // namespace attn

using namespace attn;

namespace attn {
namespace fwd {

int run(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv,
        int N, int d, float scale, int causal, float softcap, float p_drop,
        unsigned long long seed, void* stream, int window_left = -1, int window_right = -1) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  int rc = check_shape(B, H, H_kv, N, d);
  if (rc != ATTN_OK) return rc;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || scale == 0.f || std::isnan(softcap)) return ATTN_ERR_SHAPE;
  if (!(p_drop >= 0.f && p_drop < 1.f)) return ATTN_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_ALIGN;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  Params p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.H_kv = H_kv;
  p.N = N;
  p.q_blocks = (N + kBM - 1) / kBM;
  p.scale = scale;
  p.softcap = softcap > 0.f ? softcap : 0.f;
  // a negative or wider-than-N side of the window is unbounded (N)
  p.win_left = (window_left < 0 || window_left > N) ? N : window_left;
  p.win_right = causal ? 0 : ((window_right < 0 || window_right > N) ? N : window_right);
  p.dropout = p_drop > 0.f ? 1 : 0;
  p.drop.seed_lo = static_cast<uint32_t>(seed);
  p.drop.seed_hi = static_cast<uint32_t>(seed >> 32);
  p.drop.threshold = dropout_threshold(p_drop);
  p.drop.inv_keep = 1.f / (1.f - p_drop);
  p.drop.keep = 1.f - p_drop;
  p.drop.log2_inv_keep =
      static_cast<float>(-std::log2(1.0 - static_cast<double>(p_drop)));
  cudaStream_t s = as_stream(stream);
  if (d == 256) return launch<256>(p, s);
  return d == 128 ? launch<128>(p, s) : launch<64>(p, s);
}

}  // namespace fwd
}  // namespace attn

extern "C" int attn_fwd_ref(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int H_kv, int N, int d, float scale, int causal,
                            float softcap, void* stream) {
  return fwd::run(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, 0.f, 0ull, stream);
}

extern "C" int attn_fwd_ref_dropout(const void* q, const void* k, const void* v, void* o,
                                    float* lse, int B, int H, int H_kv, int N, int d, float scale,
                                    int causal, float softcap, float p_drop,
                                    unsigned long long seed, void* stream) {
  return fwd::run(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, p_drop, seed,
                  stream);
}

extern "C" int attn_fwd_ref_local(const void* q, const void* k, const void* v, void* o,
                                  float* lse, int B, int H, int H_kv, int N, int d, float scale,
                                  int causal, float softcap, int window_left, int window_right,
                                  void* stream) {
  return fwd::run(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, 0.f, 0ull, stream,
                  window_left, window_right);
}
