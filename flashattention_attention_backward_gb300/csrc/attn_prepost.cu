// attn_bwd_preprocess and attn_bwd_finalize: the two memory-bound steps
// around the main backward kernel.
//
//  * preprocess: D_i = sum_k dO_ik O_ik ("解析 FlashAttention（3）" §2.4 eq. 6;
//    "反向传播算法详解" §2.1(3): dPsum can be formed before the backward kernel
//    starts) and dq_accum := 0, in one pass. For d = 64, 128, 256 a row is
//    read by d / 8 lanes with 16-byte loads (two steps in flight per
//    thread), reduced with shuffles, and the matching fp32 dQ-accumulator
//    row is cleared with 16-byte stores; other d, one warp per row.
//  * finalize: dq = bf16(tau * dq_accum) ("解析 FlashAttention（3）" eq. 7),
//    16 bytes read / 8 bytes written per element group, four groups in
//    flight per thread.
//  * finalize_partials (deterministic dQ): dq = bf16(tau * sum over key
//    blocks n, in increasing n, of the stored partial tiles dS_mn K_n of
//    query block m) ("反向传播算法详解" §6.4: a fixed order of the
//    additions makes dQ reproducible bit for bit).
// Both grids are a multiple of the SM count and grid-stride over the rows.
#include <cstdint>
#include <cuda_bf16.h>

#include "attn_common.cuh"

namespace attn {
namespace prepost {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    preprocess_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dO,
                      float* __restrict__ dpsum, float* __restrict__ dq_accum, long long rows,
                      int d) {
  const int lane = threadIdx.x & 31;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * kThreads) >> 5;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long row = warp0; row < rows; row += nwarps) {
    const long long base = row * d;
    float acc = 0.f;
    for (int c = lane * 4; c < d; c += 128) {
      const uint2 uo = __ldcs(reinterpret_cast<const uint2*>(o + base + c));
      const uint2 ud = __ldcs(reinterpret_cast<const uint2*>(dO + base + c));
      const uint32_t wo[2] = {uo.x, uo.y}, wd[2] = {ud.x, ud.y};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        acc = fmaf(__uint_as_float(wo[e] << 16), __uint_as_float(wd[e] << 16), acc);
        acc = fmaf(__uint_as_float(wo[e] & 0xffff0000u), __uint_as_float(wd[e] & 0xffff0000u),
                   acc);
      }
      if (dq_accum != nullptr) *reinterpret_cast<float4*>(dq_accum + base + c) = zero;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) dpsum[row] = acc;
  }
}

// The same for d = 64, 128 and 256 with 16-byte loads: d / 8 lanes share a
// row (a warp covers 32 / (d / 8) rows per step), and each thread keeps two
// steps in flight, so that the loads in flight per SM cover the memory
// latency while the L2 also writes back what the backward kernel left dirty.
template <int D>
__global__ void __launch_bounds__(kThreads)
    preprocess_vec_kernel(const __nv_bfloat16* __restrict__ o,
                          const __nv_bfloat16* __restrict__ dO, float* __restrict__ dpsum,
                          float* __restrict__ dq_accum, long long rows) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerStep = 32 / kLanesPerRow;
  constexpr int kSteps = 2;
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow, li = lane % kLanesPerRow;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * kThreads) >> 5;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long r0 = warp0 * kRowsPerStep * kSteps; r0 < rows;
       r0 += nwarps * kRowsPerStep * kSteps) {
    uint4 uo[kSteps], ud[kSteps];
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
      const long long row = r0 + u * kRowsPerStep + sub;
      uo[u] = make_uint4(0u, 0u, 0u, 0u);
      ud[u] = make_uint4(0u, 0u, 0u, 0u);
      if (row < rows) {
        uo[u] = __ldcs(reinterpret_cast<const uint4*>(o + row * D) + li);
        ud[u] = __ldcs(reinterpret_cast<const uint4*>(dO + row * D) + li);
      }
    }
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
      const long long row = r0 + u * kRowsPerStep + sub;
      const uint32_t wo[4] = {uo[u].x, uo[u].y, uo[u].z, uo[u].w};
      const uint32_t wd[4] = {ud[u].x, ud[u].y, ud[u].z, ud[u].w};
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(__uint_as_float(wo[e] << 16), __uint_as_float(wd[e] << 16), acc);
        acc = fmaf(__uint_as_float(wo[e] & 0xffff0000u), __uint_as_float(wd[e] & 0xffff0000u),
                   acc);
      }
      // sum over the row's lanes (aligned groups of kLanesPerRow lanes)
#pragma unroll
      for (int off = kLanesPerRow / 2; off >= 1; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (row < rows) {
        if (li == 0) dpsum[row] = acc;
        if (dq_accum != nullptr) {
          float4* z = reinterpret_cast<float4*>(dq_accum + row * D) + 2 * li;
          z[0] = zero;
          z[1] = zero;
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads)
    finalize_kernel(const float* __restrict__ dq_accum, __nv_bfloat16* __restrict__ dq,
                    float scale, long long n4) {
  // four 16-byte loads in flight per thread before the stores
  constexpr int kUnroll = 4;
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long i0 = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i0 < n4;
       i0 += stride * kUnroll) {
    float4 a[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long i = i0 + u * stride;
      a[u] = i < n4 ? __ldcs(reinterpret_cast<const float4*>(dq_accum) + i)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long i = i0 + u * stride;
      if (i >= n4) break;
      __nv_bfloat162 lo = __floats2bfloat162_rn(a[u].x * scale, a[u].y * scale);
      __nv_bfloat162 hi = __floats2bfloat162_rn(a[u].z * scale, a[u].w * scale);
      uint2 v;
      v.x = *reinterpret_cast<uint32_t*>(&lo);
      v.y = *reinterpret_cast<uint32_t*>(&hi);
      __stcs(reinterpret_cast<uint2*>(dq) + i, v);
    }
  }
}

// Partial dQ tiles of the deterministic mode: per query head, one 128-row
// tile per (query block m, key block n) pair the mask keeps, pair index
// m (m + 1) / 2 + n (causal, n <= m) or m * n_blocks + n.
__host__ __device__ inline long long pair_index(int m, int n, int n_blocks, bool causal) {
  return causal ? static_cast<long long>(m) * (m + 1) / 2 + n
                : static_cast<long long>(m) * n_blocks + n;
}
__host__ __device__ inline long long pairs_per_head(int blocks, bool causal) {
  return causal ? static_cast<long long>(blocks) * (blocks + 1) / 2
                : static_cast<long long>(blocks) * blocks;
}

// One thread per 4 consecutive dQ elements of a row: the partials of its
// query block are added in increasing key-block order.
__global__ void __launch_bounds__(kThreads)
    finalize_partials_kernel(const float* __restrict__ part, __nv_bfloat16* __restrict__ dq,
                             float scale, long long rows, int N, int d, int blocks, int causal) {
  const long long n4 = rows * (d / 4);
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  const long long P = pairs_per_head(blocks, causal != 0);
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < n4;
       i += stride) {
    const long long row = i / (d / 4);
    const int c4 = static_cast<int>(i - row * (d / 4));
    const long long bh = row / N;
    const int qrow = static_cast<int>(row - bh * N);
    const int m = qrow >> 7, r = qrow & 127;
    const int n_end = causal ? m + 1 : blocks;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int n = 0; n < n_end; ++n) {
      const long long tile = bh * P + pair_index(m, n, blocks, causal != 0);
      const float4 a =
          __ldcs(reinterpret_cast<const float4*>(part + (tile * 128 + r) * d) + c4);
      acc.x += a.x;
      acc.y += a.y;
      acc.z += a.z;
      acc.w += a.w;
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * scale, acc.y * scale);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * scale, acc.w * scale);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    __stcs(reinterpret_cast<uint2*>(dq) + i, u);
  }
}

inline unsigned grid_for(long long work_items, int items_per_block) {
  const long long want = (work_items + items_per_block - 1) / items_per_block;
  const int sms = sm_count();
  const long long cap = static_cast<long long>(sms > 0 ? sms : 1) * 8;
  return static_cast<unsigned>(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace prepost
}  // namespace attn

using namespace attn;

extern "C" int attn_bwd_preprocess(const void* o, const void* dO, float* dpsum, float* dq_accum,
                                   int B, int H, int N, int d, void* stream) {
  if (!o || !dO || !dpsum) return ATTN_ERR_NULL;  // dq_accum may be NULL: D only
  int rc = check_shape(B, H, H > 0 ? 1 : 0, N, d);
  if (rc != ATTN_OK) return rc;
  if (d % 4 != 0) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(o) || !aligned16(dO) || !aligned16(dpsum) ||
      (dq_accum != nullptr && !aligned16(dq_accum)))
    return ATTN_ERR_ALIGN;
  const long long rows = static_cast<long long>(B) * H * N;
  if (rows == 0) return ATTN_OK;
  const auto* o16 = static_cast<const __nv_bfloat16*>(o);
  const auto* d16 = static_cast<const __nv_bfloat16*>(dO);
  cudaStream_t s = as_stream(stream);
  if (d == 64 || d == 128 || d == 256) {
    // rows per CTA per grid-stride pass: 8 warps x (256 / d) rows x 2 steps
    const unsigned grid = prepost::grid_for(rows, (prepost::kThreads / 32) * (256 / d) * 2);
    if (d == 64)
      prepost::preprocess_vec_kernel<64><<<grid, prepost::kThreads, 0, s>>>(o16, d16, dpsum,
                                                                           dq_accum, rows);
    else if (d == 128)
      prepost::preprocess_vec_kernel<128><<<grid, prepost::kThreads, 0, s>>>(o16, d16, dpsum,
                                                                            dq_accum, rows);
    else
      prepost::preprocess_vec_kernel<256><<<grid, prepost::kThreads, 0, s>>>(o16, d16, dpsum,
                                                                            dq_accum, rows);
    return launch_status();
  }
  const unsigned grid = prepost::grid_for(rows, prepost::kThreads / 32);
  prepost::preprocess_kernel<<<grid, prepost::kThreads, 0, s>>>(o16, d16, dpsum, dq_accum, rows,
                                                                d);
  return launch_status();
}

extern "C" int attn_bwd_finalize(const float* dq_accum, void* dq, float scale, int B, int H,
                                 int N, int d, void* stream) {
  if (!dq_accum || !dq) return ATTN_ERR_NULL;
  int rc = check_shape(B, H, H > 0 ? 1 : 0, N, d);
  if (rc != ATTN_OK) return rc;
  if (d % 4 != 0) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return ATTN_ERR_SHAPE;
  if (!aligned16(dq_accum) || !aligned16(dq)) return ATTN_ERR_ALIGN;
  const long long n4 = static_cast<long long>(B) * H * N * d / 4;
  if (n4 == 0) return ATTN_OK;
  const unsigned grid = prepost::grid_for(n4, prepost::kThreads * 4);
  prepost::finalize_kernel<<<grid, prepost::kThreads, 0, as_stream(stream)>>>(
      dq_accum, static_cast<__nv_bfloat16*>(dq), scale, n4);
  return launch_status();
}

extern "C" long long attn_bwd_dq_partials_bytes(int B, int H, int N, int d, int causal) {
  int rc = check_shape(B, H, H > 0 ? 1 : 0, N, d);
  if (rc != ATTN_OK) return rc;
  const int blocks = (N + 127) / 128;
  return static_cast<long long>(B) * H * prepost::pairs_per_head(blocks, causal != 0) * 128 * d *
         static_cast<long long>(sizeof(float));
}

extern "C" int attn_bwd_finalize_partials(const float* dq_partials, void* dq, float scale, int B,
                                          int H, int N, int d, int causal, void* stream) {
  if (!dq_partials || !dq) return ATTN_ERR_NULL;
  int rc = check_shape(B, H, H > 0 ? 1 : 0, N, d);
  if (rc != ATTN_OK) return rc;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return ATTN_ERR_SHAPE;
  if (!aligned16(dq_partials) || !aligned16(dq)) return ATTN_ERR_ALIGN;
  const long long rows = static_cast<long long>(B) * H * N;
  if (rows == 0) return ATTN_OK;
  const unsigned grid = prepost::grid_for(rows * (d / 4), prepost::kThreads);
  prepost::finalize_partials_kernel<<<grid, prepost::kThreads, 0, as_stream(stream)>>>(
      dq_partials, static_cast<__nv_bfloat16*>(dq), scale, rows, N, d, (N + 127) / 128,
      causal != 0 ? 1 : 0);
  return launch_status();
}
