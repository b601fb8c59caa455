// Host-side helpers shared by the translation units of the library:
// argument validation and TMA tensor-map encoding.
#pragma once

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/attnbwd.h"

namespace attn {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Shape checks common to all calls. Returns ATTN_OK, or an error code.
inline int check_shape(int B, int H, int H_kv, int N, int d) {
  if (B < 0 || H < 0 || H_kv < 0 || N < 0 || d <= 0) return ATTN_ERR_SHAPE;
  if (H > 0 && (H_kv <= 0 || H % H_kv != 0)) return ATTN_ERR_SHAPE;
  // element counts must stay below 2^31 per (batch, head) row block and the
  // flat tensors below 2^40 elements (TMA strides, 64-bit offsets)
  const long long rows = static_cast<long long>(B) * H * N;
  if (rows * d >= (1LL << 40)) return ATTN_ERR_TOO_LARGE;
  if (static_cast<long long>(N) * d >= (1LL << 31)) return ATTN_ERR_TOO_LARGE;
  return ATTN_OK;
}

// Number of SMs of the current device (cached per device); 0 on error.
inline int sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) {
    const int n = cache[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 0;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device: the attribute belongs to the device's context, so
// a process that drives several GPUs needs it on each. `done` is the calling
// launcher's own record (one per kernel instantiation).
constexpr int kMaxTrackedDevices = 64;
template <typename Kernel>
inline bool set_smem_limit_once(Kernel kern, int bytes,
                                std::atomic<bool> (&done)[kMaxTrackedDevices]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const bool tracked = dev >= 0 && dev < kMaxTrackedDevices;
  if (tracked && done[dev].load(std::memory_order_acquire)) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  if (tracked) done[dev].store(true, std::memory_order_release);
  return true;
}

inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no
// link-time dependency on libcuda).
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-D bf16 tensor map over [heads, rows, d] (innermost d), box
// {64, box_rows, 1}, 128-byte swizzle, zero fill outside the tensor.
inline bool encode_bf16_3d(CUtensorMap* map, const void* base, int d, int rows, long long heads,
                           int box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(d) * 2 * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D fp32 tensor map over [heads, rows, d] (innermost d), box
// {box_cols, box_rows, 1}; used for TMA reductions into dQaccum (rows past
// the end of a head are clipped, never written). box_cols = d: no swizzle;
// box_cols = 32 (128-byte rows): 128-byte swizzle.
inline bool encode_f32_3d(CUtensorMap* map, const void* base, int d, int rows, long long heads,
                          int box_rows, int box_cols = 0) {
  if (box_cols == 0) box_cols = d;
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                           static_cast<cuuint64_t>(d) * 4 * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   box_cols * 4 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Dropout threshold and scale for drop probability p in (0, 1): a 32-bit
// word keeps its element iff word >= round(p * 2^32).
inline uint32_t dropout_threshold(float p) {
  const double t = static_cast<double>(p) * 4294967296.0 + 0.5;  // round half up
  if (t <= 0.0) return 0u;
  if (t >= 4294967295.0) return 0xFFFFFFFFu;
  return static_cast<uint32_t>(t);
}

// Device status word of the forward kernels (attn_fwd.cu): *status := its
// value, cleared when `clear`. Returns ATTN_OK or ATTN_ERR_LAUNCH.
int fwd_status(int* status, bool clear);

// The same for the d = 256 backward kernel (attn_bwd256.cu).
int bwd256_status(int* status, bool clear);

// attn_bwd and its local, dropout and deterministic forms for d = 256
// (attn_bwd256.cu), after the caller has checked pointers, shapes, alignment,
// scale and drop probability; B, H, N > 0. With det, dq_target is the
// partials workspace of `pairs` tiles per query head, else the accumulator.
int bwd256_run(const void* q, const void* k, const void* v, const void* dO, const float* lse,
               float* dq_target, void* dk, void* dv, int B, int H, int H_kv, int N, float scale,
               int causal, float softcap, const float* dpsum, int window_left, int window_right,
               bool det, int pairs, float p_drop, unsigned long long seed, cudaStream_t s);

// attn_bwd (d = 64 or 128) with a hook: before_launch(ctx) runs after every
// argument check and tensor-map encoding has passed and right before the main
// kernel is enqueued, so a caller can enqueue work that must precede the
// kernel only once the whole call is known to be valid. A non-zero return from
// the hook ends the call with that code; d = 256 returns ATTN_ERR_UNSUPPORTED.
int bwd_run_hooked(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                   float* dq_accum, void* dk, void* dv, int B, int H, int H_kv, int N, int d,
                   float scale, int causal, float softcap, const float* dpsum, void* stream,
                   int (*before_launch)(void*), void* ctx);

}  // namespace attn
