// attn_bwd_noalloc: the full backward (preprocess -> main kernel -> finalize)
// for callers that cannot allocate device memory.
//
// The ordinary path needs two scratch buffers next to the caller's tensors:
// the fp32 dQ accumulator [B, H, N, d] and the row statistic D [B, H, N].
// Some callers cannot obtain them: code running inside a captured CUDA graph
// where allocation is not allowed, plugins handed fixed buffers by a host
// framework, or runtimes whose allocator must not be re-entered. This entry
// point takes the same inputs and outputs as the ordinary path but keeps both
// scratch buffers in one file-scope device array, so it never allocates.
//
// Limits and rules:
//  * The array holds kNoAllocScratchFloats floats (32 MiB). A problem needs
//    B*H*N*d + B*H*N floats; larger problems are rejected with
//    ATTN_ERR_TOO_LARGE before anything is launched.
//  * Every device that loads the library reserves the array until the process
//    exits.
//  * All calls share the one array and it keeps the previous call's contents;
//    the preprocess step clears the dQ accumulator at the start of every call.
//    Calls whose work overlaps on the GPU (different streams without ordering,
//    or different host threads) race on the array and give wrong results.
//  * Every argument check of the three steps runs before the first launch, so
//    a rejected call enqueues nothing and leaves the array as it was; only a
//    launch error reported by CUDA can come after a step was enqueued.
//  * The first call on a device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_common.cuh"

namespace attn {
namespace noalloc {

constexpr long long kNoAllocScratchFloats = 8LL * 1024 * 1024;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_scratch[kNoAllocScratchFloats];

// Device address of g_scratch per device, looked up once per device.
static std::atomic<float*> g_addr[kMaxDevices];
static std::mutex g_setup_mutex;

int scratch_address(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  float* p = g_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_addr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      void* sym = nullptr;
      if (cudaGetSymbolAddress(&sym, g_scratch) != cudaSuccess || sym == nullptr)
        return ATTN_ERR_LAUNCH;
      p = static_cast<float*>(sym);
      g_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return ATTN_OK;
}

}  // namespace noalloc
}  // namespace attn

using namespace attn;

namespace {

// Arguments of the preprocess step, enqueued by the main call's hook once the
// main call has passed all of its checks.
struct PreprocessArgs {
  const void* o;
  const void* dO;
  float* dpsum;
  float* dq_accum;
  int B, H, N, d;
  void* stream;
};

int enqueue_preprocess(void* ctx) {
  const PreprocessArgs* a = static_cast<const PreprocessArgs*>(ctx);
  return attn_bwd_preprocess(a->o, a->dO, a->dpsum, a->dq_accum, a->B, a->H, a->N, a->d,
                             a->stream);
}

}  // namespace

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                int B, int H, int H_kv, int N, int d, float scale, int causal,
                                float softcap, void* stream) {
  // Every check of the three steps runs here, before anything is enqueued:
  // a rejected call leaves the stream and the shared array untouched.
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return ATTN_ERR_NULL;
  int rc = check_shape(B, H, H_kv, N, d);
  if (rc != ATTN_OK) return rc;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || scale == 0.f || std::isnan(softcap)) return ATTN_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return ATTN_ERR_ALIGN;
  const long long rows = static_cast<long long>(B) * H * N;
  const long long need = rows * d + rows;  // dQ accumulator, then D
  if (need > noalloc::kNoAllocScratchFloats) return ATTN_ERR_TOO_LARGE;
  if (rows == 0) return ATTN_OK;
  float* scratch = nullptr;
  rc = noalloc::scratch_address(&scratch);
  if (rc != ATTN_OK) return rc;
  float* dq_accum = scratch;           // [B, H, N, d]; d % 4 == 0 keeps D 16-byte aligned
  float* dpsum = scratch + rows * d;   // [B, H, N]
  // The main call checks its arguments and encodes its tensor maps first; only
  // then does its hook enqueue the preprocess (D, and the accumulator
  // cleared), followed by the main kernel. Past this point an error can only
  // be a launch error reported by CUDA.
  PreprocessArgs pre{o, dO, dpsum, dq_accum, B, H, N, d, stream};
  rc = bwd_run_hooked(q, k, v, dO, lse, dq_accum, dk, dv, B, H, H_kv, N, d, scale, causal, softcap,
                      dpsum, stream, enqueue_preprocess, &pre);
  if (rc != ATTN_OK) return rc;
  return attn_bwd_finalize(dq_accum, dq, scale, B, H, N, d, stream);
}
