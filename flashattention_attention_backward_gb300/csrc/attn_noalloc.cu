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
//  * The first call on a device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture.
#include <atomic>
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

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                int B, int H, int H_kv, int N, int d, float scale, int causal,
                                float softcap, void* stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return ATTN_ERR_NULL;
  int rc = check_shape(B, H, H_kv, N, d);
  if (rc != ATTN_OK) return rc;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(B) * H * N;
  const long long need = rows * d + rows;  // dQ accumulator, then D
  if (need > noalloc::kNoAllocScratchFloats) return ATTN_ERR_TOO_LARGE;
  if (rows == 0) return ATTN_OK;
  float* scratch = nullptr;
  rc = noalloc::scratch_address(&scratch);
  if (rc != ATTN_OK) return rc;
  float* dq_accum = scratch;           // [B, H, N, d]; d % 4 == 0 keeps D 16-byte aligned
  float* dpsum = scratch + rows * d;   // [B, H, N]
  rc = attn_bwd_preprocess(o, dO, dpsum, dq_accum, B, H, N, d, stream);
  if (rc != ATTN_OK) return rc;
  rc = attn_bwd(q, k, v, o, dO, lse, dq_accum, dk, dv, B, H, H_kv, N, d, scale, causal, softcap,
                dpsum, stream);
  if (rc != ATTN_OK) return rc;
  return attn_bwd_finalize(dq_accum, dq, scale, B, H, N, d, stream);
}
