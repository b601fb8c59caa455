// attn_bwd for head dimension 256 on sm_103a (N-outer / Q-inner,
// recompute-P; "反向传播算法详解" §2-§6 and §8.3, which slices the d = 256
// GEMMs; "解析 FlashAttention（3）" §4).
//
// With 128 keys on the tensor-memory lanes, fp32 dK and dV accumulators of
// d = 256 would take all 512 columns, and K, V, Q and dO tiles of 128 rows x
// 256 would need 256 KB of shared memory. So a CTA accumulates one half of d
// (dh = 128 columns, `half` 0 or 1) for one block of 128 keys, and query
// tiles are 64 rows:
//
//   S^T  = K_j Q_i^T                 (M = 128 keys, N = 64 queries, K = 256)
//   dP^T = V_j dO_i^T                (the same shape)
//   P    = exp2(S^T * tau*log2e - LSE*log2e)   [softcap: c tanh(tau S / c)]
//   dS   = P o (dP - D)              [softcap: o (1 - tanh^2)]
//   dV_j[:, half] += P^T dO_i[:, half]    (P^T from tensor memory)
//   dK_j[:, half] += dS^T Q_i[:, half]    (dS^T from shared memory)
//   dQ_i[:, half] += dS K_j[:, half]      (transposed: dQ^T = K^T dS^T,
//                                          fp32 TMA reductions)
//
// Template flags as in the d <= 128 kernel: DROP replays the dropout keep
// mask of philox.cuh (P^T for dV is P o Z / (1 - p), and dP passes through
// the same mask before dS); DET stores each dQ tile into the partials
// workspace of attn_bwd_deterministic instead of adding it.
//
// S and dP are recomputed by the CTAs of both halves: seven GEMM-equivalents
// of 2 * 128 * 64 * 128 flops per tile and half instead of five.
//
// One CTA per unit (key block, KV head, batch entry, half); a unit walks every
// query tile of every query head of its group. K and V (64 KB each) stay in
// shared memory; Q and dO tiles (32 KB each) are single-buffered, which
// leaves room for the dS tile and the dQ staging buffer within 227 KB.
//
// Warp roles (384 threads; 512 with dropout):
//   warp 0      TMA producer: K, V once; per tile Q (+LSE, D) and dO
//   warp 1      MMA issuer (whole warp, one elected lane), tensor-memory owner
//   warps 4-7   softmax backward: thread = key row (tensor-memory lane),
//               64 query columns
//   warps 8-11  dQ drain (thread = d index of the half), then the dK/dV
//               epilogue
//   warps 12-15 with dropout only: the keep mask of the next tiles (thread =
//               key row), handed to the softmax through shared memory
//
// Tensor memory (512 columns): S^T [0,64) (P^T bf16 pairs over its first 32
// columns), dP^T [64,128), dQ^T tiles [128,192) and [192,256) alternating,
// dV [256,384), dK [384,512).
// Every mbarrier wait is bounded; on timeout the kernel records
// ATTN_ERR_DEVICE_TIMEOUT in its device status word (attn_device_status
// reads it) and returns.
#include <cstdint>
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "philox.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace bwd256 {

using namespace ptx;

constexpr int kD = 256;   // head dimension
constexpr int kDh = 128;  // the half of d one CTA accumulates
constexpr int kBc = 128;  // keys per CTA (tensor-memory lanes)
constexpr int kBr = 64;   // queries per tile
constexpr int kThreads = 384;
// With dropout the keep mask is drawn by a warpgroup of its own: Philox4x32-10
// is bound by its 32 x 32 -> 64-bit multiplies (about 1.3 calls per clock per
// SM measured), and the 2,048 calls of a tile drawn by the four softmax warps
// themselves (one per SM sub-partition, each call a chain of ten dependent
// rounds) nearly doubled the tile's time. Registers: 512 threads launch with
// 128 each; setmaxnreg gives the softmax and drain warps 168, the others 88.
template <bool DROP>
constexpr int kThreadsFor = DROP ? 512 : kThreads;
constexpr int kRegsWideDrop = 168, kRegsNarrowDrop = 88;
static_assert(256 * kRegsWideDrop + 256 * kRegsNarrowDrop <= 512 * 128, "register pool");
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitLimitCycles = 2000000000LL;  // about one second

__device__ int g_status256;  // device status word of this kernel (ATTN_OK or ATTN_ERR_*)

__device__ __noinline__ void record_status(int code) { atomicCAS(&g_status256, 0, code); }

struct Layout {
  static constexpr int kK = 0;          // [128 keys][256 d]: 4 boxes of 64 d, 16 KB each
  static constexpr int kV = 65536;      // the same
  static constexpr int kQ = 131072;     // [64 queries][256 d]: 4 boxes of 8 KB
  static constexpr int kDO = 163840;    // the same
  static constexpr int kDS = 196608;    // dS^T [128 keys][64 queries] bf16, 16 KB
  static constexpr int kDQS = 212992;   // dQ staging [32 queries][128 d] fp32, 16 KB
  static constexpr int kLSE = 229376;   // 64 fp32 (-LSE * log2e)
  static constexpr int kDsum = 229632;  // 64 fp32 (D)
  // dropout keep bits of two tiles: [tile parity][key row] x 2 words (bit j
  // of word w: query 32 w + j of the tile)
  static constexpr int kMask = 229888;
  static constexpr int kBars = kMask + 2 * 128 * 8;
  static constexpr int kNumBars = 22;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kBytes = kAbort + 12;
};
static_assert(Layout::kBytes <= 232448, "shared memory budget");

// The Q tile's two boxes of the other half of d are read only by the tile's
// S GEMM and have barriers of their own (QO), so the next tile's copies load
// while this tile's own half (QH, with LSE and D) is still in use.
enum Bar {
  BAR_KV_FULL = 0,
  BAR_QH_FULL = 1,
  BAR_QH_EMPTY = 2,
  BAR_DO_FULL = 3,
  BAR_DO_EMPTY = 4,
  BAR_S_FULL = 5,
  BAR_DP_FULL = 6,
  BAR_P_FULL = 7,
  BAR_DS_FULL = 8,
  BAR_DS_FREE = 9,
  BAR_DQ_FULL = 10,   // + buffer (tile parity)
  BAR_DQ_EMPTY = 12,  // + buffer
  BAR_UNIT_DONE = 14,
  BAR_DRAIN = 15,     // abort path only
  BAR_QO_FULL = 16,
  BAR_QO_EMPTY = 17,
  BAR_MASK_FULL = 18,   // + tile parity (dropout): keep bits written
  BAR_MASK_EMPTY = 20,  // + tile parity: the softmax has read them
};

struct Params {
  const float* lse;
  const float* dpsum;
  int B, H, H_kv, N;
  int n_blocks;  // blocks of 128 keys
  int m_blocks;  // blocks of 64 queries
  float scale;
  float softcap;
  // key j is visible to query i iff i - win_left <= j <= i + win_right (the
  // causal mask is win_right = 0; an unbounded side holds N)
  int win_left, win_right;
  // DET: dQ tiles go to partials [B*H*pairs, 128, 256]; the pair of query
  // block m (128 rows) and key block n is m (m + 1) / 2 + n (causal) or
  // m * n_blocks + n, and a 64-query tile fills rows (m0 mod 128) .. + 63
  int pairs;
  int causal;
  Dropout drop;  // DROP: keep mask of philox.cuh
};

struct Work {
  int b, g, n_block, half, G, m_start, per_head, T;
};

// Units heaviest first for a causal mask: u = 2 (n_block (H_kv B) + b H_kv + g) + half.
__device__ __forceinline__ Work work_of(const Params& p) {
  Work w;
  const int u = static_cast<int>(blockIdx.x);
  w.half = u & 1;
  const int rest = u >> 1;
  const int per_nb = p.H_kv * p.B;
  w.n_block = rest / per_nb;
  const int rem = rest - w.n_block * per_nb;
  w.b = rem / p.H_kv;
  w.g = rem - w.b * p.H_kv;
  w.G = p.H / p.H_kv;
  const int n0 = w.n_block * kBc;
  w.m_start = max(0, n0 - p.win_right) / kBr;
  const int m_end = min(p.m_blocks - 1, (n0 + kBc - 1 + p.win_left) / kBr);
  w.per_head = m_end - w.m_start + 1;  // >= 1: the band holds the diagonal
  w.T = w.G * w.per_head;
  return w;
}

// Tile t: query blocks from the last one down, the G heads of the group inner.
__device__ __forceinline__ void tile_coord(const Work& w, int t, int& h, int& m_block) {
  const int mi = t / w.G;
  h = w.g * w.G + (t - mi * w.G);
  m_block = w.m_start + w.per_head - 1 - mi;
}

struct Ctx {
  uint32_t bars;
  volatile int* abort;
};

__device__ __forceinline__ uint32_t bar_addr(const Ctx& c, int i) { return c.bars + 8u * i; }

__device__ __forceinline__ bool wait(const Ctx& c, int bar, uint32_t parity) {
  const uint32_t a = bar_addr(c, bar);
  if (mbar_try_wait(a, parity)) return true;
  const long long t0 = clock64();
  uint32_t n = 0;
  while (!mbar_try_wait(a, parity)) {
    if ((++n & 63u) == 0) {
      if (*c.abort) return false;
      if (clock64() - t0 > kWaitLimitCycles) {
        *c.abort = 1;
        record_status(ATTN_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

__device__ __forceinline__ bool wait_warp(const Ctx& c, int bar, uint32_t parity) {
  return __all_sync(0xffffffffu, wait(c, bar, parity));
}

__device__ __forceinline__ void wait_drain(const Ctx& c, int bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar_addr(c, bar), parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return;
  }
}

__device__ __forceinline__ bool tile_masked(const Params& p, int m0, int n0) {
  return n0 + kBc - 1 - m0 > p.win_right || m0 + kBr - 1 - n0 > p.win_left || n0 + kBc > p.N ||
         m0 + kBr > p.N;
}

// ------------------------------------------------------------------ producer
__device__ void producer_role(const Ctx& c, const Params& p, const Work& w, uint8_t* smem,
                              uint32_t sbase, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                              const CUtensorMap* tm_v, const CUtensorMap* tm_do) {
  using L = Layout;
  const int lane = threadIdx.x & 31;
  const int kvh = w.b * p.H_kv + w.g;
  const int n0 = w.n_block * kBc;
  if (lane == 0) {
    prefetch_tmap(tm_q);
    prefetch_tmap(tm_k);
    prefetch_tmap(tm_v);
    prefetch_tmap(tm_do);
    mbar_arrive_expect_tx(bar_addr(c, BAR_KV_FULL), 2 * 4 * 16384);
    for (int cb = 0; cb < 4; ++cb) {
      tma_load_3d(sbase + L::kK + cb * 16384, tm_k, bar_addr(c, BAR_KV_FULL), 64 * cb, n0, kvh);
      tma_load_3d(sbase + L::kV + cb * 16384, tm_v, bar_addr(c, BAR_KV_FULL), 64 * cb, n0, kvh);
    }
  }
  const uint64_t reuse = policy_evict_last();  // Q, dO tiles serve every key block of the head
  float* s_lse = reinterpret_cast<float*>(smem + L::kLSE);
  float* s_d = reinterpret_cast<float*>(smem + L::kDsum);
  int issued_q = 0, issued_qo = 0, issued_do = 0;
  bool ok = true;
  for (int t = 0; t < w.T; ++t) {
    int h, m_block;
    tile_coord(w, t, h, m_block);
    const int bh = w.b * p.H + h;
    const int m0 = m_block * kBr;
    // boxes of the other half of d: free once the previous S GEMM read them
    if (t > 0 && !(ok = wait_warp(c, BAR_QO_EMPTY, (t - 1) & 1))) break;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_addr(c, BAR_QO_FULL), 2 * 8192);
      for (int cb = 2 * (1 - w.half); cb < 2 * (1 - w.half) + 2; ++cb)
        tma_load_3d_hint(sbase + L::kQ + cb * 8192, tm_q, bar_addr(c, BAR_QO_FULL), 64 * cb, m0,
                         bh, reuse);
    }
    issued_qo = t + 1;
    if (t > 0 && !(ok = wait_warp(c, BAR_DO_EMPTY, (t - 1) & 1))) break;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_addr(c, BAR_DO_FULL), 4 * 8192);
      for (int cb = 0; cb < 4; ++cb)
        tma_load_3d_hint(sbase + L::kDO + cb * 8192, tm_do, bar_addr(c, BAR_DO_FULL), 64 * cb, m0,
                         bh, reuse);
    }
    issued_do = t + 1;
    // this CTA's half (also read by the dK GEMM), with LSE and D; the softmax
    // read the previous tile's LSE and D before DS_FULL, which precedes the
    // previous dK GEMM and hence QH_EMPTY
    if (t > 0 && !(ok = wait_warp(c, BAR_QH_EMPTY, (t - 1) & 1))) break;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_addr(c, BAR_QH_FULL), 2 * 8192);
      for (int cb = 2 * w.half; cb < 2 * w.half + 2; ++cb)
        tma_load_3d_hint(sbase + L::kQ + cb * 8192, tm_q, bar_addr(c, BAR_QH_FULL), 64 * cb, m0,
                         bh, reuse);
    }
    {
      const long long row0 = static_cast<long long>(bh) * p.N + m0;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = lane + 32 * e;
        float lv = 0.f, dv = 0.f;
        if (m0 + i < p.N) {
          lv = __ldg(p.lse + row0 + i);
          dv = __ldg(p.dpsum + row0 + i);
        }
        s_lse[i] = -lv * kLog2e;
        s_d[i] = dv;
      }
      mbar_arrive(bar_addr(c, BAR_QH_FULL));
    }
    issued_q = t + 1;
    __syncwarp();
  }
  if (!ok || *c.abort) {  // the copies issued last must land before the CTA exits
    wait_drain(c, BAR_KV_FULL, 0);
    if (issued_q > 0) wait_drain(c, BAR_QH_FULL, (issued_q - 1) & 1);
    if (issued_qo > 0) wait_drain(c, BAR_QO_FULL, (issued_qo - 1) & 1);
    if (issued_do > 0) wait_drain(c, BAR_DO_FULL, (issued_do - 1) & 1);
  }
}

// ------------------------------------------------------------------ MMA issuer
// Per tile: S^T, dP^T, then (P ready) dV, then (dS ready) dQ^T and dK. The
// next tile's S^T overwrites P^T only after this tile's dV GEMM, which reads
// it (tcgen05 MMAs of one thread run in issue order).
__device__ void mma_role(const Ctx& c, const Work& w, uint32_t sbase, uint32_t tmem) {
  using L = Layout;
  const uint32_t tS = tmem, tdP = tmem + 64, tdQ = tmem + 128, tdV = tmem + 256,
                 tdK = tmem + 384;
  constexpr uint32_t kIdS = make_idesc_bf16(kBc, kBr, false, false);   // S^T, dP^T
  constexpr uint32_t kIdKV = make_idesc_bf16(kBc, kDh, false, true);   // dV, dK (d half)
  constexpr uint32_t kIdQ = make_idesc_bf16(kDh, kBr, true, true);     // dQ^T
  // K-major tiles: k-step k (16 elements) at box k / 4, byte 32 (k % 4)
  auto kmaj_k = [](int k) { return static_cast<uint32_t>(((k >> 2) * 16384 + (k & 3) * 32) >> 4); };
  auto kmaj_q = [](int k) { return static_cast<uint32_t>(((k >> 2) * 8192 + (k & 3) * 32) >> 4); };
  auto mnmaj = [](int k) { return static_cast<uint32_t>((2048 * k) >> 4); };  // 16 rows
  const uint32_t aK = sdesc_lo(sbase + L::kK, 16), aV = sdesc_lo(sbase + L::kV, 16);
  const uint32_t bQ = sdesc_lo(sbase + L::kQ, 16), bO = sdesc_lo(sbase + L::kDO, 16);
  // MN-major views of this CTA's half of d: 64-column boxes 2 half, 2 half + 1
  const uint32_t mO = sdesc_lo(sbase + L::kDO + 2 * w.half * 8192, 8192);
  const uint32_t mQ = sdesc_lo(sbase + L::kQ + 2 * w.half * 8192, 8192);
  const uint32_t mK = sdesc_lo(sbase + L::kK + 2 * w.half * 16384, 16384);
  const uint32_t kDS = sdesc_lo(sbase + L::kDS, 16), mDS = sdesc_lo(sbase + L::kDS, 16384);
  const bool leader = elect_one_sync() != 0;
  bool ok = wait_warp(c, BAR_KV_FULL, 0);
  for (int t = 0; ok && t < w.T; ++t) {
    const uint32_t ph = t & 1;
    // S^T over the other half of d first (its Q boxes land early), then over
    // this CTA's half
    const int ko = 8 * (1 - w.half), kh = 8 * w.half;  // first k-step of each half
    if (!(ok = wait_warp(c, BAR_QO_FULL, ph))) break;
    tc_fence_after();
    if (leader) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_ss(tS, sdesc_from_lo(aK + kmaj_k(ko + k)), sdesc_from_lo(bQ + kmaj_q(ko + k)), kIdS,
               k > 0);
      mma_commit(bar_addr(c, BAR_QO_EMPTY));
    }
    if (!(ok = wait_warp(c, BAR_QH_FULL, ph))) break;
    tc_fence_after();
    if (leader) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_ss(tS, sdesc_from_lo(aK + kmaj_k(kh + k)), sdesc_from_lo(bQ + kmaj_q(kh + k)), kIdS,
               1u);
      mma_commit(bar_addr(c, BAR_S_FULL));
    }
    if (!(ok = wait_warp(c, BAR_DO_FULL, ph))) break;
    tc_fence_after();
    if (leader) {
#pragma unroll
      for (int k = 0; k < kD / 16; ++k)
        mma_ss(tdP, sdesc_from_lo(aV + kmaj_k(k)), sdesc_from_lo(bO + kmaj_q(k)), kIdS, k > 0);
      mma_commit(bar_addr(c, BAR_DP_FULL));
    }
    // dV[:, half] += P^T dO[:, half]; P^T of queries 0..63 as bf16 pairs in
    // columns 0..31 of the S region
    if (!(ok = wait_warp(c, BAR_P_FULL, ph))) break;
    tc_fence_after();
    if (leader) {
#pragma unroll
      for (int k = 0; k < kBr / 16; ++k)
        mma_ts(tdV, tS + 8 * k, sdesc_from_lo(mO + mnmaj(k)), kIdKV,
               (t > 0 || k > 0) ? 1u : 0u);
      mma_commit(bar_addr(c, BAR_DO_EMPTY));
    }
    if (!(ok = wait_warp(c, BAR_DS_FULL, ph))) break;
    tc_fence_after();
    // dK[:, half] += dS^T Q[:, half] (A = dS^T [key][query], K-major) first:
    // it is the Q tile's last reader, so the next Q tile's load starts before
    // the dQ GEMM
    if (leader) {
#pragma unroll
      for (int k = 0; k < kBr / 16; ++k)
        mma_ss(tdK, sdesc_from_lo(kDS + ((32 * k) >> 4)), sdesc_from_lo(mQ + mnmaj(k)), kIdKV,
               (t > 0 || k > 0) ? 1u : 0u);
      mma_commit(bar_addr(c, BAR_QH_EMPTY));
    }
    // the dQ buffer of tile t was drained with tile t - 2
    const int qb = t & 1;
    if (t >= 2 && !(ok = wait_warp(c, BAR_DQ_EMPTY + qb, ((t >> 1) - 1) & 1))) break;
    tc_fence_after();
    if (leader) {
      // dQ^T[:, half] = K[:, half]^T dS^T (M = d half, N = queries, K = keys)
#pragma unroll
      for (int k = 0; k < kBc / 16; ++k)
        mma_ss(tdQ + 64 * qb, sdesc_from_lo(mK + mnmaj(k)), sdesc_from_lo(mDS + mnmaj(k)), kIdQ,
               k > 0);
      mma_commit(bar_addr(c, BAR_DQ_FULL + qb));
      mma_commit(bar_addr(c, BAR_DS_FREE));
    }
  }
  if (ok && leader) mma_commit(bar_addr(c, BAR_UNIT_DONE));
  if (__any_sync(0xffffffffu, !ok || *c.abort != 0)) {
    if (leader) mma_commit(bar_addr(c, BAR_DRAIN));
    wait_drain(c, BAR_DRAIN, 0);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ softmax
// With DROP, km[] holds the keep bits of the thread's 64 query columns (bit
// j of km[w]: query m0 + 32 w + j), drawn by the mask warps; both phases use
// them.
template <bool SOFTCAP, bool MASKED, bool DROP>
__device__ __forceinline__ void softmax_tile(const Params& p, uint8_t* smem, uint32_t sbase,
                                             uint32_t tS, uint32_t tdP, int r, int key, int m0,
                                             uint64_t (&pk)[32], const uint32_t (&km)[2],
                                             bool dp_phase) {
  using L = Layout;
  const float* s_lse = reinterpret_cast<const float*>(smem + L::kLSE);
  const float* s_d = reinterpret_cast<const float*>(smem + L::kDsum);
  if (!dp_phase) {
    // P = exp2(S tau log2e - LSE log2e) -> bf16 P^T pairs in S columns 0..31
    const float c_log2 = p.scale * kLog2e;
    const float cap_in = SOFTCAP ? 2.f * kLog2e * p.scale / p.softcap : 0.f;
    const float cap_out = SOFTCAP ? p.softcap * kLog2e : 0.f;
    const uint64_t c2 = f2_make(SOFTCAP ? cap_in : c_log2, SOFTCAP ? cap_in : c_log2);
    const uint64_t out2 = f2_make(cap_out, cap_out);
    const uint64_t one2 = f2_make(1.f, 1.f), mone2 = f2_make(-1.f, -1.f),
                   mtwo2 = f2_make(-2.f, -2.f);
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      uint32_t raw[32];
      tmem_ld32(tS + 32 * pass, raw);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int j = 32 * pass + 2 * u;  // query columns j, j + 1
        const uint64_t s2 = f2_make(raw[2 * u], raw[2 * u + 1]);
        const uint64_t nl2 = f2_make(s_lse[j], s_lse[j + 1]);
        float pr[2], kp[2];
        if (SOFTCAP) {
          const uint64_t v2 = f2_mul(s2, c2);
          const uint64_t e1 = f2_add(f2_make(ex2_approx(f2_lo(v2)), ex2_approx(f2_hi(v2))), one2);
          const uint64_t th2 =
              f2_fma(f2_make(rcp_approx(f2_lo(e1)), rcp_approx(f2_hi(e1))), mtwo2, one2);
          const uint64_t y2 = f2_fma(th2, out2, nl2);
          pr[0] = ex2_approx(f2_lo(y2));
          pr[1] = ex2_approx(f2_hi(y2));
          const uint64_t k2 = f2_mul(f2_make(pr[0], pr[1]), f2_fma(th2, th2, mone2));
          kp[0] = f2_lo(k2);  // -P (1 - tanh^2)
          kp[1] = f2_hi(k2);
        } else {
          const uint64_t y2 = f2_fma(s2, c2, nl2);
          pr[0] = kp[0] = ex2_approx(f2_lo(y2));
          pr[1] = kp[1] = ex2_approx(f2_hi(y2));
        }
        if (MASKED) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int q = m0 + j + e;
            const bool ok =
                key < p.N && q < p.N && key - q <= p.win_right && q - key <= p.win_left;
            pr[e] = ok ? pr[e] : 0.f;
            kp[e] = ok ? kp[e] : 0.f;
          }
        }
        if (DROP) {
#pragma unroll
          for (int e = 0; e < 2; ++e)
            pr[e] = (km[pass] >> (2 * u + e)) & 1u ? pr[e] * p.drop.inv_keep : 0.f;
        }
        raw[u] = pack_bf16x2(pr[0], pr[1]);
        pk[16 * pass + u] = f2_make(kp[0], kp[1]);
      }
      uint32_t lo[8], hi[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        lo[u] = raw[u];
        hi[u] = raw[8 + u];
      }
      // queries 32 pass .. + 31 -> columns 16 pass .. + 15 (read already)
      tmem_st8(tS + 16 * pass, lo);
      tmem_st8(tS + 16 * pass + 8, hi);
    }
    return;
  }
  // dS = P o (dP - D) (softcap: (-P (1 - tanh^2)) o (D - dP)) -> bf16 dS^T
  // row r of the shared tile (128-byte rows, 128-byte swizzle)
  const uint32_t ds_row = sbase + L::kDS + r * 128;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    uint32_t raw[32];
    tmem_ld32(tdP + 32 * hh, raw);
    uint32_t packed[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int j = 32 * hh + 2 * u;
      uint32_t dp0 = raw[2 * u], dp1 = raw[2 * u + 1];
      if (DROP) {
        dp0 = (km[hh] >> (2 * u)) & 1u ? __float_as_uint(__uint_as_float(dp0) * p.drop.inv_keep)
                                       : 0u;
        dp1 = (km[hh] >> (2 * u + 1)) & 1u
                  ? __float_as_uint(__uint_as_float(dp1) * p.drop.inv_keep)
                  : 0u;
      }
      const uint64_t dp2 = f2_make(dp0, dp1);
      const uint64_t dd2 = f2_make(s_d[j], s_d[j + 1]);
      const uint64_t r2 =
          f2_mul(pk[16 * hh + u], SOFTCAP ? f2_sub(dd2, dp2) : f2_sub(dp2, dd2));
      packed[u] = pack_bf16x2(f2_lo(r2), f2_hi(r2));
    }
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {  // 16-byte chunks 4 hh .. 4 hh + 3
      const int chunk = 4 * hh + c4;
      st_shared_v4(ds_row + ((chunk ^ (r & 7)) << 4), packed[4 * c4], packed[4 * c4 + 1],
                   packed[4 * c4 + 2], packed[4 * c4 + 3]);
    }
  }
}

template <bool SOFTCAP, bool DROP>
__device__ void softmax_role(const Ctx& c, const Params& p, const Work& w, uint8_t* smem,
                             uint32_t sbase, uint32_t tmem) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r = ((warp & 3) << 5) + lane;
  const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
  const uint32_t tS = tmem + lane_base, tdP = tmem + lane_base + 64;
  const int n0 = w.n_block * kBc;
  const int key = n0 + r;
  uint64_t pk[32];
  uint32_t km[2] = {0xFFFFFFFFu, 0xFFFFFFFFu};  // dropout keep bits of the 64 columns
  for (int t = 0; t < w.T; ++t) {
    int h, m_block;
    tile_coord(w, t, h, m_block);
    const int m0 = m_block * kBr;
    const bool masked = tile_masked(p, m0, n0);
    const uint32_t ph = t & 1;
    if (DROP) {  // this tile's keep bits, from the mask warps
      if (!wait_warp(c, BAR_MASK_FULL + (t & 1), (t >> 1) & 1)) return;
      const uint2 kb =
          reinterpret_cast<const uint2*>(smem + Layout::kMask)[(t & 1) * 128 + r];
      km[0] = kb.x;
      km[1] = kb.y;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(c, BAR_MASK_EMPTY + (t & 1)));
    }
    // P phase: LSE and D of the tile arrive with QH_FULL
    if (!wait_warp(c, BAR_QH_FULL, ph)) return;
    if (!wait_warp(c, BAR_S_FULL, ph)) return;
    tc_fence_after();
    if (masked)
      softmax_tile<SOFTCAP, true, DROP>(p, smem, sbase, tS, tdP, r, key, m0, pk, km, false);
    else
      softmax_tile<SOFTCAP, false, DROP>(p, smem, sbase, tS, tdP, r, key, m0, pk, km, false);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_addr(c, BAR_P_FULL));
    // dS phase
    if (!wait_warp(c, BAR_DP_FULL, ph)) return;
    if (t > 0 && !wait_warp(c, BAR_DS_FREE, (t - 1) & 1)) return;
    tc_fence_after();
    if (masked)
      softmax_tile<SOFTCAP, true, DROP>(p, smem, sbase, tS, tdP, r, key, m0, pk, km, true);
    else
      softmax_tile<SOFTCAP, false, DROP>(p, smem, sbase, tS, tdP, r, key, m0, pk, km, true);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_addr(c, BAR_DS_FULL));
  }
}

// ------------------------------------------------------------------ keep mask (dropout)
// Warps 12-15: thread r draws, for every tile of the unit, the 16 Philox calls
// of key n0 + r (call g: queries m0 + 4 g .. m0 + 4 g + 3, one word each) and
// writes its two 32-query words to slot t mod 2 once the softmax has read
// tile t - 2 out of it.
__device__ void mask_role(const Ctx& c, const Params& p, const Work& w, uint8_t* smem) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r = ((warp & 3) << 5) + lane;
  const uint32_t key = static_cast<uint32_t>(w.n_block * kBc + r);
  uint32_t* mask = reinterpret_cast<uint32_t*>(smem + Layout::kMask);
  for (int t = 0; t < w.T; ++t) {
    const int slot = t & 1;
    if (t >= 2 && !wait(c, BAR_MASK_EMPTY + slot, ((t >> 1) - 1) & 1)) return;
    int h, m_block;
    tile_coord(w, t, h, m_block);
    const uint32_t qgrp = static_cast<uint32_t>(m_block * kBr) >> 2;
    const uint32_t bh = static_cast<uint32_t>(w.b * p.H + h);
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {  // queries 32 half .. 32 half + 31
      uint32_t ctr[8][4];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        ctr[g][0] = qgrp + static_cast<uint32_t>(8 * half + g);
        ctr[g][1] = key;
        ctr[g][2] = bh;
        ctr[g][3] = 0u;
      }
      philox4x32_10_batch<8, 1>(ctr, p.drop.seed_lo, p.drop.seed_hi);
      uint32_t bits = 0;
#pragma unroll
      for (int g = 0; g < 8; ++g)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          bits |= (ctr[g][e] >= p.drop.threshold ? 1u : 0u) << (4 * g + e);
      mask[(slot * 128 + r) * 2 + half] = bits;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_addr(c, BAR_MASK_FULL + slot));
  }
}

// ------------------------------------------------------------------ dQ drain and epilogue
// Thread r holds dQ[m0 + i][128 half + r] in column i of the tile's dQ^T
// buffer. Each 32-query chunk goes through the staging buffer as rows of 128
// fp32 and is added into dq_accum by one TMA reduction. After the last tile,
// dV and dK (x tau) leave tensor memory as bf16 rows through the free Q and
// dO buffers and TMA stores.
constexpr int kBarDrain = 1;  // named barrier of the drain warpgroup

template <bool DET>
__device__ void drain_role(const Ctx& c, const Params& p, const Work& w, uint32_t sbase,
                           uint32_t tmem, const CUtensorMap* tm_dq, const CUtensorMap* tm_dk,
                           const CUtensorMap* tm_dv) {
  using L = Layout;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r = ((warp & 3) << 5) + lane;
  const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
  const bool leader = r == 0;
  const uint32_t stage = sbase + L::kDQS;
  bool ok = true;
  for (int t = 0; t < w.T; ++t) {
    int h, m_block;
    tile_coord(w, t, h, m_block);
    const int m0 = m_block * kBr;
    const int bh = w.b * p.H + h;
    const int qb = t & 1;
    ok = named_bar_and(kBarDrain, 128, wait(c, BAR_DQ_FULL + qb, (t >> 1) & 1));
    if (!ok) break;
    tc_fence_after();
    uint32_t v[64];
    tmem_ld32x2(tmem + lane_base + 128 + 64 * qb, tmem + lane_base + 128 + 64 * qb + 32, v);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_addr(c, BAR_DQ_EMPTY + qb));
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      if (leader) bulk_wait_read_all();  // the previous reduction has read the buffer
      named_bar_sync(kBarDrain, 128);
#pragma unroll
      for (int q = 0; q < 32; ++q)
        st_shared_f32(stage + q * 512 + r * 4, __uint_as_float(v[32 * ch + q]));
      fence_proxy_async_smem();
      named_bar_sync(kBarDrain, 128);
      const int row = m0 + 32 * ch;
      if (DET) {
        if (leader) {
          const int m = m0 >> 7, n = w.n_block;
          const int pi = p.causal ? (m * (m + 1) >> 1) + n : m * p.n_blocks + n;
          tma_store_3d(tm_dq, stage, kDh * w.half, (m0 & 127) + 32 * ch, bh * p.pairs + pi);
          bulk_commit_group();
        }
      } else if (leader && row < p.N) {
        tma_reduce_add_3d(tm_dq, stage, kDh * w.half, row, bh);
        bulk_commit_group();
      }
    }
  }
  // epilogue: every GEMM of the unit is done, so the Q and dO buffers are free
  if (ok) ok = wait(c, BAR_UNIT_DONE, 0);
  if (named_bar_and(kBarDrain, 128, ok)) {
    tc_fence_after();
    const int kvh = w.b * p.H_kv + w.g;
    const int n0 = w.n_block * kBc;
#pragma unroll
    for (int which = 0; which < 2; ++which) {  // 0: dV -> Q buffer, 1: dK * tau -> dO buffer
      const uint32_t src = tmem + lane_base + (which ? 384 : 256);
      const uint32_t dst = sbase + (which ? L::kDO : L::kQ);
      const float mul = which ? p.scale : 1.f;
#pragma unroll
      for (int ch = 0; ch < kDh / 16; ++ch) {
        uint32_t raw[16];
        tmem_ld16(src + 16 * ch, raw);
        uint32_t packed[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          packed[u] = pack_bf16x2(__uint_as_float(raw[2 * u]) * mul,
                                  __uint_as_float(raw[2 * u + 1]) * mul);
        // columns 16 ch .. + 15 of this half: box ch / 4 ([128 rows][64 cols],
        // 16 KB), 16-byte chunks 2 (ch % 4), + 1, 128-byte swizzle
        const uint32_t row_addr = dst + (ch >> 2) * 16384 + r * 128;
        const int c0 = 2 * (ch & 3);
        st_shared_v4(row_addr + ((c0 ^ (r & 7)) << 4), packed[0], packed[1], packed[2],
                     packed[3]);
        st_shared_v4(row_addr + (((c0 + 1) ^ (r & 7)) << 4), packed[4], packed[5], packed[6],
                     packed[7]);
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(kBarDrain, 128);
    if (leader) {
      for (int bx = 0; bx < 2; ++bx) {
        tma_store_3d(tm_dv, sbase + L::kQ + bx * 16384, kDh * w.half + 64 * bx, n0, kvh);
        tma_store_3d(tm_dk, sbase + L::kDO + bx * 16384, kDh * w.half + 64 * bx, n0, kvh);
      }
      bulk_commit_group();
    }
  }
  if (leader) bulk_wait_all();  // reductions and stores complete before the CTA exits
}

// ------------------------------------------------------------------ kernel
template <bool SOFTCAP, bool DET, bool DROP>
__global__ void __launch_bounds__(kThreadsFor<DROP>, 1)
    attn_bwd256_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq,
                       const __grid_constant__ CUtensorMap tm_dk,
                       const __grid_constant__ CUtensorMap tm_dv, const Params p) {
  using L = Layout;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // the 128-byte swizzle atoms need 1024-byte alignment
    if (threadIdx.x == 0) record_status(ATTN_ERR_DEVICE);
    return;
  }
  Ctx c;
  c.bars = sbase + L::kBars;
  c.abort = reinterpret_cast<volatile int*>(smem + L::kAbort);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNumBars; ++i) mbar_init(bar_addr(c, i), 1);
    mbar_init(bar_addr(c, BAR_QH_FULL), 33);  // expect_tx arrive + 32 LSE/D lanes
    mbar_init(bar_addr(c, BAR_P_FULL), 4);   // the 4 softmax warps
    mbar_init(bar_addr(c, BAR_DS_FULL), 4);
    mbar_init(bar_addr(c, BAR_DQ_EMPTY), 4);  // the 4 drain warps
    mbar_init(bar_addr(c, BAR_DQ_EMPTY + 1), 4);
    if (DROP) {
      for (int sl = 0; sl < 2; ++sl) {
        mbar_init(bar_addr(c, BAR_MASK_FULL + sl), 4);   // the mask warps
        mbar_init(bar_addr(c, BAR_MASK_EMPTY + sl), 4);  // the softmax warps
      }
    }
    *c.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + L::kTmemSlot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);
  const Work w = work_of(p);
  if (warp < 4) {
    if constexpr (DROP) setmaxnreg_dec<kRegsNarrowDrop>();
    if (warp == 0)
      producer_role(c, p, w, smem, sbase, &tm_q, &tm_k, &tm_v, &tm_do);
    else if (warp == 1)
      mma_role(c, w, sbase, tmem);
  } else if (warp < 8) {
    if constexpr (DROP) setmaxnreg_inc<kRegsWideDrop>();
    softmax_role<SOFTCAP, DROP>(c, p, w, smem, sbase, tmem);
  } else if (warp < 12) {
    if constexpr (DROP) setmaxnreg_inc<kRegsWideDrop>();
    drain_role<DET>(c, p, w, sbase, tmem, &tm_dq, &tm_dk, &tm_dv);
  } else {
    if constexpr (DROP) {
      setmaxnreg_dec<kRegsNarrowDrop>();
      mask_role(c, p, w, smem);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool SOFTCAP, bool DET, bool DROP>
int launch(const CUtensorMap (&m)[7], const Params& p, long long grid, cudaStream_t s) {
  auto kern = attn_bwd256_kernel<SOFTCAP, DET, DROP>;
  static std::atomic<bool> configured[kMaxTrackedDevices];
  if (!set_smem_limit_once(kern, Layout::kBytes, configured)) return ATTN_ERR_LAUNCH;
  kern<<<static_cast<unsigned>(grid), kThreadsFor<DROP>, Layout::kBytes, s>>>(
      m[0], m[1], m[2], m[3], m[4], m[5], m[6], p);
  return launch_status();
}

}  // namespace bwd256

// Device status word of the d = 256 kernel (read by attn_device_status).
int bwd256_status(int* status, bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, bwd256::g_status256, sizeof(int)) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  *status = v;
  if (clear && v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(bwd256::g_status256, &zero, sizeof(int)) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

// attn_bwd (and its local, dropout and deterministic forms) with d = 256:
// the arguments have been checked by the caller (pointers, shape, alignment,
// scale, drop probability), B, H, N > 0. With det, dq_target is the partials
// workspace (`pairs` tiles per query head), else the dQ accumulator.
int bwd256_run(const void* q, const void* k, const void* v, const void* dO, const float* lse,
               float* dq_target, void* dk, void* dv, int B, int H, int H_kv, int N, float scale,
               int causal, float softcap, const float* dpsum, int window_left, int window_right,
               bool det, int pairs, float p_drop, unsigned long long seed, cudaStream_t s) {
  using namespace bwd256;
  Params p;
  p.lse = lse;
  p.dpsum = dpsum;
  p.B = B;
  p.H = H;
  p.H_kv = H_kv;
  p.N = N;
  p.n_blocks = (N + kBc - 1) / kBc;
  p.m_blocks = (N + kBr - 1) / kBr;
  p.scale = scale;
  const bool cap = softcap > 0.f;
  p.softcap = cap ? softcap : 0.f;
  p.win_left = (window_left < 0 || window_left > N) ? N : window_left;
  p.win_right = causal ? 0 : ((window_right < 0 || window_right > N) ? N : window_right);
  p.pairs = pairs;
  p.causal = causal != 0 ? 1 : 0;
  p.drop.seed_lo = static_cast<uint32_t>(seed);
  p.drop.seed_hi = static_cast<uint32_t>(seed >> 32);
  p.drop.threshold = dropout_threshold(p_drop);
  p.drop.inv_keep = 1.f / (1.f - p_drop);
  p.drop.keep = 1.f - p_drop;
  p.drop.log2_inv_keep =
      static_cast<float>(-std::log2(1.0 - static_cast<double>(p_drop)));
  const long long grid = 2LL * p.n_blocks * H_kv * B;
  if (grid > 0x7fffffffLL) return ATTN_ERR_TOO_LARGE;
  CUtensorMap m[7];  // q, k, v, dO, dq (reduce), dk, dv (store)
  const long long hq = static_cast<long long>(B) * H, hk = static_cast<long long>(B) * H_kv;
  if (!encode_bf16_3d(&m[0], q, kD, N, hq, kBr) || !encode_bf16_3d(&m[1], k, kD, N, hk, kBc) ||
      !encode_bf16_3d(&m[2], v, kD, N, hk, kBc) || !encode_bf16_3d(&m[3], dO, kD, N, hq, kBr) ||
      !(det ? encode_f32_3d(&m[4], dq_target, kD, 128, hq * pairs, 32, kDh)
            : encode_f32_3d(&m[4], dq_target, kD, N, hq, 32, kDh)) ||
      !encode_bf16_3d(&m[5], dk, kD, N, hk, kBc) || !encode_bf16_3d(&m[6], dv, kD, N, hk, kBc))
    return ATTN_ERR_LAUNCH;
  if (p_drop > 0.f)  // not combined with det
    return cap ? launch<true, false, true>(m, p, grid, s)
               : launch<false, false, true>(m, p, grid, s);
  if (det)
    return cap ? launch<true, true, false>(m, p, grid, s)
               : launch<false, true, false>(m, p, grid, s);
  return cap ? launch<true, false, false>(m, p, grid, s)
             : launch<false, false, false>(m, p, grid, s);
}

}  // namespace attn
