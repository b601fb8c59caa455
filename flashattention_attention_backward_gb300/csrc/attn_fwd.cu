// attn_fwd: attention forward on sm_103a producing O and the natural-log
// LSE the backward needs ("反向传播算法详解" §1.2-§1.3 saved tensors;
// "解析 FlashAttention（3）" §1.1 forward).
//
// One CTA owns a block of Bm = 128 queries of one query head and walks the
// key blocks (Bn = 128 keys) its mask lets it see, in two passes:
//   pass 1  S_j = Q K_j^T on the tensor cores; the softmax warps keep the
//           running row maximum m and sum l of exp2 over S_j, which gives
//           LSE exactly (in base 2: LSE2 = m + log2 l);
//   pass 2  S_j again; P_j = exp2(S_j * tau*log2e - LSE2) is already
//           normalised, goes to tensor memory as bf16 and O += P_j V_j
//           accumulates there with no rescaling.
// This spends one extra S GEMM per tile (three GEMMs instead of two) to keep
// the O accumulator free of the running-max corrections of a one-pass
// online softmax.
//
// Queries sit on the tensor-memory lanes: thread r of the softmax warpgroup
// owns query row r, so row maxima and sums need no cross-thread reduction,
// and P (bf16 pairs, keys along the columns) is the A operand of the PV GEMM
// straight from tensor memory.
//
// Warp roles (384 threads):
//   warp 0      TMA producer: Q once, K_j for every S GEMM, V_j in pass 2
//               (two-stage rings)
//   warp 1      tcgen05 MMA issuer (whole warp, one elected lane issues)
//   warps 4-11  softmax in two warpgroups, one per S buffer, then the
//               epilogue (O -> bf16 -> shared -> TMA store; LSE)
//
// Tensor memory (512 columns): S buffers at [0,128) and [128,256) (P
// overwrites the first half of its buffer), O accumulator at [256, 256 + d).
// Every mbarrier wait is bounded, as in attn_bwd.
#include <cstdint>
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace fwdtc {

using namespace ptx;

constexpr int kBm = 128;  // queries per CTA (tensor-memory lanes)
constexpr int kBn = 128;  // keys per tile
constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr long long kWaitLimitCycles = 2000000000LL;  // about one second

template <int D>
struct Layout {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kQ = 0;  // also the O staging buffer at the end
  static constexpr int kK0 = kQ + kTileBytes;
  static constexpr int kK1 = kK0 + kTileBytes;
  static constexpr int kV0 = kK1 + kTileBytes;
  static constexpr int kV1 = kV0 + kTileBytes;
  static constexpr int kStats = kV1 + kTileBytes;  // 2 x 128 rows x (m, l) fp32
  static constexpr int kBars = kStats + 2 * 128 * 8;
  static constexpr int kNumBars = 16;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  // d = 64 needs 80 KB; it asks for more than half of the SM's shared memory
  // so that a second CTA never waits on the first one's tensor memory
  static constexpr int kUsed = kAbort + 12;
  static constexpr int kBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
};

enum Bar {
  BAR_Q_FULL = 0,
  BAR_K_FULL = 1,    // + stage
  BAR_K_EMPTY = 3,   // + stage
  BAR_V_FULL = 5,    // + stage
  BAR_V_EMPTY = 7,   // + stage
  BAR_S_FULL = 9,    // + buffer
  BAR_S_FREE = 11,   // + buffer: the softmax (pass 1) or the PV GEMM (pass 2) is done with it
  BAR_P_FULL = 13,   // + buffer (pass 2 only)
  BAR_O_DONE = 15,
};

struct Params {
  float* lse;
  int B, H, H_kv, N;
  int m_blocks;
  float scale;
  float softcap;
  // visibility band: key j is visible to query i iff
  // i - win_left <= j <= i + win_right (the causal mask is win_right = 0;
  // an unbounded side holds N)
  int win_left, win_right;
};

struct Ctx {
  uint32_t bars;
  volatile int* abort;
};

__device__ __forceinline__ uint32_t bar_addr(const Ctx& c, int i) { return c.bars + 8u * i; }

__device__ int g_fwd_status;

__device__ __noinline__ void record_status(int code) { atomicCAS(&g_fwd_status, 0, code); }

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

// Work of one CTA: query block m_block of head bh (= b * H + h), against
// key blocks j0 .. j0 + nk - 1 (those holding a key of the rows' bands).
struct Work {
  int bh, kvh, m_block, j0, nk;  // nk: key blocks visited (per pass)
};

__device__ __forceinline__ Work work_of(const Params& p) {
  Work w;
  const int heads = p.B * p.H;
  const int idx = static_cast<int>(blockIdx.x);
  // heaviest query blocks first for a causal mask (the last ones see the
  // most keys)
  w.m_block = p.m_blocks - 1 - idx / heads;
  w.bh = idx - (idx / heads) * heads;
  const int b = w.bh / p.H, h = w.bh - b * p.H;
  w.kvh = b * p.H_kv + h / (p.H / p.H_kv);
  const int m0 = w.m_block * kBm;
  w.j0 = max(0, m0 - p.win_left) / kBn;
  const int j_end = min((p.N + kBn - 1) / kBn - 1, (m0 + kBm - 1 + p.win_right) / kBn);
  w.nk = j_end - w.j0 + 1;
  return w;
}

// ------------------------------------------------------------------ producer
template <int D>
__device__ void producer_role(const Ctx& c, const Work& w, uint32_t sbase, const CUtensorMap* tq,
                              const CUtensorMap* tk, const CUtensorMap* tv) {
  using L = Layout<D>;
  constexpr int kBoxes = D / 64;
  constexpr uint32_t kTileBytes = L::kTileBytes;
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    prefetch_tmap(tq);
    prefetch_tmap(tk);
    prefetch_tmap(tv);
    mbar_arrive_expect_tx(bar_addr(c, BAR_Q_FULL), kTileBytes);
    for (int cb = 0; cb < kBoxes; ++cb)
      tma_load_3d(sbase + L::kQ + cb * 16384, tq, bar_addr(c, BAR_Q_FULL), 64 * cb,
                  w.m_block * kBm, w.bh);
  }
  const uint64_t keep = policy_evict_last();  // K, V are read by every query block of the head
  int issued_k = 0, issued_v = 0;
  bool ok = true;
  for (int s = 0; s < 2 * w.nk; ++s) {
    const bool pass2 = s >= w.nk;
    const int j = pass2 ? s - w.nk : s;
    const int ks = s & 1;
    if (s >= 2 && !(ok = wait_warp(c, BAR_K_EMPTY + ks, ((s >> 1) - 1) & 1))) break;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_addr(c, BAR_K_FULL + ks), kTileBytes);
      const uint32_t dst = sbase + (ks ? L::kK1 : L::kK0);
      for (int cb = 0; cb < kBoxes; ++cb)
        tma_load_3d_hint(dst + cb * 16384, tk, bar_addr(c, BAR_K_FULL + ks), 64 * cb,
                         (w.j0 + j) * kBn, w.kvh, keep);
    }
    issued_k = s + 1;
    if (pass2) {
      const int vs = j & 1;
      if (j >= 2 && !(ok = wait_warp(c, BAR_V_EMPTY + vs, ((j >> 1) - 1) & 1))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_addr(c, BAR_V_FULL + vs), kTileBytes);
        const uint32_t dst = sbase + (vs ? L::kV1 : L::kV0);
        for (int cb = 0; cb < kBoxes; ++cb)
          tma_load_3d_hint(dst + cb * 16384, tv, bar_addr(c, BAR_V_FULL + vs), 64 * cb,
                           (w.j0 + j) * kBn, w.kvh, keep);
      }
      issued_v = j + 1;
    }
    __syncwarp();
  }
  // When aborting, the copies in flight must land before the CTA exits.
  if (!ok || *c.abort) {
    wait_drain(c, BAR_Q_FULL, 0);
    for (int s = issued_k - 2 < 0 ? 0 : issued_k - 2; s < issued_k; ++s)
      wait_drain(c, BAR_K_FULL + (s & 1), (s >> 1) & 1);
    for (int j = issued_v - 2 < 0 ? 0 : issued_v - 2; j < issued_v; ++j)
      wait_drain(c, BAR_V_FULL + (j & 1), (j >> 1) & 1);
  }
}

// P_FULL + w keeps one phase per pass-2 tile of buffer w.
__device__ __forceinline__ uint32_t p_phase(int s, int nk) {
  const int first = ((nk & 1) == (s & 1)) ? nk : nk + 1;  // first pass-2 tile of this buffer
  return static_cast<uint32_t>(((s - first) >> 1) & 1);
}

// ------------------------------------------------------------------ MMA issuer
// S GEMM s (s < nk: pass 1, else pass 2 over the same key blocks) goes to
// buffer s & 1 once the previous use of that buffer has been released; in
// pass 2, O += P V follows each P. Every barrier keeps one phase per use.
template <int D>
__device__ void mma_role(const Ctx& c, const Work& w, uint32_t sbase, uint32_t tmem) {
  using L = Layout<D>;
  const bool leader = elect_one_sync() != 0;
  constexpr uint32_t kIdS = make_idesc_bf16(kBm, kBn, false, false);  // S = Q K^T
  constexpr uint32_t kIdO = make_idesc_bf16(kBm, D, false, true);     // O += P V
  const uint32_t q_lo = sdesc_lo(sbase + L::kQ, 16);
  const uint32_t k_lo0 = sdesc_lo(sbase + L::kK0, 16), k_lo1 = sdesc_lo(sbase + L::kK1, 16);
  const uint32_t v_mn0 = sdesc_lo(sbase + L::kV0, 16384), v_mn1 = sdesc_lo(sbase + L::kV1, 16384);
  const uint32_t tO = tmem + 256;
  auto kmaj = [](int k) { return static_cast<uint32_t>(((k >> 2) * 16384 + (k & 3) * 32) >> 4); };
  auto mnmaj = [](int k) { return static_cast<uint32_t>((2048 * k) >> 4); };
  const int total = 2 * w.nk;
  bool ok = wait_warp(c, BAR_Q_FULL, 0);
  auto issue_s = [&](int s) -> bool {
    const int b = s & 1;
    if (!wait_warp(c, BAR_K_FULL + b, (s >> 1) & 1)) return false;
    if (s >= 2 && !wait_warp(c, BAR_S_FREE + b, ((s >> 1) - 1) & 1)) return false;
    tc_fence_after();
    if (leader) {
      const uint32_t kb = b ? k_lo1 : k_lo0;
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        mma_ss(tmem + b * 128, sdesc_from_lo(q_lo + kmaj(k)), sdesc_from_lo(kb + kmaj(k)), kIdS,
               k > 0);
      mma_commit(bar_addr(c, BAR_S_FULL + b));
      mma_commit(bar_addr(c, BAR_K_EMPTY + b));
    }
    return true;
  };
  if (ok) ok = issue_s(0);
  for (int s = 0; ok && s < total; ++s) {
    if (s + 1 < total && !(ok = issue_s(s + 1))) break;
    if (s >= w.nk) {
      const int j = s - w.nk, b = s & 1, vs = j & 1;
      if (!(ok = wait_warp(c, BAR_P_FULL + b, p_phase(s, w.nk)))) break;
      if (!(ok = wait_warp(c, BAR_V_FULL + vs, (j >> 1) & 1))) break;
      tc_fence_after();
      if (leader) {
        const uint32_t vb = vs ? v_mn1 : v_mn0;
        // A = P (bf16 pairs, keys along columns 8k .. of buffer b)
#pragma unroll
        for (int k = 0; k < kBn / 16; ++k)
          mma_ts(tO, tmem + b * 128 + 8 * k, sdesc_from_lo(vb + mnmaj(k)), kIdO,
                 (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar_addr(c, BAR_S_FREE + b));
        mma_commit(bar_addr(c, BAR_V_EMPTY + vs));
      }
    }
  }
  // O complete (or, when aborting, everything issued complete)
  if (leader) mma_commit(bar_addr(c, BAR_O_DONE));
  if (__any_sync(0xffffffffu, !ok || *c.abort != 0)) wait_drain(c, BAR_O_DONE, 0);
  __syncwarp();
}

// ------------------------------------------------------------------ softmax
// One S tile of one query row (this thread's tensor-memory lane), in four
// 32-key chunks. Pass 1 (PASS2 false) folds the chunk into the running
// maximum m and sum l of 2^x; pass 2 writes P = 2^(x - lse2) as bf16 pairs
// over the first half of the S buffer. MASKED tiles (the band's edges, the
// sequence's end) hide invisible keys with -inf; the others skip the test.
template <bool SOFTCAP, bool MASKED, bool PASS2>
__device__ __forceinline__ void tile_rows(const Params& p, uint32_t tS, int n0, int q,
                                          float c_log2, float cap_in, float cap_out, float& m,
                                          float& l, float lse2) {
#pragma unroll
  for (int ch = 0; ch < kBn / 32; ++ch) {
    uint32_t raw[32];
    tmem_ld32(tS + ch * 32, raw);
    float cm0 = -INFINITY, cm1 = -INFINITY;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float sv = __uint_as_float(raw[e]);
      float x;
      if (SOFTCAP) {
        // tanh(u) = 1 - 2 / (exp(2u) + 1) with u = tau s / c
        const float ex = ex2_approx(sv * cap_in);
        x = (1.f - 2.f * rcp_approx(ex + 1.f)) * cap_out;
      } else {
        x = sv * c_log2;
      }
      if (MASKED) {
        const int key = n0 + ch * 32 + e;
        if (!(key < p.N && key - q <= p.win_right && q - key <= p.win_left)) x = -INFINITY;
      }
      raw[e] = __float_as_uint(x);
      if (!PASS2) {
        if (e & 1)
          cm1 = fmaxf(cm1, x);
        else
          cm0 = fmaxf(cm0, x);
      }
    }
    if (!PASS2) {
      const float mn = fmaxf(m, fmaxf(cm0, cm1));
      // only a masked chunk (a window's edge, a padding row) can hold no
      // visible key; the shift then stays finite so that -inf - -inf never
      // arises (the exponentials of -inf are 0)
      const float sh = (MASKED && mn == -INFINITY) ? 0.f : mn;
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 32; ++e) s4[e & 3] += ex2_approx(__uint_as_float(raw[e]) - sh);
      l = l * ex2_approx(m - sh) + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
      m = mn;
    } else {
      uint32_t packed[16];
#pragma unroll
      for (int u = 0; u < 16; ++u)
        packed[u] = pack_bf16x2(ex2_approx(__uint_as_float(raw[2 * u]) - lse2),
                                ex2_approx(__uint_as_float(raw[2 * u + 1]) - lse2));
      // keys 32 ch .. 32 ch + 31 -> columns 16 ch .. 16 ch + 15, whose S
      // values were read in this or an earlier chunk
      tmem_st16(tS + ch * 16, packed);
    }
  }
}

// Two warpgroups; warpgroup w takes the S GEMMs s with s & 1 == w, i.e. S
// buffer w, so each processes one tile while the other's S GEMM runs.
// Thread = query row r (tensor-memory lane). Pass 1 keeps the running
// maximum m and sum l of 2^x over the row (x = logit * log2e) for the
// warpgroup's key blocks; the two partial statistics are combined through
// shared memory into LSE2 at the pass boundary. Pass 2 writes
// P = 2^(x - LSE2) as bf16 pairs over the first half of the S buffer, which
// the PV GEMM reads as its A operand. Then each warpgroup stores half of the
// columns of O.
template <int D, bool SOFTCAP>
__device__ void softmax_role(const Ctx& c, const Params& p, const Work& w, uint8_t* smem,
                             uint32_t sbase, uint32_t tmem, const CUtensorMap* to) {
  using L = Layout<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wg = (warp - 4) >> 2;  // 0 or 1: the S buffer this warpgroup owns
  const int r = ((warp & 3) << 5) + lane;
  const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
  const int q = w.m_block * kBm + r;
  const int bar_wg = 1 + wg;  // named barrier of this warpgroup (128 threads)
  const float c_log2 = p.scale * kLog2e;
  const float cap_in = SOFTCAP ? 2.f * kLog2e * p.scale / p.softcap : 0.f;  // 2 log2e tau/c
  const float cap_out = SOFTCAP ? p.softcap * kLog2e : 0.f;                 // c log2e
  float m = -INFINITY, l = 0.f, lse2 = 0.f;
  bool ok = true;
  const uint32_t tS = tmem + lane_base + wg * 128;
  // Both warpgroups pass the same sequence of named-barrier-3 operations on
  // every path (the votes below), so an abort can never strand one of them.
  auto tile = [&](int s) -> bool {
    const bool pass2 = s >= w.nk;
    const int j = pass2 ? s - w.nk : s;
    // the warpgroup meets at its named barrier below: one decision for all
    ok = named_bar_and(bar_wg, 128, wait(c, BAR_S_FULL + wg, (s >> 1) & 1));
    if (!ok) return false;
    tc_fence_after();
    const int n0 = (w.j0 + j) * kBn;
    const int m0 = w.m_block * kBm;
    const bool masked = n0 + kBn - 1 - m0 > p.win_right || m0 + kBm - 1 - n0 > p.win_left ||
                        n0 + kBn > p.N;
    if (pass2) {
      if (masked)
        tile_rows<SOFTCAP, true, true>(p, tS, n0, q, c_log2, cap_in, cap_out, m, l, lse2);
      else
        tile_rows<SOFTCAP, false, true>(p, tS, n0, q, c_log2, cap_in, cap_out, m, l, lse2);
    } else {
      if (masked)
        tile_rows<SOFTCAP, true, false>(p, tS, n0, q, c_log2, cap_in, cap_out, m, l, lse2);
      else
        tile_rows<SOFTCAP, false, false>(p, tS, n0, q, c_log2, cap_in, cap_out, m, l, lse2);
    }
    if (!pass2) {
      // the buffer is free for the next S GEMM once every row has read it
      tc_fence_before();
      named_bar_sync(bar_wg, 128);
      if (r == 0) mbar_arrive(bar_addr(c, BAR_S_FREE + wg));
    } else {
      tmem_wait_st();
      tc_fence_before();
      named_bar_sync(bar_wg, 128);
      if (r == 0) mbar_arrive(bar_addr(c, BAR_P_FULL + wg));
    }
    return true;
  };
  // pass 1 over this warpgroup's key blocks
  for (int s = wg; ok && s < w.nk; s += 2) ok = tile(s);
  // combine the two warpgroups' row statistics (one without pass-1 tiles
  // has m = -inf, l = 0)
  ok = named_bar_and(3, 256, ok);
  if (ok) {
    float* st = reinterpret_cast<float*>(smem + L::kStats);
    st[(wg * 128 + r) * 2] = m;
    st[(wg * 128 + r) * 2 + 1] = l;
    named_bar_sync(3, 256);
    const float mo = st[((1 - wg) * 128 + r) * 2], lo = st[((1 - wg) * 128 + r) * 2 + 1];
    const float mx = fmaxf(m, mo);
    const float sh = mx == -INFINITY ? 0.f : mx;
    lse2 = sh + __log2f(l * ex2_approx(m - sh) + lo * ex2_approx(mo - sh));
    // a padding row past N may see no key at all: its P must be 0, not NaN
    if (!(lse2 < INFINITY && lse2 > -INFINITY)) lse2 = INFINITY;
  }
  // pass 2
  for (int s = ((w.nk & 1) == wg) ? w.nk : w.nk + 1; ok && s < 2 * w.nk; s += 2) ok = tile(s);
  // ---- epilogue: O (already normalised) -> bf16 rows in the Q buffer (free
  // once every GEMM is done) -> TMA tensor store; LSE in natural log.
  // Warpgroup wg takes columns [wg * D/2, (wg + 1) * D/2) of every row.
  if (ok) ok = wait(c, BAR_O_DONE, 0);
  if (!named_bar_and(3, 256, ok)) return;  // both warpgroups reach this vote on every path
  tc_fence_after();
#pragma unroll
  for (int c16 = 0; c16 < D / 32; ++c16) {
    const int col = wg * (D / 2) + c16 * 16;
    uint32_t raw[16];
    tmem_ld16(tmem + lane_base + 256 + col, raw);
    uint32_t packed[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      packed[u] = pack_bf16x2(__uint_as_float(raw[2 * u]), __uint_as_float(raw[2 * u + 1]));
    // columns col .. col + 15: box col / 64, 16-byte chunks (col % 64) / 8, + 1
    const uint32_t row_addr = sbase + L::kQ + (col >> 6) * 16384 + r * 128;
    const int c0 = (col & 63) >> 3;
    st_shared_v4(row_addr + ((c0 ^ (r & 7)) << 4), packed[0], packed[1], packed[2], packed[3]);
    st_shared_v4(row_addr + (((c0 + 1) ^ (r & 7)) << 4), packed[4], packed[5], packed[6],
                 packed[7]);
  }
  fence_proxy_async_smem();
  named_bar_sync(3, 256);
  if (wg == 0 && r == 0) {
    for (int cb = 0; cb < D / 64; ++cb)
      tma_store_3d(to, sbase + L::kQ + cb * 16384, 64 * cb, w.m_block * kBm, w.bh);
    bulk_commit_group();
    bulk_wait_all();
  }
  if (wg == 0 && q < p.N) p.lse[static_cast<long long>(w.bh) * p.N + q] = lse2 * kLn2;
}

// ------------------------------------------------------------------ kernel
template <int D, bool SOFTCAP>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o, const Params p) {
  using L = Layout<D>;
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
  if (warp == 0) {
    producer_role<D>(c, w, sbase, &tm_q, &tm_k, &tm_v);
  } else if (warp == 1) {
    mma_role<D>(c, w, sbase, tmem);
  } else if (warp >= 4) {
    softmax_role<D, SOFTCAP>(c, p, w, smem, sbase, tmem, &tm_o);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool SOFTCAP>
int launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
           const CUtensorMap& to, const Params& p, cudaStream_t stream) {
  auto kern = attn_fwd_kernel<D, SOFTCAP>;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Layout<D>::kBytes) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
    configured = true;
  }
  const long long grid = static_cast<long long>(p.m_blocks) * p.B * p.H;
  if (grid > 0x7fffffffLL) return ATTN_ERR_TOO_LARGE;
  kern<<<static_cast<unsigned>(grid), kThreads, Layout<D>::kBytes, stream>>>(tq, tk, tv, to, p);
  return launch_status();
}

}  // namespace fwdtc

// Device status of the forward kernels (read by attn_device_status).
int fwd_status(int* status, bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, fwdtc::g_fwd_status, sizeof(int)) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  *status = v;
  if (clear && v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(fwdtc::g_fwd_status, &zero, sizeof(int)) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

}  // namespace attn

using namespace attn;

namespace attn {
namespace fwdtc {

int run(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv,
        int N, int d, float scale, int causal, float softcap, int window_left, int window_right,
        void* stream) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  int rc = check_shape(B, H, H_kv, N, d);
  if (rc != ATTN_OK) return rc;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || scale == 0.f || std::isnan(softcap)) return ATTN_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_ALIGN;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  CUtensorMap tq, tk, tv, to;
  const long long hq = static_cast<long long>(B) * H, hk = static_cast<long long>(B) * H_kv;
  if (!encode_bf16_3d(&tq, q, d, N, hq, kBm) || !encode_bf16_3d(&tk, k, d, N, hk, kBn) ||
      !encode_bf16_3d(&tv, v, d, N, hk, kBn) || !encode_bf16_3d(&to, o, d, N, hq, kBm))
    return ATTN_ERR_LAUNCH;
  Params p;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.H_kv = H_kv;
  p.N = N;
  p.m_blocks = (N + kBm - 1) / kBm;
  p.scale = scale;
  const bool cap = softcap > 0.f;
  p.softcap = cap ? softcap : 0.f;
  // a negative or wider-than-N side of the window is unbounded (N); the
  // causal mask bounds the right side at 0
  p.win_left = (window_left < 0 || window_left > N) ? N : window_left;
  p.win_right = causal ? 0 : ((window_right < 0 || window_right > N) ? N : window_right);
  cudaStream_t s = as_stream(stream);
  if (d == 128)
    return cap ? launch<128, true>(tq, tk, tv, to, p, s) : launch<128, false>(tq, tk, tv, to, p, s);
  return cap ? launch<64, true>(tq, tk, tv, to, p, s) : launch<64, false>(tq, tk, tv, to, p, s);
}

}  // namespace fwdtc
}  // namespace attn

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int H_kv, int N, int d, float scale, int causal, float softcap,
                        void* stream) {
  return fwdtc::run(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, -1, -1, stream);
}

extern "C" int attn_fwd_local(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int H_kv, int N, int d, float scale, int causal,
                              float softcap, int window_left, int window_right, void* stream) {
  return fwdtc::run(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, window_left,
                    window_right, stream);
}
