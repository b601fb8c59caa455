// attn_bwd: attention backward on sm_103a, N-outer / Q-inner, recompute-P.
//
// Method ("反向传播算法详解" §2-§6; "解析 FlashAttention（3）" §3-§4):
// the unit of work is a block of Bc = 128 keys of one KV head (block
// coordinate (n_block, kv_head, batch), "反向传播算法详解" §3.3). Its CTA
// loads K_j, V_j once (§4.5) and keeps the fp32 accumulators dK_j, dV_j in
// tensor memory while it walks every query block i (Br = 128 rows) of every
// query head of the KV head's group. Per (i, j) tile it runs the five GEMMs
// of §5.2 on the tcgen05 tensor cores and the elementwise softmax backward in
// registers:
//
//   S^T  = K_j Q_i^T                (M = keys, N = queries, K = d)
//   dP^T = V_j dO_i^T
//   P    = exp2(S^T * tau*log2e - LSE*log2e)   [softcap: tau*S -> c tanh(tau*S/c)]
//   dS   = P o (dP - D)              [softcap: o (1 - tanh^2)]
//   dV_j += P^T dO_i                 (P^T taken from tensor memory)
//   dK_j += dS^T Q_i                 (dS^T from shared memory)
//   dQ_i += dS K_j                   (dS from shared memory; fp32 TMA
//                                     reductions into dq_accum)
//
// Because S^T is computed with keys on the tensor-memory lanes, P^T already
// sits in the layout the dV GEMM wants as its A operand and never passes
// through shared memory (the analogue of feeding P from registers to the dV
// GEMM, "反向传播算法详解" §8.2). dK/dV are summed over the GQA group on chip
// (§8.5 sums them in fp32 HBM buffers instead), so they need no atomics;
// only dQ is accumulated globally (§3.2, §6).
//
// The kernel is persistent: one CTA per SM walks units in snake order, with
// the next unit's K and V loaded as soon as the last GEMMs that read the
// current ones are done.
//
// Warp roles (640 threads, five warpgroups; registers 80 / 128 / 72 after
// setmaxnreg):
//   warp 0       TMA producer: per tile Q_i (+LSE_i, D_i) and dO_i into rings
//                (the two pipelines of §4.3); per unit K_j, V_j
//   warp 1       tcgen05 MMA issuer (the whole warp runs the loop, one
//                elected lane issues), tensor-memory owner
//   warps 4-11   softmax backward: two warpgroups, one per half of the
//                query columns; thread = key row (tensor-memory lane)
//   warps 12-19  dQ drain: two warpgroups, each loads its share of the dQ
//                tile from tensor memory and frees it, then stages it in
//                shared memory and adds it into dq_accum with TMA tensor
//                reductions; after a unit's last tile, its dK/dV epilogue
//
// MMA issue order per tile: dP_t, dV_t, S_{t+1}, dQ_t, dK_t. The P phase of
// tile t+1 overlaps dQ_t/dK_t, dK_t overlaps the dQ drain, and only
// dP -> dS -> dQ -> drain forms the per-tile dependency chain. The dQ
// reduction (bounded by the L2 reduction rate, about 6 TB/s on GB300)
// overlaps the next tile instead of stalling it.
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   [  0,128)  S^T (fp32); P^T (bf16 pairs) overwrites the read part
//   [128,256)  dP^T (fp32), then the dQ tile of the same query block
//   [256,384)  dV accumulator     [384,512)  dK accumulator
// dS^T goes to shared memory only ([key][query], 128-byte swizzle): it is the
// K-major A operand of dK += dS^T Q and the MN-major B operand of the dQ GEMM.
//
// Every wait on an mbarrier is bounded: on timeout the kernel records
// ATTN_ERR_DEVICE_TIMEOUT in the device status word and all roles return.
#include <cstdint>
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "philox.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace bwd {

using namespace ptx;

constexpr int kBc = 128;  // keys per CTA (tensor-memory lanes)
constexpr int kBr = 128;  // queries per tile
constexpr int kThreads = 640;
// registers per thread after setmaxnreg (launch: 640 x 96)
constexpr int kRegsCtl = 80, kRegsSoftmax = 128, kRegsDq = 72;
static_assert(128 * (kRegsCtl + 2 * kRegsSoftmax + 2 * kRegsDq) <= kThreads * 96, "register pool");
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitLimitCycles = 2000000000LL;  // about one second

__device__ int g_status;  // device status word (ATTN_OK or ATTN_ERR_*)

template <int D>
struct Layout {
  static constexpr int kTileBytes = kBr * D * 2;  // one Q / dO / K / V tile
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ0 = kV + kTileBytes;
  static constexpr int kQ1 = kQ0 + kTileBytes;
  // d = 128: one dO stage, and the freed 32 KB stage the dQ tile for TMA
  // reductions (two 16 KB buffers, [32 queries][128 d] fp32). d = 64: two
  // dO stages and two 4 KB buffers per drain warp ([32 queries][32 d] fp32).
  static constexpr int kDOStages = D == 128 ? 1 : 2;
  static constexpr int kDO0 = kQ1 + kTileBytes;
  static constexpr int kDO1 = kDO0 + (kDOStages - 1) * kTileBytes;
  static constexpr int kDS = kDO0 + kDOStages * kTileBytes;  // dS^T, [key][query], 32 KB
  static constexpr int kDQS = kDS + kBc * kBr * 2;            // dQ staging
  static constexpr int kDQSBytes = D == 128 ? 2 * 16384 : 8 * 2 * 4096;
  static constexpr int kLSE = kDQS + kDQSBytes;  // 2 stages x 128 fp32 (-LSE*log2e)
  static constexpr int kDsum = kLSE + 2 * kBr * 4;  // 2 stages x 128 fp32 (D)
  static constexpr int kBars = kDsum + 2 * kBr * 4;
  static constexpr int kNumBars = 21;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kBytes = kAbort + 12;
};
static_assert(Layout<128>::kBytes <= 232448, "shared memory budget");

enum Bar {
  BAR_K_FULL = 0,
  BAR_Q_FULL = 1,    // + stage
  BAR_Q_EMPTY = 3,   // + stage
  BAR_DO_FULL = 5,   // + stage
  BAR_DO_EMPTY = 7,  // + stage
  BAR_S_FULL = 9,
  BAR_P_FULL = 10,
  BAR_DP_FULL = 11,
  BAR_DS_FULL = 12,
  BAR_DQ_FULL = 13,
  BAR_DQ_EMPTY = 14,
  BAR_UNIT_DONE = 15,  // every GEMM of a unit done: the epilogue may read dK, dV
  BAR_DS_FREE = 16,
  BAR_V_FULL = 17,
  BAR_DRAIN = 18,      // abort path only: completion of everything issued
  BAR_ACC_FREE = 19,   // dK, dV of the previous unit read out: the next may overwrite them
  BAR_DSBUF_FREE = 20, // the epilogue's stores have read the dS buffer
};

struct Params {
  const float* lse;
  const float* dpsum;
  float* dq_accum;
  int B, H, H_kv, N;
  int n_blocks, m_blocks;
  int n_units;  // n_blocks * H_kv * B
  // deterministic dQ (kernel template flag DET): tiles are stored into
  // dq_accum viewed as partials [B*H*pairs, 128, d] (pair of query block m
  // and key block n: causal m (m + 1) / 2 + n, else m * n_blocks + n)
  // instead of being added
  int pairs;    // pairs per query head
  Dropout drop; // kernel template flag DROP: keep mask of philox.cuh
  float scale;
  float softcap;
  // visibility band: key j is visible to query i iff
  // i - win_left <= j <= i + win_right (the causal mask is win_right = 0;
  // an unbounded side holds N)
  int win_left, win_right;
};

// One unit of work: a block of 128 keys of one KV head of one batch entry,
// with the query tiles it visits.
struct Work {
  int b, g, n_block;
  int G, m_start, per_head, T;
};

// Units in heaviest-first order are u = n_block * (H_kv * B) + b * H_kv + g
// (for a causal mask, key block 0 sees every query block). A persistent CTA
// takes one unit per pass in snake order (pass r visits CTAs 0..grid-1 when
// r is even, grid-1..0 when odd), which balances the shrinking causal units.
__device__ __forceinline__ int unit_of(int r, int n_units) {
  const int grid = static_cast<int>(gridDim.x);
  const int cta = static_cast<int>(blockIdx.x);
  const int u = r * grid + ((r & 1) ? grid - 1 - cta : cta);
  return u < n_units ? u : -1;
}

// The query blocks a key block meets are those holding a query of its
// visibility band: queries n0 - win_right .. n0 + 127 + win_left. The band
// always holds the diagonal, so every unit has at least one tile per head.
__device__ __forceinline__ void unit_work(const Params& p, int u, Work& w) {
  const int per_nb = p.H_kv * p.B;
  w.n_block = u / per_nb;
  const int rem = u - w.n_block * per_nb;
  w.b = rem / p.H_kv;
  w.g = rem - w.b * p.H_kv;
  w.G = p.H / p.H_kv;
  const int n0 = w.n_block * kBc;
  w.m_start = max(0, n0 - p.win_right) / kBr;
  const int m_end = min(p.m_blocks - 1, (n0 + kBc - 1 + p.win_left) / kBr);
  w.per_head = m_end - w.m_start + 1;
  w.T = w.G * w.per_head;
}

// A tile needs the elementwise mask unless every (query, key) pair in it is
// inside the band and inside the sequence.
__device__ __forceinline__ bool tile_masked(const Params& p, int m0, int n0) {
  return n0 + kBc - 1 - m0 > p.win_right || m0 + kBr - 1 - n0 > p.win_left || n0 + kBc > p.N ||
         m0 + kBr > p.N;
}

struct Ctx {
  uint32_t bars;
  volatile int* abort;
};

__device__ __forceinline__ uint32_t bar_addr(const Ctx& c, int i) { return c.bars + 8u * i; }

__device__ __noinline__ void record_status(int code) { atomicCAS(&g_status, 0, code); }

// Bounded wait; returns false if the kernel is aborting (another role gave
// up) or if this wait ran out (it then raises the abort flag and records
// ATTN_ERR_DEVICE_TIMEOUT).
__device__ __forceinline__ bool wait(const Ctx& c, int bar, uint32_t parity,
                                     long long limit = kWaitLimitCycles) {
  const uint32_t a = bar_addr(c, bar);
  if (mbar_try_wait(a, parity)) return true;
  const long long t0 = clock64();
  uint32_t n = 0;
  while (!mbar_try_wait(a, parity)) {
    if ((++n & 63u) == 0) {
      if (*c.abort) return false;
      if (clock64() - t0 > limit) {
        *c.abort = 1;
        record_status(ATTN_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ void wait_drain(const Ctx& c, int bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar_addr(c, bar), parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return;
  }
}

// wait() taken by a whole warp with one outcome for all lanes.
__device__ __forceinline__ bool wait_warp(const Ctx& c, int bar, uint32_t parity) {
  return __all_sync(0xffffffffu, wait(c, bar, parity));
}

// Tile t of a unit: query blocks from the last one down to m_start, the G
// query heads of the group inner. Units that start together then visit the
// same query block of the same heads at the same time, so the Q and dO tiles
// they share and the dQ accumulator rows they all add into are touched
// within a short window and stay in L2.
__device__ __forceinline__ void tile_coord(const Work& w, int t, int& h, int& m_block) {
  const int mi = t / w.G;
  h = w.g * w.G + (t - mi * w.G);
  m_block = w.m_start + w.per_head - 1 - mi;
}

// ------------------------------------------------------------------ producer
// Streams, per tile, Q (+LSE, D) and dO into two-stage rings, and per unit K
// and V. A unit's V is requested as soon as the previous unit's last dP GEMM
// has completed and its K as soon as the last dQ GEMM has, so the loads
// overlap the previous unit's final GEMMs and its dK/dV epilogue.
template <int D, bool CAUSAL>
__device__ void producer_role(const Ctx& c, const Params& p, uint8_t* smem, uint32_t sbase,
                              const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                              const CUtensorMap* tm_v, const CUtensorMap* tm_do) {
  using L = Layout<D>;
  constexpr int kBoxes = D / 64;
  constexpr uint32_t kTileBytes = L::kTileBytes;
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    prefetch_tmap(tm_q);
    prefetch_tmap(tm_k);
    prefetch_tmap(tm_v);
    prefetch_tmap(tm_do);
  }
  const uint64_t once = policy_evict_first();
  // Q/dO tiles are re-read by every key block of the head: keep them in L2.
  const uint64_t reuse = policy_evict_last();
  int issued_q = 0, issued_do = 0, issued_k = 0, issued_v = 0;
  bool ok = true;
  int tg = 0;  // tiles of all earlier units
  for (int r = 0; ok; ++r) {
    const int u = unit_of(r, p.n_units);
    if (u < 0) break;
    Work w;
    unit_work(p, u, w);
    for (int tl = 0; tl < w.T; ++tl) {
      const int t = tg + tl;
      const int st = t & 1;
      const uint32_t ph = (t >> 1) & 1;
      int h, m_block;
      tile_coord(w, tl, h, m_block);
      const int bh = w.b * p.H + h;
      const int m0 = m_block * kBr;
      if (t >= 2 && !(ok = wait(c, BAR_Q_EMPTY + st, ph ^ 1))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_addr(c, BAR_Q_FULL + st), kTileBytes);
        const uint32_t dst = sbase + (st ? L::kQ1 : L::kQ0);
        for (int cb = 0; cb < kBoxes; ++cb)
          tma_load_3d_hint(dst + cb * 16384, tm_q, bar_addr(c, BAR_Q_FULL + st), 64 * cb, m0, bh,
                           reuse);
      }
      {
        float* s_lse = reinterpret_cast<float*>(smem + L::kLSE) + st * kBr;
        float* s_d = reinterpret_cast<float*>(smem + L::kDsum) + st * kBr;
        const long long row0 = static_cast<long long>(bh) * p.N + m0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = lane + 32 * e;
          float lv = 0.f, dv = 0.f;
          if (m0 + i < p.N) {
            lv = __ldg(p.lse + row0 + i);
            dv = __ldg(p.dpsum + row0 + i);
          }
          s_lse[i] = -lv * kLog2e;
          s_d[i] = dv;
        }
        mbar_arrive(bar_addr(c, BAR_Q_FULL + st));
      }
      issued_q = t + 1;
      const int kvh = w.b * p.H_kv + w.g;
      if (tl == 0) {
        // V of this unit once the previous unit's last dP GEMM has read V.
        // (Q_EMPTY of tile t-2, waited above, implies dP of t-2 is complete,
        // so the parity below cannot match an older phase.)
        if (t > 0 && !(ok = wait(c, BAR_DP_FULL, (t - 1) & 1))) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_addr(c, BAR_V_FULL), kTileBytes);
          for (int cb = 0; cb < kBoxes; ++cb)
            tma_load_3d_hint(sbase + L::kV + cb * 16384, tm_v, bar_addr(c, BAR_V_FULL), 64 * cb,
                             w.n_block * kBc, kvh, once);
        }
        issued_v = r + 1;
      }
      const int ost = t % L::kDOStages;
      const uint32_t oph = (t / L::kDOStages) & 1;
      if (t >= L::kDOStages && !(ok = wait(c, BAR_DO_EMPTY + ost, oph ^ 1))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_addr(c, BAR_DO_FULL + ost), kTileBytes);
        const uint32_t dst = sbase + (ost ? L::kDO1 : L::kDO0);
        for (int cb = 0; cb < kBoxes; ++cb)
          tma_load_3d_hint(dst + cb * 16384, tm_do, bar_addr(c, BAR_DO_FULL + ost), 64 * cb, m0,
                           bh, reuse);
      }
      issued_do = t + 1;
      if (tl == 0) {
        // K of this unit once the previous unit's last dQ GEMM has read K
        if (t > 0 && !(ok = wait(c, BAR_DQ_FULL, (t - 1) & 1))) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_addr(c, BAR_K_FULL), kTileBytes);
          for (int cb = 0; cb < kBoxes; ++cb)
            tma_load_3d_hint(sbase + L::kK + cb * 16384, tm_k, bar_addr(c, BAR_K_FULL), 64 * cb,
                             w.n_block * kBc, kvh, once);
        }
        issued_k = r + 1;
      }
      __syncwarp();
    }
    tg += w.T;
  }
  // When aborting, the copies issued last must land before the CTA exits.
  if (*c.abort) {
    if (issued_k > 0) wait_drain(c, BAR_K_FULL, (issued_k - 1) & 1);
    if (issued_v > 0) wait_drain(c, BAR_V_FULL, (issued_v - 1) & 1);
    for (int t = issued_q - 2 < 0 ? 0 : issued_q - 2; t < issued_q; ++t)
      wait_drain(c, BAR_Q_FULL + (t & 1), (t >> 1) & 1);
    for (int t = issued_do - L::kDOStages < 0 ? 0 : issued_do - L::kDOStages; t < issued_do; ++t)
      wait_drain(c, BAR_DO_FULL + t % L::kDOStages, (t / L::kDOStages) & 1);
  }
}

// ------------------------------------------------------------------ MMA issuer
template <int D>
struct Mma {
  static constexpr int kKSteps = D / 16;      // S, dP: reduction over d
  static constexpr int kQSteps = kBr / 16;    // dV, dK: reduction over queries
  static constexpr int kKeySteps = kBc / 16;  // dQ: reduction over keys
  static constexpr uint32_t kIdS = make_idesc_bf16(kBc, kBr, false, false);
  static constexpr uint32_t kIdKV = make_idesc_bf16(kBc, D, false, true);
  // d = 128: dQ^T = K^T dS^T (M = d lanes, N = queries), drained coalesced
  // d =  64: dQ   = dS K     (M = query lanes, N = d)
  static constexpr uint32_t kIdQ =
      D == 128 ? make_idesc_bf16(D, kBr, true, true) : make_idesc_bf16(kBr, D, true, true);
  // byte offset of K-step k in a K-major 128-byte-swizzled tile (64 elements
  // per 16 KB column block) and in an MN-major one (16 rows = 2 KB per step)
  static __device__ __forceinline__ constexpr uint32_t kmaj(int k) {
    return ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
  }
  static __device__ __forceinline__ constexpr uint32_t mnmaj(int k) { return (2048 * k) >> 4; }

  // S^T = K Q^T or dP^T = V dO^T (both operands K-major); a, b = low words
  static __device__ __forceinline__ void nt(uint32_t d_tmem, uint32_t a, uint32_t b) {
#pragma unroll
    for (int k = 0; k < kKSteps; ++k)
      mma_ss(d_tmem, sdesc_from_lo(a + kmaj(k)), sdesc_from_lo(b + kmaj(k)), kIdS, k > 0);
  }
  // dV += P^T dO: A (bf16 pairs) from tensor memory, B MN-major
  static __device__ __forceinline__ void tn(uint32_t d_tmem, uint32_t a_tmem, uint32_t b,
                                            bool accumulate) {
#pragma unroll
    for (int k = 0; k < kQSteps; ++k) {
      const uint32_t acol = 8 * k + (k >= 4 ? 32 : 0);
      mma_ts(d_tmem, a_tmem + acol, sdesc_from_lo(b + mnmaj(k)), kIdKV,
             (accumulate || k > 0) ? 1u : 0u);
    }
  }
  // dK += dS^T Q: A = dS^T from the shared tile ([key][query], which is the
  // K-major layout of an M = keys, K = queries operand), B = Q MN-major
  static __device__ __forceinline__ void dk(uint32_t d_tmem, uint32_t ds_k, uint32_t q_mn,
                                            bool accumulate) {
#pragma unroll
    for (int k = 0; k < kQSteps; ++k)
      mma_ss(d_tmem, sdesc_from_lo(ds_k + kmaj(k)), sdesc_from_lo(q_mn + mnmaj(k)), kIdKV,
             (accumulate || k > 0) ? 1u : 0u);
  }
  // dQ tile from the shared dS^T tile and K (both MN-major low words)
  static __device__ __forceinline__ void dq(uint32_t d_tmem, uint32_t k_mn, uint32_t ds_mn) {
#pragma unroll
    for (int k = 0; k < kKeySteps; ++k) {
      if (D == 128)
        mma_ss(d_tmem, sdesc_from_lo(k_mn + mnmaj(k)), sdesc_from_lo(ds_mn + mnmaj(k)), kIdQ,
               k > 0);
      else
        mma_ss(d_tmem, sdesc_from_lo(ds_mn + mnmaj(k)), sdesc_from_lo(k_mn + mnmaj(k)), kIdQ,
               k > 0);
    }
  }
};

// Tensor-memory reuse relies on tcgen05 MMAs of one thread running in issue
// order: a GEMM that overwrites a region is always issued after the GEMM that
// reads what the region held (P^T before S, dS^T before the dQ tile).
// Descriptor low words are formed once; the loop only adds constants, which
// keeps the single issuing thread ahead of the tensor cores.
//
// Tiles are numbered t over all units of the CTA, so every per-tile barrier
// keeps one phase per tile across unit boundaries. A unit starts with dP of
// its first tile (V and dO usually land before K); its first dV and dK
// overwrite the accumulators only after ACC_FREE, i.e. once the drain warps
// have read the previous unit's dK, dV out of tensor memory.
template <int D, bool CAUSAL>
__device__ void mma_role(const Ctx& c, const Params& p, uint32_t sbase, uint32_t tmem) {
  using L = Layout<D>;
  using M = Mma<D>;
  const uint32_t tS = tmem + 0, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;
  const uint32_t kK = sdesc_lo(sbase + L::kK, 16), kV = sdesc_lo(sbase + L::kV, 16);
  const uint32_t kQ0 = sdesc_lo(sbase + L::kQ0, 16), kQ1 = sdesc_lo(sbase + L::kQ1, 16);
  const uint32_t kO0 = sdesc_lo(sbase + L::kDO0, 16), kO1 = sdesc_lo(sbase + L::kDO1, 16);
  const uint32_t mK = sdesc_lo(sbase + L::kK, 16384), mDS = sdesc_lo(sbase + L::kDS, 16384);
  const uint32_t kDS = sdesc_lo(sbase + L::kDS, 16);
  const uint32_t mQ0 = sdesc_lo(sbase + L::kQ0, 16384), mQ1 = sdesc_lo(sbase + L::kQ1, 16384);
  const uint32_t mO0 = sdesc_lo(sbase + L::kDO0, 16384), mO1 = sdesc_lo(sbase + L::kDO1, 16384);
  auto ph = [](int t) { return static_cast<uint32_t>((t >> 1) & 1); };
  auto oph = [](int t) { return static_cast<uint32_t>((t / L::kDOStages) & 1); };
  // The whole warp runs the loop, so descriptor arithmetic stays warp-uniform;
  // one elected lane issues the tensor-core instructions.
  const bool leader = elect_one_sync() != 0;

  bool ok = true;
  int tg = 0;
  for (int r = 0; ok; ++r) {
    const int u = unit_of(r, p.n_units);
    if (u < 0) break;
    Work w;
    unit_work(p, u, w);
    // unit prologue: dP of the first tile, then S
    {
      const int ost = tg % L::kDOStages;
      if (!(ok = wait_warp(c, BAR_V_FULL, r & 1))) break;
      if (!(ok = wait_warp(c, BAR_DO_FULL + ost, oph(tg)))) break;
      if (tg > 0 && !(ok = wait_warp(c, BAR_DQ_EMPTY, (tg - 1) & 1))) break;
      tc_fence_after();
      if (leader) M::nt(tdP, kV, ost ? kO1 : kO0);
      if (leader) mma_commit(bar_addr(c, BAR_DP_FULL));
      if (!(ok = wait_warp(c, BAR_K_FULL, r & 1))) break;
      if (!(ok = wait_warp(c, BAR_Q_FULL + (tg & 1), ph(tg)))) break;
      tc_fence_after();
      if (leader) M::nt(tS, kK, (tg & 1) ? kQ1 : kQ0);
      if (leader) mma_commit(bar_addr(c, BAR_S_FULL));
    }
    for (int tl = 0; tl < w.T; ++tl) {
      const int t = tg + tl;
      const bool more = tl + 1 < w.T;
      const int st = t & 1;
      const int ost = t % L::kDOStages, ostn = (t + 1) % L::kDOStages;
      const uint32_t kQn = st ? kQ0 : kQ1, kOn = ostn ? kO1 : kO0;
      const uint32_t mQ = st ? mQ1 : mQ0, mO = ost ? mO1 : mO0;
      // dV += P_t^T dO_t (A = P_t^T in the S region)
      if (!(ok = wait_warp(c, BAR_P_FULL, t & 1))) break;
      // the first dV and dK of a unit overwrite the accumulators: the
      // previous unit's epilogue must have read them out
      if (tl == 0 && r > 0 && !(ok = wait_warp(c, BAR_ACC_FREE, (r - 1) & 1))) break;
      tc_fence_after();
      if (leader) M::tn(tdV, tS, mO, tl > 0);
      if (leader) mma_commit(bar_addr(c, BAR_DO_EMPTY + ost));  // dP_t and dV_t were dO_t's readers
      // S_{t+1} = K Q_{t+1}^T into the S region (P_t^T there was read by dV_t)
      if (more) {
        if (!(ok = wait_warp(c, BAR_Q_FULL + (st ^ 1), ph(t + 1)))) break;
        tc_fence_after();
        if (leader) M::nt(tS, kK, kQn);
        if (leader) mma_commit(bar_addr(c, BAR_S_FULL));
      }
      // dQ tile of t into the dP region (the softmax has read dP_t), then
      // dK += dS_t^T Q_t, both from the shared dS tile
      if (!(ok = wait_warp(c, BAR_DS_FULL, t & 1))) break;
      tc_fence_after();
      if (leader) M::dq(tdP, mK, mDS);
      if (leader) mma_commit(bar_addr(c, BAR_DQ_FULL));
      if (leader) M::dk(tdK, kDS, mQ, tl > 0);
      if (leader) mma_commit(bar_addr(c, BAR_Q_EMPTY + st));
      if (leader) mma_commit(bar_addr(c, BAR_DS_FREE));
      // dP_{t+1} = V dO_{t+1}^T once the dQ tile has been drained
      if (more) {
        if (!(ok = wait_warp(c, BAR_DO_FULL + ostn, oph(t + 1)))) break;
        if (!(ok = wait_warp(c, BAR_DQ_EMPTY, t & 1))) break;
        tc_fence_after();
        if (leader) M::nt(tdP, kV, kOn);
        if (leader) mma_commit(bar_addr(c, BAR_DP_FULL));
      }
    }
    if (!ok) break;
    // completion of the unit's GEMMs: the epilogue may read dK, dV
    if (leader) mma_commit(bar_addr(c, BAR_UNIT_DONE));
    tg += w.T;
  }
  if (__any_sync(0xffffffffu, *c.abort != 0)) {
    // completion of everything issued before tensor memory is released
    if (leader) mma_commit(bar_addr(c, BAR_DRAIN));
    wait_drain(c, BAR_DRAIN, 0);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ softmax
// One tile, one half of its query columns. Thread = key row r (tensor-memory
// lane r); columns [64*half, 64*half + 64).
// With dropout (DROP), P^T for dV is P o Z / (1 - p) and dP passes through the
// same mask (dP o Z / (1 - p)) before dS = P o (dP - D); the keep bits of the
// thread's 64 columns are drawn in the P phase (one Philox call per four
// queries of its key) and kept in km[] for the dS phase.
template <int D, bool SOFTCAP, bool CAUSAL, bool MASKED, bool DROP>
__device__ __forceinline__ bool softmax_tile(const Ctx& c, const Params& p, uint8_t* smem,
                                             uint32_t sbase, uint32_t tmem, int t, int half,
                                             int r, int key, int m0, int dsbuf_parity,
                                             uint32_t bh) {
  using L = Layout<D>;
  const int st = t & 1;
  const int lane = threadIdx.x & 31;
  const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
  const float* s_lse = reinterpret_cast<const float*>(smem + L::kLSE) + st * kBr;
  const float* s_d = reinterpret_cast<const float*>(smem + L::kDsum) + st * kBr;
  const float c_log2 = p.scale * kLog2e;                                  // tau*log2e
  const float cap_in = SOFTCAP ? 2.f * kLog2e * p.scale / p.softcap : 0.f;  // 2 log2e tau/c
  const float cap_out = SOFTCAP ? p.softcap * kLog2e : 0.f;                 // c log2e
  // pairs of columns go through the f32x2 arithmetic (same roundings as the
  // scalar forms, half the instructions)
  const uint64_t c2 = f2_make(SOFTCAP ? cap_in : c_log2, SOFTCAP ? cap_in : c_log2);
  const uint64_t out2 = f2_make(cap_out, cap_out);
  const uint64_t one2 = f2_make(1.f, 1.f), mone2 = f2_make(-1.f, -1.f),
                 mtwo2 = f2_make(-2.f, -2.f);
  // P, or with a softcap -P (1 - tanh^2) (the sign is undone in the dS
  // phase), for this thread's 64 columns as 32 pairs
  uint64_t pk[32];
  uint32_t km[2] = {0xFFFFFFFFu, 0xFFFFFFFFu};  // dropout keep bits of the 64 columns

  // ---- P = exp(S - LSE) -> bf16 P^T in tensor memory
  if (!wait(c, BAR_S_FULL, t & 1)) return false;
  tc_fence_after();
  // In kPasses column groups: with a softcap each element takes three MUFU
  // operations in a dependent chain, and loading half the row at a time
  // leaves the registers for more of those chains in flight. P^T of a group
  // (bf16 pairs) lands in columns whose S values were read by this or an
  // earlier group.
  constexpr int kPasses = (SOFTCAP || DROP) ? 2 : 1;
  constexpr int kCols = 64 / kPasses;
#pragma unroll
  for (int pass = 0; pass < kPasses; ++pass) {
    uint32_t raw[kCols];
    const uint32_t src = tmem + lane_base + half * 64 + pass * kCols;
    if constexpr (kPasses == 1)
      tmem_ld32x2(src, src + 32, raw);
    else
      tmem_ld32(src, raw);
#pragma unroll
    for (int j4 = 0; j4 < kCols / 4; ++j4) {
      // -LSE*log2e of the four query columns
      const float4 l4 =
          *reinterpret_cast<const float4*>(s_lse + half * 64 + pass * kCols + 4 * j4);
      const uint64_t nl2[2] = {f2_make(l4.x, l4.y), f2_make(l4.z, l4.w)};
      uint32_t kb = 0xFu;
      if (DROP) {
        const int cc = pass * kCols + 4 * j4;  // first of the four columns
        const PhiloxOut rr = philox4x32_10(
            static_cast<uint32_t>((m0 + half * 64 + cc) >> 2), static_cast<uint32_t>(key), bh,
            0u, p.drop.seed_lo, p.drop.seed_hi);
        kb = 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e) kb |= (rr.w[e] >= p.drop.threshold ? 1u : 0u) << e;
        km[cc >> 5] = (km[cc >> 5] & ~(0xFu << (cc & 31))) | (kb << (cc & 31));
      }
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int j = 4 * j4 + 2 * e2;  // columns j, j + 1 of this group
        const uint64_t s2 = f2_make(raw[j], raw[j + 1]);
        float pr[2], kp[2];
        if (SOFTCAP) {
          // tanh(u) = 1 - 2 / (exp(2u) + 1) with u = tau s / c
          const uint64_t u2 = f2_mul(s2, c2);
          const uint64_t e1 = f2_add(f2_make(ex2_approx(f2_lo(u2)), ex2_approx(f2_hi(u2))), one2);
          const uint64_t th2 =
              f2_fma(f2_make(rcp_approx(f2_lo(e1)), rcp_approx(f2_hi(e1))), mtwo2, one2);
          const uint64_t y2 = f2_fma(th2, out2, nl2[e2]);
          pr[0] = ex2_approx(f2_lo(y2));
          pr[1] = ex2_approx(f2_hi(y2));
          // -P (1 - tanh^2) = P (tanh^2 - 1)
          const uint64_t k2 = f2_mul(f2_make(pr[0], pr[1]), f2_fma(th2, th2, mone2));
          kp[0] = f2_lo(k2);
          kp[1] = f2_hi(k2);
        } else {
          const uint64_t y2 = f2_fma(s2, c2, nl2[e2]);
          pr[0] = kp[0] = ex2_approx(f2_lo(y2));
          pr[1] = kp[1] = ex2_approx(f2_hi(y2));
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          if (MASKED) {
            const int q = m0 + half * 64 + pass * kCols + j + h2;
            const bool ok =
                key < p.N && q < p.N && key - q <= p.win_right && q - key <= p.win_left;
            pr[h2] = ok ? pr[h2] : 0.f;
            kp[h2] = ok ? kp[h2] : 0.f;
          }
          if (DROP) pr[h2] = (kb >> (2 * e2 + h2)) & 1u ? pr[h2] * p.drop.inv_keep : 0.f;
          raw[j + h2] = __float_as_uint(pr[h2]);
        }
        pk[(pass * kCols + j) >> 1] = f2_make(kp[0], kp[1]);
      }
    }
#pragma unroll
    for (int ch = 0; ch < kCols / 16; ++ch) {
      uint32_t packed[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        packed[u] = pack_bf16x2(__uint_as_float(raw[16 * ch + 2 * u]),
                                __uint_as_float(raw[16 * ch + 2 * u + 1]));
      tmem_st8(tmem + lane_base + half * 64 + pass * (kCols / 2) + ch * 8, packed);
    }
  }
  tmem_wait_st();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar_addr(c, BAR_P_FULL));

  // ---- dS = P o (dP - D) -> bf16 dS^T in shared memory
  if (!wait(c, BAR_DP_FULL, t & 1)) return false;
  // the previous tile's dQ and dK GEMMs must be done reading the shared dS tile
  if (t > 0 && !wait(c, BAR_DS_FREE, (t - 1) & 1)) return false;
  // first tile of a unit: the previous unit's dK/dV stores must have read
  // the buffer first
  if (dsbuf_parity >= 0 && !wait(c, BAR_DSBUF_FREE, static_cast<uint32_t>(dsbuf_parity)))
    return false;
  tc_fence_after();
  const uint32_t ds_row = sbase + L::kDS + half * 16384 + r * 128;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int col0 = half * 64 + hh * 32;
    uint32_t raw[32];
    tmem_ld32(tmem + lane_base + 128 + col0, raw);
#pragma unroll
    for (int j4 = 0; j4 < 8; ++j4) {
      const float4 d4 = *reinterpret_cast<const float4*>(s_d + col0 + 4 * j4);
      const uint64_t dd2[2] = {f2_make(d4.x, d4.y), f2_make(d4.z, d4.w)};
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int j = 4 * j4 + 2 * e2;
        uint32_t dp0 = raw[j], dp1 = raw[j + 1];
        if (DROP) {
          dp0 = (km[hh] >> j) & 1u ? __float_as_uint(__uint_as_float(dp0) * p.drop.inv_keep) : 0u;
          dp1 = (km[hh] >> (j + 1)) & 1u ? __float_as_uint(__uint_as_float(dp1) * p.drop.inv_keep)
                                         : 0u;
        }
        const uint64_t dp2 = f2_make(dp0, dp1);
        // dS = P (dP - D); with a softcap (-P (1 - tanh^2)) (D - dP)
        const uint64_t r2 =
            f2_mul(pk[(hh * 32 + j) >> 1], SOFTCAP ? f2_sub(dd2[e2], dp2) : f2_sub(dp2, dd2[e2]));
        raw[j] = static_cast<uint32_t>(r2);
        raw[j + 1] = static_cast<uint32_t>(r2 >> 32);
      }
    }
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      uint32_t packed[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        packed[u] = pack_bf16x2(__uint_as_float(raw[16 * ch + 2 * u]),
                                __uint_as_float(raw[16 * ch + 2 * u + 1]));
      const int c16 = hh * 2 + ch;  // 16-query chunk within this half
      // dS^T row r, queries [16 c16, 16 c16 + 16) of this half: 16-byte chunks
      // 2 c16, 2 c16 + 1 of the 128-byte row, placed by the 128-byte swizzle
      st_shared_v4(ds_row + (((2 * c16) ^ (r & 7)) << 4), packed[0], packed[1], packed[2],
                   packed[3]);
      st_shared_v4(ds_row + (((2 * c16 + 1) ^ (r & 7)) << 4), packed[4], packed[5], packed[6],
                   packed[7]);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar_addr(c, BAR_DS_FULL));
  return true;
}

template <int D, bool CAUSAL, bool SOFTCAP, bool DROP>
__device__ void softmax_role(const Ctx& c, const Params& p, uint8_t* smem, uint32_t sbase,
                             uint32_t tmem) {
  const int warp = threadIdx.x >> 5;
  const int half = (warp - 4) >> 2;
  const int r = ((warp & 3) << 5) + (threadIdx.x & 31);
  bool ok = true;
  int tg = 0;
  for (int ur = 0; ok; ++ur) {
    const int u = unit_of(ur, p.n_units);
    if (u < 0) break;
    Work w;
    unit_work(p, u, w);
    const int n0 = w.n_block * kBc;
    const int key = n0 + r;
    for (int tl = 0; tl < w.T && ok; ++tl) {
      const int t = tg + tl;
      int h, m_block;
      tile_coord(w, tl, h, m_block);
      const int m0 = m_block * kBr;
      if (!(ok = wait(c, BAR_Q_FULL + (t & 1), (t >> 1) & 1))) break;
      const bool masked = tile_masked(p, m0, n0);
      const int dsbuf = (tl == 0 && ur > 0) ? ((ur - 1) & 1) : -1;
      const uint32_t bh = static_cast<uint32_t>(w.b * p.H + h);
      if (masked)
        ok = softmax_tile<D, SOFTCAP, CAUSAL, true, DROP>(c, p, smem, sbase, tmem, t, half, r,
                                                          key, m0, dsbuf, bh);
      else
        ok = softmax_tile<D, SOFTCAP, CAUSAL, false, DROP>(c, p, smem, sbase, tmem, t, half, r,
                                                           key, m0, dsbuf, bh);
    }
    tg += w.T;
  }
}

// ------------------------------------------------------------------ dQ drain
// Two warpgroups, each owning half of the dQ tile's columns. A thread loads
// its share from tensor memory, the warp frees the region (DQ_EMPTY), and
// only then is the share added into dq_accum, so the reduction overlaps the
// next tile's GEMMs. After a unit's last tile the same warps write its dK and
// dV (the epilogue), so the softmax warps go on with the next unit at once.

constexpr int kBarDqAll = 3;  // named barrier of both drain warpgroups (ids 1, 2: one each)

// 16-column pieces of this thread's tensor-memory row -> bf16 -> 16-byte
// chunks chunk0, chunk0 + 1, ... of a 128-byte shared-memory row, placed by
// the 128-byte swizzle (chunk c of row r at c ^ (r & 7)).
template <int COLS>
__device__ __forceinline__ void stage_row_bf16(uint32_t taddr, float mul, uint32_t row_addr,
                                               int chunk0, int r) {
#pragma unroll
  for (int ch = 0; ch < COLS / 16; ++ch) {
    uint32_t raw[16];
    tmem_ld16(taddr + ch * 16, raw);
    uint32_t packed[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      packed[u] = pack_bf16x2(__uint_as_float(raw[2 * u]) * mul,
                              __uint_as_float(raw[2 * u + 1]) * mul);
    const int c0 = chunk0 + 2 * ch;
    st_shared_v4(row_addr + ((c0 ^ (r & 7)) << 4), packed[0], packed[1], packed[2], packed[3]);
    st_shared_v4(row_addr + (((c0 + 1) ^ (r & 7)) << 4), packed[4], packed[5], packed[6],
                 packed[7]);
  }
}

// dK (x tau) and dV of a finished unit: fp32 tensor memory -> bf16 rows in
// shared memory -> TMA tensor stores, which write whole lines. Thread = key
// row r (tensor-memory lane). Each 64-column box is 128 rows x 128 bytes with
// the swizzle of the tensor maps.
//   d = 128: warpgroup `part` handles box `part` (columns 64*part ..) of each
//            matrix: dV into the dS buffer (free once the unit's GEMMs are
//            done), dK into its own dQ staging buffer (once its last
//            reduction has read it).
//   d =  64: dV and dK fill the two halves of the dS buffer; warpgroup
//            `part` writes 32 columns of each row.
// ACC_FREE is arrived on as soon as tensor memory has been read; DSBUF_FREE
// once the stores have read the dS buffer. Returns false when aborting.
template <int D>
__device__ __forceinline__ bool dq_epilogue(const Ctx& c, const Params& p, int kvh, int row0,
                                            uint32_t sbase, uint32_t tmem, uint32_t stage,
                                            int part, int r, int ur, bool leader,
                                            const CUtensorMap* tm_dk, const CUtensorMap* tm_dv) {
  using L = Layout<D>;
  const int lane = threadIdx.x & 31;
  const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
  // the threads that meet at the named barriers below decide together
  bool ok = wait(c, BAR_UNIT_DONE, ur & 1);
  ok = D == 128 ? named_bar_and(1 + part, 128, ok) : named_bar_and(kBarDqAll, 256, ok);
  if (!ok) return false;
  tc_fence_after();
  if (D == 128) {
    stage_row_bf16<64>(tmem + lane_base + 256 + part * 64, 1.f,
                       sbase + L::kDS + part * 16384 + r * 128, 0, r);
    if (leader) bulk_wait_read_all();  // the last dQ reduction has read the staging buffer
    named_bar_sync(1 + part, 128);
    stage_row_bf16<64>(tmem + lane_base + 384 + part * 64, p.scale, stage + r * 128, 0, r);
  } else {
    stage_row_bf16<32>(tmem + lane_base + 256 + part * 32, 1.f, sbase + L::kDS + r * 128,
                       4 * part, r);
    stage_row_bf16<32>(tmem + lane_base + 384 + part * 32, p.scale,
                       sbase + L::kDS + 16384 + r * 128, 4 * part, r);
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar_addr(c, BAR_ACC_FREE));
  fence_proxy_async_smem();
  if (D == 128) {
    named_bar_sync(1 + part, 128);
    if (leader) {
      tma_store_3d(tm_dv, sbase + L::kDS + part * 16384, 64 * part, row0, kvh);
      tma_store_3d(tm_dk, stage, 64 * part, row0, kvh);
      bulk_commit_group();
      bulk_wait_read_all();
      mbar_arrive(bar_addr(c, BAR_DSBUF_FREE));
    }
  } else {
    named_bar_sync(kBarDqAll, 256);
    if (leader && part == 0) {
      tma_store_3d(tm_dv, sbase + L::kDS, 0, row0, kvh);
      tma_store_3d(tm_dk, sbase + L::kDS + 16384, 0, row0, kvh);
      bulk_commit_group();
      bulk_wait_read_all();
      mbar_arrive(bar_addr(c, BAR_DSBUF_FREE));
    }
  }
  return true;
}

template <int D, bool CAUSAL, bool DET>
__device__ void dq_role(const Ctx& c, const Params& p, uint8_t* smem, uint32_t sbase,
                        uint32_t tmem, const CUtensorMap* tm_dq, const CUtensorMap* tm_dk,
                        const CUtensorMap* tm_dv) {
  using L = Layout<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int part = (warp - 12) >> 2;  // which half of the tile
  const int r = ((warp & 3) << 5) + lane;
  const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
  // d = 128: this warpgroup's staging buffer and the thread that issues its
  // TMA reductions and stores (the bulk async-group is per thread)
  const uint32_t stage = sbase + L::kDQS + part * 16384;
  const bool leader = (warp & 3) == 0 && lane == 0;
  (void)smem;
  bool ok = true;
  int tg = 0, T = 0, head0 = 0, kvh = 0, row0 = 0, hh = 0, m_block = 0;
  const int G = p.H / p.H_kv;
  for (int ur = 0, tl = 0; ok; ++tl) {
    if (tl == T) {  // unit boundary: epilogue of the finished unit, then the next unit
      if (ur > 0 && !(ok = dq_epilogue<D>(c, p, kvh, row0, sbase, tmem, stage, part, r, ur - 1,
                                          leader, tm_dk, tm_dv)))
        break;
      tg += T;
      tl = 0;
      const int u = unit_of(ur++, p.n_units);
      if (u < 0) break;
      Work w;
      unit_work(p, u, w);
      kvh = w.b * p.H_kv + w.g;
      row0 = w.n_block * kBc;
      T = w.T;
      head0 = w.b * p.H + w.g * G;
      hh = 0;
      m_block = w.m_start + w.per_head - 1;
    }
    {
      const int t = tg + tl;
      const int m0 = m_block * kBr;
      const long long bh = head0 + hh;
      if (++hh == G) {
        hh = 0;
        --m_block;
      }
      // the threads that meet at named barriers (each warpgroup for d = 128,
      // both in the d = 64 epilogue) take the same decision
      ok = wait(c, BAR_DQ_FULL, t & 1);
      ok = D == 128 ? named_bar_and(1 + part, 128, ok) : named_bar_and(kBarDqAll, 256, ok);
      if (!ok) break;
      tc_fence_after();
      if (D == 128) {
        // lane r holds dQ[m0 + i][r] in column 128 + i. The tile leaves tensor
        // memory at once; each 32-query chunk is then written to the staging
        // buffer as rows of 128 floats and added into dq_accum by one TMA
        // reduction, which keeps the atomics off the load/store path the
        // softmax warps use.
        uint32_t v[64];
        tmem_ld32x2(tmem + lane_base + 128 + part * 64, tmem + lane_base + 128 + part * 64 + 32,
                    v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr(c, BAR_DQ_EMPTY));
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          if (leader) bulk_wait_read_all();  // previous reduction has read the buffer
          named_bar_sync(1 + part, 128);
#pragma unroll
          for (int q = 0; q < 32; ++q)
            st_shared_f32(stage + q * 512 + r * 4, __uint_as_float(v[ch * 32 + q]));
          fence_proxy_async_smem();
          named_bar_sync(1 + part, 128);
          const int row = m0 + part * 64 + ch * 32;
          if (leader) {
            if (DET) {
              const int m = m0 >> 7, n = row0 >> 7;
              const int pi = CAUSAL ? (m * (m + 1) >> 1) + n : m * p.n_blocks + n;
              tma_store_3d(tm_dq, stage, 0, part * 64 + ch * 32,
                           static_cast<int>(bh) * p.pairs + pi);
              bulk_commit_group();
            } else if (row < p.N) {
              tma_reduce_add_3d(tm_dq, stage, 0, row, static_cast<int>(bh));
              bulk_commit_group();
            }
          }
        }
      } else {
        // lane r holds query row m0 + r; columns 128 + [0, 64) are dQ[m0 + r][:]
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + 128 + part * 32, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr(c, BAR_DQ_EMPTY));
        // the warp's 32 rows x 32 columns go to one of its two 4 KB buffers
        // (128-byte rows, 128-byte swizzle) and out with one TMA reduce-add
        const uint32_t buf = sbase + L::kDQS + ((warp - 12) * 2 + (t & 1)) * 4096;
        if (lane == 0) bulk_wait_read_1();  // the reduction of two tiles ago has read it
        __syncwarp();
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          st_shared_v4(buf + lane * 128 + ((c4 ^ (lane & 7)) << 4), v[4 * c4], v[4 * c4 + 1],
                       v[4 * c4 + 2], v[4 * c4 + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int row = m0 + 32 * (warp & 3);
          if (DET) {
            const int m = m0 >> 7, n = row0 >> 7;
            const int pi = CAUSAL ? (m * (m + 1) >> 1) + n : m * p.n_blocks + n;
            tma_store_3d(tm_dq, buf, 32 * part, 32 * (warp & 3),
                         static_cast<int>(bh) * p.pairs + pi);
          } else if (row < p.N) {
            tma_reduce_add_3d(tm_dq, buf, 32 * part, row, static_cast<int>(bh));
          }
          bulk_commit_group();  // one group per tile, empty or not
        }
      }
    }
  }
  // the reductions and stores must complete before the CTA exits (each
  // lane 0 may have issued some)
  if (lane == 0) bulk_wait_all();
}

// ------------------------------------------------------------------ kernel
template <int D, bool CAUSAL, bool SOFTCAP, bool DET, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq,
                    const __grid_constant__ CUtensorMap tm_dk,
                    const __grid_constant__ CUtensorMap tm_dv, const Params p) {
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
    mbar_init(bar_addr(c, BAR_K_FULL), 1);
    mbar_init(bar_addr(c, BAR_V_FULL), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_addr(c, BAR_Q_FULL + s), 33);  // expect_tx arrive + 32 LSE/D lanes
      mbar_init(bar_addr(c, BAR_Q_EMPTY + s), 1);
      mbar_init(bar_addr(c, BAR_DO_FULL + s), 1);
      mbar_init(bar_addr(c, BAR_DO_EMPTY + s), 1);
    }
    mbar_init(bar_addr(c, BAR_S_FULL), 1);
    mbar_init(bar_addr(c, BAR_P_FULL), 8);
    mbar_init(bar_addr(c, BAR_DP_FULL), 1);
    mbar_init(bar_addr(c, BAR_DS_FULL), 8);
    mbar_init(bar_addr(c, BAR_DQ_FULL), 1);
    mbar_init(bar_addr(c, BAR_DQ_EMPTY), 8);
    mbar_init(bar_addr(c, BAR_UNIT_DONE), 1);
    mbar_init(bar_addr(c, BAR_DS_FREE), 1);
    mbar_init(bar_addr(c, BAR_DRAIN), 1);
    mbar_init(bar_addr(c, BAR_ACC_FREE), 8);                   // the 8 drain warps
    mbar_init(bar_addr(c, BAR_DSBUF_FREE), D == 128 ? 2 : 1);  // the store-issuing threads
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

  if (warp < 4) {
    setmaxnreg_dec<kRegsCtl>();
    if (warp == 0) {
      producer_role<D, CAUSAL>(c, p, smem, sbase, &tm_q, &tm_k, &tm_v, &tm_do);
    } else if (warp == 1) {
      mma_role<D, CAUSAL>(c, p, sbase, tmem);
    }
  } else if (warp < 12) {
    setmaxnreg_inc<kRegsSoftmax>();
    softmax_role<D, CAUSAL, SOFTCAP, DROP>(c, p, smem, sbase, tmem);
  } else {
    setmaxnreg_dec<kRegsDq>();
    dq_role<D, CAUSAL, DET>(c, p, smem, sbase, tmem, &tm_dq, &tm_dk, &tm_dv);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Exercises the bounded wait of the kernels above on the device: warp 0
// waits on an mbarrier that nothing arrives on, gives up after
// `limit_cycles`, raises the abort flag and records ATTN_ERR_DEVICE_TIMEOUT;
// warp 1, waiting on another such barrier with a far longer limit, returns
// on the abort flag. Nothing faults or traps; the context stays usable.
__global__ void __launch_bounds__(64, 1) wait_timeout_probe(long long limit_cycles) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  Ctx c;
  c.bars = smem_u32(bars);
  c.abort = &abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(c.bars, 1);
    mbar_init(c.bars + 8, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x < 32)
    (void)wait(c, 0, 0, limit_cycles);
  else
    (void)wait(c, 1, 0, 64 * limit_cycles);
  __syncthreads();
}

// Tensor maps of one call: loads of Q, K, V, dO; reductions into dq_accum;
// stores of dK, dV.
struct Maps {
  CUtensorMap q, k, v, dO, dq, dk, dv;
};

template <int D, bool CAUSAL, bool SOFTCAP, bool DET, bool DROP>
int launch(const Maps& m, const Params& p, cudaStream_t stream) {
  auto kern = attn_bwd_kernel<D, CAUSAL, SOFTCAP, DET, DROP>;
  static std::atomic<bool> configured[kMaxTrackedDevices];
  if (!set_smem_limit_once(kern, Layout<D>::kBytes, configured)) return ATTN_ERR_LAUNCH;
  // persistent: one CTA per SM (or per unit, if there are fewer units)
  const int sms = sm_count();
  if (sms <= 0) return ATTN_ERR_LAUNCH;
  const int grid = p.n_units < sms ? p.n_units : sms;
  kern<<<grid, kThreads, Layout<D>::kBytes, stream>>>(m.q, m.k, m.v, m.dO, m.dq, m.dk, m.dv, p);
  return launch_status();
}

}  // namespace bwd
}  // namespace attn

using namespace attn;

namespace attn {
namespace bwd {

template <bool DET, bool DROP>
int dispatch(const Maps& m, const Params& p, cudaStream_t s, int d, bool cs, bool cap) {
  if (d == 128) {
    if (cs)
      return cap ? launch<128, true, true, DET, DROP>(m, p, s)
                 : launch<128, true, false, DET, DROP>(m, p, s);
    return cap ? launch<128, false, true, DET, DROP>(m, p, s)
               : launch<128, false, false, DET, DROP>(m, p, s);
  }
  if (cs)
    return cap ? launch<64, true, true, DET, DROP>(m, p, s)
               : launch<64, true, false, DET, DROP>(m, p, s);
  return cap ? launch<64, false, true, DET, DROP>(m, p, s)
             : launch<64, false, false, DET, DROP>(m, p, s);
}

// Shared by attn_bwd (dQ added into dq_target) and attn_bwd_deterministic
// (dQ tiles stored into the partials buffer dq_target).
// `before_launch`, when given, runs once every argument check and tensor-map
// encoding has passed, right before the kernel is enqueued (d = 64 and 128
// only); a non-zero return ends the call with that code and nothing more is
// enqueued.
int run(const void* q, const void* k, const void* v, const void* dO, const float* lse,
        float* dq_target, void* dk, void* dv, int B, int H, int H_kv, int N, int d, float scale,
        int causal, float softcap, const float* dpsum, void* stream, bool det, float p_drop = 0.f,
        unsigned long long seed = 0, int window_left = -1, int window_right = -1,
        int (*before_launch)(void*) = nullptr, void* before_ctx = nullptr) {
  if (!q || !k || !v || !dO || !lse || !dq_target || !dk || !dv || !dpsum) return ATTN_ERR_NULL;
  int rc = check_shape(B, H, H_kv, N, d);
  if (rc != ATTN_OK) return rc;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;  // d = 256: its own kernel
  if (!std::isfinite(scale) || scale == 0.f || std::isnan(softcap)) return ATTN_ERR_SHAPE;
  if (!(p_drop >= 0.f && p_drop < 1.f)) return ATTN_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(lse) ||
      !aligned16(dq_target) || !aligned16(dk) || !aligned16(dv) || !aligned16(dpsum))
    return ATTN_ERR_ALIGN;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (d == 256 && before_launch != nullptr) return ATTN_ERR_UNSUPPORTED;
  if (d == 256) {
    // dQ partials: one tile of 128 query rows per (query block, key block)
    // pair, as for d <= 128
    const long long mb = (N + kBr - 1) / kBr, nb = (N + kBc - 1) / kBc;
    const long long pairs256 = causal ? mb * (mb + 1) / 2 : mb * nb;
    if (det && static_cast<long long>(B) * H * pairs256 > 0x7fffffffLL) return ATTN_ERR_TOO_LARGE;
    return bwd256_run(q, k, v, dO, lse, dq_target, dk, dv, B, H, H_kv, N, scale, causal, softcap,
                      dpsum, window_left, window_right, det, static_cast<int>(pairs256), p_drop,
                      seed, as_stream(stream));
  }

  Params p;
  p.lse = lse;
  p.dpsum = dpsum;
  p.dq_accum = dq_target;
  p.B = B;
  p.H = H;
  p.H_kv = H_kv;
  p.N = N;
  p.n_blocks = (N + kBc - 1) / kBc;
  p.m_blocks = (N + kBr - 1) / kBr;
  const long long units = static_cast<long long>(p.n_blocks) * H_kv * B;
  if (units > 0x7fffffffLL) return ATTN_ERR_TOO_LARGE;
  p.n_units = static_cast<int>(units);
  const long long pairs = causal ? static_cast<long long>(p.m_blocks) * (p.m_blocks + 1) / 2
                                 : static_cast<long long>(p.m_blocks) * p.n_blocks;
  if (det && static_cast<long long>(B) * H * pairs > 0x7fffffffLL) return ATTN_ERR_TOO_LARGE;
  p.pairs = static_cast<int>(pairs);
  p.scale = scale;
  const bool cap = softcap > 0.f;
  p.softcap = cap ? softcap : 0.f;
  // a negative or wider-than-N side of the window is unbounded (N); the
  // causal mask bounds the right side at 0
  p.win_left = (window_left < 0 || window_left > N) ? N : window_left;
  p.win_right = causal ? 0 : ((window_right < 0 || window_right > N) ? N : window_right);
  const bool drop = p_drop > 0.f;
  p.drop.seed_lo = static_cast<uint32_t>(seed);
  p.drop.seed_hi = static_cast<uint32_t>(seed >> 32);
  p.drop.threshold = dropout_threshold(p_drop);
  p.drop.inv_keep = 1.f / (1.f - p_drop);
  p.drop.keep = 1.f - p_drop;
  p.drop.log2_inv_keep =
      static_cast<float>(-std::log2(1.0 - static_cast<double>(p_drop)));

  Maps m;
  const long long hq = static_cast<long long>(B) * H, hk = static_cast<long long>(B) * H_kv;
  const bool dq_ok =
      det ? encode_f32_3d(&m.dq, dq_target, d, kBr, hq * pairs, 32, d == 128 ? d : 32)
          : encode_f32_3d(&m.dq, dq_target, d, N, hq, 32, d == 128 ? d : 32);
  if (!encode_bf16_3d(&m.q, q, d, N, hq, kBr) || !encode_bf16_3d(&m.k, k, d, N, hk, kBc) ||
      !encode_bf16_3d(&m.v, v, d, N, hk, kBc) || !encode_bf16_3d(&m.dO, dO, d, N, hq, kBr) ||
      !dq_ok || !encode_bf16_3d(&m.dk, dk, d, N, hk, kBc) ||
      !encode_bf16_3d(&m.dv, dv, d, N, hk, kBc))
    return ATTN_ERR_LAUNCH;

  if (before_launch != nullptr) {
    rc = before_launch(before_ctx);
    if (rc != ATTN_OK) return rc;
  }
  cudaStream_t s = as_stream(stream);
  const bool cs = causal != 0;
  if (drop) return dispatch<false, true>(m, p, s, d, cs, cap);  // not combined with det
  return det ? dispatch<true, false>(m, p, s, d, cs, cap)
             : dispatch<false, false>(m, p, s, d, cs, cap);
}

}  // namespace bwd
}  // namespace attn

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* o,
                        const void* dO, const float* lse, float* dq_accum, void* dk, void* dv,
                        int B, int H, int H_kv, int N, int d, float scale, int causal,
                        float softcap, const float* dpsum, void* stream) {
  (void)o;  // D = rowsum(dO o O) arrives precomputed in dpsum
  return bwd::run(q, k, v, dO, lse, dq_accum, dk, dv, B, H, H_kv, N, d, scale, causal, softcap,
                  dpsum, stream, false);
}

extern "C" int attn_bwd_dropout(const void* q, const void* k, const void* v, const void* o,
                                const void* dO, const float* lse, float* dq_accum, void* dk,
                                void* dv, int B, int H, int H_kv, int N, int d, float scale,
                                int causal, float softcap, const float* dpsum, float p_drop,
                                unsigned long long seed, void* stream) {
  (void)o;
  return bwd::run(q, k, v, dO, lse, dq_accum, dk, dv, B, H, H_kv, N, d, scale, causal, softcap,
                  dpsum, stream, false, p_drop, seed);
}

extern "C" int attn_bwd_local(const void* q, const void* k, const void* v, const void* o,
                              const void* dO, const float* lse, float* dq_accum, void* dk,
                              void* dv, int B, int H, int H_kv, int N, int d, float scale,
                              int causal, float softcap, const float* dpsum, int window_left,
                              int window_right, void* stream) {
  (void)o;
  return bwd::run(q, k, v, dO, lse, dq_accum, dk, dv, B, H, H_kv, N, d, scale, causal, softcap,
                  dpsum, stream, false, 0.f, 0, window_left, window_right);
}

extern "C" int attn_bwd_deterministic(const void* q, const void* k, const void* v,
                                      const void* o, const void* dO, const float* lse,
                                      float* dq_partials, void* dk, void* dv, int B, int H,
                                      int H_kv, int N, int d, float scale, int causal,
                                      float softcap, const float* dpsum, void* stream) {
  (void)o;
  return bwd::run(q, k, v, dO, lse, dq_partials, dk, dv, B, H, H_kv, N, d, scale, causal,
                  softcap, dpsum, stream, true);
}

namespace attn {

int bwd_run_hooked(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                   float* dq_accum, void* dk, void* dv, int B, int H, int H_kv, int N, int d,
                   float scale, int causal, float softcap, const float* dpsum, void* stream,
                   int (*before_launch)(void*), void* ctx) {
  return bwd::run(q, k, v, dO, lse, dq_accum, dk, dv, B, H, H_kv, N, d, scale, causal, softcap,
                  dpsum, stream, false, 0.f, 0, -1, -1, before_launch, ctx);
}

}  // namespace attn

extern "C" int attn_device_status(int* status, int clear, void* stream) {
  if (!status) return ATTN_ERR_NULL;
  cudaStream_t s = as_stream(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_LAUNCH;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, bwd::g_status, sizeof(int)) != cudaSuccess) return ATTN_ERR_LAUNCH;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(bwd::g_status, &zero, sizeof(int)) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
  }
  int vf = 0, v256 = 0;  // the forward and d = 256 kernels keep their own words
  if (fwd_status(&vf, clear != 0) != ATTN_OK) return ATTN_ERR_LAUNCH;
  if (bwd256_status(&v256, clear != 0) != ATTN_OK) return ATTN_ERR_LAUNCH;
  *status = v != 0 ? v : (vf != 0 ? vf : v256);
  return ATTN_OK;
}

extern "C" int attn_selftest_wait_timeout(int* status, void* stream) {
  if (!status) return ATTN_ERR_NULL;
  cudaStream_t s = as_stream(stream);
  const int zero = 0;
  if (cudaMemcpyToSymbolAsync(bwd::g_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return ATTN_ERR_LAUNCH;
  bwd::wait_timeout_probe<<<1, 64, 0, s>>>(1000000LL);  // about half a millisecond
  const int rc = launch_status();
  if (rc != ATTN_OK) return rc;
  return attn_device_status(status, 1, stream);
}

extern "C" const char* attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "success";
    case ATTN_ERR_NULL: return "a required pointer is NULL";
    case ATTN_ERR_SHAPE: return "invalid shape or scalar argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported head dimension";
    case ATTN_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case ATTN_ERR_LAUNCH: return "CUDA launch or runtime error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel timed out waiting on a barrier";
    case ATTN_ERR_DEVICE: return "a kernel detected an internal fault";
    case ATTN_ERR_TOO_LARGE: return "a size exceeds the supported range";
    default: return "unknown error code";
  }
}
