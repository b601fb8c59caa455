// attn_fwd: attention forward on sm_103a producing O and the natural-log
// LSE the backward needs ("反向传播算法详解" §1.2-§1.3 saved tensors;
// "解析 FlashAttention（3）" §1.1 forward and §3.2 eq. 9-12, the running
// (max, sum) statistics of the online softmax).
//
// Queries sit on the tensor-memory lanes: thread r of a softmax warpgroup
// owns query row r, so row maxima and sums need no reduction across rows.
// Per key block j:
//   S(j)  = Q K_j^T                             (tensor cores, fp32 in TMEM)
//   m     = running row maximum of x = logit * log2e; the shift m_used is
//           moved only when the maximum grows by more than kRescale (in
//           log2 units), and then O and l are multiplied by
//           2^(m_used_old - m_used_new)
//   P(j)  = 2^(x - m_used) as bf16 pairs over the S buffer, l += sum P
//   O    += P(j) V_j                            (P read from TMEM)
// and at the end O = O / l, LSE = (m_used + log2 l) ln 2. The values of P
// stay below 2^kRescale, so neither the bf16 P nor the fp32 O can overflow.
//
// A tile is one block of 128 queries of one query head, and the CTAs are
// persistent: one per SM, each walking its tiles heaviest first in snake
// order. A tile's key blocks alternate between two S buffers ([0,128) and
// [128,256)), so S(j + 1) runs on the tensor cores while the softmax works on
// S(j); O sits at [256, 256 + d), and at d <= 128 the tiles alternate
// between two O buffers. The next tile's Q (two Q stages at d <= 128), K and
// V blocks load while the current tile finishes, so the launch, the first
// loads and the epilogue of a tile do not stand alone. Both softmax
// warpgroups work on the one tile, warpgroup h on keys 64 h .. 64 h + 63 of
// each block and on columns h d/2 .. of O; they exchange the half-row maxima
// through shared memory once per block.
//   warp 0      Q of each tile; K_j in a ring of 2 stages (d <= 128) or 1
//   warp 2      V_j in the same kind of ring
//   warp 1      MMA issuer: per tile S(0), then per block S(j + 1), P(j) V
//   warps 4-11  softmax, then the tile's epilogue (O staged in the tile's Q
//               stage, TMA stores; LSE)
//   warps 12-19 with dropout only: the keep mask, one key block ahead
// Every mbarrier wait is bounded, as in attn_bwd.
#include <cstdint>
#include <cuda_bf16.h>

#include <type_traits>

#include "attn_common.cuh"
#include "philox.cuh"
#include "sm103_ptx.cuh"
#include "softcap_math.cuh"

namespace attn {
namespace fwdtc {

using namespace ptx;

constexpr int kBm = 128;  // queries per tile (tensor-memory lanes)
constexpr int kBn = 128;  // keys per block
constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.f;  // move the shift only when the maximum grows by more
constexpr long long kWaitLimitCycles = 2000000000LL;  // about one second

// With dropout the keep mask is drawn by warps of its own (warps 12-19, two
// per SM sub-partition). Philox4x32-10 is bound by its 32 x 32 -> 64-bit
// multiplies (measured on this GPU: about 1.3 calls per clock per SM, some
// 3,000 cycles for the 4,096 calls of a 128 x 128 block), about as long as
// the softmax of a block; drawn inline it adds to the softmax's critical
// path, drawn for block g + 1 while the softmax works on block g it runs
// beside it. The CTA then has 640 threads; setmaxnreg gives the softmax
// warps 128 registers and the other twelve warps 72.
template <bool DROP>
constexpr int kThreadsFor = DROP ? 640 : kThreads;
constexpr int kMaskWarps = 8;  // two per SM sub-partition
constexpr int kRegsSoftmaxDrop = 128, kRegsOtherDrop = 72;
static_assert(256 * kRegsSoftmaxDrop + 384 * kRegsOtherDrop <= 640 * 96, "register pool");
// Without dropout at d = 256 (384 threads launched at 168 registers), the
// softmax warps' state does not fit in 168: setmaxnreg moves registers to
// them from the loaders and the MMA warp.
constexpr int kRegsSoftmax256 = 200, kRegsCtl256 = 56;
static_assert(256 * kRegsSoftmax256 + 128 * kRegsCtl256 <= 384 * 168, "register pool");
template <int D, bool DROP>
constexpr bool kSplitRegs256 = D == 256 && !DROP;

template <int D>
struct Layout {
  static constexpr int kTileBytes = 128 * D * 2;
  // K and V stages: two where they fit (d <= 128), one at d = 256. Q stages
  // likewise: the next tile's Q loads while the current one finishes, and a
  // tile's Q stage stages its O for the TMA store at the end.
  static constexpr int kStages = D <= 128 ? 2 : 1;
  static constexpr int kQStages = D <= 128 ? 2 : 1;
  // O accumulators in tensor memory (after the two S buffers): two at
  // d <= 128, so a tile's P V GEMMs never wait for the previous tile's
  // epilogue to read O; one at d = 256
  static constexpr int kOBufs = D <= 128 ? 2 : 1;
  static constexpr int kQ0 = 0;
  static constexpr int kQ1 = kQ0 + (kQStages - 1) * kTileBytes;
  static constexpr int kK0 = kQ1 + kTileBytes;
  static constexpr int kK1 = kK0 + (kStages - 1) * kTileBytes;
  static constexpr int kV0 = kK1 + kTileBytes;
  static constexpr int kV1 = kV0 + (kStages - 1) * kTileBytes;
  // the two softmax warpgroups' half-row maxima (two blocks in flight) and
  // row sums: [2][2][128] + [2][128] fp32
  static constexpr int kXchg = kV1 + kTileBytes;
  // dropout keep bits of two key blocks: [block parity][key half][row] x
  // 2 words (bit j of word w: key 64 half + 32 w + j of the block)
  static constexpr int kMask = kXchg + 6 * 128 * 4;
  static constexpr int kBars = kMask + 2 * 2048;
  static constexpr int kNumBars = 26;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kUsed = kAbort + 12;
  // more than half of the SM's shared memory (d = 64 uses about 104 KB), so
  // that a second CTA never waits on the first one's tensor memory
  static constexpr int kBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
};
static_assert(Layout<128>::kBytes <= 232448, "shared memory budget");
static_assert(Layout<256>::kBytes <= 232448, "shared memory budget");
static_assert(2 * 128 + Layout<128>::kOBufs * 128 <= 512, "tensor memory");
static_assert(2 * 128 + Layout<256>::kOBufs * 256 <= 512, "tensor memory");

enum Bar {
  BAR_Q_FULL = 0,       // + Q stage: the tile's Q loaded
  BAR_K_FULL = 2,       // + stage
  BAR_K_EMPTY = 4,      // + stage
  BAR_V_FULL = 6,       // + stage
  BAR_V_EMPTY = 8,      // + stage
  BAR_S_FULL = 10,      // + S buffer (block parity): S of the block written
  BAR_P_FULL = 12,      // + S buffer: P of the block written (and O rescaled if needed)
  BAR_O_DONE = 14,      // P V of a block completed (one phase per key block)
  BAR_DRAIN = 16,       // abort path only: completion of everything issued
  BAR_MASK_FULL = 17,   // + block parity (dropout): keep bits written
  BAR_MASK_EMPTY = 19,  // + block parity: the softmax has read them
  BAR_Q_EMPTY = 21,     // + Q stage: the tile's O store has read the stage
  BAR_O_FREE = 23,      // + O buffer: the tile's epilogue has read O
  BAR_O_LAST = 25,      // the tile's last P V completed (one phase per tile)
};

struct Params {
  float* lse;
  int B, H, H_kv, N;
  int tiles;  // query tiles per head (blocks of 128 queries)
  float scale;
  float softcap;
  // visibility band: key j is visible to query i iff
  // i - win_left <= j <= i + win_right (the causal mask is win_right = 0;
  // an unbounded side holds N)
  int win_left, win_right;
  Dropout drop;  // kernel template flag DROP: keep mask of philox.cuh
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

// The CTAs are persistent: min(#SMs, tiles) of them, CTA c taking tile
// index r * grid + c in even passes r and r * grid + (grid - 1 - c) in odd
// ones (snake order over the tiles, heaviest first for a causal mask), so the
// next tile's Q and first K, V blocks load and its first S GEMM runs while
// the current tile finishes. Every per-block barrier keeps one phase per key
// block across the CTA's tiles (global block index g), the per-tile ones one
// phase per tile.
struct Tile {
  int bh, kvh, m0, j0, nt;
};

__device__ __forceinline__ int cta_tile(int r, int n_tiles) {
  const int grid = static_cast<int>(gridDim.x);
  const int cta = static_cast<int>(blockIdx.x);
  const int idx = r * grid + ((r & 1) ? grid - 1 - cta : cta);
  return idx < n_tiles ? idx : -1;
}

// Tile idx: query block pair (heaviest first) of head bh.
__device__ __forceinline__ Tile tile_of(const Params& p, int idx) {
  Tile t;
  const int heads = p.B * p.H;
  const int blk = p.tiles - 1 - idx / heads;
  t.bh = idx - (idx / heads) * heads;
  const int b = t.bh / p.H, h = t.bh - b * p.H;
  t.kvh = b * p.H_kv + h / (p.H / p.H_kv);
  t.m0 = blk * kBm;
  const int last_block = (p.N + kBn - 1) / kBn - 1;
  t.j0 = max(0, t.m0 - p.win_left) / kBn;
  const int j_end = min(last_block, (t.m0 + kBm - 1 + p.win_right) / kBn);
  t.nt = j_end - t.j0 + 1;  // >= 1: the band holds the diagonal
  return t;
}

// ------------------------------------------------------------------ loaders and MMA issuer
// The loaders. Warp 0 loads Q and the K blocks, warp 2 the
// V blocks, each into its own ring of kStages stages: K(g) once S(g - kStages)
// has read its stage, V(g) once P(g - kStages) V has, Q of tile i once the O
// store of tile i - kQStages has read its stage. Each warp waits on its own
// barriers in the order the tensor cores finish them, so no load waits
// behind another operand's.
template <int D>
__device__ void loader_role(const Ctx& c, const Params& p, uint32_t sbase,
                                const CUtensorMap* tq, const CUtensorMap* tkv, bool is_v) {
  using L = Layout<D>;
  constexpr int kBoxes = D / 64;
  constexpr uint32_t kTileBytes = L::kTileBytes;
  constexpr int kS = L::kStages, kQS = L::kQStages;
  const int lane = threadIdx.x & 31;
  const int n_tiles = p.tiles * p.B * p.H;
  if (lane == 0) {
    prefetch_tmap(tkv);
    if (!is_v) prefetch_tmap(tq);
  }
  const uint64_t keep = policy_evict_last();  // K, V are read by every query block of the head
  const int bar_full = is_v ? BAR_V_FULL : BAR_K_FULL;
  const int bar_empty = is_v ? BAR_V_EMPTY : BAR_K_EMPTY;
  const uint32_t base = sbase + (is_v ? L::kV0 : L::kK0);
  int g = 0, i = 0;  // blocks and tiles issued
  bool ok = true;
  for (int r = 0; ok; ++r, ++i) {
    const int idx = cta_tile(r, n_tiles);
    if (idx < 0) break;
    const Tile tl = tile_of(p, idx);
    if (!is_v) {
      const int qs = i % kQS;
      if (i >= kQS && !(ok = wait_warp(c, BAR_Q_EMPTY + qs, ((i / kQS) - 1) & 1))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_addr(c, BAR_Q_FULL + qs), kTileBytes);
        for (int cb = 0; cb < kBoxes; ++cb)
          tma_load_3d(sbase + L::kQ0 + qs * kTileBytes + cb * 16384, tq,
                      bar_addr(c, BAR_Q_FULL + qs), 64 * cb, tl.m0, tl.bh);
      }
    }
    for (int t = 0; t < tl.nt; ++t, ++g) {
      const int st = g % kS;
      if (g >= kS && !(ok = wait_warp(c, bar_empty + st, ((g / kS) - 1) & 1))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_addr(c, bar_full + st), kTileBytes);
        for (int cb = 0; cb < kBoxes; ++cb)
          tma_load_3d_hint(base + st * kTileBytes + cb * 16384, tkv, bar_addr(c, bar_full + st),
                           64 * cb, (tl.j0 + t) * kBn, tl.kvh, keep);
      }
      __syncwarp();
    }
  }
  // When aborting, the copies in flight must land before the CTA exits: the
  // last kStages blocks and the last kQStages Q tiles issued.
  if (!ok || *c.abort) {
    for (int gg = g - kS < 0 ? 0 : g - kS; gg < g; ++gg)
      wait_drain(c, bar_full + gg % kS, (gg / kS) & 1);
    if (!is_v)
      for (int ii = i - kQS < 0 ? 0 : i - kQS; ii < i; ++ii)
        wait_drain(c, BAR_Q_FULL + ii % kQS, (ii / kQS) & 1);
  }
}

// The MMA issuer, per tile: S(0); then per key block t,
// S(t + 1) into the other S buffer (its P(t - 1) was read by P(t - 1) V,
// issued before), then P(t) V into the tile's O buffer once the softmax has
// written P(t) (the first one once the epilogue of the tile kOBufs before has
// read that buffer).
template <int D>
__device__ void mma_role(const Ctx& c, const Params& p, uint32_t sbase, uint32_t tmem) {
  using L = Layout<D>;
  constexpr int kS = L::kStages, kQS = L::kQStages, kOB = L::kOBufs;
  const bool leader = elect_one_sync() != 0;
  constexpr uint32_t kIdS = make_idesc_bf16(kBm, kBn, false, false);  // S = Q K^T
  constexpr uint32_t kIdO = make_idesc_bf16(kBm, D, false, true);     // O += P V
  const uint32_t k_lo[2] = {sdesc_lo(sbase + L::kK0, 16), sdesc_lo(sbase + L::kK1, 16)};
  const uint32_t v_mn[2] = {sdesc_lo(sbase + L::kV0, 16384), sdesc_lo(sbase + L::kV1, 16384)};
  auto kmaj = [](int k) { return static_cast<uint32_t>(((k >> 2) * 16384 + (k & 3) * 32) >> 4); };
  auto mnmaj = [](int k) { return static_cast<uint32_t>((2048 * k) >> 4); };
  const int n_tiles = p.tiles * p.B * p.H;
  bool ok = true;
  int g = 0;  // global index of the tile's first block
  for (int r = 0, i = 0; ok; ++r, ++i) {
    const int idx = cta_tile(r, n_tiles);
    if (idx < 0) break;
    const int nt = tile_of(p, idx).nt;
    const int qs = i % kQS, ob = i % kOB;
    const uint32_t q_lo = sdesc_lo(sbase + L::kQ0 + qs * L::kTileBytes, 16);
    const uint32_t t_o = tmem + 256 + ob * D;
    auto issue_s = [&](int gb) -> bool {
      const int st = gb % kS;
      if (!wait_warp(c, BAR_K_FULL + st, (gb / kS) & 1)) return false;
      tc_fence_after();
      if (leader) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tmem + (gb & 1) * 128, sdesc_from_lo(q_lo + kmaj(k)),
                 sdesc_from_lo(k_lo[st] + kmaj(k)), kIdS, k > 0);
        mma_commit(bar_addr(c, BAR_S_FULL + (gb & 1)));
        mma_commit(bar_addr(c, BAR_K_EMPTY + st));
      }
      return true;
    };
    ok = wait_warp(c, BAR_Q_FULL + qs, (i / kQS) & 1);
    if (ok) ok = issue_s(g);
    for (int t = 0; ok && t < nt; ++t) {
      const int gb = g + t;
      if (t + 1 < nt && !(ok = issue_s(gb + 1))) break;
      if (!(ok = wait_warp(c, BAR_P_FULL + (gb & 1), (gb >> 1) & 1))) break;
      const int vs = gb % kS;
      if (!(ok = wait_warp(c, BAR_V_FULL + vs, (gb / kS) & 1))) break;
      if (t == 0 && i >= kOB && !(ok = wait_warp(c, BAR_O_FREE + ob, ((i / kOB) - 1) & 1)))
        break;
      tc_fence_after();
      if (leader) {
        // A = P (bf16 pairs in the S buffer of block gb: keys 0-63 in columns
        // 0-31, keys 64-127 in columns 64-95, one half per softmax warpgroup)
#pragma unroll
        for (int k = 0; k < kBn / 16; ++k)
          mma_ts(t_o, tmem + (gb & 1) * 128 + 8 * k + (k >= 4 ? 32 : 0),
                 sdesc_from_lo(v_mn[vs] + mnmaj(k)), kIdO, (t > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar_addr(c, BAR_O_DONE));
        mma_commit(bar_addr(c, BAR_V_EMPTY + vs));
        if (t == nt - 1) mma_commit(bar_addr(c, BAR_O_LAST));
      }
    }
    g += nt;
  }
  if (__any_sync(0xffffffffu, !ok || *c.abort != 0)) {
    // completion of everything issued before tensor memory is released
    if (leader) mma_commit(bar_addr(c, BAR_DRAIN));
    wait_drain(c, BAR_DRAIN, 0);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ softmax
// Row maximum over 64 keys (key0 .. key0 + 63, S columns src .. src + 63)
// of raw scores; with tau > 0 the logit grows with the score, softcap
// included. MASKED chunks (a band's edge, the sequence's end) leave
// invisible keys out.
template <bool MASKED>
__device__ __forceinline__ float chunk_max_regs(const Params& p, const uint32_t (&raw)[64],
                                                int key0, int qrow) {
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int e = 0; e < 64; ++e) {
    float s = __uint_as_float(raw[e]);
    if (MASKED) {
      const int key = key0 + e;
      if (!(key < p.N && key - qrow <= p.win_right && qrow - key <= p.win_left)) s = -INFINITY;
    }
    if (e & 1)
      m1 = fmaxf(m1, s);
    else
      m0 = fmaxf(m0, s);
  }
  return fmaxf(m0, m1);
}

// Scores of keys key0 .. key0 + 63 that the band or the sequence's end hides
// set to -inf, so that the unmasked maximum and P code (exp2(-inf) = 0) then
// serve the block too. A separate masked copy of that code runs once per
// tile and was found cold in the instruction cache every time.
__device__ __forceinline__ void mask_scores(const Params& p, uint32_t (&raw)[64], int key0,
                                            int qrow) {
  // key0 + e is visible iff lo <= e <= hi
  const int hi = min(p.N - 1, qrow + p.win_right) - key0;
  const int lo = qrow - p.win_left - key0;
#pragma unroll
  for (int e = 0; e < 64; ++e)
    if (e < lo || e > hi) raw[e] = 0xff800000u;  // -inf
}

// P = 2^(x - shift) of 64 keys (key0 .. key0 + 63, S columns src .. src +
// 63) as bf16 pairs in columns dst .. dst + 31; returns their sum of P (fp32,
// before rounding and before dropout). With DROP the bf16 values are
// P o Z / (1 - p), Z the keep mask whose bit j of kb0 (kb1) belongs to key
// key0 + j (key0 + 32 + j): the exponent carries log2(1 / (1 - p)), so exp2
// gives P / (1 - p), and the sum returned is that of P / (1 - p) over every
// key (the caller multiplies the row sum by 1 - p at the end). dst may
// overlap src: every S value of the chunk is read before the first P is
// written.
template <bool SOFTCAP, bool MASKED, bool DROP>
__device__ __forceinline__ float chunk_p_regs(const Params& p, const uint32_t (&raw)[64],
                                              uint32_t dst, int key0, int qrow, float c_log2,
                                              float cap_in, float cap_out, float shift,
                                              uint32_t kb0, uint32_t kb1) {
  const uint64_t c2v = f2_make(SOFTCAP ? cap_in : c_log2, SOFTCAP ? cap_in : c_log2);
  const uint64_t out2 = f2_make(cap_out, cap_out);
  const float cap_u = SOFTCAP ? p.scale / p.softcap : 0.f;  // u = tau s / c
  const uint64_t cu2 = f2_make(cap_u, cap_u);
  const float nsh = DROP ? p.drop.log2_inv_keep - shift : -shift;
  const uint64_t nsh2 = f2_make(nsh, nsh);
  uint64_t sum2 = f2_make(0.f, 0.f);
  uint32_t packed[32];
  // FAST: tanh by the polynomial (every |u| of the warp's 64 keys <= 1)
  auto p_group = [&](auto fast_tag) {
    constexpr bool FAST = decltype(fast_tag)::value;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const uint64_t s2 = f2_make(raw[2 * u], raw[2 * u + 1]);
      uint64_t y2;
      if (SOFTCAP) {
        // tanh(v), v = tau s / c
        const uint64_t th2 = FAST ? softcap::tanh_poly2(f2_mul(s2, cu2))
                                  : softcap::tanh_mufu2(f2_mul(s2, c2v));
        y2 = f2_fma(th2, out2, nsh2);
      } else {
        y2 = f2_fma(s2, c2v, nsh2);
      }
      float y0 = f2_lo(y2), y1 = f2_hi(y2);
      if (MASKED) {
        const int key = key0 + 2 * u;
        if (!(key < p.N && key - qrow <= p.win_right && qrow - key <= p.win_left)) y0 = -INFINITY;
        if (!(key + 1 < p.N && key + 1 - qrow <= p.win_right && qrow - key - 1 <= p.win_left))
          y1 = -INFINITY;
      }
      const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
      sum2 = f2_add(sum2, f2_make(p0, p1));
      if (DROP) {
        const uint32_t kb = u < 16 ? kb0 : kb1;
        const int bit = (2 * u) & 31;
        const float d0 = (kb >> bit) & 1u ? p0 : 0.f;
        const float d1 = (kb >> (bit + 1)) & 1u ? p1 : 0.f;
        packed[u] = pack_bf16x2(d0, d1);
      } else {
        packed[u] = pack_bf16x2(p0, p1);
      }
    }
  };
  if constexpr (SOFTCAP) {
    if (__all_sync(0xffffffffu, softcap::max_abs(raw) * cap_u <= softcap::kPolyMax))
      p_group(std::true_type{});
    else
      p_group(std::false_type{});
  } else {
    p_group(std::false_type{});
  }
  uint32_t lo[16], hi[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    lo[u] = packed[u];
    hi[u] = packed[16 + u];
  }
  tmem_st16(dst, lo);
  tmem_st16(dst + 16, hi);
  return f2_lo(sum2) + f2_hi(sum2);
}

// The keep mask with dropout (warps 12-19, two per SM
// sub-partition). For each key block of the CTA's tiles, warp 12 + w and lane
// q draw the Philox calls of the query quad q (rows 4q .. 4q + 3, counter
// word 0 = (m0 + 4q) / 4) and of the 16 keys 16 w .. 16 w + 15 of the block:
// call g gives the four rows' words of key g, so the thread ends with 16 bits
// of each of its four rows, half of a 32-key word. Block g (counted over
// the CTA's tiles) goes to slot g mod 2 once the softmax has read block g - 2
// out of it; the softmax reads block g's words while the one after is drawn.
template <int D>
__device__ void mask_role(const Ctx& c, const Params& p, uint8_t* smem) {
  using L = Layout<D>;
  const int lane = threadIdx.x & 31;
  const int mw = (static_cast<int>(threadIdx.x) >> 5) - 12;  // 16-key group of a block
  uint16_t* mask = reinterpret_cast<uint16_t*>(smem + L::kMask);
  const int n_tiles = p.tiles * p.B * p.H;
  int g = 0;  // global block index
  for (int r = 0;; ++r) {
    const int idx = cta_tile(r, n_tiles);
    if (idx < 0) return;
    const Tile tl = tile_of(p, idx);
    const uint32_t qgrp = static_cast<uint32_t>(tl.m0 >> 2) + static_cast<uint32_t>(lane);
    const uint32_t bh = static_cast<uint32_t>(tl.bh);
    for (int t = 0; t < tl.nt; ++t, ++g) {
      const int slot = g & 1;
      if (g >= 2 && !wait(c, BAR_MASK_EMPTY + slot, ((g >> 1) - 1) & 1)) return;
      const uint32_t k0 = static_cast<uint32_t>((tl.j0 + t) * kBn + 16 * mw);
      uint32_t bits[4] = {0u, 0u, 0u, 0u};
      constexpr int kNB = 8;  // calls in flight
#pragma unroll 1
      for (int g0 = 0; g0 < 16; g0 += kNB) {
        uint32_t ctr[kNB][4];
#pragma unroll
        for (int u = 0; u < kNB; ++u) {
          ctr[u][0] = qgrp;
          ctr[u][1] = k0 + static_cast<uint32_t>(g0 + u);
          ctr[u][2] = bh;
          ctr[u][3] = 0u;
        }
        philox4x32_10_batch<kNB, 10>(ctr, p.drop.seed_lo, p.drop.seed_hi);
#pragma unroll
        for (int u = 0; u < kNB; ++u)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            bits[e] |= (ctr[u][e] >= p.drop.threshold ? 1u : 0u) << (g0 + u);
      }
      // row 4 lane + e: 32-key word mw / 2 (key half mw / 4, word (mw / 2)
      // mod 2), 16-bit half mw mod 2
      const int kg = mw >> 1;
      uint16_t* dst = mask + slot * 1024 + ((kg >> 1) * 256 + (kg & 1)) * 2 + (mw & 1);
#pragma unroll
      for (int e = 0; e < 4; ++e) dst[(4 * lane + e) * 4] = static_cast<uint16_t>(bits[e]);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(c, BAR_MASK_FULL + slot));
    }
  }
}

// The softmax: the two warpgroups share the tile, warpgroup
// h taking keys 64 h .. 64 h + 63 of every key block (thread = query row r
// in both). Per block they exchange the half-row maxima through shared
// memory, so both take the same shift; each keeps the row sum of its half,
// writes P of its keys (warpgroup 1 into columns 64-95, so that it never
// overwrites S values warpgroup 0 still reads) and rescales its half of the
// O row. At the end the two row sums are added, and warpgroup h writes
// columns h d/2 .. of O. Every decision is taken by both warpgroups together
// (a 256-thread barrier with an AND), so an abort leaves none of them behind.
constexpr int kBarBoth = 3;  // named barrier of both softmax warpgroups

template <int D, bool SOFTCAP, bool DROP>
__device__ void softmax_role(const Ctx& c, const Params& p, uint8_t* smem, uint32_t sbase,
                                   uint32_t tmem, const CUtensorMap* to) {
  using L = Layout<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = (warp - 4) >> 2;  // which half of the keys (and of O's columns)
  const int r = ((warp & 3) << 5) + lane;
  const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
  float* xmax = reinterpret_cast<float*>(smem + L::kXchg);  // [block parity][half][row]
  float* xsum = xmax + 4 * 128;                              // [half][row]
  const int bar_wg = 1 + h;
  const float c_log2 = p.scale * kLog2e;
  const float cap_in = SOFTCAP ? 2.f * kLog2e * p.scale / p.softcap : 0.f;  // 2 log2e tau/c
  const float cap_out = SOFTCAP ? p.softcap * kLog2e : 0.f;                 // c log2e
  const int n_tiles = p.tiles * p.B * p.H;
  bool ok = true;
  int g = 0;  // global index of the tile's first key block
  int q_empty_pending = 0;  // Q stage + 1 whose O stores this thread has yet to hand back
  for (int rr = 0, i = 0; ok; ++rr, ++i) {
    const int idx = cta_tile(rr, n_tiles);
    if (idx < 0) break;
    const Tile tl = tile_of(p, idx);
    const int nt = tl.nt, m0 = tl.m0, qrow = m0 + r;
    const int qs = i % L::kQStages, ob = i % L::kOBufs;
    const uint32_t tO = tmem + lane_base + 256 + ob * D + h * (D / 2);
    float m_used = -INFINITY, l = 0.f;
    for (int t = 0; t < nt; ++t) {
      const int gb = g + t;  // this block over the CTA's tiles
      const int n0 = (tl.j0 + t) * kBn;
      const int key0 = n0 + 64 * h;
      const uint32_t tS = tmem + lane_base + (gb & 1) * 128;
      const uint32_t src = tS + 64 * h;
      // the keep bits of this half's 64 keys, drawn by the mask warpgroup
      uint32_t kb0 = 0xFFFFFFFFu, kb1 = 0xFFFFFFFFu;
      if (DROP) {
        const int slot = gb & 1;
        if (wait(c, BAR_MASK_FULL + slot, (gb >> 1) & 1)) {
          const uint2 kb =
              reinterpret_cast<const uint2*>(smem + L::kMask)[slot * 256 + h * 128 + r];
          kb0 = kb.x;
          kb1 = kb.y;
        } else {
          ok = false;  // voted on at this block's barrier
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr(c, BAR_MASK_EMPTY + slot));
      }
      // The scores are read from tensor memory once and kept in registers for
      // the maximum and P. The one barrier of both warpgroups per block carries
      // the half-row maxima and the abort decision (a wait that gave up, here
      // or at the previous block's O rescale).
      const bool got = wait(c, BAR_S_FULL + (gb & 1), (gb >> 1) & 1);
      uint32_t raw[64];
      if (got) {
        tc_fence_after();
        tmem_ld32x2(src, src + 32, raw);
      } else {
  #pragma unroll
        for (int e = 0; e < 64; ++e) raw[e] = 0u;
      }
      const bool masked =
          n0 + kBn - 1 - m0 > p.win_right || m0 + kBm - 1 - n0 > p.win_left || n0 + kBn > p.N;
      // without the softcap, hidden keys become -inf scores (tanh would make
      // -inf a finite logit, so the softcap keeps its masked code)
      if (!SOFTCAP && masked) mask_scores(p, raw, key0, qrow);
      const bool mask_code = SOFTCAP && masked;
      const float hmax = mask_code ? chunk_max_regs<true>(p, raw, key0, qrow)
                                   : chunk_max_regs<false>(p, raw, key0, qrow);
      float* slot = xmax + (gb & 1) * 256;
      slot[h * 128 + r] = hmax;
      ok = named_bar_and(kBarBoth, 256, ok && got);
      if (!ok) break;
      const float smax = fmaxf(hmax, slot[(1 - h) * 128 + r]);
      float m_tile = -INFINITY;  // row maximum of x = logit * log2e over this block
      if (smax > -INFINITY) {
        if (SOFTCAP) {
          const float ex = ex2_approx(smax * cap_in);
          m_tile = (1.f - 2.f * rcp_approx(ex + 1.f)) * cap_out;
        } else {
          m_tile = smax * c_log2;
        }
      }
      // move the shift when the maximum outgrows it by more than kRescale (the
      // same decision in both warpgroups: they see the same maxima)
      const bool need = m_tile > m_used + kRescale;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? m_tile : m_used;
        const float f = need ? ex2_approx(m_used - m_new) : 1.f;  // 0 while m_used = -inf
        // this half of the O row, once P(t - 1) V has completed; a wait that
        // gives up is voted on at the next barrier
        if (__any_sync(0xffffffffu, need && m_used > -INFINITY) && t > 0) {
          if (!wait_warp(c, BAR_O_DONE, (gb - 1) & 1)) ok = false;
          if (ok) {
            tc_fence_after();
            const uint64_t f2 = f2_make(f, f);
  #pragma unroll
            for (int c32 = 0; c32 < D / 64; ++c32) {
              uint32_t o[32];
              tmem_ld32(tO + c32 * 32, o);
  #pragma unroll
              for (int u = 0; u < 16; ++u) {
                const uint64_t v = f2_mul(f2_make(o[2 * u], o[2 * u + 1]), f2);
                o[2 * u] = static_cast<uint32_t>(v);
                o[2 * u + 1] = static_cast<uint32_t>(v >> 32);
              }
              uint32_t lo[16], hi[16];
  #pragma unroll
              for (int u = 0; u < 16; ++u) {
                lo[u] = o[u];
                hi[u] = o[16 + u];
              }
              tmem_st16(tO + c32 * 32, lo);
              tmem_st16(tO + c32 * 32 + 16, hi);
            }
          }
        }
        l *= f;
        m_used = m_new;
      }
      const float shift = m_used > -INFINITY ? m_used : 0.f;
      const uint32_t dst = tS + 64 * h;  // keys 0-63 -> columns 0-31, 64-127 -> 64-95
      l += mask_code ? chunk_p_regs<SOFTCAP, true, DROP>(p, raw, dst, key0, qrow, c_log2, cap_in,
                                                         cap_out, shift, kb0, kb1)
                     : chunk_p_regs<SOFTCAP, false, DROP>(p, raw, dst, key0, qrow, c_log2,
                                                          cap_in, cap_out, shift, kb0, kb1);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(c, BAR_P_FULL + (gb & 1)));  // one arrival per warp
      // The previous tile's O stores have long read their Q stage: hand it
      // back now (the loader needs it two tiles on), not at the end of that
      // tile's epilogue, where the wait held this warp back.
      if (q_empty_pending) {
        bulk_wait_read_all();
        mbar_arrive(bar_addr(c, BAR_Q_EMPTY + q_empty_pending - 1));
        q_empty_pending = 0;
      }
    }
    // ---- epilogue, once the tile's last P V has completed. Its own barrier
    // (one phase per tile) is waited on, not O_DONE: by the time the softmax
    // gets here both of the tile's last P V phases of O_DONE may have
    // completed, and O_DONE would then stand at the parity of the first of
    // them again (a wait on that parity would last until the next tile's
    // first P V, which needs this softmax: a deadlock, seen on the GPU as a
    // rare wait timeout).
    if (ok) ok = wait(c, BAR_O_LAST, i & 1);
    xsum[h * 128 + r] = l;
    if (!named_bar_and(kBarBoth, 256, ok)) break;
    tc_fence_after();
    // with dropout the sums were of P / (1 - p)
    const float lt = (xsum[r] + xsum[128 + r]) * (DROP ? p.drop.keep : 1.f);
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    const uint64_t inv2 = f2_make(inv, inv);
    // O / l of this half's columns -> bf16 rows in the tile's Q stage (free
    // once the last S GEMM is done, which precedes the last P V) -> TMA tensor
    // stores; O_FREE once tensor memory is read, Q_EMPTY once the stores have
    // read the stage
    const uint32_t buf = sbase + L::kQ0 + qs * L::kTileBytes;
  #pragma unroll
    for (int c16 = 0; c16 < D / 32; ++c16) {
      const int col = h * (D / 2) + c16 * 16;  // column of O
      uint32_t raw[16];
      tmem_ld16(tO + c16 * 16, raw);
      uint32_t packed[8];
  #pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint64_t v = f2_mul(f2_make(raw[2 * u], raw[2 * u + 1]), inv2);
        packed[u] = pack_bf16x2(f2_lo(v), f2_hi(v));
      }
      // columns col .. col + 15: box col / 64, 16-byte chunks (col % 64) / 8, + 1
      const uint32_t row_addr = buf + (col >> 6) * 16384 + r * 128;
      const int c0 = (col & 63) >> 3;
      st_shared_v4(row_addr + ((c0 ^ (r & 7)) << 4), packed[0], packed[1], packed[2], packed[3]);
      st_shared_v4(row_addr + (((c0 + 1) ^ (r & 7)) << 4), packed[4], packed[5], packed[6],
                   packed[7]);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_addr(c, BAR_O_FREE + ob));
    fence_proxy_async_smem();
    // d >= 128: each warpgroup stores its own 64-column boxes; d = 64: the one
    // box holds both halves and is stored once both warpgroups have written it
    if (D >= 128)
      named_bar_sync(bar_wg, 128);
    else
      named_bar_sync(kBarBoth, 256);
    if (r == 0 && (D >= 128 || h == 0)) {
      constexpr int kBoxesWg = D >= 128 ? D / 128 : 1;  // boxes one thread stores
      for (int cb = h * kBoxesWg; cb < (h + 1) * kBoxesWg; ++cb)
        tma_store_3d(to, buf + cb * 16384, 64 * cb, m0, tl.bh);
      bulk_commit_group();
      if (L::kQStages >= 2) {
        q_empty_pending = qs + 1;  // handed back after the next tile's first block
      } else {
        bulk_wait_read_all();
        mbar_arrive(bar_addr(c, BAR_Q_EMPTY + qs));
      }
    }
    if (h == 0 && qrow < p.N)
      p.lse[static_cast<long long>(tl.bh) * p.N + qrow] =
          lt > 0.f ? (m_used + __log2f(lt)) * kLn2 : -INFINITY;
    g += nt;
  }
  // the O stores complete before the CTA exits
  if (q_empty_pending) mbar_arrive(bar_addr(c, BAR_Q_EMPTY + q_empty_pending - 1));
  if (r == 0) bulk_wait_all();
}

// ------------------------------------------------------------------ kernel
template <int D, bool SOFTCAP, bool DROP>
__global__ void __launch_bounds__(kThreadsFor<DROP>, 1)
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
    for (int sl = 0; sl < 2; ++sl) {
      mbar_init(bar_addr(c, BAR_P_FULL + sl), 8);  // one arrival per softmax warp
      mbar_init(bar_addr(c, BAR_Q_EMPTY + sl), D >= 128 ? 2 : 1);  // the O-storing threads
      mbar_init(bar_addr(c, BAR_O_FREE + sl), 8);  // the softmax warps
      if (DROP) {
        mbar_init(bar_addr(c, BAR_MASK_FULL + sl), kMaskWarps);
        mbar_init(bar_addr(c, BAR_MASK_EMPTY + sl), 8);  // the softmax warps
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
  if (warp < 4) {
    if constexpr (DROP) setmaxnreg_dec<kRegsOtherDrop>();
    if constexpr (kSplitRegs256<D, DROP>) setmaxnreg_dec<kRegsCtl256>();
    if (warp == 0)
      loader_role<D>(c, p, sbase, &tm_q, &tm_k, false);
    else if (warp == 1)
      mma_role<D>(c, p, sbase, tmem);
    else if (warp == 2)
      loader_role<D>(c, p, sbase, &tm_q, &tm_v, true);
  } else if (warp < 12) {
    if constexpr (DROP) setmaxnreg_inc<kRegsSoftmaxDrop>();
    if constexpr (kSplitRegs256<D, DROP>) setmaxnreg_inc<kRegsSoftmax256>();
    softmax_role<D, SOFTCAP, DROP>(c, p, smem, sbase, tmem, &tm_o);
  } else {
    if constexpr (DROP) {
      setmaxnreg_dec<kRegsOtherDrop>();
      mask_role<D>(c, p, smem);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool SOFTCAP, bool DROP>
int launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
           const CUtensorMap& to, const Params& p, cudaStream_t stream) {
  auto kern = attn_fwd_kernel<D, SOFTCAP, DROP>;
  static std::atomic<bool> configured[kMaxTrackedDevices];
  if (!set_smem_limit_once(kern, Layout<D>::kBytes, configured)) return ATTN_ERR_LAUNCH;
  // persistent: one CTA per SM, or per tile if there are fewer
  long long grid = static_cast<long long>(p.tiles) * p.B * p.H;
  if (grid > 0x7fffffffLL) return ATTN_ERR_TOO_LARGE;
  const int sms = sm_count();
  if (sms <= 0) return ATTN_ERR_LAUNCH;
  if (grid > sms) grid = sms;
  kern<<<static_cast<unsigned>(grid), kThreadsFor<DROP>, Layout<D>::kBytes, stream>>>(tq, tk, tv,
                                                                                        to, p);
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

template <bool DROP>
int dispatch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
             const CUtensorMap& to, const Params& p, cudaStream_t s, int d, bool cap) {
  if (d == 256)
    return cap ? launch<256, true, DROP>(tq, tk, tv, to, p, s)
               : launch<256, false, DROP>(tq, tk, tv, to, p, s);
  if (d == 128)
    return cap ? launch<128, true, DROP>(tq, tk, tv, to, p, s)
               : launch<128, false, DROP>(tq, tk, tv, to, p, s);
  return cap ? launch<64, true, DROP>(tq, tk, tv, to, p, s)
             : launch<64, false, DROP>(tq, tk, tv, to, p, s);
}

int run(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv,
        int N, int d, float scale, int causal, float softcap, int window_left, int window_right,
        void* stream, float p_drop = 0.f, unsigned long long seed = 0) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  int rc = check_shape(B, H, H_kv, N, d);
  if (rc != ATTN_OK) return rc;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  // tau > 0: the kernel takes a row's largest logit at its largest score
  if (!std::isfinite(scale) || !(scale > 0.f) || std::isnan(softcap)) return ATTN_ERR_SHAPE;
  if (!(p_drop >= 0.f && p_drop < 1.f)) return ATTN_ERR_SHAPE;
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
  p.tiles = (N + kBm - 1) / kBm;
  p.scale = scale;
  const bool cap = softcap > 0.f;
  p.softcap = cap ? softcap : 0.f;
  // a negative or wider-than-N side of the window is unbounded (N); the
  // causal mask bounds the right side at 0
  p.win_left = (window_left < 0 || window_left > N) ? N : window_left;
  p.win_right = causal ? 0 : ((window_right < 0 || window_right > N) ? N : window_right);
  p.drop.seed_lo = static_cast<uint32_t>(seed);
  p.drop.seed_hi = static_cast<uint32_t>(seed >> 32);
  p.drop.threshold = dropout_threshold(p_drop);
  p.drop.inv_keep = 1.f / (1.f - p_drop);
  p.drop.keep = 1.f - p_drop;
  p.drop.log2_inv_keep =
      static_cast<float>(-std::log2(1.0 - static_cast<double>(p_drop)));
  cudaStream_t s = as_stream(stream);
  return p_drop > 0.f ? dispatch<true>(tq, tk, tv, to, p, s, d, cap)
                      : dispatch<false>(tq, tk, tv, to, p, s, d, cap);
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

extern "C" int attn_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int H_kv, int N, int d, float scale, int causal,
                                float softcap, float p_drop, unsigned long long seed,
                                void* stream) {
  return fwdtc::run(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, -1, -1, stream,
                    p_drop, seed);
}
