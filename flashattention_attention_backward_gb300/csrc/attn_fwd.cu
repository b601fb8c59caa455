// attn_fwd: attention forward on sm_103a producing O and the natural-log
// LSE the backward needs ("反向传播算法详解" §1.2-§1.3 saved tensors;
// "解析 FlashAttention（3）" §1.1 forward and §3.2 eq. 9-12, the running
// (max, sum) statistics of the online softmax).
//
// Two forms share the per-block arithmetic below. Queries sit on the
// tensor-memory lanes: thread r of a softmax warpgroup owns query row r, so
// row maxima and sums need no reduction across rows. Per key block j:
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
// Two-tile form (d = 64). One CTA owns two blocks of 128 queries (tiles 0
// and 1) of one query head and walks, once, the key blocks their masks let
// them see. The tiles ping-pong on the tensor cores: while the softmax of
// tile 0 works on S_0(j), the tensor cores run P_1(j-1) V and S_1(j), and the
// other way round; K_j and V_j serve both tiles.
//   warp 0      TMA producer: Q_0, Q_1 once; K_j, V_j in two-stage rings
//   warp 1      tcgen05 MMA issuer (whole warp, one elected lane issues)
//   warps 4-7   softmax of tile 0, then its epilogue (O / l -> bf16 ->
//               shared -> TMA store; LSE)
//   warps 8-11  the same for tile 1
// Tensor memory: S buffers of the tiles at [0,128) and [128,256) (P
// overwrites the first half of its buffer), O_0 at [256, 256 + d), O_1 at
// [256 + d, 256 + 2d).
//
// One-tile form (d = 128 and 256; two tiles' S and O would need 768 columns
// at d = 256). A tile is one block of 128 queries, and the CTAs are
// persistent: one per SM, each walking its tiles in snake order. A tile's key
// blocks alternate between two S buffers ([0,128) and [128,256)), so
// S(j + 1) runs on the tensor cores while the softmax works on S(j); O sits
// at [256, 256 + d), and at d = 128 the tiles alternate between two O
// buffers ([256, 384) and [384, 512)). The next tile's Q (two Q stages at
// d = 128), K and V blocks load while the current tile finishes, so the
// launch, the first loads and the epilogue of a tile no longer stand alone.
// Both softmax warpgroups work on the one tile, warpgroup h on keys
// 64 h .. 64 h + 63 of each block and on columns h d/2 .. of O; they
// exchange the half-row maxima through shared memory once per block.
//   warp 0      Q of each tile; K_j in a ring of 2 stages (d = 128) or 1
//   warp 2      V_j in the same kind of ring
//   warp 1      MMA issuer: per tile S(0), then per block S(j + 1), P(j) V
//   warps 4-11  softmax, then the tile's epilogue (each warpgroup its half of
//               O, staged in the tile's Q stage)
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

template <int D>
struct Layout {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kQ0 = 0;  // Q of tile 0; its O staging buffer at the end
  static constexpr int kQ1 = kQ0 + kTileBytes;
  static constexpr int kK0 = kQ1 + kTileBytes;
  static constexpr int kK1 = kK0 + kTileBytes;
  static constexpr int kV0 = kK1 + kTileBytes;
  static constexpr int kV1 = kV0 + kTileBytes;
  static constexpr int kBars = kV1 + kTileBytes;
  static constexpr int kNumBars = 17;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  // d = 64 needs 96 KB; it asks for more than half of the SM's shared memory
  // so that a second CTA never waits on the first one's tensor memory
  static constexpr int kUsed = kAbort + 12;
  static constexpr int kBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
};
static_assert(Layout<128>::kBytes <= 232448, "shared memory budget");

// The one-tile form (d = 256): one query tile per CTA and one K and one V
// stage; the Q buffer stages O at the end. It asks for more than half of the
// SM's shared memory, so that a second CTA never waits on the first one's
// tensor memory.
template <int D>
constexpr bool kOneTile = D >= 128;

// With dropout the one-tile form draws the keep mask in a warpgroup of its
// own. Philox4x32-10 is bound by the 32 x 32 -> 64-bit multiplies (measured
// on this GPU: about 1.3 calls per clock per SM, some 3,000 cycles for the
// 4,096 calls of a 128 x 128 block), about as long as the softmax of a
// block; drawn inline it adds to the softmax's critical path, drawn by
// warps 12-15 for block j + 1 while the softmax works on block j it runs
// beside it. The CTA then has 640 threads; setmaxnreg gives the softmax
// warps 128 registers and the other twelve warps 72.
template <int D, bool DROP>
constexpr bool kMaskRole = kOneTile<D> && DROP;
template <int D, bool DROP>
constexpr int kThreadsFor = kMaskRole<D, DROP> ? 640 : kThreads;
constexpr int kMaskWarps = 8;  // two per SM sub-partition
constexpr int kRegsSoftmaxDrop = 128, kRegsOtherDrop = 72;
static_assert(256 * kRegsSoftmaxDrop + 384 * kRegsOtherDrop <= 640 * 96, "register pool");

template <int D>
struct LayoutOne {
  static constexpr int kTileBytes = 128 * D * 2;
  // K and V stages: two where they fit (d <= 128), one at d = 256. Q stages
  // likewise: the next tile's Q loads while the current one finishes, and a
  // tile's Q stage stages its O for the TMA store at the end.
  static constexpr int kStages = D <= 128 ? 2 : 1;
  static constexpr int kQStages = D <= 128 ? 2 : 1;
  // O accumulators in tensor memory (after the two S buffers): two at
  // d = 128, so a tile's P V GEMMs never wait for the previous tile's
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
  static constexpr int kNumBars = 25;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kUsed = kAbort + 12;
  static constexpr int kBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
};
static_assert(LayoutOne<128>::kBytes <= 232448, "shared memory budget");
static_assert(LayoutOne<256>::kBytes <= 232448, "shared memory budget");
static_assert(2 * 128 + LayoutOne<128>::kOBufs * 128 <= 512, "tensor memory");
static_assert(2 * 128 + LayoutOne<256>::kOBufs * 256 <= 512, "tensor memory");

template <int D>
using LayoutFor = std::conditional_t<kOneTile<D>, LayoutOne<D>, Layout<D>>;

enum Bar {
  BAR_Q_FULL = 0,    // + tile
  BAR_K_FULL = 2,    // + stage
  BAR_K_EMPTY = 4,   // + stage
  BAR_V_FULL = 6,    // + stage
  BAR_V_EMPTY = 8,   // + stage
  BAR_S_FULL = 10,   // + tile (d = 256: + S buffer): S_q(j) in its buffer
  BAR_P_FULL = 12,   // + tile (d = 256: + S buffer): P_q(j) written (and O_q rescaled if needed)
  BAR_O_DONE = 14,   // + tile: P_q(j) V_j completed (one phase per key block of the tile)
  BAR_DRAIN = 16,    // abort path only: completion of everything issued
  BAR_MASK_FULL = 17,   // + block parity (one-tile form with dropout): keep bits written
  BAR_MASK_EMPTY = 19,  // + block parity: the softmax has read them
  BAR_Q_EMPTY = 21,     // + Q stage (one-tile form): the tile's O store has read the stage
  BAR_O_FREE = 23,      // + O buffer (one-tile form): the tile's epilogue has read O
};

struct Params {
  float* lse;
  int B, H, H_kv, N;
  int pairs;  // CTAs per query head: ceil(query blocks / 2) (d = 256: query blocks)
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

// Work of one CTA: query tiles m0[0] = 256 * pair and m0[1] = m0[0] + 128
// of head bh (= b * H + h). Tile q sees key blocks j0[q] .. j0[q] + nt[q] - 1
// (nt[q] = 0: the tile lies past N); together they span jlo .. jhi.
struct Work {
  int bh, kvh;
  int m0[2], j0[2], nt[2];
  int jlo, jhi;
  __device__ __forceinline__ bool has(int q, int j) const {
    return j >= j0[q] && j < j0[q] + nt[q];
  }
  __device__ __forceinline__ int uses(int j) const {
    return (has(0, j) ? 1 : 0) + (has(1, j) ? 1 : 0);
  }
};

// The one-tile form: m0[0] = 128 * pair; tile 1 is empty.
template <int D>
__device__ __forceinline__ Work work_of(const Params& p) {
  Work w;
  const int heads = p.B * p.H;
  const int idx = static_cast<int>(blockIdx.x);
  // heaviest query blocks first for a causal mask (the last ones see the
  // most keys)
  const int pair = p.pairs - 1 - idx / heads;
  w.bh = idx - (idx / heads) * heads;
  const int b = w.bh / p.H, h = w.bh - b * p.H;
  w.kvh = b * p.H_kv + h / (p.H / p.H_kv);
  const int last_block = (p.N + kBn - 1) / kBn - 1;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    w.m0[q] = kOneTile<D> ? (q == 0 ? pair * kBm : p.N) : pair * 2 * kBm + q * kBm;
    if (w.m0[q] >= p.N) {
      w.j0[q] = 0;
      w.nt[q] = 0;
      continue;
    }
    w.j0[q] = max(0, w.m0[q] - p.win_left) / kBn;
    const int j_end = min(last_block, (w.m0[q] + kBm - 1 + p.win_right) / kBn);
    w.nt[q] = j_end - w.j0[q] + 1;  // >= 1: the band holds the diagonal
  }
  // tile 1 starts and ends no earlier than tile 0, and their ranges touch
  w.jlo = w.j0[0];
  w.jhi = w.nt[1] > 0 ? w.j0[1] + w.nt[1] - 1 : w.j0[0] + w.nt[0] - 1;
  return w;
}

// The one-tile form is persistent: min(#SMs, tiles) CTAs, CTA c taking tile
// index r * grid + c in even passes r and r * grid + (grid - 1 - c) in odd
// ones (snake order over the tiles, heaviest first for a causal mask), so the
// next tile's Q and first K, V blocks load and its first S GEMM runs while
// the current tile finishes. Every per-block barrier keeps one phase per key
// block across the CTA's tiles (global block index g), the per-tile ones one
// phase per tile.
struct TileOne {
  int bh, kvh, m0, j0, nt;
};

__device__ __forceinline__ int cta_tile(int r, int n_tiles) {
  const int grid = static_cast<int>(gridDim.x);
  const int cta = static_cast<int>(blockIdx.x);
  const int idx = r * grid + ((r & 1) ? grid - 1 - cta : cta);
  return idx < n_tiles ? idx : -1;
}

// Tile idx: query block pair (heaviest first) of head bh.
__device__ __forceinline__ TileOne tile_one(const Params& p, int idx) {
  TileOne t;
  const int heads = p.B * p.H;
  const int blk = p.pairs - 1 - idx / heads;
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
    for (int q = 0; q < 2; ++q) {
      if (w.nt[q] == 0) continue;
      mbar_arrive_expect_tx(bar_addr(c, BAR_Q_FULL + q), kTileBytes);
      for (int cb = 0; cb < kBoxes; ++cb)
        tma_load_3d(sbase + (q ? L::kQ1 : L::kQ0) + cb * 16384, tq, bar_addr(c, BAR_Q_FULL + q),
                    64 * cb, w.m0[q], w.bh);
    }
  }
  const uint64_t keep = policy_evict_last();  // K, V are read by every query block of the head
  int issued = 0;
  bool ok = true;
  for (int j = w.jlo; j <= w.jhi; ++j) {
    const int kb = j - w.jlo, st = kb & 1;
    const uint32_t ph = ((kb >> 1) - 1) & 1;
    if (kb >= 2 && !(ok = wait_warp(c, BAR_K_EMPTY + st, ph))) break;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_addr(c, BAR_K_FULL + st), kTileBytes);
      for (int cb = 0; cb < kBoxes; ++cb)
        tma_load_3d_hint(sbase + (st ? L::kK1 : L::kK0) + cb * 16384, tk,
                         bar_addr(c, BAR_K_FULL + st), 64 * cb, j * kBn, w.kvh, keep);
    }
    if (kb >= 2 && !(ok = wait_warp(c, BAR_V_EMPTY + st, ph))) {
      issued = 2 * kb + 1;
      break;
    }
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_addr(c, BAR_V_FULL + st), kTileBytes);
      for (int cb = 0; cb < kBoxes; ++cb)
        tma_load_3d_hint(sbase + (st ? L::kV1 : L::kV0) + cb * 16384, tv,
                         bar_addr(c, BAR_V_FULL + st), 64 * cb, j * kBn, w.kvh, keep);
    }
    issued = 2 * kb + 2;
    __syncwarp();
  }
  // When aborting, the copies in flight must land before the CTA exits.
  if (!ok || *c.abort) {
    for (int q = 0; q < 2; ++q)
      if (w.nt[q] > 0) wait_drain(c, BAR_Q_FULL + q, 0);
    // issued counts K and V loads in order K_0, V_0, K_1, V_1, ...
    const int first = issued - 4 < 0 ? 0 : issued - 4;
    for (int i = first; i < issued; ++i) {
      const int kb = i >> 1;
      wait_drain(c, ((i & 1) ? BAR_V_FULL : BAR_K_FULL) + (kb & 1), (kb >> 1) & 1);
    }
  }
}

// ------------------------------------------------------------------ MMA issuer
// Issue order: S_0(first), S_1(first), then for every key block j and tile q
// that sees it: P_q(j) V_j, then S_q(j + 1). S_q(j + 1) overwrites the S
// buffer holding P_q(j) only after P_q(j) V_j, which reads it (tcgen05 MMAs of
// one thread run in issue order). K_j and V_j stages are released after their
// last use by either tile.
template <int D>
__device__ void mma_role(const Ctx& c, const Work& w, uint32_t sbase, uint32_t tmem) {
  using L = Layout<D>;
  const bool leader = elect_one_sync() != 0;
  constexpr uint32_t kIdS = make_idesc_bf16(kBm, kBn, false, false);  // S = Q K^T
  constexpr uint32_t kIdO = make_idesc_bf16(kBm, D, false, true);     // O += P V
  const uint32_t q_lo[2] = {sdesc_lo(sbase + L::kQ0, 16), sdesc_lo(sbase + L::kQ1, 16)};
  const uint32_t k_lo[2] = {sdesc_lo(sbase + L::kK0, 16), sdesc_lo(sbase + L::kK1, 16)};
  const uint32_t v_mn[2] = {sdesc_lo(sbase + L::kV0, 16384), sdesc_lo(sbase + L::kV1, 16384)};
  auto kmaj = [](int k) { return static_cast<uint32_t>(((k >> 2) * 16384 + (k & 3) * 32) >> 4); };
  auto mnmaj = [](int k) { return static_cast<uint32_t>((2048 * k) >> 4); };
  // uses of the K / V block each stage holds that are still to be issued
  int k_left[2] = {0, 0}, v_left[2] = {0, 0}, k_blk[2] = {-1, -1}, v_blk[2] = {-1, -1};
  bool ok = true;

  auto issue_s = [&](int q, int j) -> bool {
    const int kb = j - w.jlo, st = kb & 1;
    if (!wait_warp(c, BAR_K_FULL + st, (kb >> 1) & 1)) return false;
    if (k_blk[st] != j) {
      k_blk[st] = j;
      k_left[st] = w.uses(j);
    }
    tc_fence_after();
    if (leader) {
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        mma_ss(tmem + q * 128, sdesc_from_lo(q_lo[q] + kmaj(k)), sdesc_from_lo(k_lo[st] + kmaj(k)),
               kIdS, k > 0);
      mma_commit(bar_addr(c, BAR_S_FULL + q));
      if (k_left[st] == 1) mma_commit(bar_addr(c, BAR_K_EMPTY + st));
    }
    --k_left[st];
    return true;
  };

  for (int q = 0; q < 2 && ok; ++q) {
    if (w.nt[q] == 0) continue;
    if (!(ok = wait_warp(c, BAR_Q_FULL + q, 0))) break;
    ok = issue_s(q, w.j0[q]);
  }
  for (int j = w.jlo; ok && j <= w.jhi; ++j) {
    const int kb = j - w.jlo, st = kb & 1;
    for (int q = 0; q < 2; ++q) {
      if (!w.has(q, j)) continue;
      const int t = j - w.j0[q];
      if (!(ok = wait_warp(c, BAR_P_FULL + q, t & 1))) break;
      if (!(ok = wait_warp(c, BAR_V_FULL + st, (kb >> 1) & 1))) break;
      if (v_blk[st] != j) {
        v_blk[st] = j;
        v_left[st] = w.uses(j);
      }
      tc_fence_after();
      if (leader) {
        // A = P (bf16 pairs, keys along columns 8k .. of the tile's S buffer)
#pragma unroll
        for (int k = 0; k < kBn / 16; ++k)
          mma_ts(tmem + 256 + q * D, tmem + q * 128 + 8 * k, sdesc_from_lo(v_mn[st] + mnmaj(k)),
                 kIdO, (t > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar_addr(c, BAR_O_DONE + q));
        if (v_left[st] == 1) mma_commit(bar_addr(c, BAR_V_EMPTY + st));
      }
      --v_left[st];
      if (w.has(q, j + 1) && !(ok = issue_s(q, j + 1))) break;
    }
  }
  if (__any_sync(0xffffffffu, !ok || *c.abort != 0)) {
    // completion of everything issued before tensor memory is released
    if (leader) mma_commit(bar_addr(c, BAR_DRAIN));
    wait_drain(c, BAR_DRAIN, 0);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ one-tile roles
// Loaders of the one-tile form. Warp 0 loads Q and the K blocks, warp 2 the
// V blocks, each into its own ring of kStages stages: K(g) once S(g - kStages)
// has read its stage, V(g) once P(g - kStages) V has, Q of tile i once the O
// store of tile i - kQStages has read its stage. Each warp waits on its own
// barriers in the order the tensor cores finish them, so no load waits
// behind another operand's.
template <int D>
__device__ void loader_role_one(const Ctx& c, const Params& p, uint32_t sbase,
                                const CUtensorMap* tq, const CUtensorMap* tkv, bool is_v) {
  using L = LayoutOne<D>;
  constexpr int kBoxes = D / 64;
  constexpr uint32_t kTileBytes = L::kTileBytes;
  constexpr int kS = L::kStages, kQS = L::kQStages;
  const int lane = threadIdx.x & 31;
  const int n_tiles = p.pairs * p.B * p.H;
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
    const TileOne tl = tile_one(p, idx);
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

// MMA issuer of the one-tile form, per tile: S(0); then per key block t,
// S(t + 1) into the other S buffer (its P(t - 1) was read by P(t - 1) V,
// issued before), then P(t) V into the tile's O buffer once the softmax has
// written P(t) (the first one once the epilogue of the tile kOBufs before has
// read that buffer).
template <int D>
__device__ void mma_role_one(const Ctx& c, const Params& p, uint32_t sbase, uint32_t tmem) {
  using L = LayoutOne<D>;
  constexpr int kS = L::kStages, kQS = L::kQStages, kOB = L::kOBufs;
  const bool leader = elect_one_sync() != 0;
  constexpr uint32_t kIdS = make_idesc_bf16(kBm, kBn, false, false);  // S = Q K^T
  constexpr uint32_t kIdO = make_idesc_bf16(kBm, D, false, true);     // O += P V
  const uint32_t k_lo[2] = {sdesc_lo(sbase + L::kK0, 16), sdesc_lo(sbase + L::kK1, 16)};
  const uint32_t v_mn[2] = {sdesc_lo(sbase + L::kV0, 16384), sdesc_lo(sbase + L::kV1, 16384)};
  auto kmaj = [](int k) { return static_cast<uint32_t>(((k >> 2) * 16384 + (k & 3) * 32) >> 4); };
  auto mnmaj = [](int k) { return static_cast<uint32_t>((2048 * k) >> 4); };
  const int n_tiles = p.pairs * p.B * p.H;
  bool ok = true;
  int g = 0;  // global index of the tile's first block
  for (int r = 0, i = 0; ok; ++r, ++i) {
    const int idx = cta_tile(r, n_tiles);
    if (idx < 0) break;
    const int nt = tile_one(p, idx).nt;
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

template <bool MASKED>
__device__ __forceinline__ float chunk_max(const Params& p, uint32_t src, int key0, int qrow) {
  uint32_t raw[64];
  tmem_ld32x2(src, src + 32, raw);  // two 32-column loads per wait
  return chunk_max_regs<MASKED>(p, raw, key0, qrow);
}

// Row maximum of one S tile (both 64-key chunks).
template <bool MASKED>
__device__ __forceinline__ float tile_max(const Params& p, uint32_t tS, int n0, int qrow) {
  return fmaxf(chunk_max<MASKED>(p, tS, n0, qrow), chunk_max<MASKED>(p, tS + 64, n0 + 64, qrow));
}

// Dropout keep bits of keys k0 .. k0 + 31 for this thread's query row.
// One Philox call gives the words of four consecutive query rows of one key,
// and those rows sit in the four lanes of a quad: lane t of the quad draws
// the call of key k0 + 4 g + t, and a 4 x 4 transpose by shuffles hands
// every lane its own row's word of each of the four keys. In round k a lane
// offers word (t - k) mod 4 of its call and reads from quad lane
// (t + k) mod 4, which offers word t, for key k0 + 4 g + (t + k) mod 4.
// Everything that depends on t is done with masks, not selects on t: the
// offered words come from one rotation of the four words by t (two masked
// swaps), round k's bit goes to the fixed position 4 g + k, and a rotation of
// every nibble by t at the end moves it to 4 g + (t + k) mod 4.
__device__ __forceinline__ uint32_t keep_bits32(const Params& p, int qrow, int k0, uint32_t bh) {
  const int lane = threadIdx.x & 31;
  const uint32_t t = static_cast<uint32_t>(lane & 3);
  const uint32_t qgrp = static_cast<uint32_t>(qrow) >> 2;
  const uint32_t m1 = 0u - (t & 1u), m2 = 0u - ((t >> 1) & 1u);
  uint32_t bits = 0;
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const PhiloxOut w = philox4x32_10(qgrp, static_cast<uint32_t>(k0 + 4 * g) + t, bh, 0u,
                                      p.drop.seed_lo, p.drop.seed_hi);
    // offer[k] = word (t - k) mod 4: the words in the order 0, 3, 2, 1,
    // rotated by t (t & 1 by one place, t & 2 by two)
    const uint32_t u[4] = {w.w[0], w.w[3], w.w[2], w.w[1]};
    uint32_t r1[4], offer[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) r1[k] = (u[(k + 3) & 3] & m1) | (u[k] & ~m1);
#pragma unroll
    for (int k = 0; k < 4; ++k) offer[k] = (r1[(k + 2) & 3] & m2) | (r1[k] & ~m2);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t got =
          k == 0 ? offer[0]
                 : __shfl_sync(0xffffffffu, offer[k], (lane & ~3) | static_cast<int>((t + k) & 3));
      bits |= (got >= p.drop.threshold ? 1u : 0u) << (4 * g + k);
    }
  }
  // nibble bit k -> bit (k + t) mod 4, in all eight nibbles
  const uint32_t hi_mask = 0x11111111u * ((0xFu << t) & 0xFu);
  const uint32_t lo_mask = 0x11111111u * (0xFu >> (4u - t));
  return ((bits << t) & hi_mask) | ((bits >> (4u - t)) & lo_mask);
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

template <bool SOFTCAP, bool MASKED, bool DROP>
__device__ __forceinline__ float chunk_p(const Params& p, uint32_t src, uint32_t dst, int key0,
                                         int qrow, float c_log2, float cap_in, float cap_out,
                                         float shift, uint32_t kb0, uint32_t kb1) {
  uint32_t raw[64];
  tmem_ld32x2(src, src + 32, raw);  // two 32-column loads per wait
  return chunk_p_regs<SOFTCAP, MASKED, DROP>(p, raw, dst, key0, qrow, c_log2, cap_in, cap_out,
                                             shift, kb0, kb1);
}

// P of one S tile over the first half of its buffer: keys 64 c .. 64 c + 63
// land in columns 32 c .. 32 c + 31, whose S values were read in this or an
// earlier chunk; returns the row sum of P.
template <bool SOFTCAP, bool MASKED, bool DROP>
__device__ __forceinline__ float tile_p(const Params& p, uint32_t tS, int n0, int qrow,
                                        float c_log2, float cap_in, float cap_out, float shift,
                                        const uint32_t (&kbits)[kBn / 32]) {
  const float s0 = chunk_p<SOFTCAP, MASKED, DROP>(p, tS, tS, n0, qrow, c_log2, cap_in, cap_out,
                                                  shift, kbits[0], kbits[1]);
  const float s1 = chunk_p<SOFTCAP, MASKED, DROP>(p, tS + 64, tS + 32, n0 + 64, qrow, c_log2,
                                                  cap_in, cap_out, shift, kbits[2], kbits[3]);
  return s0 + s1;
}

// Softmax warpgroup q (thread = query row r of tile q): per key block, the
// row maximum, the shift update (with the rescale of O_q and l when the shift
// moves), and P; then the epilogue of the tile.
template <int D, bool SOFTCAP, bool DROP>
__device__ void softmax_role(const Ctx& c, const Params& p, const Work& w, uint32_t sbase,
                             uint32_t tmem, const CUtensorMap* to) {
  using L = LayoutFor<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q = (warp - 4) >> 2;  // the tile this warpgroup owns
  const int r = ((warp & 3) << 5) + lane;
  const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
  // the one-tile form: its key blocks alternate between the S buffers
  constexpr bool kAlt = kOneTile<D>;
  const uint32_t tO = tmem + lane_base + 256 + q * D;
  const int qrow = w.m0[q] + r;
  const int bar_wg = 1 + q;  // named barrier of this warpgroup (128 threads)
  const float c_log2 = p.scale * kLog2e;
  const float cap_in = SOFTCAP ? 2.f * kLog2e * p.scale / p.softcap : 0.f;  // 2 log2e tau/c
  const float cap_out = SOFTCAP ? p.softcap * kLog2e : 0.f;                 // c log2e
  const int nt = w.nt[q];
  if (nt == 0) return;
  float m_used = -INFINITY, l = 0.f;
  bool ok = true;
  const uint32_t bh = static_cast<uint32_t>(w.bh);
  for (int t = 0; t < nt; ++t) {
    const int n0 = (w.j0[q] + t) * kBn;
    const int m0 = w.m0[q];
    const uint32_t tS = tmem + lane_base + (kAlt ? (t & 1) : q) * 128;
    const int bar_s = kAlt ? BAR_S_FULL + (t & 1) : BAR_S_FULL + q;
    const uint32_t par_s = kAlt ? (t >> 1) & 1 : t & 1;
    // The keep mask depends on no score: it is drawn while the S GEMM of this
    // block runs, with no tensor-memory rows held in registers, so that many
    // Philox calls are in flight at once.
    uint32_t kbits[kBn / 32];
#pragma unroll
    for (int i = 0; i < kBn / 32; ++i)
      kbits[i] = DROP ? keep_bits32(p, qrow, n0 + 32 * i, bh) : 0xFFFFFFFFu;
    // the warpgroup meets at its named barrier below: one decision for all
    ok = named_bar_and(bar_wg, 128, wait(c, bar_s, par_s));
    if (!ok) break;
    tc_fence_after();
    const bool masked =
        n0 + kBn - 1 - m0 > p.win_right || m0 + kBm - 1 - n0 > p.win_left || n0 + kBn > p.N;
    const float smax = masked ? tile_max<true>(p, tS, n0, qrow) : tile_max<false>(p, tS, n0, qrow);
    float m_tile = -INFINITY;  // row maximum of x = logit * log2e over this block
    if (smax > -INFINITY) {
      if (SOFTCAP) {
        const float ex = ex2_approx(smax * cap_in);
        m_tile = (1.f - 2.f * rcp_approx(ex + 1.f)) * cap_out;
      } else {
        m_tile = smax * c_log2;
      }
    }
    // move the shift when the maximum outgrows it by more than kRescale
    const bool need = m_tile > m_used + kRescale;
    if (__any_sync(0xffffffffu, need)) {
      const float m_new = need ? m_tile : m_used;
      const float f = need ? ex2_approx(m_used - m_new) : 1.f;  // 0 while m_used = -inf
      // O_q holds a nonzero row only once the shift is finite; P_q(t - 1) V
      // must have completed before the row is read
      if (__any_sync(0xffffffffu, need && m_used > -INFINITY) && t > 0) {
        if (!wait_warp(c, BAR_O_DONE + q, (t - 1) & 1)) ok = false;
        if (ok) {
          tc_fence_after();
          const uint64_t f2 = f2_make(f, f);
#pragma unroll
          for (int c32 = 0; c32 < D / 32; ++c32) {
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
    ok = named_bar_and(bar_wg, 128, ok);
    if (!ok) break;
    const float shift = m_used > -INFINITY ? m_used : 0.f;
    l += masked ? tile_p<SOFTCAP, true, DROP>(p, tS, n0, qrow, c_log2, cap_in, cap_out, shift,
                                              kbits)
                : tile_p<SOFTCAP, false, DROP>(p, tS, n0, qrow, c_log2, cap_in, cap_out, shift,
                                               kbits);
    tmem_wait_st();
    tc_fence_before();
    named_bar_sync(bar_wg, 128);
    if (r == 0) mbar_arrive(bar_addr(c, (kAlt ? BAR_P_FULL + (t & 1) : BAR_P_FULL + q)));
  }
  // ---- epilogue: O / l -> bf16 rows in the tile's Q buffer (free once its
  // last S GEMM is done, which precedes the last P V) -> TMA tensor store;
  // LSE in natural log
  // the one-tile form issues S(j + 1) before P(j) V, so P(nt - 2) V may still run:
  // its phase of O_DONE completes first (a wait on the parity of the last
  // phase would pass while the one before it is still open)
  if (ok && kAlt && nt >= 2) ok = wait(c, BAR_O_DONE + q, (nt - 2) & 1);
  if (ok) ok = wait(c, BAR_O_DONE + q, (nt - 1) & 1);
  if (!named_bar_and(bar_wg, 128, ok)) return;
  tc_fence_after();
  if (DROP) l *= p.drop.keep;  // the sums were of P / (1 - p)
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const uint64_t inv2 = f2_make(inv, inv);
  const uint32_t buf = sbase + (q ? L::kQ1 : L::kQ0);
#pragma unroll
  for (int c16 = 0; c16 < D / 16; ++c16) {
    const int col = c16 * 16;
    uint32_t raw[16];
    tmem_ld16(tO + col, raw);
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
  fence_proxy_async_smem();
  named_bar_sync(bar_wg, 128);
  if (r == 0) {
    for (int cb = 0; cb < D / 64; ++cb)
      tma_store_3d(to, buf + cb * 16384, 64 * cb, w.m0[q], w.bh);
    bulk_commit_group();
    bulk_wait_all();
  }
  if (qrow < p.N)
    p.lse[static_cast<long long>(w.bh) * p.N + qrow] =
        l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
}

// The keep mask of the one-tile form with dropout (warps 12-19, two per SM
// sub-partition). For each key block of the CTA's tiles, warp 12 + w and lane
// q draw the Philox calls of the query quad q (rows 4q .. 4q + 3, counter
// word 0 = (m0 + 4q) / 4) and of the 16 keys 16 w .. 16 w + 15 of the block:
// call g gives the four rows' words of key g, so the thread ends with 16 bits
// of each of its four rows, half of a 32-key word. Block g (counted over
// the CTA's tiles) goes to slot g mod 2 once the softmax has read block g - 2
// out of it; the softmax reads block g's words while the one after is drawn.
template <int D>
__device__ void mask_role(const Ctx& c, const Params& p, uint8_t* smem) {
  using L = LayoutOne<D>;
  const int lane = threadIdx.x & 31;
  const int mw = (static_cast<int>(threadIdx.x) >> 5) - 12;  // 16-key group of a block
  uint16_t* mask = reinterpret_cast<uint16_t*>(smem + L::kMask);
  const int n_tiles = p.pairs * p.B * p.H;
  int g = 0;  // global block index
  for (int r = 0;; ++r) {
    const int idx = cta_tile(r, n_tiles);
    if (idx < 0) return;
    const TileOne tl = tile_one(p, idx);
    const uint32_t qgrp = static_cast<uint32_t>(tl.m0 >> 2) + static_cast<uint32_t>(lane);
    const uint32_t bh = static_cast<uint32_t>(tl.bh);
    for (int t = 0; t < tl.nt; ++t, ++g) {
      const int slot = g & 1;
      if (g >= 2 && !wait(c, BAR_MASK_EMPTY + slot, ((g >> 1) - 1) & 1)) return;
      const uint32_t k0 = static_cast<uint32_t>((tl.j0 + t) * kBn + 16 * mw);
      uint32_t bits[4] = {0u, 0u, 0u, 0u};
      constexpr int kNB = 4;  // calls in flight
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

// Softmax of the one-tile form: the two warpgroups share the tile, warpgroup
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
__device__ void softmax_role_split(const Ctx& c, const Params& p, uint8_t* smem, uint32_t sbase,
                                   uint32_t tmem, const CUtensorMap* to) {
  using L = LayoutOne<D>;
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
  const int n_tiles = p.pairs * p.B * p.H;
  bool ok = true;
  int g = 0;  // global index of the tile's first key block
  for (int rr = 0, i = 0; ok; ++rr, ++i) {
    const int idx = cta_tile(rr, n_tiles);
    if (idx < 0) break;
    const TileOne tl = tile_one(p, idx);
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
      const float hmax = masked ? chunk_max_regs<true>(p, raw, key0, qrow)
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
      l += masked ? chunk_p_regs<SOFTCAP, true, DROP>(p, raw, dst, key0, qrow, c_log2, cap_in,
                                                      cap_out, shift, kb0, kb1)
                  : chunk_p_regs<SOFTCAP, false, DROP>(p, raw, dst, key0, qrow, c_log2, cap_in,
                                                       cap_out, shift, kb0, kb1);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_addr(c, BAR_P_FULL + (gb & 1)));  // one arrival per warp
    }
    // ---- epilogue. S(j + 1) is issued before P(j) V, so P(nt - 2) V may still
    // run: its phase of O_DONE completes first (a wait on the parity of the
    // last phase alone would pass while the one before it is still open).
    if (ok && nt >= 2) ok = wait(c, BAR_O_DONE, (g + nt - 2) & 1);
    if (ok) ok = wait(c, BAR_O_DONE, (g + nt - 1) & 1);
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
    named_bar_sync(bar_wg, 128);
    if (r == 0) {
      for (int cb = h * (D / 128); cb < (h + 1) * (D / 128); ++cb)
        tma_store_3d(to, buf + cb * 16384, 64 * cb, m0, tl.bh);
      bulk_commit_group();
      bulk_wait_read_all();
      mbar_arrive(bar_addr(c, BAR_Q_EMPTY + qs));
    }
    if (h == 0 && qrow < p.N)
      p.lse[static_cast<long long>(tl.bh) * p.N + qrow] =
          lt > 0.f ? (m_used + __log2f(lt)) * kLn2 : -INFINITY;
    g += nt;
  }
  // the O stores complete before the CTA exits
  if (r == 0) bulk_wait_all();
}

// ------------------------------------------------------------------ kernel
template <int D, bool SOFTCAP, bool DROP>
__global__ void __launch_bounds__(kThreadsFor<D, DROP>, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o, const Params p) {
  using L = LayoutFor<D>;
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
    if (kOneTile<D>) {  // P of a block: one arrival per softmax warp
      mbar_init(bar_addr(c, BAR_P_FULL), 8);
      mbar_init(bar_addr(c, BAR_P_FULL + 1), 8);
    }
    if (kOneTile<D>) {
      for (int sl = 0; sl < 2; ++sl) {
        mbar_init(bar_addr(c, BAR_Q_EMPTY + sl), 2);  // the two O-storing threads
        mbar_init(bar_addr(c, BAR_O_FREE + sl), 8);   // the softmax warps
      }
    }
    if (kMaskRole<D, DROP>) {
      for (int sl = 0; sl < 2; ++sl) {
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
  const Work w = work_of<D>(p);
  if (warp < 4) {
    if constexpr (kMaskRole<D, DROP>) setmaxnreg_dec<kRegsOtherDrop>();
    if (warp == 0) {
      if constexpr (kOneTile<D>)
        loader_role_one<D>(c, p, sbase, &tm_q, &tm_k, false);
      else
        producer_role<D>(c, w, sbase, &tm_q, &tm_k, &tm_v);
    } else if (warp == 1) {
      if constexpr (kOneTile<D>)
        mma_role_one<D>(c, p, sbase, tmem);
      else
        mma_role<D>(c, w, sbase, tmem);
    } else if (warp == 2) {
      if constexpr (kOneTile<D>) loader_role_one<D>(c, p, sbase, &tm_q, &tm_v, true);
    }
  } else if (warp < 12) {
    if constexpr (kMaskRole<D, DROP>) setmaxnreg_inc<kRegsSoftmaxDrop>();
    if constexpr (kOneTile<D>)
      softmax_role_split<D, SOFTCAP, DROP>(c, p, smem, sbase, tmem, &tm_o);
    else
      softmax_role<D, SOFTCAP, DROP>(c, p, w, sbase, tmem, &tm_o);
  } else {
    if constexpr (kMaskRole<D, DROP>) {
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
  if (!set_smem_limit_once(kern, LayoutFor<D>::kBytes, configured)) return ATTN_ERR_LAUNCH;
  long long grid = static_cast<long long>(p.pairs) * p.B * p.H;
  if (grid > 0x7fffffffLL) return ATTN_ERR_TOO_LARGE;
  if (kOneTile<D>) {  // persistent: one CTA per SM (or per tile, if fewer)
    const int sms = sm_count();
    if (sms <= 0) return ATTN_ERR_LAUNCH;
    if (grid > sms) grid = sms;
  }
  kern<<<static_cast<unsigned>(grid), kThreadsFor<D, DROP>, LayoutFor<D>::kBytes, stream>>>(
      tq, tk, tv, to, p);
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
  const bool one_tile = d == 256 ? kOneTile<256> : (d == 128 ? kOneTile<128> : kOneTile<64>);
  p.pairs = one_tile ? (N + kBm - 1) / kBm : ((N + kBm - 1) / kBm + 1) / 2;
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
