// Philox4x32-10 counter-based generator on the device, written from its
// published definition (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011): a 128-bit counter and a 64-bit
// key; each of the ten rounds multiplies counter words 0 and 2 by
// 0xD2511F53 and 0xCD9E8D57 (32 x 32 -> 64 bits) and mixes
//   (c0, c1, c2, c3) <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0),
// and the key is bumped by 0x9E3779B9, 0xBB67AE85 between rounds.
//
// Dropout keep mask used by the kernels ("解析 FlashAttention（3）" §3.3 and
// Algorithm 4 of §4): element (query i, key j) of query head bh is kept iff
// word (i mod 4) of Philox(counter = (i / 4, j, bh, 0), key = (seed_lo,
// seed_hi)) is >= the threshold round(p * 2^32); kept elements are scaled by
// 1 / (1 - p). One call gives the words of four consecutive queries of a
// key, which is how the backward (thread = key row) walks its columns.
#pragma once

#include <cstdint>

namespace attn {

struct PhiloxOut {
  uint32_t w[4];
};

__device__ __forceinline__ PhiloxOut philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                                   uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int rnd = 0; rnd < 10; ++rnd) {
    if (rnd > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  PhiloxOut o;
  o.w[0] = c0;
  o.w[1] = c1;
  o.w[2] = c2;
  o.w[3] = c3;
  return o;
}

// NB independent calls of the same key in one pass: rounds outermost, so the
// multiplies of different calls interleave (one call alone is a chain of ten
// dependent rounds, and the multiply pipe is the bound). ctr[u] holds call
// u's counter on entry and its four output words on return. UNROLL rounds
// are unrolled: all ten suit a small batch, whose rounds are too short to
// hide their own latency; a rolled loop suits a large batch in a kernel
// whose other warps' loops need the instruction cache (fully unrolled, a
// batch of eight would take much of it).
template <int NB, int UNROLL>
__device__ __forceinline__ void philox4x32_10_batch(uint32_t (&ctr)[NB][4], uint32_t k0,
                                                    uint32_t k1) {
#pragma unroll(UNROLL)
  for (int rnd = 0; rnd < 10; ++rnd) {
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const uint32_t hi0 = __umulhi(0xD2511F53u, ctr[u][0]), lo0 = 0xD2511F53u * ctr[u][0];
      const uint32_t hi1 = __umulhi(0xCD9E8D57u, ctr[u][2]), lo1 = 0xCD9E8D57u * ctr[u][2];
      const uint32_t n0 = hi1 ^ ctr[u][1] ^ k0, n2 = hi0 ^ ctr[u][3] ^ k1;
      ctr[u][0] = n0;
      ctr[u][1] = lo1;
      ctr[u][2] = n2;
      ctr[u][3] = lo0;
    }
    k0 += 0x9E3779B9u;  // the key of the next round
    k1 += 0xBB67AE85u;
  }
}

// Dropout parameters shared by the kernels (p_drop > 0 enables it).
struct Dropout {
  uint32_t seed_lo, seed_hi;
  uint32_t threshold;   // keep iff word >= threshold
  float inv_keep;       // 1 / (1 - p)
  float keep;           // 1 - p
  float log2_inv_keep;  // log2(1 / (1 - p)): the tensor-core forward adds it to
                        // the exponent, so exp2 gives P / (1 - p) directly
};

}  // namespace attn
