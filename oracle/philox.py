"""Philox4x32-10 counter-based generator and the dropout keep mask, for the
oracle. Test infrastructure only (see the package docstring).

Generator (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
1, 2, 3", SC 2011, Philox4x32 with 10 rounds): a 128-bit counter
(c0, c1, c2, c3) and a 64-bit key (k0, k1). One round:
    hi0:lo0 = 0xD2511F53 * c0      hi1:lo1 = 0xCD9E8D57 * c2   (32x32 -> 64)
    (c0, c1, c2, c3) <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0)
and the key is bumped by the Weyl constants (0x9E3779B9, 0xBB67AE85)
between rounds. The output is the counter after ten rounds.

Dropout keep mask (dropout as the pages apply it to P,
"解析 FlashAttention（3）" §3.3 and Algorithm 4 of §4): element (query i, key j)
of query head bh is kept iff the 32-bit word (i mod 4) of
Philox(counter = (floor(i / 4), j, bh, 0), key = (seed mod 2^32, seed >> 32))
is >= round(p * 2^32); a kept element is scaled by 1 / (1 - p).
"""
import math

import numpy as np

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = np.uint64(0x9E3779B9)
_W1 = np.uint64(0xBB67AE85)
_MASK = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10: arrays (or scalars) of 32-bit counters and
    keys -> four uint32 arrays."""
    c = [np.asarray(x, dtype=np.uint64) & _MASK for x in (c0, c1, c2, c3)]
    k0 = np.asarray(k0, dtype=np.uint64) & _MASK
    k1 = np.asarray(k1, dtype=np.uint64) & _MASK
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        p0 = _M0 * c[0]
        p1 = _M1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return [x.astype(np.uint32) for x in c]


def keep_threshold(p_drop):
    """32-bit threshold: a word u keeps its element iff u >= threshold, for
    the float32 value of p_drop (what the library receives), rounded half
    up."""
    t = float(np.float32(p_drop)) * 4294967296.0
    return int(min(max(math.floor(t + 0.5), 0), 4294967295))


def dropout_keep_mask(seed, bh, n_q, n_k, p_drop):
    """Boolean [n_q, n_k] keep mask of query head `bh` (= b * H + h)."""
    i = np.arange(n_q, dtype=np.uint64)[:, None]
    j = np.arange(n_k, dtype=np.uint64)[None, :]
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    words = philox4x32_10(i >> np.uint64(2), np.broadcast_to(j, (n_q, n_k)), bh, 0,
                          seed & 0xFFFFFFFF, seed >> 32)
    sel = (i & np.uint64(3)).astype(np.int64)
    w = np.choose(np.broadcast_to(sel, (n_q, n_k)), words)
    return w >= np.uint32(keep_threshold(p_drop))
