"""Host-side arithmetic of bench.py (no GPU): the count of visible (query,
key) pairs that the local-window FLOP figures are based on, against a
brute-force count of the band on small sizes."""
import numpy as np
import pytest

import bench


def _brute(N, causal, left, right):
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    ok = np.ones((N, N), dtype=bool)
    if left >= 0:
        ok &= j >= i - left
    if right >= 0:
        ok &= j <= i + right
    if causal:
        ok &= j <= i
    return int(ok.sum())


@pytest.mark.parametrize("N", [1, 7, 128, 300])
@pytest.mark.parametrize("causal,left,right",
                         [(False, -1, -1), (True, -1, -1), (True, 5, -1), (False, 3, 9),
                          (False, 0, 0), (True, 1023, 40), (False, -1, 2), (False, 400, 400)])
def test_visible_pairs_matches_brute_force(N, causal, left, right):
    assert bench.visible_pairs(N, causal, left, right) == _brute(N, causal, left, right)


def test_visible_pairs_closed_forms():
    N = 4096
    assert bench.visible_pairs(N, False, -1, -1) == N * N
    assert bench.visible_pairs(N, True, -1, -1) == N * (N + 1) // 2
    L = 1023  # causal window of L + 1 keys: row i sees min(i, L) + 1 keys
    assert bench.visible_pairs(N, True, L, -1) == (L + 1) * (L + 2) // 2 + (N - L - 1) * (L + 1)
