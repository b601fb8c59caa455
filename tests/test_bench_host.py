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


@pytest.mark.parametrize("B,H,N,d", [(2, 32, 4096, 128), (1, 2, 256, 64), (8, 16, 1024, 64)])
def test_hbm_bytes_of_the_memory_bound_kernels(B, H, N, d):
    """The algorithmic bytes of preprocess and finalize are the sizes of the
    tensors each one reads and writes once."""
    import torch

    def nbytes(shape, dtype):
        return torch.empty(shape, dtype=dtype, device="meta").nbytes

    o = do = nbytes((B, H, N, d), torch.bfloat16)
    dpsum = nbytes((B, H, N), torch.float32)
    dq_accum = nbytes((B, H, N, d), torch.float32)
    dq = nbytes((B, H, N, d), torch.bfloat16)
    assert bench.hbm_bytes_preprocess(B, H, N, d) == o + do + dpsum + dq_accum
    assert bench.hbm_bytes_finalize(B, H, N, d) == dq_accum + dq


def test_step_kernels_fractions():
    class W:
        B, H, N, d = 2, 32, 4096, 128
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0}
    k = bench.step_kernels(W, [0.05, 0.05], [0.5, 0.7], [0.04, 0.02], peaks)
    assert k["attn_bwd"]["ms"] == pytest.approx(0.6)
    pre = k["attn_bwd_preprocess"]
    assert pre["GB/s"] == pytest.approx(bench.hbm_bytes_preprocess(2, 32, 4096, 128) / 0.05e-3 / 1e9)
    assert pre["frac"] == pytest.approx(pre["GB/s"] / 6000.0)
    assert k["attn_bwd_finalize"]["ms"] == pytest.approx(0.03)
