"""Bit-exact check of the dropout keep mask between the CUDA kernels and the
oracle.

The backward replays the forward's keep mask Z ("解析 FlashAttention（3）"
§3.3 and Algorithm 4 of §4: the same Z_ij drops P in the forward and dP in
the backward). Whether an element is kept is an integer decision, so the
kernels' masks must equal the oracle's element for element, not only within
the float tolerances of the gradients. Each mask is read out through a
one-hot operand:

* forward: V is one-hot over d keys (64, 128 or 256), V_j = e_(j - j0) for
  j0 <= j < j0 + d and 0 elsewhere. Then O[i, c] = P~[i, j0 + c] with
  P~ = P o Z / (1 - p), so O is zero exactly where the key is dropped (or
  masked by causality) and nonzero where it is kept: inputs of small spread
  keep every P far from underflow.
* backward: dO of one query head h* per KV group is one-hot over a query
  block, dO_i = e_(i - i0), and zero for the group's other heads. Then
  dV[j, c] = P~[i0 + c, j] of head h*, so dV's zero pattern is the mask of
  head b * H + h*, transposed.

Ragged N (333: the last quad of rows holds one row), several key and query
blocks (block-aligned and straddling), b * H + h > 0 and a seed >= 2^32 are
covered; both tensor-core kernels and the fp32 forward are checked.
"""
import numpy as np
import pytest
import torch

from flashattention_attention_backward_gb300 import runner
from flashattention_attention_backward_gb300.inputs import Workload, make_inputs
from oracle.philox import dropout_keep_mask

pytestmark = pytest.mark.gpu

P_DROP = float(np.float32(0.2))
SEED = 2**40 + 7


def _inputs(B, H, H_kv, N, d, seed_base):
    w = Workload("mask", B, H, H_kv, N, d, False, sigma_qkv=0.5, seed_base=seed_base)
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    return w, x["q"].to(dev), x["k"].to(dev), x["v"].to(dev)


def _visible(N, causal):
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    return (j <= i) if causal else np.ones((N, N), dtype=bool)


def _one_hot_rows(shape, start, d, device):
    """[..., N, d] zeros with row start + c equal to e_c for the c that fit."""
    t = torch.zeros(shape, dtype=torch.bfloat16)
    N = shape[-2]
    for c in range(min(d, N - start)):
        t[..., start + c, c] = 1.0
    return t.to(device)


@pytest.mark.parametrize("impl", ["tc", "ref"])
@pytest.mark.parametrize("N,d,causal,j0s", [
    (333, 128, False, (0, 100, 256)),
    (333, 128, True, (0, 128, 205)),
    (200, 64, False, (0, 64, 136)),
    (200, 64, True, (37, 136)),
    (333, 256, False, (0, 100)),
    (333, 256, True, (77,)),
])
def test_forward_keep_mask_bit_exact(impl, N, d, causal, j0s):
    B, H, H_kv = 2, 2, 1
    w, q, k, _ = _inputs(B, H, H_kv, N, d, seed_base=4242 + N + d)
    vis = _visible(N, causal)
    for j0 in j0s:
        v = _one_hot_rows((B, H_kv, N, d), j0, d, q.device)
        o, _ = runner.forward(q, k, v, w.scale, causal, dropout=(P_DROP, SEED), impl=impl)
        torch.cuda.synchronize()
        nz = (o.float() != 0).cpu().numpy()
        width = min(d, N - j0)
        for b in range(B):
            for h in range(H):
                keep = dropout_keep_mask(SEED, b * H + h, N, N, P_DROP)
                want = (keep & vis)[:, j0:j0 + width]
                got = nz[b, h, :, :width]
                bad = np.argwhere(got != want)
                assert bad.size == 0, ("b=%d h=%d j0=%d: %d mismatches, first (i, c) %s"
                                       % (b, h, j0, len(bad), bad[:4].tolist()))
                assert not nz[b, h, :, width:].any()
    import flashattention_attention_backward_gb300 as attn
    rc, status = attn.attn_device_status(clear=True)
    assert rc == 0 and status == 0


@pytest.mark.parametrize("N,d,causal,i0s", [
    (333, 128, False, (0, 100, 256)),
    (333, 128, True, (128, 205)),
    (200, 64, False, (0, 136)),
    (200, 64, True, (64, 150)),
    (333, 256, False, (0, 77)),
    (333, 256, True, (0,)),
])
def test_backward_keep_mask_bit_exact(N, d, causal, i0s):
    B, H, H_kv = 2, 4, 2
    G = H // H_kv
    w, q, k, v = _inputs(B, H, H_kv, N, d, seed_base=5353 + N + d)
    o, lse = runner.forward(q, k, v, w.scale, causal, dropout=(P_DROP, SEED))
    vis = _visible(N, causal)
    for i0 in i0s:
        do = torch.zeros((B, H, N, d), dtype=torch.bfloat16)
        hstar = [g * G + (g + i0) % G for g in range(H_kv)]  # one head per group
        for b in range(B):
            for g in range(H_kv):
                do[b, hstar[g]] = _one_hot_rows((N, d), i0, d, "cpu")
        do = do.to(q.device)
        _, _, dv = runner.backward(q, k, v, o, do, lse, w.scale, causal, dropout=(P_DROP, SEED))
        torch.cuda.synchronize()
        nz = (dv.float() != 0).cpu().numpy()
        width = min(d, N - i0)
        for b in range(B):
            for g in range(H_kv):
                h = hstar[g]
                keep = dropout_keep_mask(SEED, b * H + h, N, N, P_DROP)
                want = (keep & vis)[i0:i0 + width, :].T
                got = nz[b, g, :, :width]
                bad = np.argwhere(got != want)
                assert bad.size == 0, ("b=%d h=%d i0=%d: %d mismatches, first (j, c) %s"
                                       % (b, h, i0, len(bad), bad[:4].tolist()))
                assert not nz[b, g, :, width:].any()
    import flashattention_attention_backward_gb300 as attn
    rc, status = attn.attn_device_status(clear=True)
    assert rc == 0 and status == 0
