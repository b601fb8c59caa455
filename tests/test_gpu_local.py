"""GPU parity of the local (sliding-window) mask: attn_fwd_local,
attn_fwd_ref_local and attn_bwd_local against the fp64 oracle under the same
window, with the tolerances of the other parity tests (dQ, dK, dV max-rel
<= 2e-2 and Frobenius <= 5e-3; O max-rel <= 2e-2; LSE abs <= 1e-5).

Key j is visible to query i iff i - left <= j <= i + right (a negative bound
is unbounded), intersected with the causal mask when causal is set.
"""
import numpy as np
import pytest
import torch

import flashattention_attention_backward_gb300 as attn
from flashattention_attention_backward_gb300 import runner
from flashattention_attention_backward_gb300.inputs import WORKLOADS, Workload, make_inputs, \
    sample_slices
from oracle import attention_backward, attention_forward

pytestmark = pytest.mark.gpu

from parity_helpers import LSE_ABS, O_MAX_REL, check_grad, rel_max  # noqa: E402


def _w(name, B, H, H_kv, N, d, causal, softcap=0.0, sigma_qkv=1.0, seed=31):
    return Workload(name, B, H, H_kv, N, d, causal, softcap, sigma_qkv, 1.0, seed)


CASES = [
    # (workload, window): windows that cut through blocks, ragged tails, GQA,
    # both head dims, one-sided and two-sided bands, softcap, many units
    (_w("sliding_causal_d128", 1, 4, 2, 700, 128, True), (200, -1)),
    (_w("band_d64", 2, 2, 2, 513, 64, False), (64, 64)),
    (_w("future_only_d128", 1, 2, 1, 640, 128, False), (0, 300)),
    (_w("right_only_d128", 1, 2, 2, 384, 128, False), (-1, 37)),
    (_w("softcap_band_d64", 1, 2, 2, 333, 64, False, softcap=2.0, sigma_qkv=2.0), (100, 20)),
    (_w("causal_right_ignored_d64", 1, 3, 3, 300, 64, True), (150, 40)),
    (_w("narrow_causal_d128", 1, 2, 2, 520, 128, True), (5, -1)),
    (_w("many_units_causal_d128", 16, 8, 4, 300, 128, True), (130, -1)),
    (_w("wider_than_n_d64", 1, 2, 2, 256, 64, False), (5000, 5000)),
]


def _run(w, win, x=None):
    if x is None:
        x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, w.causal, w.softcap, window=win)
    o_r, lse_r = runner.forward(q, k, v, w.scale, w.causal, w.softcap, impl="ref", window=win)
    dq, dk, dv = runner.backward(q, k, v, o, do, lse, w.scale, w.causal, w.softcap, window=win)
    torch.cuda.synchronize()
    rc, status = attn.attn_device_status(clear=True)
    assert rc == 0 and status == 0, "device status %d (rc %d)" % (status, rc)
    out = {"o": o.cpu(), "lse": lse.cpu(), "o_ref": o_r.cpu(), "lse_ref": lse_r.cpu(),
           "dq": dq.cpu(), "dk": dk.cpu(), "dv": dv.cpu()}
    return x, out


def _check_forward(w, win, out, O, LSE, sl=(slice(None),)):
    for tag in ("", "_ref"):
        lse_err = float(np.abs(out["lse" + tag][sl].double().numpy() - LSE).max())
        assert lse_err <= LSE_ABS, "%s LSE%s abs err %.3e" % (w.name, tag, lse_err)
        o_err = rel_max(out["o" + tag][sl].double().numpy(), O)
        assert o_err <= O_MAX_REL, "%s O%s max-rel %.3e" % (w.name, tag, o_err)


@pytest.mark.parametrize("w,win", CASES, ids=lambda c: c.name if hasattr(c, "name") else str(c))
def test_local_against_oracle(w, win):
    x, out = _run(w, win)
    f64 = {n: x[n].double().numpy() for n in ("q", "k", "v", "do")}
    O, LSE = attention_forward(f64["q"], f64["k"], f64["v"], w.scale, w.causal, w.softcap,
                               window=win)
    _check_forward(w, win, out, O, LSE)
    dQ, dK, dV = attention_backward(f64["q"], f64["k"], f64["v"], f64["do"], w.scale, w.causal,
                                    w.softcap, window=win)
    check_grad("dQ", out["dq"], dQ)
    check_grad("dK", out["dk"], dK)
    check_grad("dV", out["dv"], dV)


def test_diagonal_window():
    """Window (0, 0): each query sees only its own key, so P = 1, O = V,
    dV = dO (summed over the group) and the exact dQ and dK vanish; the GPU
    result is then rounding noise far below the O(1) size of a gradient."""
    w = _w("diagonal_d64", 1, 4, 2, 300, 64, False)
    x, out = _run(w, (0, 0))
    f64 = {n: x[n].double().numpy() for n in ("q", "k", "v", "do")}
    O, LSE = attention_forward(f64["q"], f64["k"], f64["v"], w.scale, False, 0.0, window=(0, 0))
    _check_forward(w, (0, 0), out, O, LSE)
    _, _, dV = attention_backward(f64["q"], f64["k"], f64["v"], f64["do"], w.scale, False, 0.0,
                                  window=(0, 0))
    check_grad("dV", out["dv"], dV)
    assert float(out["dq"].float().abs().max()) <= 1e-3
    assert float(out["dk"].float().abs().max()) <= 1e-3


def test_unbounded_window_equals_plain_calls():
    """(-1, -1) is the plain call and (-1, 0) without causal is the causal
    mask: the same kernels on the same band, hence the same bits (dK and dV
    are summed on chip in a fixed order; dQ only up to atomic order)."""
    w = _w("equiv_d128", 1, 4, 2, 400, 128, False)
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    for causal, win in ((False, (-1, -1)), (True, (-1, 0))):
        o, lse = runner.forward(q, k, v, w.scale, causal)
        o_l, lse_l = runner.forward(q, k, v, w.scale, False, window=win)
        assert torch.equal(o, o_l) and torch.equal(lse, lse_l)
        o_r, lse_r = runner.forward(q, k, v, w.scale, causal, impl="ref")
        o_rl, lse_rl = runner.forward(q, k, v, w.scale, False, impl="ref", window=win)
        assert torch.equal(o_r, o_rl) and torch.equal(lse_r, lse_rl)
        dq, dk, dv = (t.clone() for t in runner.backward(q, k, v, o, do, lse, w.scale, causal))
        dq_l, dk_l, dv_l = runner.backward(q, k, v, o, do, lse, w.scale, False, window=win)
        torch.cuda.synchronize()
        assert torch.equal(dk, dk_l) and torch.equal(dv, dv_l)
        assert torch.allclose(dq.float(), dq_l.float(), rtol=1e-2, atol=1e-3)
    rc, status = attn.attn_device_status(clear=True)
    assert rc == 0 and status == 0


def test_sliding_window_causal_gqa_sampled():
    """The causal GQA shape (B=2, H=32, H_kv=8, N=4096, d=128) under a causal
    sliding window of 1024 keys, checked on a seeded sample of (batch, KV
    head) slices."""
    w = WORKLOADS["causal_gqa"]
    win = (1023, -1)
    x, out = _run(w, win)
    G = w.G
    for (b, g) in sample_slices(w, 2):
        heads = slice(g * G, (g + 1) * G)
        q = x["q"][b:b + 1, heads].double().numpy()
        do = x["do"][b:b + 1, heads].double().numpy()
        k = x["k"][b:b + 1, g:g + 1].double().numpy()
        v = x["v"][b:b + 1, g:g + 1].double().numpy()
        O, LSE = attention_forward(q, k, v, w.scale, True, 0.0, window=win)
        _check_forward(w, win, out, O[0], LSE[0], (b, heads))
        dQ, dK, dV = attention_backward(q, k, v, do, w.scale, True, 0.0, window=win)
        check_grad("dQ%s" % ((b, g),), out["dq"][b, heads], dQ[0])
        check_grad("dK%s" % ((b, g),), out["dk"][b, g], dK[0, 0])
        check_grad("dV%s" % ((b, g),), out["dv"][b, g], dV[0, 0])
        del O, LSE, dQ, dK, dV
