"""GPU parity of the tensor-core forward (attn_fwd) against the fp64 oracle
and against the plain fp32 forward (attn_fwd_ref): O max|err|/max|ref| <=
2e-2, LSE abs <= 1e-5. (Every other GPU test also runs attn_fwd, through
runner.forward, before the backward.)"""
import numpy as np
import pytest
import torch

from flashattention_attention_backward_gb300 import runner
from flashattention_attention_backward_gb300.inputs import Workload, make_inputs
from oracle import attention_forward

pytestmark = pytest.mark.gpu

from parity_helpers import O_MAX_REL, lse_tol, rel_max  # noqa: E402


def _w(name, B, H, H_kv, N, d, causal, softcap=0.0, sigma_qkv=1.0, seed=7):
    return Workload(name, B, H, H_kv, N, d, causal, softcap, sigma_qkv, 1.0, seed)


CASES = [
    _w("d128_causal_ragged", 1, 4, 2, 333, 128, True),
    _w("d128_noncausal", 2, 2, 1, 256, 128, False),
    _w("d64_causal", 1, 3, 3, 300, 64, True),
    _w("d64_softcap_sat", 1, 2, 2, 200, 64, False, softcap=2.0, sigma_qkv=2.0),
    _w("d128_softcap30_causal", 1, 2, 1, 384, 128, True, softcap=30.0, sigma_qkv=2.0),
    _w("single_row", 1, 1, 1, 1, 64, True),
    _w("many_blocks", 3, 8, 2, 1030, 128, True),
    # sharper scores (logit std about 9): later key blocks often raise a row
    # maximum past the one-pass forward's rescale threshold
    _w("sharp_d128", 1, 2, 2, 700, 128, False, sigma_qkv=3.0),
    _w("sharp_d64_causal", 1, 3, 1, 900, 64, True, sigma_qkv=3.0),
    # an odd number of query blocks: the last CTA's second tile is empty
    _w("odd_blocks_d128", 2, 2, 1, 3 * 128, 128, True),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fwd_against_oracle(w):
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o, lse = runner.forward(q, k, v, w.scale, w.causal, w.softcap, impl="tc")
    o_r, lse_r = runner.forward(q, k, v, w.scale, w.causal, w.softcap, impl="ref")
    torch.cuda.synchronize()
    O, LSE = attention_forward(*(x[n].double().numpy() for n in ("q", "k", "v")), w.scale,
                               w.causal, w.softcap)
    lse_err = float(np.abs(lse.cpu().double().numpy() - LSE).max())
    assert lse_err <= lse_tol(LSE), "LSE abs err %.3e" % lse_err
    o_err = rel_max(o.cpu().double().numpy(), O)
    assert o_err <= O_MAX_REL, "O max-rel %.3e" % o_err
    # the two GPU forwards agree as closely as bf16 outputs allow
    assert float((lse - lse_r).abs().max()) <= 2 * lse_tol(LSE)
    assert rel_max(o.cpu().double().numpy(), o_r.cpu().double().numpy()) <= O_MAX_REL


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_growing_logits(causal):
    """K rows scaled by 1 + 6 j / N along the sequence, so that nearly every
    key block raises the row maxima (logit std from 1 to 7): the one-pass
    forward must rescale its O accumulator repeatedly and still agree with
    the oracle and with the fp32 forward on the same bf16 inputs."""
    w = _w("ramp", 1, 2, 1, 1024, 128, causal, seed=11)
    x = make_inputs(w)
    ramp = 1.0 + 6.0 * torch.arange(w.N, dtype=torch.float32) / w.N
    x["k"] = (x["k"].float() * ramp[None, None, :, None]).to(torch.bfloat16)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o, lse = runner.forward(q, k, v, w.scale, causal, impl="tc")
    o_r, lse_r = runner.forward(q, k, v, w.scale, causal, impl="ref")
    torch.cuda.synchronize()
    O, LSE = attention_forward(*(x[n].double().numpy() for n in ("q", "k", "v")), w.scale,
                               causal)
    assert float(np.abs(lse.cpu().double().numpy() - LSE).max()) <= lse_tol(LSE)
    assert float(np.abs(lse_r.cpu().double().numpy() - LSE).max()) <= lse_tol(LSE)
    assert rel_max(o.cpu().double().numpy(), O) <= O_MAX_REL
    assert rel_max(o_r.cpu().double().numpy(), O) <= O_MAX_REL
