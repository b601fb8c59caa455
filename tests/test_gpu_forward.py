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

from parity_helpers import LSE_ABS, O_MAX_REL, rel_max  # noqa: E402


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
    assert lse_err <= LSE_ABS, "LSE abs err %.3e" % lse_err
    o_err = rel_max(o.cpu().double().numpy(), O)
    assert o_err <= O_MAX_REL, "O max-rel %.3e" % o_err
    # the two GPU forwards agree as closely as bf16 outputs allow
    assert float((lse - lse_r).abs().max()) <= 2 * LSE_ABS
    assert rel_max(o.cpu().double().numpy(), o_r.cpu().double().numpy()) <= O_MAX_REL
