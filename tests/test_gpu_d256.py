"""GPU parity of the head-dimension-256 backward (its own kernel: a CTA
accumulates one half of d for 128 keys over 64-query tiles) against the fp64
oracle, with the tolerances of the other parity tests; O and LSE come from
attn_fwd_ref (d = 256)."""
import pytest
import torch

from flashattention_attention_backward_gb300.inputs import Workload, make_inputs, sample_slices

pytestmark = pytest.mark.gpu

from parity_helpers import compare_full, compare_slices, run_gpu  # noqa: E402


def _w(name, B, H, H_kv, N, causal, softcap=0.0, sigma_qkv=1.0, seed=41):
    return Workload(name, B, H, H_kv, N, 256, causal, softcap, sigma_qkv, 1.0, seed)


CASES = [
    _w("d256_noncausal", 1, 2, 2, 256, False),
    _w("d256_causal_ragged_gqa", 1, 4, 2, 333, True),
    _w("d256_softcap_sat", 2, 2, 1, 200, False, softcap=2.0, sigma_qkv=2.0),
    _w("d256_single_row", 1, 1, 1, 1, True),
    _w("d256_many_blocks", 3, 4, 2, 640, True),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_d256_against_oracle(w):
    x, out = run_gpu(w)
    compare_full(w, x, out)


def test_d256_causal_gqa_sampled():
    """B=2, H=16, H_kv=4, N=2048, d=256 causal on two sampled (batch, KV
    head) slices."""
    w = _w("d256_gqa_2048", 2, 16, 4, 2048, True, seed=43)
    x, out = run_gpu(w)
    compare_slices(w, x, out, sample_slices(w, 2))


def test_d256_local_window():
    """The local band reaches the d = 256 kernel through attn_bwd_local."""
    import numpy as np
    from flashattention_attention_backward_gb300 import runner
    from oracle import attention_backward
    from parity_helpers import check_grad
    w = _w("d256_window", 1, 2, 1, 520, True)
    win = (150, -1)
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, True, window=win)
    dq, dk, dv = runner.backward(q, k, v, o, do, lse, w.scale, True, window=win)
    torch.cuda.synchronize()
    f64 = {n: x[n].double().numpy() for n in ("q", "k", "v", "do")}
    dQ, dK, dV = attention_backward(f64["q"], f64["k"], f64["v"], f64["do"], w.scale, True, 0.0,
                                    window=win)
    check_grad("dQ", dq.cpu(), dQ)
    check_grad("dK", dk.cpu(), dK)
    check_grad("dV", dv.cpu(), dV)
    assert np.isfinite(lse.cpu().numpy()).all()
