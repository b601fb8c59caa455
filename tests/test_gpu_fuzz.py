"""Seeded random configurations of the whole path against the fp64 oracle.

Each case draws a head dimension (64, 128, 256), a sequence length that
often sits next to a block edge (127, 128, 129, 255, 256, 257, ...), a GQA
ratio, the causal mask, a softcap, a local window, dropout or the
deterministic dQ mode (the combinations the library offers), runs the
forward (tensor cores) and the backward through the C ABI, and compares O,
LSE, dQ, dK and dV with the oracle at the parity tolerances. The draws come
from a fixed seed, so the cases are the same on every run.

With a single key (N = 1) P = 1 and the exact dS = P (dP - D) is zero, so
the exact dQ and dK vanish; what the kernels return there is rounding: with
dropout O = V / (1 - p) is no bf16 value (P~ and O are each rounded to bf16
once), and dS keeps sum_c dO_c (O_c - V_c / (1 - p)) of it. Those cases are
checked for what the arithmetic fixes instead of element by element (see
_check_single_key).
"""
import numpy as np
import pytest
import torch

from flashattention_attention_backward_gb300 import runner
from flashattention_attention_backward_gb300.inputs import Workload, make_inputs
from oracle import attention_backward, attention_forward

pytestmark = pytest.mark.gpu

from parity_helpers import O_MAX_REL, check_grad, lse_tol, rel_max  # noqa: E402

U = 2.0 ** -8          # unit roundoff of bf16 (8 significant bits)
STRUCT = 4 * U         # a product rounded once to bf16, against a least-squares fit
LAMBDA = 6.0           # probabilistic bound: fails with probability < 2 exp(-18)

EDGES = [1, 2, 63, 64, 65, 127, 128, 129, 191, 255, 256, 257, 383, 384, 385, 511]


def _check_single_key(w, f64, O, dq, dk):
    """N = 1: the exact dS of head h is 0; the kernels' is a scalar r_h.

    Then dQ_h = beta_h K_0 and dK_0 = the sum over the group's heads of
    beta_h q_h, with beta_h = scale * r_h (times 1 - tanh^2 with a softcap),
    each up to one bf16 rounding of the product. r_h is what the rounding of
    O leaves of dP - D: the stored O_c is (x V_c)(1 + d0)(1 + d_c) with x =
    1 / (1 - p) for a kept key (1 without dropout), d0 a rounding of P~ to
    bf16 common to every c, and d_c the rounding of O_c itself (|d| <= u).
    So |r_h| <= u |sum_c dO_c O_c| + |sum_c dO_c O_c d_c|; the second sum is
    bounded by LAMBDA u ||dO o O||_2 in the probabilistic model of rounding
    (independent, mean-zero d_c; Higham and Mary 2019, "A new approach to
    probabilistic rounding error analysis", Hoeffding's inequality), since
    the worst case grows with d where a mistake (dP missing the factor 1 /
    (1 - p)) grows with sqrt(d) too. A dropped key has O = 0 and dP = 0:
    r = 0.
    """
    dq, dk = dq[:, :, 0], dk[:, :, 0]                       # [B, H, d], [B, H_kv, d]
    K = np.repeat(f64["k"][:, :, 0], w.G, axis=1)           # K_0 of each query head
    q = f64["q"][:, :, 0]
    beta = (dq * K).sum(-1) / np.maximum((K * K).sum(-1), 1e-30)       # [B, H]
    bK = beta[..., None] * K
    tiny = 2.0 ** -20 * np.abs(bK).max(axis=-1, keepdims=True) + 1e-30
    assert np.all(np.abs(dq - bK) <= STRUCT * np.abs(bK) + tiny), "dQ not parallel to K_0"
    bq = (beta[..., None] * q).reshape(w.B, w.H_kv, w.G, w.d)
    want, spread = bq.sum(2), np.abs(bq).sum(2)
    assert np.all(np.abs(dk - want) <= STRUCT * spread + 2.0 ** -20 * spread.max() + 1e-30), \
        "dK_0 is not the group's sum of beta_h q_h"
    a = f64["do"][:, :, 0] * O[:, :, 0]                     # dO_c O_c of each head
    r_max = (U * np.abs(a.sum(-1)) + LAMBDA * U * np.sqrt((a * a).sum(-1))
             + 1e-6 * np.abs(a).sum(-1))                    # + fp32 sums of D and dP
    bound = w.scale * (1 + U) ** 2 * r_max
    assert np.all(np.abs(beta) <= bound + 1e-30), (np.abs(beta).max(), bound.min())


def _draw(i):
    rng = np.random.default_rng(90210 + i)
    d = int(rng.choice([64, 128, 256]))
    N = int(rng.choice(EDGES)) if rng.random() < 0.6 else int(rng.integers(1, 700))
    H_kv = int(rng.choice([1, 2]))
    G = int(rng.choice([1, 2, 4]))
    B = int(rng.choice([1, 2]))
    causal = bool(rng.random() < 0.5)
    softcap = float(rng.choice([0.0, 0.0, 5.0]))
    sigma = 2.0 if softcap else 1.0
    mode = str(rng.choice(["plain", "plain", "window", "dropout", "deterministic"]))
    window = None
    if mode == "window":
        window = (int(rng.integers(0, N + 1)), -1 if causal else int(rng.integers(0, N + 1)))
    dropout = (float(np.float32(rng.choice([0.1, 0.3]))), int(rng.integers(0, 2**40))) \
        if mode == "dropout" else None
    w = Workload("fuzz%d" % i, B, H_kv * G, H_kv, N, d, causal, softcap, sigma, 1.0,
                 4000 + 17 * i)
    return w, mode, window, dropout


CASES = [_draw(i) for i in range(24)]


def _id(case):
    w, mode, window, dropout = case
    return "%s-d%d-N%d-G%d-%s%s%s" % (w.name, w.d, w.N, w.G, "c" if w.causal else "nc",
                                      "-cap" if w.softcap else "", "-" + mode)


@pytest.mark.parametrize("case", CASES, ids=[_id(c) for c in CASES])
def test_fuzz_against_oracle(case):
    w, mode, window, dropout = case
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, w.causal, w.softcap, dropout=dropout, window=window)
    dq, dk, dv = runner.backward(q, k, v, o, do, lse, w.scale, w.causal, w.softcap,
                                 deterministic=(mode == "deterministic"), dropout=dropout,
                                 window=window)
    torch.cuda.synchronize()
    import flashattention_attention_backward_gb300 as attn
    rc, status = attn.attn_device_status(clear=True)
    assert rc == 0 and status == 0, (rc, status)
    f64 = {n: x[n].double().numpy() for n in ("q", "k", "v", "do")}
    O, LSE = attention_forward(f64["q"], f64["k"], f64["v"], w.scale, w.causal, w.softcap,
                               dropout=dropout, window=window)
    assert float(np.abs(lse.cpu().double().numpy() - LSE).max()) <= lse_tol(LSE)
    assert rel_max(o.cpu().double().numpy(), O) <= O_MAX_REL
    dQ, dK, dV = attention_backward(f64["q"], f64["k"], f64["v"], f64["do"], w.scale, w.causal,
                                    w.softcap, dropout=dropout, window=window)
    check_grad("dV", dv.cpu(), dV)
    if w.N == 1:
        _check_single_key(w, f64, O, dq.cpu().double().numpy(), dk.cpu().double().numpy())
    else:
        check_grad("dQ", dq.cpu(), dQ)
        check_grad("dK", dk.cpu(), dK)
