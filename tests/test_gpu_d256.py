"""GPU parity at head dimension 256 against the fp64 oracle, with the
tolerances of the other parity tests: the backward (its own kernel: a CTA
accumulates one half of d for 128 keys over 64-query tiles) with its local,
dropout and deterministic forms, and the tensor-core forward (one query tile
per CTA), which produces O and LSE for the backward cases."""
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


# ---------------------------------------------------------------- forward
FWD_CASES = CASES + [
    # sharper scores (logit std about 9): the running shift moves often
    _w("d256_sharp", 1, 2, 2, 700, False, sigma_qkv=3.0),
    _w("d256_softcap30_causal", 1, 2, 1, 384, True, softcap=30.0, sigma_qkv=2.0),
]


@pytest.mark.parametrize("w", FWD_CASES, ids=lambda w: w.name)
def test_d256_forward_tensor_cores(w):
    """attn_fwd at d = 256 (one query tile per CTA, two S buffers) against
    the oracle and against the fp32 attn_fwd_ref."""
    import numpy as np
    from flashattention_attention_backward_gb300 import runner
    from oracle import attention_forward
    from parity_helpers import O_MAX_REL, lse_tol, rel_max
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o, lse = runner.forward(q, k, v, w.scale, w.causal, w.softcap, impl="tc")
    o_r, lse_r = runner.forward(q, k, v, w.scale, w.causal, w.softcap, impl="ref")
    torch.cuda.synchronize()
    import flashattention_attention_backward_gb300 as attn
    rc, status = attn.attn_device_status(clear=True)
    assert rc == 0 and status == 0
    O, LSE = attention_forward(*(x[n].double().numpy() for n in ("q", "k", "v")), w.scale,
                               w.causal, w.softcap)
    lse_err = float(np.abs(lse.cpu().double().numpy() - LSE).max())
    assert lse_err <= lse_tol(LSE), "LSE abs err %.3e" % lse_err
    o_err = rel_max(o.cpu().double().numpy(), O)
    assert o_err <= O_MAX_REL, "O max-rel %.3e" % o_err
    assert float((lse - lse_r).abs().max()) <= 2 * lse_tol(LSE)
    assert rel_max(o.cpu().double().numpy(), o_r.cpu().double().numpy()) <= O_MAX_REL


@pytest.mark.parametrize("causal", [False, True])
def test_d256_forward_growing_logits(causal):
    """K rows scaled by 1 + 6 j / N along the sequence: nearly every key block
    raises the row maxima, so the O accumulator (256 columns) is rescaled
    repeatedly."""
    import numpy as np
    from flashattention_attention_backward_gb300 import runner
    from oracle import attention_forward
    from parity_helpers import O_MAX_REL, lse_tol, rel_max
    w = _w("d256_ramp", 1, 2, 1, 1024, causal, seed=47)
    x = make_inputs(w)
    ramp = 1.0 + 6.0 * torch.arange(w.N, dtype=torch.float32) / w.N
    x["k"] = (x["k"].float() * ramp[None, None, :, None]).to(torch.bfloat16)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o, lse = runner.forward(q, k, v, w.scale, causal, impl="tc")
    torch.cuda.synchronize()
    O, LSE = attention_forward(*(x[n].double().numpy() for n in ("q", "k", "v")), w.scale,
                               causal)
    assert float(np.abs(lse.cpu().double().numpy() - LSE).max()) <= lse_tol(LSE)
    assert rel_max(o.cpu().double().numpy(), O) <= O_MAX_REL


@pytest.mark.parametrize("win,causal", [((150, -1), True), ((40, 60), False)])
def test_d256_forward_local_window(win, causal):
    """attn_fwd_local at d = 256: key blocks outside the band are skipped,
    those at its edge masked."""
    import numpy as np
    from flashattention_attention_backward_gb300 import runner
    from oracle import attention_forward
    from parity_helpers import O_MAX_REL, lse_tol, rel_max
    w = _w("d256_fwd_window", 1, 2, 1, 520, causal, seed=49)
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o, lse = runner.forward(q, k, v, w.scale, causal, window=win)
    torch.cuda.synchronize()
    O, LSE = attention_forward(*(x[n].double().numpy() for n in ("q", "k", "v")), w.scale,
                               causal, 0.0, window=win)
    assert float(np.abs(lse.cpu().double().numpy() - LSE).max()) <= lse_tol(LSE)
    assert rel_max(o.cpu().double().numpy(), O) <= O_MAX_REL


# ---------------------------------------------------------------- dropout, deterministic dQ
@pytest.mark.parametrize("w,p_drop,seed", [
    (_w("d256_drop_causal_gqa", 1, 4, 2, 333, True), 0.1, 1234),
    (_w("d256_drop_softcap", 2, 2, 1, 200, False, softcap=5.0, sigma_qkv=2.0), 0.25, 2**40 + 7),
], ids=lambda c: getattr(c, "name", str(c)))
def test_d256_dropout_against_oracle(w, p_drop, seed):
    """attn_fwd_dropout, attn_fwd_ref_dropout and attn_bwd_dropout at
    d = 256 with the same (p, seed) as the oracle."""
    import numpy as np
    from flashattention_attention_backward_gb300 import runner
    from oracle import attention_backward, attention_forward
    from parity_helpers import LSE_ABS, O_MAX_REL, check_grad, rel_max
    p32 = float(np.float32(p_drop))
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, w.causal, w.softcap, dropout=(p32, seed))
    o_r, lse_r = runner.forward(q, k, v, w.scale, w.causal, w.softcap, dropout=(p32, seed),
                                impl="ref")
    dq, dk, dv = runner.backward(q, k, v, o, do, lse, w.scale, w.causal, w.softcap,
                                 dropout=(p32, seed))
    torch.cuda.synchronize()
    import flashattention_attention_backward_gb300 as attn
    rc, status = attn.attn_device_status(clear=True)
    assert rc == 0 and status == 0
    f64 = {n: x[n].double().numpy() for n in ("q", "k", "v", "do")}
    O, LSE = attention_forward(f64["q"], f64["k"], f64["v"], w.scale, w.causal, w.softcap,
                               dropout=(p32, seed))
    for o_, lse_ in ((o, lse), (o_r, lse_r)):
        assert float(np.abs(lse_.cpu().double().numpy() - LSE).max()) <= LSE_ABS
        assert rel_max(o_.cpu().double().numpy(), O) <= O_MAX_REL
    dQ, dK, dV = attention_backward(f64["q"], f64["k"], f64["v"], f64["do"], w.scale, w.causal,
                                    w.softcap, dropout=(p32, seed))
    check_grad("dQ", dq.cpu(), dQ)
    check_grad("dK", dk.cpu(), dK)
    check_grad("dV", dv.cpu(), dV)


@pytest.mark.parametrize("w", [
    _w("d256_det_causal_gqa", 1, 4, 2, 333, True),
    _w("d256_det_noncausal_softcap", 2, 2, 1, 300, False, softcap=2.0, sigma_qkv=2.0),
], ids=lambda w: w.name)
def test_d256_deterministic(w):
    """attn_bwd_deterministic at d = 256: parity with the oracle, dQ
    identical bit for bit across two runs, dK and dV identical to the
    default path."""
    from flashattention_attention_backward_gb300 import runner
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, w.causal, w.softcap)
    outs = []
    for _ in range(2):
        dq, dk, dv = runner.backward(q, k, v, o, do, lse, w.scale, w.causal, w.softcap,
                                     deterministic=True)
        outs.append((dq.clone(), dk.clone(), dv.clone()))
    dq_d, dk_d, dv_d = runner.backward(q, k, v, o, do, lse, w.scale, w.causal, w.softcap)
    torch.cuda.synchronize()
    import flashattention_attention_backward_gb300 as attn
    rc, status = attn.attn_device_status(clear=True)
    assert rc == 0 and status == 0
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], dk_d) and torch.equal(outs[0][2], dv_d)
    compare_full(w, x, {"o": o.cpu(), "lse": lse.cpu(), "dq": outs[0][0].cpu(),
                        "dk": outs[0][1].cpu(), "dv": outs[0][2].cpu()})
