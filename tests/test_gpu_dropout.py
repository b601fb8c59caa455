"""GPU parity with dropout (Philox keep mask, drawn independently on each
side): attn_fwd_dropout (tensor cores), attn_fwd_ref_dropout (fp32) and
attn_bwd_dropout against the fp64 oracle with the same (p_drop, seed). The
keep decision is an integer one taken from the same 32-bit words on both
sides, so any mask mismatch shows up as a gross error; the float tolerances
are the usual ones."""
import numpy as np
import pytest
import torch

from flashattention_attention_backward_gb300 import runner
from flashattention_attention_backward_gb300.inputs import Workload, make_inputs
from oracle import attention_backward, attention_forward

pytestmark = pytest.mark.gpu

from parity_helpers import LSE_ABS, O_MAX_REL, check_grad, rel_max  # noqa: E402


def _w(name, B, H, H_kv, N, d, causal, softcap=0.0, sigma_qkv=1.0, seed=21):
    return Workload(name, B, H, H_kv, N, d, causal, softcap, sigma_qkv, 1.0, seed)


CASES = [
    (_w("drop_d128_causal_gqa", 1, 4, 2, 300, 128, True), 0.1, 1234),
    (_w("drop_d64_noncausal", 2, 2, 2, 256, 64, False), 0.5, 99),
    (_w("drop_d128_softcap", 1, 2, 1, 200, 128, False, softcap=5.0, sigma_qkv=2.0), 0.25,
     2**40 + 7),
    (_w("drop_many_units_d128", 16, 8, 4, 260, 128, True), 0.2, 5),
]


@pytest.mark.parametrize("w,p_drop,seed", CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_dropout_fwd_bwd_against_oracle(w, p_drop, seed):
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


def test_dropout_zero_matches_plain():
    w = _w("drop0", 1, 2, 2, 200, 128, True)
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    for impl in ("ref", "tc"):
        o, lse = runner.forward(q, k, v, w.scale, w.causal, w.softcap, impl=impl)
        o0, lse0 = runner.forward(q, k, v, w.scale, w.causal, w.softcap, dropout=(0.0, 3),
                                  impl=impl)
        assert torch.equal(o, o0) and torch.equal(lse, lse0)
    a = [t.clone() for t in runner.backward(q, k, v, o, do, lse, w.scale, w.causal, w.softcap)]
    b = runner.backward(q, k, v, o, do, lse, w.scale, w.causal, w.softcap, dropout=(0.0, 3))
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_dropout_fwd_keep_rate_and_rows():
    """attn_fwd_dropout on a key-independent V (every row of V equal to 1):
    O_i = (sum of the kept P_ij) / (1 - p), whose mean over many rows is 1,
    and rows of different quads of lanes draw different masks."""
    w = _w("drop_rate", 1, 1, 1, 1024, 64, False, seed=5)
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k = (x[n].to(dev) for n in ("q", "k"))
    v = torch.ones_like(k)
    o, _ = runner.forward(q, k, v, w.scale, False, dropout=(0.3, 77))
    torch.cuda.synchronize()
    row = o[0, 0, :, 0].float()
    assert abs(float(row.mean()) - 1.0) < 0.03
    assert float(row.std()) > 0.01  # the mask differs from row to row


def test_dropout_causal_gqa_full_size_sampled():
    """The causal GQA workload at full size (B=2, H=32, H_kv=8, N=4096,
    d=128) with p = 0.1, the launch configuration the bench times: O and LSE
    of attn_fwd_dropout and dQ, dK, dV of attn_bwd_dropout against the oracle
    on one seeded (batch, KV head) slice. The oracle runs per query head with
    the keep mask of the library's head index b * H + h."""
    from flashattention_attention_backward_gb300.inputs import WORKLOADS, sample_slices
    from oracle.attention import head_backward
    from oracle.philox import dropout_keep_mask
    w = WORKLOADS["causal_gqa"]
    p32, seed = float(np.float32(0.1)), 1234
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, True, dropout=(p32, seed))
    dq, dk, dv = runner.backward(q, k, v, o, do, lse, w.scale, True, dropout=(p32, seed))
    torch.cuda.synchronize()
    import flashattention_attention_backward_gb300 as attn
    rc, status = attn.attn_device_status(clear=True)
    assert rc == 0 and status == 0
    G = w.G
    for (b, g) in sample_slices(w, 1):
        kk = x["k"][b, g].double().numpy()
        vv = x["v"][b, g].double().numpy()
        dK = np.zeros_like(kk)
        dV = np.zeros_like(vv)
        for h in range(g * G, (g + 1) * G):
            keep = dropout_keep_mask(seed, b * w.H + h, w.N, w.N, p32)
            r = head_backward(x["q"][b, h].double().numpy(), kk, vv,
                              x["do"][b, h].double().numpy(), w.scale, True, 0.0, keep=keep,
                              p_drop=p32)
            assert float(np.abs(lse[b, h].cpu().double().numpy() - r["LSE"]).max()) <= LSE_ABS
            assert rel_max(o[b, h].cpu().double().numpy(), r["O"]) <= O_MAX_REL
            check_grad("dQ[%d]" % h, dq[b, h].cpu(), r["dQ"])
            dK += r["dK"]
            dV += r["dV"]
            del r, keep
        check_grad("dK", dk[b, g].cpu(), dK)
        check_grad("dV", dv[b, g].cpu(), dV)
