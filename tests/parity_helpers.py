"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare with the fp64 oracle using the stated tolerances."""
import numpy as np
import torch

import flashattention_attention_backward_gb300 as attn
from flashattention_attention_backward_gb300 import runner
from flashattention_attention_backward_gb300.inputs import make_inputs
from oracle import attention_backward, attention_forward

# Tolerances of the attention-backward parity bar.
GRAD_MAX_REL = 2e-2    # max |err| / max |ref| for dQ, dK, dV
GRAD_FRO_REL = 5e-3    # ||err||_F / ||ref||_F for dQ, dK, dV
O_MAX_REL = 2e-2       # forward O, max |err| / max |ref|
LSE_ABS = 1e-5         # forward LSE, max |err| (for |LSE| <= LSE_SCALE_FROM)
# fp32 scores resolve a logit of size |x| only to a few ulps of |x|; beyond
# |LSE| = 16 (the five workloads stay below it) the LSE bound keeps the same
# number of ulps, i.e. grows with |LSE| / 16.
LSE_SCALE_FROM = 16.0
# Where the exact gradient vanishes (e.g. a single key: P = 1 so dS = 0), a
# relative error is undefined; errors are then measured against this floor.
REF_FLOOR = 1e-4


def lse_tol(lse_ref):
    """LSE_ABS, widened in proportion to |LSE| past LSE_SCALE_FROM."""
    return LSE_ABS * max(1.0, float(np.abs(lse_ref).max()) / LSE_SCALE_FROM)


def run_gpu(w, x=None):
    """Forward + backward of workload `w` on cuda:0; returns CPU tensors."""
    if x is None:
        x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, w.causal, w.softcap)
    dq, dk, dv = runner.backward(q, k, v, o, do, lse, w.scale, w.causal, w.softcap)
    torch.cuda.synchronize()
    rc, status = attn.attn_device_status(clear=True)
    assert rc == 0 and status == 0, "device status %d (rc %d)" % (status, rc)
    return x, {"o": o.cpu(), "lse": lse.cpu(), "dq": dq.cpu(), "dk": dk.cpu(), "dv": dv.cpu()}


def rel_max(got, ref, floor=1e-30):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), floor))


def rel_fro(got, ref, floor=1e-30):
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), floor))


def check_grad(name, got, ref):
    g = got.double().numpy() if torch.is_tensor(got) else got
    assert np.isfinite(g).all(), name + " has non-finite values"
    m, f = rel_max(g, ref, REF_FLOOR), rel_fro(g, ref, REF_FLOOR * np.sqrt(ref.size))
    assert m <= GRAD_MAX_REL and f <= GRAD_FRO_REL, "%s: max-rel %.3e fro-rel %.3e" % (name, m, f)
    return m, f


def compare_full(w, x, out):
    f64 = {n: x[n].double().numpy() for n in ("q", "k", "v", "do")}
    O, LSE = attention_forward(f64["q"], f64["k"], f64["v"], w.scale, w.causal, w.softcap)
    lse_err = float(np.abs(out["lse"].double().numpy() - LSE).max())
    assert lse_err <= LSE_ABS, "LSE abs err %.3e" % lse_err
    o_err = rel_max(out["o"].double().numpy(), O)
    assert o_err <= O_MAX_REL, "O max-rel %.3e" % o_err
    dQ, dK, dV = attention_backward(f64["q"], f64["k"], f64["v"], f64["do"], w.scale, w.causal,
                                    w.softcap)
    res = {"dq": check_grad("dQ", out["dq"], dQ), "dk": check_grad("dK", out["dk"], dK),
           "dv": check_grad("dV", out["dv"], dV)}
    return res


def compare_slices(w, x, out, slices):
    """Oracle on selected (batch, kv_head) slices only (dK/dV need the group)."""
    G = w.G
    worst = {}
    for (b, g) in slices:
        heads = slice(g * G, (g + 1) * G)
        q = x["q"][b:b + 1, heads].double().numpy()
        do = x["do"][b:b + 1, heads].double().numpy()
        k = x["k"][b:b + 1, g:g + 1].double().numpy()
        v = x["v"][b:b + 1, g:g + 1].double().numpy()
        O, LSE = attention_forward(q, k, v, w.scale, w.causal, w.softcap)
        lse_err = float(np.abs(out["lse"][b, heads].double().numpy() - LSE[0]).max())
        assert lse_err <= LSE_ABS, "slice %s: LSE abs err %.3e" % ((b, g), lse_err)
        assert rel_max(out["o"][b, heads].double().numpy(), O[0]) <= O_MAX_REL
        dQ, dK, dV = attention_backward(q, k, v, do, w.scale, w.causal, w.softcap)
        worst[(b, g)] = (check_grad("dQ%s" % ((b, g),), out["dq"][b, heads], dQ[0]),
                         check_grad("dK%s" % ((b, g),), out["dk"][b, g], dK[0, 0]),
                         check_grad("dV%s" % ((b, g),), out["dv"][b, g], dV[0, 0]))
        del O, LSE, dQ, dK, dV
    return worst
