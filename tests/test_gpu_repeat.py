"""Repeated launches of the persistent forward with the device status checked.

A wait on a barrier parity can alias when the barrier runs two phases ahead
of the waiter, and then lasts until a later phase that needs the waiter: a
deadlock that the kernels' bounded waits turn into a device timeout status.
Such a race shows only on some runs (the forward's epilogue once had one,
about one run in thirty on the d = 256 shape below), so these cases repeat
the launches many times on multi-tile shapes and check the status after each
batch, as well as the result against the fp32 reference forward once.
"""
import numpy as np
import pytest
import torch

import flashattention_attention_backward_gb300 as attn
from flashattention_attention_backward_gb300 import runner
from flashattention_attention_backward_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _status_clean():
    torch.cuda.synchronize()
    rc, status = attn.attn_device_status(clear=True)
    return rc == 0 and status == 0


@pytest.mark.parametrize("B,H,H_kv,N,d,reps", [
    (2, 16, 4, 4096, 256, 60),   # seven tiles per CTA, one Q / K / V / O buffer each
    (2, 32, 8, 2048, 128, 60),
    (4, 16, 16, 2048, 64, 60),
])
def test_forward_repeated_launches_keep_status_clean(B, H, H_kv, N, d, reps):
    w = Workload("repeat", B, H, H_kv, N, d, True, seed_base=777 + d)
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    assert _status_clean()
    o_ref, lse_ref = runner.forward(q, k, v, w.scale, True, impl="ref")
    bufs = runner.BackwardBuffers(q, k)
    bad = []
    for rep in range(reps):
        o, lse = runner.forward(q, k, v, w.scale, True)
        if not _status_clean():
            bad.append(("forward", rep))
        if d == 256 and rep % 4 == 0:  # the backward between forwards, as in the bench
            runner.backward(q, k, v, o, do, lse, w.scale, True, bufs=bufs)
            if not _status_clean():
                bad.append(("backward", rep))
    assert not bad, bad
    err = float((o.float() - o_ref.float()).abs().max())
    assert err <= 2e-2 * float(o_ref.float().abs().max())
    assert float(np.abs((lse - lse_ref).cpu().numpy()).max()) <= 1e-4


@pytest.mark.parametrize("d,reps", [(128, 30), (256, 30), (64, 30)])
def test_dropout_paths_repeated_keep_status_clean(d, reps):
    """The dropout forward (mask warps beside the softmax) and backward (at
    d = 256 a mask warpgroup of its own) hand the keep bits over through
    double-buffered shared memory with their own barriers; repeated launches
    must all finish with a clean status and the same result."""
    B, H, H_kv, N = 2, 8, 2, 2048
    w = Workload("repeat_drop", B, H, H_kv, N, d, True, seed_base=888 + d)
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    drop = (0.2, 2 ** 35 + 11)
    assert _status_clean()
    o0, lse0 = runner.forward(q, k, v, w.scale, True, dropout=drop)
    g0 = [t.clone() for t in runner.backward(q, k, v, o0, do, lse0, w.scale, True, dropout=drop)]
    assert _status_clean()
    bufs = runner.BackwardBuffers(q, k)
    bad = []
    for rep in range(reps):
        o, lse = runner.forward(q, k, v, w.scale, True, dropout=drop)
        if not _status_clean():
            bad.append(("forward", rep))
        if not torch.equal(o, o0):
            bad.append(("forward differs", rep))
        if rep % 3 == 0:
            dq, dk, dv = runner.backward(q, k, v, o, do, lse, w.scale, True, bufs=bufs,
                                         dropout=drop)
            if not _status_clean():
                bad.append(("backward", rep))
            # dK and dV are summed on chip in a fixed order: bitwise repeatable
            if not (torch.equal(dk, g0[1]) and torch.equal(dv, g0[2])):
                bad.append(("backward dK/dV differ", rep))
    assert not bad, bad


def test_deterministic_backward_repeated_keep_status_clean():
    w = Workload("repeat_det", 2, 8, 2, 2048, 128, True, seed_base=999)
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, True)
    first = None
    for rep in range(20):
        dq, dk, dv = runner.backward(q, k, v, o, do, lse, w.scale, True, deterministic=True)
        assert _status_clean(), rep
        if first is None:
            first = [t.clone() for t in (dq, dk, dv)]
        else:
            assert all(torch.equal(a, b) for a, b in zip((dq, dk, dv), first)), rep
