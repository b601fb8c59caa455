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
