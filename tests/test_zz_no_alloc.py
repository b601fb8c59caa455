"""The allocation-free backward entry point (attn_bwd_noalloc).

Some callers cannot allocate device memory (graph-captured code, plugins that
get fixed buffers); attn_bwd_noalloc serves them by keeping the dQ
accumulator and D in a fixed device array inside the library. These tests
call it through the C ABI and check it against the ordinary path
(attn_bwd_preprocess -> attn_bwd -> attn_bwd_finalize with caller-allocated
scratch), twice in a row, since every call reuses the same array.
"""
import numpy as np
import pytest
import torch

import flashattention_attention_backward_gb300 as attn
from flashattention_attention_backward_gb300 import runner
from flashattention_attention_backward_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu

MAX_REL = 2e-2   # max |err| / max |ref|, as in the parity tests
FRO_REL = 5e-3   # relative Frobenius error


def _close(got, ref, name):
    g, r = got.double().cpu().numpy(), ref.double().cpu().numpy()
    m = float(np.abs(g - r).max() / max(np.abs(r).max(), 1e-4))
    f = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-4 * np.sqrt(r.size)))
    assert m <= MAX_REL and f <= FRO_REL, "%s: max-rel %.3e fro-rel %.3e" % (name, m, f)


@pytest.mark.parametrize("w", [
    Workload("noalloc_d128_gqa_causal", 1, 4, 2, 300, 128, True, seed_base=777),
    Workload("noalloc_d64_softcap", 2, 2, 2, 256, 64, False, softcap=5.0, sigma_qkv=2.0,
             seed_base=778),
], ids=lambda w: w.name)
def test_noalloc_matches_ordinary_path_twice(w):
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, w.causal, w.softcap)
    ref_dq, ref_dk, ref_dv = (t.clone() for t in
                              runner.backward(q, k, v, o, do, lse, w.scale, w.causal, w.softcap))
    s = torch.cuda.current_stream()
    for _ in range(2):
        dq = torch.full_like(q, float("nan"))
        dk = torch.full_like(k, float("nan"))
        dv = torch.full_like(v, float("nan"))
        rc = attn.attn_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, w.B, w.H, w.H_kv, w.N, w.d,
                                   w.scale, w.causal, w.softcap, s)
        assert rc == attn.ATTN_OK, attn.attn_strerror(rc)
        torch.cuda.synchronize()
        rc, status = attn.attn_device_status(clear=True)
        assert rc == 0 and status == 0
        _close(dq, ref_dq, "dQ")
        _close(dk, ref_dk, "dK")
        _close(dv, ref_dv, "dV")


def test_noalloc_rejects_problems_beyond_its_array():
    t = torch.zeros(16, device="cuda:0")
    p = t.data_ptr()
    # B*H*N*d + B*H*N = 2*16*4096*128 + ... floats, far beyond 8,388,608
    rc = attn.attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, 2, 16, 16, 4096, 128, 0.1, 1, 0.0)
    assert rc == attn.ATTN_ERR_TOO_LARGE


def test_noalloc_rejected_calls_enqueue_nothing():
    """A rejected call returns before its first launch: dq, dk and dv keep
    the sentinel they held, and a valid call afterwards is still correct."""
    w = Workload("noalloc_reject", 1, 2, 1, 256, 128, True, seed_base=779)
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, w.causal, w.softcap)
    ref_dq, ref_dk, ref_dv = (t.clone() for t in
                              runner.backward(q, k, v, o, do, lse, w.scale, w.causal, w.softcap))
    # spare room so that a pointer one element past the start is misaligned
    dq_buf = torch.full((q.numel() + 8,), 7.0, dtype=q.dtype, device=dev)
    dk_buf = torch.full((k.numel() + 8,), 7.0, dtype=k.dtype, device=dev)
    dv = torch.full_like(v, 7.0)
    dq, dk = dq_buf[:q.numel()].view_as(q), dk_buf[:k.numel()].view_as(k)
    s = torch.cuda.current_stream()
    args = (w.B, w.H, w.H_kv, w.N, w.d)
    cases = [
        ((q, k, v, o, do, lse, dq, dk, dv), float("nan"), 0.0, attn.ATTN_ERR_SHAPE),
        ((q, k, v, o, do, lse, dq, dk, dv), 0.0, 0.0, attn.ATTN_ERR_SHAPE),
        ((q, k, v, o, do, lse, dq, dk, dv), w.scale, float("nan"), attn.ATTN_ERR_SHAPE),
        ((q, k, v, o, do, lse, dq_buf.data_ptr() + 2, dk, dv), w.scale, 0.0, attn.ATTN_ERR_ALIGN),
        ((q, k, v, o, do, lse, dq, dk_buf.data_ptr() + 2, dv), w.scale, 0.0, attn.ATTN_ERR_ALIGN),
    ]
    for ptrs, scale, cap, want in cases:
        rc = attn.attn_bwd_noalloc(*ptrs, *args, scale, w.causal, cap, s)
        assert rc == want, (rc, want)
    torch.cuda.synchronize()
    assert bool((dq_buf == 7.0).all()) and bool((dk_buf == 7.0).all()) and bool((dv == 7.0).all())
    rc, status = attn.attn_device_status(clear=True)
    assert rc == 0 and status == 0
    rc = attn.attn_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, *args, w.scale, w.causal, 0.0, s)
    assert rc == attn.ATTN_OK, attn.attn_strerror(rc)
    torch.cuda.synchronize()
    _close(dq, ref_dq, "dQ")
    _close(dk, ref_dk, "dK")
    _close(dv, ref_dv, "dV")


def test_noalloc_largest_problem_that_fits():
    """B*H*N*(d + 1) exactly at the array's limit side: N = 65027 rows of
    d = 128 fit (8,388,483 of 8,388,608 floats) and match the ordinary path;
    one row more is rejected."""
    w = Workload("noalloc_limit", 1, 1, 1, 65027, 128, True, seed_base=780)
    x = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, w.causal, w.softcap)
    ref_dq, ref_dk, ref_dv = (t.clone() for t in
                              runner.backward(q, k, v, o, do, lse, w.scale, w.causal, w.softcap))
    s = torch.cuda.current_stream()
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    rc = attn.attn_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, w.B, w.H, w.H_kv, w.N, w.d,
                               w.scale, w.causal, w.softcap, s)
    assert rc == attn.ATTN_OK, attn.attn_strerror(rc)
    torch.cuda.synchronize()
    rc, status = attn.attn_device_status(clear=True)
    assert rc == 0 and status == 0
    _close(dq, ref_dq, "dQ")
    _close(dk, ref_dk, "dK")
    _close(dv, ref_dv, "dV")
    rc = attn.attn_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, w.B, w.H, w.H_kv, w.N + 1, w.d,
                               w.scale, w.causal, w.softcap, s)
    assert rc == attn.ATTN_ERR_TOO_LARGE
