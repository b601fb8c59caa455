"""The whole path driven from plain C (tests/c_abi_client.c: cudaMalloc'd
buffers, its own stream, attn_fwd -> attn_bwd_preprocess -> attn_bwd ->
attn_bwd_finalize, status word checked) gives the same results as the
Python binding on the same inputs: O, LSE, dK and dV bit for bit, dQ up to
the order of its fp32 atomic additions (and within the oracle tolerances)."""
import subprocess

import numpy as np
import pytest
import torch

from flashattention_attention_backward_gb300 import runner
from flashattention_attention_backward_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu

from c_client_build import build_client  # noqa: E402
from parity_helpers import compare_full  # noqa: E402


def test_c_client_matches_python_binding(tmp_path):
    w = Workload("c_abi", 1, 4, 2, 300, 128, True, seed_base=77)
    x = make_inputs(w)
    exe = build_client(str(tmp_path / "c_abi_client"))
    src = tmp_path / "in.bin"
    dst = tmp_path / "out.bin"
    with open(src, "wb") as f:
        for n in ("q", "k", "v", "do"):
            f.write(x[n].contiguous().view(torch.int16).numpy().tobytes())
    r = subprocess.run([exe, str(src), str(dst), str(w.B), str(w.H), str(w.H_kv), str(w.N),
                        str(w.d), "1"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
    raw = np.fromfile(dst, dtype=np.uint8)
    nq, nk, nr = w.B * w.H * w.N * w.d, w.B * w.H_kv * w.N * w.d, w.B * w.H * w.N
    sizes = [("o", nq * 2), ("lse", nr * 4), ("dq", nq * 2), ("dk", nk * 2), ("dv", nk * 2)]
    out, at = {}, 0
    for name, nbytes in sizes:
        chunk = raw[at:at + nbytes].copy()
        at += nbytes
        if name == "lse":
            out[name] = torch.from_numpy(chunk.view(np.float32)).reshape(w.B, w.H, w.N)
        else:
            shape = (w.B, w.H if name in ("o", "dq") else w.H_kv, w.N, w.d)
            out[name] = torch.from_numpy(chunk.view(np.int16)).view(torch.bfloat16).reshape(shape)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, True)
    dq, dk, dv = runner.backward(q, k, v, o, do, lse, w.scale, True)
    torch.cuda.synchronize()
    assert torch.equal(out["o"], o.cpu()) and torch.equal(out["lse"], lse.cpu())
    assert torch.equal(out["dk"], dk.cpu()) and torch.equal(out["dv"], dv.cpu())
    assert torch.allclose(out["dq"].float(), dq.cpu().float(), rtol=1e-2, atol=1e-3)
    compare_full(w, x, out)
