"""Convenience wrappers that allocate device memory with torch and call the
C ABI in stream order: forward (O, LSE), then preprocess -> attn_bwd ->
finalize. No arithmetic happens here; torch provides memory and streams.
"""
import torch

from . import (attn_bwd, attn_bwd_deterministic, attn_bwd_dq_partials_bytes, attn_bwd_dropout,
               attn_bwd_finalize, attn_bwd_finalize_partials, attn_bwd_local, attn_bwd_preprocess,
               attn_fwd, attn_fwd_dropout, attn_fwd_local, attn_fwd_ref, attn_fwd_ref_dropout,
               attn_fwd_ref_local, check)


def _dims(q, k, *others):
    """(B, H, H_kv, N, d) of q [B,H,N,d] and k [B,H_kv,N,d], after checking
    what the C ABI assumes of its pointers: contiguous bf16 tensors on one
    CUDA device, with matching shapes (k, v alike; q, o, dO alike)."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be 4-D ([B, heads, N, d])")
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    if k.shape != (B, H_kv, N, d):
        raise ValueError("k has shape %s, expected %s" % (tuple(k.shape), (B, H_kv, N, d)))
    for t in others:
        if t.shape not in (q.shape, k.shape):
            raise ValueError("tensor of shape %s matches neither q nor k" % (tuple(t.shape),))
    for t in (q, k) + others:
        if t.dtype != torch.bfloat16:
            raise ValueError("expected bfloat16 tensors, got %s" % t.dtype)
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous (row-major [B, heads, N, d])")
    for t in (q, k) + others:
        if t.device != q.device or t.device.type != "cuda":
            raise ValueError("all tensors must be on the same CUDA device")
    return B, H, H_kv, N, d


def _check_lse(lse, B, H, N, device):
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, N) \
            or lse.device != device:
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor on the inputs' device")


def _stream(stream):
    return stream if stream is not None else torch.cuda.current_stream()


def forward(q, k, v, scale, causal, softcap=0.0, stream=None, impl="tc", dropout=None,
            window=None):
    """O [B,H,N,d] bf16 and LSE [B,H,N] fp32: attn_fwd (tensor cores, impl
    "tc") or attn_fwd_ref (plain fp32, impl "ref"). dropout = (p_drop, seed)
    runs attn_fwd_dropout or attn_fwd_ref_dropout; window = (left, right) runs
    attn_fwd_local or attn_fwd_ref_local."""
    B, H, H_kv, N, d = _dims(q, k, v)
    if v.shape != k.shape:
        raise ValueError("v must have the shape of k")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if dropout is not None:
        fn = {"tc": attn_fwd_dropout, "ref": attn_fwd_ref_dropout}[impl]
        check(fn(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, dropout[0],
                 dropout[1], _stream(stream)))
        return o, lse
    if window is not None:
        fn = {"tc": attn_fwd_local, "ref": attn_fwd_ref_local}[impl]
        check(fn(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, window[0], window[1],
                 _stream(stream)))
        return o, lse
    fn = {"tc": attn_fwd, "ref": attn_fwd_ref}[impl]
    check(fn(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, softcap, _stream(stream)))
    return o, lse


class BackwardBuffers:
    """Outputs and scratch of one backward problem, reusable across calls."""

    def __init__(self, q, k):
        B, H, H_kv, N, d = _dims(q, k)
        dev = q.device
        self.dq = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
        self.dk = torch.empty((B, H_kv, N, d), dtype=torch.bfloat16, device=dev)
        self.dv = torch.empty((B, H_kv, N, d), dtype=torch.bfloat16, device=dev)
        self.dq_accum = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
        self.dpsum = torch.empty((B, H, N), dtype=torch.float32, device=dev)


def backward(q, k, v, o, do, lse, scale, causal, softcap=0.0, stream=None, bufs=None,
             deterministic=False, dropout=None, window=None):
    """dQ, dK, dV (bf16) via preprocess -> attn_bwd -> finalize, or, with
    deterministic=True, preprocess -> attn_bwd_deterministic ->
    finalize_partials (dQ identical bit for bit from run to run). window =
    (left, right) runs attn_bwd_local in place of attn_bwd."""
    B, H, H_kv, N, d = _dims(q, k, v, o, do)
    if v.shape != k.shape or o.shape != q.shape or do.shape != q.shape:
        raise ValueError("v must have the shape of k, and o, dO that of q")
    _check_lse(lse, B, H, N, q.device)
    s = _stream(stream)
    if bufs is None:
        bufs = BackwardBuffers(q, k)
    if dropout is not None:
        check(attn_bwd_preprocess(o, do, bufs.dpsum, bufs.dq_accum, B, H, N, d, s))
        check(attn_bwd_dropout(q, k, v, o, do, lse, bufs.dq_accum, bufs.dk, bufs.dv, B, H, H_kv,
                               N, d, scale, causal, softcap, bufs.dpsum, dropout[0], dropout[1],
                               s))
        check(attn_bwd_finalize(bufs.dq_accum, bufs.dq, scale, B, H, N, d, s))
        return bufs.dq, bufs.dk, bufs.dv
    if window is not None:
        if deterministic:
            raise ValueError("the local window has no deterministic variant")
        check(attn_bwd_preprocess(o, do, bufs.dpsum, bufs.dq_accum, B, H, N, d, s))
        check(attn_bwd_local(q, k, v, o, do, lse, bufs.dq_accum, bufs.dk, bufs.dv, B, H, H_kv, N,
                             d, scale, causal, softcap, bufs.dpsum, window[0], window[1], s))
        check(attn_bwd_finalize(bufs.dq_accum, bufs.dq, scale, B, H, N, d, s))
        return bufs.dq, bufs.dk, bufs.dv
    if not deterministic:
        check(attn_bwd_preprocess(o, do, bufs.dpsum, bufs.dq_accum, B, H, N, d, s))
        check(attn_bwd(q, k, v, o, do, lse, bufs.dq_accum, bufs.dk, bufs.dv, B, H, H_kv, N, d,
                       scale, causal, softcap, bufs.dpsum, s))
        check(attn_bwd_finalize(bufs.dq_accum, bufs.dq, scale, B, H, N, d, s))
        return bufs.dq, bufs.dk, bufs.dv
    nbytes = attn_bwd_dq_partials_bytes(B, H, N, d, causal)
    if nbytes < 0:
        check(int(nbytes))
    if getattr(bufs, "dq_partials", None) is None or bufs.dq_partials.numel() * 4 < nbytes:
        bufs.dq_partials = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device=q.device)
    check(attn_bwd_preprocess(o, do, bufs.dpsum, None, B, H, N, d, s))
    check(attn_bwd_deterministic(q, k, v, o, do, lse, bufs.dq_partials, bufs.dk, bufs.dv, B, H,
                                 H_kv, N, d, scale, causal, softcap, bufs.dpsum, s))
    check(attn_bwd_finalize_partials(bufs.dq_partials, bufs.dq, scale, B, H, N, d, causal, s))
    return bufs.dq, bufs.dk, bufs.dv
