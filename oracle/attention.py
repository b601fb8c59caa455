"""Plain fp64 CPU attention forward and backward that materialises P.

Test infrastructure only (see the package docstring): nothing on the product
path may import this module.

What it computes is the exact gradient of standard attention. Tiling and
recomputation change only the order of the arithmetic, so the oracle is the
materialised chain written out once, in the pages' order:

  forward   ("解析 FlashAttention（3）" §1.1; "反向传播算法详解" §1.2, §2.1(3))
      Z   = tau * Q K^T
      S   = c * tanh(Z / c)             if a softcap c > 0, else S = Z
      S_ij = -inf for key j > query i   if causal (lower-triangular mask,
                                        "解析 FlashAttention（3）" §4 line 12)
      LSE_i = m_i + ln sum_j exp(S_ij - m_i),  m_i = max_j S_ij
      P   = exp(S - LSE 1^T)            (eq. 9 with LSE = m + ln l)
      O   = P V
  backward  ("解析 FlashAttention（3）" §2.7, eq. 1-8)
      dV  = P^T dO                      (eq. 1)
      dP  = dO V^T                      (eq. 2)
      D   = rowsum(dO o O)              (eq. 6)
      dS  = P o (dP - D 1^T)            (eq. 5)
      dZ  = dS o (1 - T^2)              if softcap ("反向传播算法详解" §2.1(3))
      dQ  = tau * dZ K                  (eq. 7)
      dK  = tau * dZ^T Q                (eq. 8)

Local window ("反向传播算法详解" §3.4, the local-attention masking), optional:
window = (left, right) hides key j from query i unless i - left <= j <= i + right
(a negative bound is unbounded); it combines with the causal mask.

Dropout ("解析 FlashAttention（3）" §3.3, Algorithm 4 of §4), optional: with a
keep mask Z (from oracle.philox, drop probability p),
      P~  = P o Z / (1 - p)             O = P~ V; LSE is that of P
      dV  = P~^T dO                     dP = (dO V^T) o Z / (1 - p)
and the rest as above; D = rowsum(dO o O) still equals rowsum(P o dP).

Grouped KV heads ("反向传播算法详解" §8.5): query head h reads KV head
floor(h / G) with G = H / H_kv, and dK, dV of a KV head are the sums over the
G query heads of its group.

Layout: Q, O, dO are [B, H, N, d]; K, V are [B, H_kv, N, d]; LSE is [B, H, N].
All arithmetic is float64; inputs of any float dtype are converted exactly.
Library matrix products (numpy ``@``) are the only primitives used; there is
no blocking or reordering beyond the definitions above.
"""
import numpy as np

from .philox import dropout_keep_mask


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def head_forward(q, k, v, scale, causal=False, softcap=0.0, keep=None, p_drop=0.0,
                 window=None):
    """Forward pass of one query head against its KV head.

    q: [Nq, d], k, v: [Nk, d] (Nq == Nk when causal). Returns a dict with
    Z (tau Q K^T), T (tanh(Z/c) or None), S (masked logits), LSE, P and O,
    all float64. With a boolean keep mask [Nq, Nk], O = (P o keep / (1 - p)) V.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Z = scale * (q @ k.T)
    if softcap > 0.0:
        T = np.tanh(Z / softcap)
        S = softcap * T
    else:
        T = None
        S = Z.copy()
    nq, nk = S.shape
    i = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    if causal:
        S = np.where(j > i, -np.inf, S)
    if window is not None:
        left, right = window
        if left >= 0:
            S = np.where(j < i - left, -np.inf, S)
        if right >= 0:
            S = np.where(j > i + right, -np.inf, S)
    m = S.max(axis=1)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    ell = np.exp(S - m_safe[:, None]).sum(axis=1)
    with np.errstate(divide="ignore"):
        LSE = np.where(finite, m_safe + np.log(ell), -np.inf)
    lse_safe = np.where(finite, LSE, 0.0)
    P = np.where(finite[:, None], np.exp(S - lse_safe[:, None]), 0.0)
    Pd = P if keep is None else np.where(keep, P / (1.0 - p_drop), 0.0)
    O = Pd @ v
    return {"Z": Z, "T": T, "S": S, "LSE": LSE, "P": P, "Pd": Pd, "O": O}


def head_backward(q, k, v, do, scale, causal=False, softcap=0.0, o=None, keep=None, p_drop=0.0,
                  window=None):
    """Backward pass of one query head (materialised P, dP, dS).

    Returns a dict with dQ [Nq, d], dK and dV [Nk, d] (this head's share,
    not yet summed over a GQA group) and the intermediates P, dP, D, dS, dZ,
    O and LSE. If ``o`` is given, D is formed from that O instead of the
    oracle's own (used to separate forward error from backward error).
    """
    fw = head_forward(q, k, v, scale, causal, softcap, keep, p_drop, window)
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    P = fw["P"]
    O = fw["O"] if o is None else _f64(o)
    dV = fw["Pd"].T @ do                            # eq. 1 (dropped P)
    dP = do @ v.T                                   # eq. 2
    if keep is not None:
        dP = np.where(keep, dP / (1.0 - p_drop), 0.0)  # through the dropout
    D = (do * O).sum(axis=1)                        # eq. 6
    dS = P * (dP - D[:, None])                      # eq. 5
    if softcap > 0.0:
        dZ = dS * (1.0 - fw["T"] ** 2)              # softcap derivative
    else:
        dZ = dS
    dQ = scale * (dZ @ k)                           # eq. 7
    dK = scale * (dZ.T @ q)                         # eq. 8
    return {"dQ": dQ, "dK": dK, "dV": dV, "P": P, "dP": dP, "D": D,
            "dS": dS, "dZ": dZ, "O": fw["O"], "LSE": fw["LSE"]}


def _check_shapes(Q, K):
    B, H, N, d = Q.shape
    Bk, H_kv, Nk, dk = K.shape
    if Bk != B or dk != d or H % H_kv != 0:
        raise ValueError("inconsistent shapes Q%s K%s" % (Q.shape, K.shape))
    return B, H, H_kv, N, Nk, d


def _keep(dropout, b, h, H, nq, nk):
    """Keep mask of head (b, h) for dropout = (p_drop, seed), or None."""
    if dropout is None or dropout[0] <= 0.0:
        return None, 0.0
    p_drop, seed = dropout
    return dropout_keep_mask(seed, b * H + h, nq, nk, p_drop), float(p_drop)


def attention_forward(Q, K, V, scale, causal=False, softcap=0.0, dropout=None, window=None):
    """O [B,H,N,d] and natural-log LSE [B,H,N] for the whole batch.
    dropout = (p_drop, seed) applies the Philox keep mask of oracle.philox;
    window = (left, right) the local-attention mask."""
    B, H, H_kv, N, Nk, d = _check_shapes(Q, K)
    G = H // H_kv
    O = np.empty((B, H, N, d), dtype=np.float64)
    LSE = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            g = h // G
            keep, pd = _keep(dropout, b, h, H, N, Nk)
            fw = head_forward(Q[b, h], K[b, g], V[b, g], scale, causal, softcap, keep, pd,
                              window)
            O[b, h] = fw["O"]
            LSE[b, h] = fw["LSE"]
    return O, LSE


def attention_backward(Q, K, V, dO, scale, causal=False, softcap=0.0,
                       slices=None, O=None, dropout=None, window=None):
    """dQ, dK, dV for the batch, or for selected (batch, kv_head) slices.

    With ``slices=None`` returns arrays dQ [B,H,N,d], dK, dV [B,H_kv,N,d].
    With ``slices=[(b, g), ...]`` returns a dict mapping (b, g) to a dict
    {"dQ": [G,N,d], "dK": [N,d], "dV": [N,d], "heads": [h...]} where dK and
    dV are summed over the G query heads of KV head g. ``O`` optionally
    supplies the forward output used for D (same shape as Q). dropout =
    (p_drop, seed) applies the Philox keep mask of oracle.philox; window =
    (left, right) the local-attention mask.
    """
    B, H, H_kv, N, Nk, d = _check_shapes(Q, K)
    G = H // H_kv

    def one_slice(b, g):
        heads = list(range(g * G, (g + 1) * G))
        dQ = np.empty((G, N, d), dtype=np.float64)
        dK = np.zeros((Nk, d), dtype=np.float64)
        dV = np.zeros((Nk, d), dtype=np.float64)
        for r, h in enumerate(heads):
            keep, pd = _keep(dropout, b, h, H, N, Nk)
            res = head_backward(Q[b, h], K[b, g], V[b, g], dO[b, h], scale,
                                causal, softcap,
                                None if O is None else O[b, h], keep, pd, window)
            dQ[r] = res["dQ"]
            dK += res["dK"]                         # GQA group sum
            dV += res["dV"]
            del res
        return {"dQ": dQ, "dK": dK, "dV": dV, "heads": heads}

    if slices is not None:
        return {(b, g): one_slice(b, g) for (b, g) in slices}
    dQ = np.empty((B, H, N, d), dtype=np.float64)
    dK = np.empty((B, H_kv, Nk, d), dtype=np.float64)
    dV = np.empty((B, H_kv, Nk, d), dtype=np.float64)
    for b in range(B):
        for g in range(H_kv):
            r = one_slice(b, g)
            dQ[b, g * G:(g + 1) * G] = r["dQ"]
            dK[b, g] = r["dK"]
            dV[b, g] = r["dV"]
    return dQ, dK, dV
