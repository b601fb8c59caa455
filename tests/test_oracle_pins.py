"""Pins of the fp64 oracle to facts other than itself (CPU only).

* hand-derived N=2, d=2 worked examples (tests/golden/n2_d2_worked.json),
  following the element formulas of "解析 FlashAttention（3）" §2.2-2.5;
* the N=2, d=2 element formulas evaluated in separate scalar code;
* an independent brute-force scalar forward (pure Python loops) for O, LSE;
* central finite differences of L = sum(dO o O) through that scalar forward
  against the oracle's dQ, dK, dV (causal, GQA and softcap included);
* invariants: rowsum(dS) = 0, D_i = sum_j P_ij dP_ij, column sums of dV,
  column sums of dK, rows of P sum to 1, GQA == repeated-KV MHA;
* special cases: equal keys, equal values, causal first row / last key,
  huge softcap, rescaled Q and tau;
* planted mistakes: mutated copies of the backward must fail the FD pin.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import attention_backward, attention_forward, head_backward, head_forward

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "n2_d2_worked.json")


# --------------------------------------------------------------------------
# hand-derived worked examples
# --------------------------------------------------------------------------
def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_worked_example(case):
    q, k, v, do = (np.array(case[n], dtype=np.float64) for n in ("q", "k", "v", "do"))
    res = head_backward(q, k, v, do, case["scale"], case["causal"], case["softcap"])
    fw = head_forward(q, k, v, case["scale"], case["causal"], case["softcap"])
    got = {"P": fw["P"], "O": fw["O"], "LSE": fw["LSE"], "dP": res["dP"],
           "D": res["D"], "dS": res["dS"], "dV": res["dV"], "dQ": res["dQ"],
           "dK": res["dK"]}
    for name, want in case["expect"].items():
        np.testing.assert_allclose(got[name], np.array(want, dtype=np.float64),
                                   rtol=0, atol=1e-14, err_msg=name)


# --------------------------------------------------------------------------
# element formulas of the N=2, d=2 derivation, scalar code
# --------------------------------------------------------------------------
def test_element_formulas_n2_d2():
    tau = 0.7
    q = [[0.5, -1.0], [1.0, 0.25]]
    k = [[-0.5, 1.0], [0.75, 0.5]]
    v = [[1.0, -2.0], [0.5, 3.0]]
    dO = [[0.25, -1.0], [2.0, 0.5]]
    # S_ij = tau (q_i1 k_j1 + q_i2 k_j2)
    s = [[tau * (q[i][0] * k[j][0] + q[i][1] * k[j][1]) for j in range(2)] for i in range(2)]
    # two-element softmax per row
    p = []
    for i in range(2):
        e0, e1 = math.exp(s[i][0]), math.exp(s[i][1])
        p.append([e0 / (e0 + e1), e1 / (e0 + e1)])
    O = [[p[i][0] * v[0][c] + p[i][1] * v[1][c] for c in range(2)] for i in range(2)]
    # dL/dv11 = dO11 p11 + dO21 p21, and the other three entries
    dv = [[dO[0][c] * p[0][j] + dO[1][c] * p[1][j] for c in range(2)] for j in range(2)]
    # dL/dp_ij = dO_i1 v_j1 + dO_i2 v_j2
    dp = [[dO[i][0] * v[j][0] + dO[i][1] * v[j][1] for j in range(2)] for i in range(2)]
    # D_i = p_i1 dp_i1 + p_i2 dp_i2 ; ds_ij = p_ij (dp_ij - D_i)
    D = [p[i][0] * dp[i][0] + p[i][1] * dp[i][1] for i in range(2)]
    ds = [[p[i][j] * (dp[i][j] - D[i]) for j in range(2)] for i in range(2)]
    # dL/dq_i c = tau (ds_i1 k_1c + ds_i2 k_2c); dL/dk_j c = tau (ds_1j q_1c + ds_2j q_2c)
    dq = [[tau * (ds[i][0] * k[0][c] + ds[i][1] * k[1][c]) for c in range(2)] for i in range(2)]
    dk = [[tau * (ds[0][j] * q[0][c] + ds[1][j] * q[1][c]) for c in range(2)] for j in range(2)]
    # D_1 also equals dO_11 O_11 + dO_12 O_12
    for i in range(2):
        assert abs(D[i] - (dO[i][0] * O[i][0] + dO[i][1] * O[i][1])) < 1e-14

    res = head_backward(np.array(q), np.array(k), np.array(v), np.array(dO), tau)
    np.testing.assert_allclose(res["O"], O, atol=1e-13, rtol=0)
    np.testing.assert_allclose(res["dV"], dv, atol=1e-13, rtol=0)
    np.testing.assert_allclose(res["dP"], dp, atol=1e-13, rtol=0)
    np.testing.assert_allclose(res["D"], D, atol=1e-13, rtol=0)
    np.testing.assert_allclose(res["dS"], ds, atol=1e-13, rtol=0)
    np.testing.assert_allclose(res["dQ"], dq, atol=1e-13, rtol=0)
    np.testing.assert_allclose(res["dK"], dk, atol=1e-13, rtol=0)


# --------------------------------------------------------------------------
# independent brute-force scalar forward
# --------------------------------------------------------------------------
def brute_forward(Q, K, V, scale, causal, softcap, keep=None, p_drop=0.0, window=None):
    """Pure-Python loops: O and LSE for [B,H,N,d] / [B,H_kv,N,d] nested lists.
    keep[b][h][i][j] (optional) drops P_ij where false and scales the rest by
    1 / (1 - p_drop)."""
    B, H, N, d = len(Q), len(Q[0]), len(Q[0][0]), len(Q[0][0][0])
    H_kv = len(K[0])
    G = H // H_kv
    O = [[[[0.0] * d for _ in range(N)] for _ in range(H)] for _ in range(B)]
    LSE = [[[0.0] * N for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            g = h // G
            for i in range(N):
                logits = []
                for j in range(N):
                    if causal and j > i:
                        continue
                    if window is not None and ((window[0] >= 0 and j < i - window[0]) or
                                               (window[1] >= 0 and j > i + window[1])):
                        continue
                    raw = 0.0
                    for c in range(d):
                        raw += Q[b][h][i][c] * K[b][g][j][c]
                    raw *= scale
                    if softcap > 0:
                        raw = softcap * math.tanh(raw / softcap)
                    logits.append((j, raw))
                mx = max(x for _, x in logits)
                tot = sum(math.exp(x - mx) for _, x in logits)
                lse = mx + math.log(tot)
                LSE[b][h][i] = lse
                for j, x in logits:
                    pij = math.exp(x - lse)
                    if keep is not None:
                        pij = pij / (1.0 - p_drop) if keep[b][h][i][j] else 0.0
                    for c in range(d):
                        O[b][h][i][c] += pij * V[b][g][j][c]
    return O, LSE


def _rand(rng, shape, sigma=1.0):
    return rng.normal(0.0, sigma, size=shape)


SMALL_CASES = [
    # B, H, H_kv, N, d, causal, softcap
    (1, 1, 1, 3, 2, False, 0.0),
    (1, 2, 2, 5, 4, True, 0.0),
    (1, 2, 1, 5, 2, False, 2.0),
    (1, 2, 1, 3, 4, True, 2.0),
    (2, 4, 2, 4, 3, True, 0.0),
]


@pytest.mark.parametrize("case", SMALL_CASES)
def test_forward_matches_brute_force(case):
    B, H, H_kv, N, d, causal, cap = case
    rng = np.random.default_rng(11)
    Q, K, V = _rand(rng, (B, H, N, d)), _rand(rng, (B, H_kv, N, d)), _rand(rng, (B, H_kv, N, d))
    scale = 1.0 / math.sqrt(d)
    O, LSE = attention_forward(Q, K, V, scale, causal, cap)
    Ob, LSEb = brute_forward(Q.tolist(), K.tolist(), V.tolist(), scale, causal, cap)
    np.testing.assert_allclose(O, np.array(Ob), atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE, np.array(LSEb), atol=1e-12, rtol=0)


def _fd_grads(Q, K, V, dO, scale, causal, cap, h=1e-6):
    """Central differences of L = sum(dO o O) through the scalar forward."""
    def loss(Qx, Kx, Vx):
        O, _ = brute_forward(Qx.tolist(), Kx.tolist(), Vx.tolist(), scale, causal, cap)
        return float((np.array(O) * dO).sum())

    grads = []
    for which in range(3):
        base = [Q, K, V][which]
        g = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            args_p = [Q.copy(), K.copy(), V.copy()]
            args_m = [Q.copy(), K.copy(), V.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            g[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        grads.append(g)
    return grads


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


def _fd_case(case, seed=5):
    B, H, H_kv, N, d, causal, cap = case
    rng = np.random.default_rng(seed)
    Q, K, V = _rand(rng, (B, H, N, d)), _rand(rng, (B, H_kv, N, d)), _rand(rng, (B, H_kv, N, d))
    dO = _rand(rng, (B, H, N, d))
    return Q, K, V, dO, 1.0 / math.sqrt(d), causal, cap


@pytest.mark.parametrize("case", SMALL_CASES)
def test_backward_matches_finite_differences(case):
    Q, K, V, dO, scale, causal, cap = _fd_case(case)
    dQ, dK, dV = attention_backward(Q, K, V, dO, scale, causal, cap)
    fQ, fK, fV = _fd_grads(Q, K, V, dO, scale, causal, cap)
    assert _rel(dQ, fQ) < 1e-7
    assert _rel(dK, fK) < 1e-7
    assert _rel(dV, fV) < 1e-7


# --------------------------------------------------------------------------
# planted mistakes must be caught by the FD pin
# --------------------------------------------------------------------------
def _mutant_backward(kind):
    def bwd(q, k, v, do, scale, causal=False, softcap=0.0):
        fw = head_forward(q, k, v, scale, causal, softcap)
        P, O, T = fw["P"], fw["O"], fw["T"]
        dV = P.T @ do
        dP = do @ v.T
        D = (do * O).sum(axis=1)
        if kind == "dropped_D":
            dS = P * dP
        elif kind == "sign_D":
            dS = P * (dP + D[:, None])
        else:
            dS = P * (dP - D[:, None])
        if softcap > 0.0 and kind != "no_dtanh":
            dS = dS * (1.0 - T ** 2)
        if kind == "transposed_dK":
            dK = scale * (dS @ q)
        else:
            dK = scale * (dS.T @ q)
        if kind == "dQ_no_scale":
            dQ = dS @ k
        else:
            dQ = scale * (dS @ k)
        if kind == "dV_untransposed":
            dV = P @ do
        return dQ, dK, dV
    return bwd


@pytest.mark.parametrize("kind", ["dropped_D", "sign_D", "no_dtanh", "transposed_dK",
                                  "dQ_no_scale", "dV_untransposed"])
def test_planted_mistakes_fail_fd(kind):
    case = (1, 1, 1, 4, 3, True, 2.0)
    Q, K, V, dO, scale, causal, cap = _fd_case(case, seed=9)
    fQ, fK, fV = _fd_grads(Q, K, V, dO, scale, causal, cap)
    dQ, dK, dV = _mutant_backward(kind)(Q[0, 0], K[0, 0], V[0, 0], dO[0, 0], scale, causal, cap)
    worst = max(_rel(dQ, fQ[0, 0]), _rel(dK, fK[0, 0]), _rel(dV, fV[0, 0]))
    assert worst > 1e-3, kind


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_invariants(causal):
    rng = np.random.default_rng(3)
    N, d = 37, 8
    q, k, v, do = (_rand(rng, (N, d)) for _ in range(4))
    scale = 1.0 / math.sqrt(d)
    r = head_backward(q, k, v, do, scale, causal)
    np.testing.assert_allclose(r["P"].sum(axis=1), 1.0, atol=1e-13)
    np.testing.assert_allclose(r["dS"].sum(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose(r["D"], (r["P"] * r["dP"]).sum(axis=1), atol=1e-12)
    np.testing.assert_allclose(r["dV"].sum(axis=0), do.sum(axis=0), atol=1e-12)
    np.testing.assert_allclose(r["dK"].sum(axis=0), 0.0, atol=1e-12)
    if causal:
        assert np.all(r["P"][np.triu_indices(N, 1)] == 0.0)


def test_gqa_equals_repeated_mha():
    rng = np.random.default_rng(4)
    B, H, H_kv, N, d = 2, 6, 2, 9, 4
    G = H // H_kv
    Q, dO = _rand(rng, (B, H, N, d)), _rand(rng, (B, H, N, d))
    K, V = _rand(rng, (B, H_kv, N, d)), _rand(rng, (B, H_kv, N, d))
    scale = 0.4
    dQ, dK, dV = attention_backward(Q, K, V, dO, scale, True, 0.0)
    Kr, Vr = np.repeat(K, G, axis=1), np.repeat(V, G, axis=1)
    dQm, dKm, dVm = attention_backward(Q, Kr, Vr, dO, scale, True, 0.0)
    np.testing.assert_allclose(dQ, dQm, atol=1e-13)
    np.testing.assert_allclose(dK, dKm.reshape(B, H_kv, G, N, d).sum(axis=2), atol=1e-12)
    np.testing.assert_allclose(dV, dVm.reshape(B, H_kv, G, N, d).sum(axis=2), atol=1e-12)
    # the group column sums of dV equal the group's dO column sums
    np.testing.assert_allclose(dV.sum(axis=2), dO.reshape(B, H_kv, G, N, d).sum(axis=(2, 3)),
                               atol=1e-12)
    # slice API agrees with the full API
    sl = attention_backward(Q, K, V, dO, scale, True, 0.0, slices=[(1, 1)])[(1, 1)]
    np.testing.assert_allclose(sl["dK"], dK[1, 1], atol=0)
    np.testing.assert_allclose(sl["dQ"], dQ[1, G:2 * G], atol=0)


# --------------------------------------------------------------------------
# special cases
# --------------------------------------------------------------------------
def test_equal_keys_give_zero_dq():
    rng = np.random.default_rng(6)
    N, d = 16, 4
    q, v, do = (_rand(rng, (N, d)) for _ in range(3))
    k = np.tile(_rand(rng, (1, d)), (N, 1))
    r = head_backward(q, k, v, do, 0.5)
    np.testing.assert_allclose(r["P"], 1.0 / N, atol=1e-15)
    np.testing.assert_allclose(r["dQ"], 0.0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_values_give_zero_dq_dk(causal):
    rng = np.random.default_rng(8)
    N, d = 16, 4
    q, k, do = (_rand(rng, (N, d)) for _ in range(3))
    v = np.tile(_rand(rng, (1, d)), (N, 1))
    r = head_backward(q, k, v, do, 0.5, causal)
    np.testing.assert_allclose(r["dS"], 0.0, atol=1e-13)
    np.testing.assert_allclose(r["dQ"], 0.0, atol=1e-13)
    np.testing.assert_allclose(r["dK"], 0.0, atol=1e-13)


def test_causal_first_row_and_last_key():
    rng = np.random.default_rng(12)
    N, d = 11, 4
    q, k, v, do = (_rand(rng, (N, d)) for _ in range(4))
    r = head_backward(q, k, v, do, 0.5, causal=True)
    assert r["P"][0, 0] == 1.0
    np.testing.assert_allclose(r["dS"][0], 0.0, atol=1e-15)
    np.testing.assert_allclose(r["dQ"][0], 0.0, atol=1e-15)
    np.testing.assert_allclose(r["dV"][N - 1], r["P"][N - 1, N - 1] * do[N - 1], atol=1e-14)


def test_huge_softcap_matches_plain():
    rng = np.random.default_rng(13)
    N, d = 12, 4
    q, k, v, do = (_rand(rng, (N, d)) for _ in range(4))
    a = head_backward(q, k, v, do, 0.5, True, 0.0)
    b = head_backward(q, k, v, do, 0.5, True, 1e6)
    for name in ("dQ", "dK", "dV"):
        np.testing.assert_allclose(b[name], a[name], atol=1e-9)


def test_rescaled_q_and_tau():
    rng = np.random.default_rng(14)
    N, d = 10, 4
    q, k, v, do = (_rand(rng, (N, d)) for _ in range(4))
    a = head_backward(q, k, v, do, 0.5)
    b = head_backward(3.0 * q, k, v, do, 0.5 / 3.0)
    np.testing.assert_allclose(b["P"], a["P"], atol=1e-14)
    np.testing.assert_allclose(b["dQ"], a["dQ"] / 3.0, atol=1e-13)
    np.testing.assert_allclose(b["dK"], a["dK"], atol=1e-13)


def test_saturated_softcap_kills_gradient():
    # with c small and large logits, tanh saturates: dZ -> 0 where |Z/c| >> 1
    N, d = 4, 1
    q = np.array([[10.0], [10.0], [10.0], [10.0]])
    k = np.array([[10.0], [-10.0], [10.0], [-10.0]])
    v = np.array([[1.0], [2.0], [3.0], [4.0]])
    do = np.ones((N, d))
    r = head_backward(q, k, v, do, 1.0, False, 1.0)
    assert np.abs(r["dZ"]).max() < 1e-60 or np.abs(r["dQ"]).max() < 1e-12


# --------------------------------------------------------------------------
# dropout: the Philox generator and the dropped forward/backward
# --------------------------------------------------------------------------
from oracle import dropout_keep_mask, keep_threshold, philox4x32_10  # noqa: E402

# Known-answer vectors of Philox4x32-10 (counter, key -> output) published
# with the Random123 library of Salmon et al.
PHILOX_KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,out", PHILOX_KAT)
def test_philox_known_answers(ctr, key, out):
    got = philox4x32_10(*ctr, *key)
    assert tuple(int(x) for x in got) == out


def test_keep_mask_rate_and_layout():
    p = 0.3
    keep = dropout_keep_mask(12345, 3, 256, 256, p)
    assert abs(keep.mean() - (1 - p)) < 0.01
    # word i % 4 of the counter (i // 4, j, bh, 0)
    w = philox4x32_10(5, 7, 3, 0, 12345, 0)
    for i in range(20, 24):
        assert keep[i, 7] == (int(w[i - 20]) >= keep_threshold(p))
    assert dropout_keep_mask(1, 0, 8, 8, 0.0).all()


# The keep threshold for drop probability p is round(p32 * 2^32), half up,
# where p32 is the float32 value of p: the library receives p as a C float,
# and the keep decision is an integer decision both sides must take alike.
# Values worked out by hand from float32 bit patterns:
#   0.5  = 2^-1                 -> 2^31
#   0.25 = 2^-2                 -> 2^30
#   float32(0.1) = 13421773 * 2^-27 (0x3DCCCCCD) -> 13421773 * 2^5 = 429496736
#       (a float64 p would give 0.1 * 2^32 = 429496729.6 -> 429496730)
#   2^-33                       -> 0.5 exactly -> 1 (half up; half-even and
#                                  truncation both give 0)
#   3 * 2^-33                   -> 1.5 -> 2
#   1 - 2^-24 (largest float32 below 1) -> 2^32 - 2^8 = 4294967040
#   0                           -> 0 (every word keeps)
KEEP_THRESHOLD_PINS = [
    (0.5, 2**31),
    (0.25, 2**30),
    (np.float32(0.1), 429496736),
    (0.1, 429496736),
    (2.0**-33, 1),
    (3 * 2.0**-33, 2),
    (1.0 - 2.0**-24, 4294967040),
    (0.0, 0),
]


@pytest.mark.parametrize("p,want", KEEP_THRESHOLD_PINS)
def test_keep_threshold_hand_values(p, want):
    assert keep_threshold(p) == want


def test_keep_threshold_float32_reading_differs_from_float64():
    # 0.1 as float64 times 2^32 rounds to 429496730; the float32 reading taken
    # here must not give that
    assert keep_threshold(0.1) != 429496730
    assert keep_threshold(np.float64(0.1)) == keep_threshold(np.float32(0.1))


def test_keep_mask_seed_words_and_threshold_edge():
    """A seed of 2^40 + 7 splits into key (7, 256); a word equal to the
    threshold keeps its element and one below it drops (u >= threshold)."""
    seed, bh, p = 2**40 + 7, 5, 0.2
    keep = dropout_keep_mask(seed, bh, 12, 9, p)
    thr = keep_threshold(p)
    for i in range(12):
        for j in range(9):
            w = philox4x32_10(i // 4, j, bh, 0, 7, 256)
            assert keep[i, j] == (int(w[i % 4]) >= thr)
    # choose p so that the threshold equals one of the words exactly: that
    # element is kept, and with the threshold one above it, dropped
    w00 = int(philox4x32_10(0, 0, bh, 0, 7, 256)[0])
    p_eq = float(np.float32(w00 / 2.0**32))
    t_eq = keep_threshold(p_eq)
    assert dropout_keep_mask(seed, bh, 1, 1, p_eq)[0, 0] == (w00 >= t_eq)
    assert abs(t_eq - w00) <= 256  # float32 p resolves the word to 2^8 at most


DROP_CASES = [
    # B, H, H_kv, N, d, causal, softcap, p_drop
    (1, 1, 1, 5, 2, False, 0.0, 0.4),
    (1, 2, 1, 5, 3, True, 0.0, 0.25),
    (1, 2, 2, 4, 2, True, 2.0, 0.5),
]


def _drop_case(case, seed=9):
    B, H, H_kv, N, d, causal, cap, p = case
    rng = np.random.default_rng(seed)
    Q, K, V = _rand(rng, (B, H, N, d)), _rand(rng, (B, H_kv, N, d)), _rand(rng, (B, H_kv, N, d))
    dO = _rand(rng, (B, H, N, d))
    keep = [[dropout_keep_mask(77, b * H + h, N, N, p).tolist() for h in range(H)]
            for b in range(B)]
    return Q, K, V, dO, 1.0 / math.sqrt(d), causal, cap, p, keep


@pytest.mark.parametrize("case", DROP_CASES)
def test_dropout_forward_matches_brute_force(case):
    Q, K, V, dO, scale, causal, cap, p, keep = _drop_case(case)
    O, LSE = attention_forward(Q, K, V, scale, causal, cap, dropout=(p, 77))
    Ob, LSEb = brute_forward(Q.tolist(), K.tolist(), V.tolist(), scale, causal, cap, keep, p)
    np.testing.assert_allclose(O, np.array(Ob), atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE, np.array(LSEb), atol=1e-12, rtol=0)


def _fd_dropout(Q, K, V, dO, scale, causal, cap, keep, p, h=1e-6):
    def loss(Qx, Kx, Vx):
        O, _ = brute_forward(Qx.tolist(), Kx.tolist(), Vx.tolist(), scale, causal, cap, keep, p)
        return float((np.array(O) * dO).sum())

    grads = []
    for which in range(3):
        base = [Q, K, V][which]
        g = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            args_p = [Q.copy(), K.copy(), V.copy()]
            args_m = [Q.copy(), K.copy(), V.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            g[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        grads.append(g)
    return grads


@pytest.mark.parametrize("case", DROP_CASES)
def test_dropout_backward_matches_finite_differences(case):
    Q, K, V, dO, scale, causal, cap, p, keep = _drop_case(case)
    dQ, dK, dV = attention_backward(Q, K, V, dO, scale, causal, cap, dropout=(p, 77))
    fQ, fK, fV = _fd_dropout(Q, K, V, dO, scale, causal, cap, keep, p)
    assert _rel(dQ, fQ) < 1e-7
    assert _rel(dK, fK) < 1e-7
    assert _rel(dV, fV) < 1e-7


def test_dropout_zero_is_plain_and_d_identity():
    Q, K, V, dO, scale, causal, cap, p, keep = _drop_case(DROP_CASES[1])
    a = attention_backward(Q, K, V, dO, scale, causal, cap)
    b = attention_backward(Q, K, V, dO, scale, causal, cap, dropout=(0.0, 77))
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    # D = rowsum(dO o O) = rowsum(P o dP) with dP taken through the dropout
    km = np.array(keep[0][1])
    r = head_backward(Q[0, 1], K[0, 0], V[0, 0], dO[0, 1], scale, causal, cap, None, km, p)
    np.testing.assert_allclose(r["D"], (r["P"] * r["dP"]).sum(axis=1), atol=1e-12)


def test_dropout_missing_rescale_fails_fd():
    """A backward that forgets the 1 / (1 - p) on dP is caught."""
    Q, K, V, dO, scale, causal, cap, p, keep = _drop_case(DROP_CASES[0])
    km = np.array(keep[0][0])
    fw = head_forward(Q[0, 0], K[0, 0], V[0, 0], scale, causal, cap, km, p)
    dP = np.where(km, dO[0, 0] @ V[0, 0].T, 0.0)  # mistake: no 1 / (1 - p)
    D = (dO[0, 0] * fw["O"]).sum(axis=1)
    dS = fw["P"] * (dP - D[:, None])
    dQ = scale * dS @ K[0, 0]
    fQ, _, _ = _fd_dropout(Q, K, V, dO, scale, causal, cap, keep, p)
    assert _rel(dQ[None, None], fQ) > 1e-3


# --------------------------------------------------------------------------
# local window
# --------------------------------------------------------------------------
WIN_CASES = [
    # B, H, H_kv, N, d, causal, softcap, (left, right)
    (1, 1, 1, 6, 2, False, 0.0, (1, 2)),
    (1, 2, 1, 6, 3, True, 0.0, (2, -1)),
    (1, 2, 2, 5, 2, False, 2.0, (0, 0)),
    (1, 1, 1, 7, 2, False, 0.0, (-1, 1)),
]


def _win_case(case, seed=13):
    B, H, H_kv, N, d, causal, cap, win = case
    rng = np.random.default_rng(seed)
    Q, K, V = _rand(rng, (B, H, N, d)), _rand(rng, (B, H_kv, N, d)), _rand(rng, (B, H_kv, N, d))
    dO = _rand(rng, (B, H, N, d))
    return Q, K, V, dO, 1.0 / math.sqrt(d), causal, cap, win


@pytest.mark.parametrize("case", WIN_CASES)
def test_window_forward_matches_brute_force(case):
    Q, K, V, dO, scale, causal, cap, win = _win_case(case)
    O, LSE = attention_forward(Q, K, V, scale, causal, cap, window=win)
    Ob, LSEb = brute_forward(Q.tolist(), K.tolist(), V.tolist(), scale, causal, cap, window=win)
    np.testing.assert_allclose(O, np.array(Ob), atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE, np.array(LSEb), atol=1e-12, rtol=0)


@pytest.mark.parametrize("case", WIN_CASES)
def test_window_backward_matches_finite_differences(case):
    Q, K, V, dO, scale, causal, cap, win = _win_case(case)
    dQ, dK, dV = attention_backward(Q, K, V, dO, scale, causal, cap, window=win)

    def loss(Qx, Kx, Vx):
        O, _ = brute_forward(Qx.tolist(), Kx.tolist(), Vx.tolist(), scale, causal, cap,
                             window=win)
        return float((np.array(O) * dO).sum())

    h = 1e-6
    for which, got in enumerate((dQ, dK, dV)):
        base = [Q, K, V][which]
        g = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            ap = [Q.copy(), K.copy(), V.copy()]
            am = [Q.copy(), K.copy(), V.copy()]
            ap[which][idx] += h
            am[which][idx] -= h
            g[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        # relative to the gradient's size, or absolute where it vanishes
        # (window (0, 0) leaves dQ = dK = 0 exactly)
        assert np.abs(got - g).max() <= 1e-7 * max(np.abs(g).max(), 1.0)


def test_window_special_cases():
    Q, K, V, dO, scale, causal, cap, win = _win_case((1, 2, 1, 6, 2, False, 0.0, (0, 0)))
    # an unbounded or wider-than-N window is no window; (-1, 0) is causal
    plain = attention_backward(Q, K, V, dO, scale, False, 0.0)
    for w in ((-1, -1), (10, 10), (6, 6)):
        for x, y in zip(plain, attention_backward(Q, K, V, dO, scale, False, 0.0, window=w)):
            np.testing.assert_array_equal(x, y)
    causal_ = attention_backward(Q, K, V, dO, scale, True, 0.0)
    for x, y in zip(causal_, attention_backward(Q, K, V, dO, scale, False, 0.0, window=(-1, 0))):
        np.testing.assert_array_equal(x, y)
    # window (0, 0): every query sees only its own key, P = 1, dS = 0
    dQ, dK, dV = attention_backward(Q, K, V, dO, scale, False, 0.0, window=(0, 0))
    np.testing.assert_allclose(dQ, 0.0, atol=1e-15)
    np.testing.assert_allclose(dK, 0.0, atol=1e-15)
    np.testing.assert_allclose(dV[0, 0], dO[0, 0] + dO[0, 1], atol=1e-14)
