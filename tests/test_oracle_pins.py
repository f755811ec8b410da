"""Pins for the float64 oracle: closed forms, invariants and a library routine.

Each test checks the oracle against something other than itself, chosen so
that a plausible slip (a dropped 1/sqrt(d_k), a flipped causal mask, a wrong
GQA head map, a transposed gate column order, a missing sigmoid, an
off-by-one on the first token) fails at least one of them:

  * the hand-derived golden cases (tests/golden/hand_cases.json);
  * torch's CPU float64 scaled_dot_product_attention (a library routine);
  * numpy matmul + scipy's expit for the gate (library routines);
  * closed forms: equal scores give the (prefix) mean of V; V = 1 gives the
    gate itself; one key gives V (.) gate; Q = 0 gives the harmonic first-token
    share H_L / L; logits of +-200 give plain SDPA or zero;
  * invariants: GQA == MHA with K/V repeated per group, causal prefix,
    bottom-right alignment == suffix of the square case, batch independence,
    linearity in V, headwise == elementwise with columns tiled, row sampling.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def rnd(seed, *shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def make(seed, B=2, Lq=9, Lk=9, Hq=4, Hkv=2, dk=8, dm=12, gate="elementwise", wscale=0.3):
    X = rnd(seed, B, Lq, dm)
    Q = rnd(seed + 1, B, Lq, Hq, dk)
    K = rnd(seed + 2, B, Lk, Hkv, dk)
    V = rnd(seed + 3, B, Lk, Hkv, dk)
    cols = Hq * dk if gate == "elementwise" else Hq
    W = rnd(seed + 4, dm, cols, scale=wscale)
    return X, Q, K, V, W


def torch_sdpa_f64(Q, K, V, causal):
    """Library reference: torch SDPA in float64 on the CPU, K/V repeated per group."""
    Hq, Hkv = Q.shape[2], K.shape[2]
    q = torch.from_numpy(Q).permute(0, 2, 1, 3)
    k = torch.from_numpy(K).permute(0, 2, 1, 3).repeat_interleave(Hq // Hkv, dim=1)
    v = torch.from_numpy(V).permute(0, 2, 1, 3).repeat_interleave(Hq // Hkv, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal)
    return o.permute(0, 2, 1, 3).numpy()


# --------------------------------------------------------------------------- golden

@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_derived_cases(case):
    a = {k: np.array(case[k], dtype=np.float64) for k in ("X", "Q", "K", "V", "W_g")}
    O, p0 = oracle.gated_sdpa(a["X"], a["Q"], a["K"], a["V"], a["W_g"],
                              gate=case["gate"], causal=case["causal"])
    np.testing.assert_allclose(O, np.array(case["expected_O"]), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(p0, np.array(case["expected_p0"]), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle.sink_share(p0), np.array(case["expected_sink"]), rtol=1e-13)


# --------------------------------------------------------------------------- library routine

@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (6, 1)])
@pytest.mark.parametrize("dk", [1, 4, 64])
def test_ungated_matches_torch_sdpa(causal, Hq, Hkv, dk):
    X, Q, K, V, W = make(10 + dk + Hkv, Hq=Hq, Hkv=Hkv, dk=dk, Lq=17, Lk=17)
    O, _ = oracle.gated_sdpa(None, Q, K, V, None, gate="none", causal=causal)
    np.testing.assert_allclose(O, torch_sdpa_f64(Q, K, V, causal), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("gate", ["elementwise", "headwise"])
def test_gate_plus_200_is_plain_sdpa(gate):
    X, Q, K, V, W = make(3, gate=gate)
    dm = X.shape[-1]
    X1 = np.ones_like(X)
    W1 = np.full_like(W, 200.0 / dm)
    O, _ = oracle.gated_sdpa(X1, Q, K, V, W1, gate=gate, causal=True)
    np.testing.assert_allclose(O, torch_sdpa_f64(Q, K, V, True), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("gate", ["elementwise", "headwise"])
def test_gate_minus_200_is_zero(gate):
    X, Q, K, V, W = make(4, gate=gate)
    dm = X.shape[-1]
    O, _ = oracle.gated_sdpa(np.ones_like(X), Q, K, V, np.full_like(W, -200.0 / dm),
                             gate=gate, causal=True)
    assert np.max(np.abs(O)) < 1e-80


@pytest.mark.parametrize("gate", ["elementwise", "headwise"])
def test_v_ones_gives_the_gate(gate):
    """V = 1 makes y = 1 (rows sum to 1), so O is the gate: sigmoid(X W_g), head-major."""
    X, Q, K, V, W = make(5, gate=gate, Hq=3, Hkv=3, dk=5)
    O, _ = oracle.gated_sdpa(X, Q, K, np.ones_like(V), W, gate=gate, causal=True)
    B, L, Hq, dk = O.shape
    logits = X @ W                                   # library matmul
    if gate == "elementwise":
        g = expit(logits).reshape(B, L, Hq, dk)      # column h*d_k + c
    else:
        g = np.broadcast_to(expit(logits)[..., None], (B, L, Hq, dk))
    np.testing.assert_allclose(O, g, rtol=1e-13, atol=1e-14)


# --------------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("causal", [True, False])
def test_softmax_rows_sum_to_one(causal):
    X, Q, K, V, W = make(6, Lq=7, Lk=13)
    O, _ = oracle.gated_sdpa(None, Q * 3.0, K, np.ones_like(V), None, gate="none", causal=causal)
    np.testing.assert_allclose(O, 1.0, rtol=0, atol=1e-14)


@pytest.mark.parametrize("Lq,Lk", [(11, 11), (4, 11), (1, 11)])
def test_equal_scores_give_prefix_mean(Lq, Lk):
    X, Q, K, V, W = make(7, Lq=Lq, Lk=Lk, Hq=4, Hkv=2)
    O, _ = oracle.gated_sdpa(None, np.zeros_like(Q), K, V, None, gate="none", causal=True)
    Hq, Hkv = Q.shape[2], K.shape[2]
    csum = np.cumsum(V, axis=1)
    for i in range(Lq):
        a = Lk - Lq + i
        mean = csum[:, a] / (a + 1)                       # [B, Hkv, dk]
        expect = np.repeat(mean, Hq // Hkv, axis=1)       # contiguous groups
        np.testing.assert_allclose(O[:, i], expect, rtol=1e-13, atol=1e-14)
    On, _ = oracle.gated_sdpa(None, np.zeros_like(Q), K, V, None, gate="none", causal=False)
    np.testing.assert_allclose(On, np.repeat(V.mean(axis=1, keepdims=True), Hq // Hkv, axis=2)
                               .repeat(Lq, axis=1), rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("gate", ["elementwise", "headwise"])
def test_single_key(gate):
    X, Q, K, V, W = make(8, Lq=1, Lk=1, gate=gate)
    O, p0 = oracle.gated_sdpa(X, Q, K, V, W, gate=gate, causal=True)
    B, _, Hq, dk = O.shape
    Hkv = K.shape[2]
    g = expit(X @ W)
    g = g.reshape(B, 1, Hq, dk) if gate == "elementwise" else g[..., None]
    expect = np.repeat(V, Hq // Hkv, axis=2) * g
    np.testing.assert_allclose(O, expect, rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(p0, 1.0)


@pytest.mark.parametrize("L", [1, 2, 7, 64])
def test_sink_share_harmonic(L):
    X, Q, K, V, W = make(9, Lq=L, Lk=L)
    _, p0 = oracle.gated_sdpa(None, np.zeros_like(Q), K, V, None, gate="none", causal=True)
    harmonic = sum(1.0 / i for i in range(1, L + 1)) / L
    np.testing.assert_allclose(oracle.sink_share(p0), harmonic, rtol=1e-13)


def test_p0_matches_torch_softmax():
    X, Q, K, V, W = make(11, Lq=6, Lk=10, Hq=4, Hkv=2, dk=8)
    _, p0 = oracle.gated_sdpa(None, Q, K, V, None, gate="none", causal=True)
    Lq, Lk = 6, 10
    q = torch.from_numpy(Q).permute(0, 2, 1, 3)
    k = torch.from_numpy(K).permute(0, 2, 1, 3).repeat_interleave(2, dim=1)
    s = (q @ k.transpose(-1, -2)) / math.sqrt(8)
    vis = torch.ones(Lq, Lk, dtype=torch.bool).tril(diagonal=Lk - Lq)   # bottom-right
    s = s.masked_fill(~vis, float("-inf"))
    ref = torch.softmax(s, dim=-1)[..., 0].permute(0, 2, 1).numpy()
    np.testing.assert_allclose(p0, ref, rtol=1e-12)


# --------------------------------------------------------------------------- invariants

@pytest.mark.parametrize("gate", ["none", "elementwise", "headwise"])
def test_gqa_equals_repeated_mha(gate):
    X, Q, K, V, W = make(12, Hq=6, Hkv=2, gate=gate if gate != "none" else "elementwise")
    Wg = None if gate == "none" else W
    Xg = None if gate == "none" else X
    O1, p1 = oracle.gated_sdpa(Xg, Q, K, V, Wg, gate=gate, causal=True)
    Kr, Vr = np.repeat(K, 3, axis=2), np.repeat(V, 3, axis=2)
    O2, p2 = oracle.gated_sdpa(Xg, Q, Kr, Vr, Wg, gate=gate, causal=True)
    np.testing.assert_allclose(O1, O2, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(p1, p2, rtol=1e-14)


def test_causal_prefix_invariance():
    X, Q, K, V, W = make(13, Lq=12, Lk=12)
    O1, _ = oracle.gated_sdpa(X, Q, K, V, W, causal=True)
    i = 5
    X2, Q2, K2, V2 = X.copy(), Q.copy(), K.copy(), V.copy()
    for a in (X2, Q2, K2, V2):
        a[:, i + 1:] = rnd(99, *a[:, i + 1:].shape)
    O2, _ = oracle.gated_sdpa(X2, Q2, K2, V2, W, causal=True)
    np.testing.assert_array_equal(O1[:, :i + 1], O2[:, :i + 1])
    assert np.max(np.abs(O1[:, i + 1:] - O2[:, i + 1:])) > 1e-3


def test_bottom_right_alignment_is_suffix_of_square():
    X, Q, K, V, W = make(14, Lq=12, Lk=12)
    Of, pf = oracle.gated_sdpa(X, Q, K, V, W, causal=True)
    for Lq in (1, 5):
        O, p = oracle.gated_sdpa(X[:, -Lq:], Q[:, -Lq:], K, V, W, causal=True)
        np.testing.assert_allclose(O, Of[:, -Lq:], rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(p, pf[:, -Lq:], rtol=1e-14)


def test_single_query_causal_sees_whole_cache():
    X, Q, K, V, W = make(15, Lq=1, Lk=20)
    O1, _ = oracle.gated_sdpa(X, Q, K, V, W, causal=True)
    O2, _ = oracle.gated_sdpa(X, Q, K, V, W, causal=False)
    np.testing.assert_array_equal(O1, O2)


def test_batch_independence_and_linearity_in_v():
    X, Q, K, V, W = make(16, B=3)
    O, _ = oracle.gated_sdpa(X, Q, K, V, W)
    O1, _ = oracle.gated_sdpa(X[1:2], Q[1:2], K[1:2], V[1:2], W)
    np.testing.assert_array_equal(O[1:2], O1)
    O3, _ = oracle.gated_sdpa(X, Q, K, -2.5 * V, W)
    np.testing.assert_allclose(O3, -2.5 * O, rtol=1e-13, atol=1e-15)


def test_headwise_equals_elementwise_with_tiled_columns():
    X, Q, K, V, W = make(17, gate="headwise", Hq=4, Hkv=2, dk=8)
    Oh, _ = oracle.gated_sdpa(X, Q, K, V, W, gate="headwise")
    We = np.repeat(W, 8, axis=1)       # column h*d_k + c = W[:, h]
    Oe, _ = oracle.gated_sdpa(X, Q, K, V, We, gate="elementwise")
    np.testing.assert_allclose(Oh, Oe, rtol=1e-14, atol=1e-15)


def test_row_sampling_matches_full():
    X, Q, K, V, W = make(18, B=2, Lq=9, Lk=14)
    O, p = oracle.gated_sdpa(X, Q, K, V, W)
    rows = [(1, 8), (0, 0), (1, 3)]
    Os, ps = oracle.gated_sdpa(X, Q, K, V, W, rows=rows)
    for r, (b, i) in enumerate(rows):
        np.testing.assert_array_equal(Os[r], O[b, i])
        np.testing.assert_array_equal(ps[r], p[b, i])


def test_rejects_bad_shapes():
    X, Q, K, V, W = make(19, Lq=9, Lk=5)
    with pytest.raises(ValueError):
        oracle.gated_sdpa(X, Q, K, V, W)            # L_q > L_k
    X, Q, K, V, W = make(19, Hq=3, Hkv=2)
    with pytest.raises(ValueError):
        oracle.gated_sdpa(X, Q, K, V, W[:, :3 * 8])  # H_q % H_kv != 0
