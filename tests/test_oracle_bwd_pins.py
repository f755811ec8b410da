"""Pins for the oracle's backward pass and its log-sum-exp output.

Each check is independent of the oracle's own arithmetic:
- torch's CPU float64 autograd through ``scaled_dot_product_attention`` (a
  library routine) and the gate's sigmoid-multiply;
- central finite differences of the forward oracle (itself pinned in
  ``test_oracle_pins.py``);
- invariants of the softmax: shifting a row's scores changes nothing, so the
  keys' gradients of a row sum to zero; rows of p sum to one, so the values'
  gradients sum to the rows' dy;
- grouped-query heads equal multi-head attention with repeated K/V;
- closed forms: one key (the scores carry no gradient), gate logits +-200
  (plain attention gradients / no gradient through the values).
The backward pass is the chain rule of the layer; the gate's part follows
"解密NeurIPS最佳论文：Gated Attention…", sec. 2.2 (the gradient on the gate's
input is the upstream gradient times the ungated context times sigma (1 - sigma)).
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _inputs(B, Lq, Lk, Hq, Hkv, dk, d_model, gate, seed, w_scale=0.3):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((B, Lq, d_model))
    Q = rng.standard_normal((B, Lq, Hq, dk))
    K = rng.standard_normal((B, Lk, Hkv, dk))
    V = rng.standard_normal((B, Lk, Hkv, dk))
    G = Hq * dk if gate == "elementwise" else Hq
    W = rng.standard_normal((d_model, G)) * w_scale
    dO = rng.standard_normal((B, Lq, Hq, dk))
    return X, Q, K, V, W, dO


def _torch_grads(X, Q, K, V, W, dO, gate, causal):
    """The layer through torch float64 autograd (bottom-right causal mask)."""
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in
         dict(X=X, Q=Q, K=K, V=V, W=W).items()}
    B, Lq, Hq, dk = Q.shape
    Lk, Hkv = K.shape[1], K.shape[2]
    grp = Hq // Hkv
    q = t["Q"].transpose(1, 2)
    k = t["K"].repeat_interleave(grp, dim=2).transpose(1, 2)
    v = t["V"].repeat_interleave(grp, dim=2).transpose(1, 2)
    mask = None
    if causal:
        i = torch.arange(Lq)[:, None] + (Lk - Lq)
        j = torch.arange(Lk)[None, :]
        mask = j <= i
    y = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask).transpose(1, 2)
    if gate == "elementwise":
        g = torch.sigmoid(t["X"] @ t["W"]).reshape(B, Lq, Hq, dk)
    elif gate == "headwise":
        g = torch.sigmoid(t["X"] @ t["W"]).reshape(B, Lq, Hq, 1)
    else:
        g = torch.ones(1, dtype=torch.float64)
    loss = (y * g * torch.tensor(dO)).sum()
    loss.backward()
    out = {"dQ": t["Q"].grad.numpy(), "dK": t["K"].grad.numpy(), "dV": t["V"].grad.numpy()}
    if gate != "none":
        out["dX"] = t["X"].grad.numpy()
        out["dW_g"] = t["W"].grad.numpy()
    return out


CASES = [
    # B, Lq, Lk, Hq, Hkv, dk, d_model, gate, causal
    (1, 7, 7, 2, 2, 4, 5, "elementwise", True),
    (2, 6, 6, 4, 2, 8, 6, "headwise", True),
    (1, 5, 9, 4, 1, 4, 3, "elementwise", True),      # bottom-right alignment, MQA
    (2, 6, 6, 2, 1, 8, 4, "none", False),
    (1, 8, 8, 3, 3, 2, 7, "headwise", False),
    (1, 1, 6, 4, 2, 4, 5, "elementwise", True),      # one decode query
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}_Lq{c[1]}_Lk{c[2]}_H{c[3]}-{c[4]}_d{c[5]}_{c[7]}_{'causal' if c[8] else 'full'}")
def test_bwd_matches_torch_autograd(case):
    B, Lq, Lk, Hq, Hkv, dk, dm, gate, causal = case
    X, Q, K, V, W, dO = _inputs(B, Lq, Lk, Hq, Hkv, dk, dm, gate, seed=hash(case) % 1000)
    got = oracle.gated_sdpa_bwd(X, Q, K, V, W, dO, gate=gate, causal=causal)
    ref = _torch_grads(X, Q, K, V, W, dO, gate, causal)
    assert set(got) == set(ref)
    for k in ref:
        np.testing.assert_allclose(got[k], ref[k], rtol=1e-9, atol=1e-11, err_msg=k)


@pytest.mark.parametrize("gate", ["elementwise", "headwise", "none"])
def test_bwd_finite_differences(gate):
    B, Lq, Lk, Hq, Hkv, dk, dm = 1, 4, 6, 4, 2, 3, 5
    X, Q, K, V, W, dO = _inputs(B, Lq, Lk, Hq, Hkv, dk, dm, gate, seed=7)
    got = oracle.gated_sdpa_bwd(X, Q, K, V, W, dO, gate=gate, causal=True)
    args = dict(X=X, Q=Q, K=K, V=V, W_g=W)
    grad_name = {"X": "dX", "Q": "dQ", "K": "dK", "V": "dV", "W_g": "dW_g"}

    def loss(a):
        O, _ = oracle.gated_sdpa(a["X"], a["Q"], a["K"], a["V"], a["W_g"], gate=gate, causal=True)
        return float((O * dO).sum())

    rng = np.random.default_rng(3)
    eps = 1e-6
    names = ["Q", "K", "V"] + (["X", "W_g"] if gate != "none" else [])
    for name in names:
        arr = args[name]
        for _ in range(6):
            idx = tuple(int(rng.integers(s)) for s in arr.shape)
            plus = {k: v.copy() for k, v in args.items()}
            minus = {k: v.copy() for k, v in args.items()}
            plus[name][idx] += eps
            minus[name][idx] -= eps
            fd = (loss(plus) - loss(minus)) / (2 * eps)
            assert abs(fd - got[grad_name[name]][idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd)


def test_bwd_invariants():
    # non-causal rows see every key: the keys' gradients of each (b, kv head) sum to zero
    B, Lq, Lk, Hq, Hkv, dk, dm = 2, 5, 7, 4, 2, 4, 3
    X, Q, K, V, W, dO = _inputs(B, Lq, Lk, Hq, Hkv, dk, dm, "none", seed=11)
    g = oracle.gated_sdpa_bwd(X, Q, K, V, W, dO, gate="none", causal=False)
    np.testing.assert_allclose(g["dK"].sum(axis=1), 0.0, atol=1e-12)
    # rows of p sum to one: sum_j dV_j = sum over the group's rows of dy (= dO without a gate)
    grp = Hq // Hkv
    dy_sum = dO.reshape(B, Lq, Hkv, grp, dk).sum(axis=(1, 3))
    np.testing.assert_allclose(g["dV"].sum(axis=1), dy_sum, rtol=1e-12, atol=1e-12)
    # the same holds causally for dV (every row's p still sums to one)
    gc = oracle.gated_sdpa_bwd(X, Q, K, V, W, dO, gate="none", causal=True)
    np.testing.assert_allclose(gc["dV"].sum(axis=1), dy_sum, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("gate", ["elementwise", "headwise"])
def test_bwd_gqa_equals_mha_with_repeated_kv(gate):
    B, Lq, Lk, Hq, Hkv, dk, dm = 1, 6, 6, 4, 2, 4, 5
    X, Q, K, V, W, dO = _inputs(B, Lq, Lk, Hq, Hkv, dk, dm, gate, seed=5)
    grp = Hq // Hkv
    g = oracle.gated_sdpa_bwd(X, Q, K, V, W, dO, gate=gate, causal=True)
    Kr, Vr = np.repeat(K, grp, axis=2), np.repeat(V, grp, axis=2)
    m = oracle.gated_sdpa_bwd(X, Q, Kr, Vr, W, dO, gate=gate, causal=True)
    np.testing.assert_allclose(g["dQ"], m["dQ"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g["dX"], m["dX"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g["dW_g"], m["dW_g"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g["dK"], m["dK"].reshape(B, Lk, Hkv, grp, dk).sum(axis=3), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g["dV"], m["dV"].reshape(B, Lk, Hkv, grp, dk).sum(axis=3), rtol=1e-12, atol=1e-13)


def test_bwd_one_key():
    # one key: p = 1 whatever the score, so Q and K get no gradient; y = V
    B, Hq, Hkv, dk, dm = 2, 4, 2, 4, 5
    X, Q, K, V, W, dO = _inputs(B, 1, 1, Hq, Hkv, dk, dm, "elementwise", seed=9)
    g = oracle.gated_sdpa_bwd(X, Q, K, V, W, dO, gate="elementwise", causal=True)
    np.testing.assert_allclose(g["dQ"], 0.0, atol=1e-15)
    np.testing.assert_allclose(g["dK"], 0.0, atol=1e-15)
    sig = 1.0 / (1.0 + np.exp(-(X @ W)))                   # [B, 1, Hq*dk]
    grp = Hq // Hkv
    dy = (dO.reshape(B, 1, Hq * dk) * sig).reshape(B, 1, Hkv, grp, dk).sum(axis=3)
    np.testing.assert_allclose(g["dV"], dy, rtol=1e-12)
    y = np.repeat(V, grp, axis=2).reshape(B, 1, Hq * dk)
    dgl = dO.reshape(B, 1, Hq * dk) * y * sig * (1 - sig)
    np.testing.assert_allclose(g["dW_g"], np.einsum("bim,bic->mc", X, dgl), rtol=1e-12)
    np.testing.assert_allclose(g["dX"], np.einsum("bic,mc->bim", dgl, W), rtol=1e-12)


@pytest.mark.parametrize("sign", [+1, -1])
def test_bwd_saturated_gates(sign):
    # logits +-200: sigma = 1 (plain attention gradients) or 0 (no gradient
    # through the attention), and sigma (1 - sigma) = 0 for the gate itself
    B, Lq, Hq, Hkv, dk, dm = 1, 5, 2, 2, 4, 3
    _, Q, K, V, _, dO = _inputs(B, Lq, Lq, Hq, Hkv, dk, dm, "elementwise", seed=13)
    X = np.ones((B, Lq, dm))
    W = np.full((dm, Hq * dk), sign * 200.0 / dm)
    g = oracle.gated_sdpa_bwd(X, Q, K, V, W, dO, gate="elementwise", causal=True)
    np.testing.assert_allclose(g["dX"], 0.0, atol=1e-60)
    np.testing.assert_allclose(g["dW_g"], 0.0, atol=1e-60)
    if sign > 0:
        plain = oracle.gated_sdpa_bwd(None, Q, K, V, None, dO, gate="none", causal=True)
        for k in ("dQ", "dK", "dV"):
            np.testing.assert_allclose(g[k], plain[k], rtol=1e-12, atol=1e-14)
    else:
        for k in ("dQ", "dK", "dV"):
            np.testing.assert_allclose(g[k], 0.0, atol=1e-60)


def test_lse_closed_forms():
    # equal scores: lse = log(number of visible keys); one key: lse = its score
    B, Lq, Lk, Hq, Hkv, dk = 1, 4, 6, 2, 1, 4
    Q = np.zeros((B, Lq, Hq, dk))
    rng = np.random.default_rng(2)
    K = rng.standard_normal((B, Lk, Hkv, dk))
    V = rng.standard_normal((B, Lk, Hkv, dk))
    _, _, lse = oracle.gated_sdpa(None, Q, K, V, None, gate="none", causal=True, return_lse=True)
    visible = np.arange(Lq) + (Lk - Lq) + 1
    np.testing.assert_allclose(lse[0], np.log(visible)[:, None].repeat(Hq, 1), rtol=1e-14)
    Q1 = rng.standard_normal((1, 1, Hq, dk))
    K1 = rng.standard_normal((1, 1, Hkv, dk))
    _, _, lse1 = oracle.gated_sdpa(None, Q1, K1, K1, None, gate="none", causal=True, return_lse=True)
    np.testing.assert_allclose(lse1[0, 0], (Q1[0, 0] @ K1[0, 0, 0]) / np.sqrt(dk), rtol=1e-14)
    # against torch's logsumexp of the scores (library routine), causal bottom-right
    Qr = rng.standard_normal((B, Lq, Hq, dk))
    _, _, lse2 = oracle.gated_sdpa(None, Qr, K, V, None, gate="none", causal=True, return_lse=True)
    s = torch.einsum("bihc,bjc->bhij", torch.tensor(Qr), torch.tensor(K[:, :, 0])) / np.sqrt(dk)
    mask = (torch.arange(Lk)[None, :] <= torch.arange(Lq)[:, None] + (Lk - Lq))
    ref = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1).permute(0, 2, 1).numpy()
    np.testing.assert_allclose(lse2, ref, rtol=1e-13)


@pytest.mark.parametrize("case", [(2, 7, 9, 4, 2, 4, 5, "elementwise", True), (1, 6, 6, 2, 2, 8, 3, "headwise", False),
                                  (1, 5, 5, 3, 1, 4, 0, "none", True)], ids=["gqa_elementwise_causal",
                                                                             "headwise_full", "mqa_none"])
def test_bwd_rows_equals_full_backward(case):
    # the sampled-row form (used at sizes the full form cannot reach) against the pinned full form
    B, Lq, Lk, Hq, Hkv, dk, dm, gate, causal = case
    X, Q, K, V, W, dO = _inputs(B, Lq, Lk, Hq, Hkv, dk, max(dm, 1), gate, seed=21)
    full = oracle.gated_sdpa_bwd(X, Q, K, V, W, dO, gate=gate, causal=causal)
    q_rows = [(b, i) for b in range(B) for i in range(Lq)]
    k_rows = [(b, j) for b in range(B) for j in range(Lk)]
    rows = oracle.gated_sdpa_bwd_rows(X, Q, K, V, W, dO, q_rows, k_rows, gate=gate, causal=causal)
    np.testing.assert_allclose(rows["dQ"], full["dQ"].reshape(-1, Hq, dk), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(rows["dK"], full["dK"].reshape(-1, Hkv, dk), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(rows["dV"], full["dV"].reshape(-1, Hkv, dk), rtol=1e-10, atol=1e-13)
    if gate == "none":
        assert "dX" not in rows
    else:
        np.testing.assert_allclose(rows["dX"], full["dX"].reshape(-1, dm), rtol=1e-10, atol=1e-13)
