"""Pins of the oracle's whole layer (projections, attention, output
projection; "GatedAttention [2025]", sec. 1.2.1 and 1.2.2), along a path that
does not call the attention oracle: with W_Q = 0 every score of a row is equal,
so each head's attention output is the mean of the visible values (a causal
prefix mean, computed here with cumulative sums); and linearity in W_O."""
import numpy as np
import pytest
from scipy.special import expit

import oracle


def _inputs(B=2, L=6, dm=5, Hq=4, Hkv=2, dk=3, gated=True, seed=0):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((B, L, dm))
    n_in = (Hq + 2 * Hkv) * dk + (Hq * dk if gated else 0)
    W_in = rng.standard_normal((dm, n_in))
    W_O = rng.standard_normal((Hq * dk, dm))
    return X, W_in, W_O


@pytest.mark.parametrize("gate", ["elementwise", "none"])
@pytest.mark.parametrize("causal", [True, False])
def test_zero_query_weights_give_the_prefix_mean_of_the_values(gate, causal):
    B, L, dm, Hq, Hkv, dk = 2, 6, 5, 4, 2, 3
    X, W_in, W_O = _inputs(gated=gate != "none")
    W_in[:, :Hq * dk] = 0.0                       # Q = 0: all scores 0
    Y = oracle.gated_attention_layer(X, W_in, W_O, Hq, Hkv, dk, gate=gate, causal=causal)
    qc, kc = Hq * dk, Hkv * dk
    V = (X @ W_in[:, qc + kc:qc + 2 * kc]).reshape(B, L, Hkv, dk)
    if causal:
        mean = np.cumsum(V, axis=1) / np.arange(1, L + 1)[None, :, None, None]
    else:
        mean = np.broadcast_to(V.mean(axis=1, keepdims=True), V.shape)
    O = np.repeat(mean, Hq // Hkv, axis=2).reshape(B, L, qc)   # head h reads kv head h // (Hq/Hkv)
    if gate != "none":
        O = O * expit(X @ W_in[:, qc + 2 * kc:])
    np.testing.assert_allclose(Y, O @ W_O, rtol=1e-12, atol=1e-12)


def test_linear_in_the_output_projection():
    X, W_in, W_O = _inputs(seed=1)
    W2 = np.random.default_rng(2).standard_normal(W_O.shape)
    a = oracle.gated_attention_layer(X, W_in, W_O, 4, 2, 3)
    b = oracle.gated_attention_layer(X, W_in, W2, 4, 2, 3)
    c = oracle.gated_attention_layer(X, W_in, W_O + 2 * W2, 4, 2, 3)
    np.testing.assert_allclose(c, a + 2 * b, rtol=1e-12, atol=1e-12)


def test_rows_form_equals_the_full_layer():
    X, W_in, W_O = _inputs(seed=3)
    full = oracle.gated_attention_layer(X, W_in, W_O, 4, 2, 3)
    rows = [(0, 0), (1, 5), (0, 3)]
    got = oracle.gated_attention_layer(X, W_in, W_O, 4, 2, 3, rows=rows)
    np.testing.assert_allclose(got, np.stack([full[b, i] for b, i in rows]), rtol=1e-13, atol=1e-13)


def test_headwise_layer_equals_elementwise_with_each_heads_column_repeated():
    # the headwise gate (one scalar per head and token, "GatedAttention [2025]"
    # sec. 1.2.2) is the elementwise gate whose d_k columns of head h all equal
    # column h: the two layers agree when W_in's gate block is widened that way
    Hq, Hkv, dk = 4, 2, 3
    X, W_in, W_O = _inputs(seed=4, gated=False)
    Wg_head = np.random.default_rng(5).standard_normal((X.shape[-1], Hq))
    head = oracle.gated_attention_layer(X, np.concatenate([W_in, Wg_head], axis=1), W_O, Hq, Hkv, dk,
                                        gate="headwise")
    elem = oracle.gated_attention_layer(X, np.concatenate([W_in, np.repeat(Wg_head, dk, axis=1)], axis=1), W_O,
                                        Hq, Hkv, dk, gate="elementwise")
    np.testing.assert_allclose(head, elem, rtol=1e-12, atol=1e-12)
