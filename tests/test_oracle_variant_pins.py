"""Pins of the oracle's gate variants ("GatedAttention [2025]", sec. 1.2.2
items (3)-(5), sec. 1.4.1 and sec. 1.4.2), each against something other than
the variant's own code path:

* the head-shared and input-independent shapes equal the (pinned) head-specific
  elementwise / headwise gate with the weights rearranged;
* the additive gates minus the ungated output equal the gate computed with a
  numpy matmul;
* NS-sigmoid is the mean of the ungated and the sigmoid-gated outputs;
* SiLU of the output and the per-head RMSNorm follow from the (pinned) ungated
  output in numpy, and the RMSNorm rows have unit mean square.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _inputs(B=2, Lq=5, Lk=7, Hq=4, Hkv=2, dk=8, dm=6, seed=0):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((B, Lq, dm))
    Q = rng.standard_normal((B, Lq, Hq, dk))
    K = rng.standard_normal((B, Lk, Hkv, dk))
    V = rng.standard_normal((B, Lk, Hkv, dk))
    return X, Q, K, V, rng


def _none(X, Q, K, V, causal):
    return oracle.gated_sdpa_variant(X, Q, K, V, None, gate="none", causal=causal)[0]


def _sig(x):
    return 1.0 / (1.0 + np.exp(-x))


@pytest.mark.parametrize("causal", [True, False])
def test_elementwise_shared_equals_tiled_head_specific(causal):
    X, Q, K, V, rng = _inputs(seed=1)
    B, Lq, Hq, dk = Q.shape
    Ws = rng.standard_normal((X.shape[-1], dk))
    got = oracle.gated_sdpa_variant(X, Q, K, V, Ws, gate="elementwise_shared", causal=causal)[0]
    Wfull = np.tile(Ws, (1, Hq))                      # column h*dk + c = Ws[:, c]
    ref = oracle.gated_sdpa(X, Q, K, V, Wfull, gate="elementwise", causal=causal)[0]
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)


def test_headwise_shared_equals_tiled_headwise():
    X, Q, K, V, rng = _inputs(seed=2)
    Hq = Q.shape[2]
    Ws = rng.standard_normal((X.shape[-1], 1))
    got = oracle.gated_sdpa_variant(X, Q, K, V, Ws, gate="headwise_shared")[0]
    ref = oracle.gated_sdpa(X, Q, K, V, np.tile(Ws, (1, Hq)), gate="headwise")[0]
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)


def test_static_gate_equals_elementwise_with_a_constant_input():
    # sigma(theta) is the elementwise gate of an input that is 1 in its only column
    X, Q, K, V, rng = _inputs(seed=3)
    B, Lq, Hq, dk = Q.shape
    theta = rng.standard_normal((Hq, dk))
    got = oracle.gated_sdpa_variant(None, Q, K, V, theta, gate="static")[0]
    ones = np.ones((B, Lq, 1))
    ref = oracle.gated_sdpa(ones, Q, K, V, theta.reshape(1, Hq * dk), gate="elementwise")[0]
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)
    # zero-initialised theta (sec. 1.4.2 (iii)): the gate is 1/2 everywhere
    half = oracle.gated_sdpa_variant(None, Q, K, V, np.zeros((Hq, dk)), gate="static")[0]
    np.testing.assert_allclose(half, 0.5 * _none(X, Q, K, V, True), rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("gate", ["elementwise", "headwise", "elementwise_shared", "headwise_shared"])
def test_additive_gates_minus_ungated_equal_the_gate(gate):
    X, Q, K, V, rng = _inputs(seed=4)
    B, Lq, Hq, dk = Q.shape
    G = {"elementwise": Hq * dk, "headwise": Hq, "elementwise_shared": dk, "headwise_shared": 1}[gate]
    W = 0.5 * rng.standard_normal((X.shape[-1], G))
    y = _none(X, Q, K, V, True)
    gl = X @ W                                        # [B, Lq, G]
    if gate == "elementwise":
        gl = gl.reshape(B, Lq, Hq, dk)
    elif gate == "headwise":
        gl = np.broadcast_to(gl[..., None], (B, Lq, Hq, dk))
    elif gate == "elementwise_shared":
        gl = np.broadcast_to(gl[:, :, None, :], (B, Lq, Hq, dk))
    else:
        gl = np.broadcast_to(gl[..., None], (B, Lq, Hq, dk))
    for fn, g in (("sigmoid_add", _sig(gl)), ("silu_add", gl * _sig(gl)), ("identity_add", gl)):
        got = oracle.gated_sdpa_variant(X, Q, K, V, W, gate=gate, gate_fn=fn)[0]
        np.testing.assert_allclose(got - y, g, rtol=1e-12, atol=1e-13, err_msg=fn)
    mul = oracle.gated_sdpa_variant(X, Q, K, V, W, gate=gate, gate_fn="sigmoid_mul")[0]
    np.testing.assert_allclose(mul, y * _sig(gl), rtol=1e-12, atol=1e-14)


def test_ns_sigmoid_is_the_mean_of_ungated_and_gated():
    # y (0.5 + 0.5 s) = (y + y s) / 2; and the factor lies in [0.5, 1]
    X, Q, K, V, rng = _inputs(seed=5)
    W = rng.standard_normal((X.shape[-1], Q.shape[2] * Q.shape[3]))
    ns = oracle.gated_sdpa_variant(X, Q, K, V, W, gate="elementwise", gate_fn="ns_sigmoid_mul")[0]
    y = _none(X, Q, K, V, True)
    g = oracle.gated_sdpa(X, Q, K, V, W, gate="elementwise")[0]
    np.testing.assert_allclose(ns, 0.5 * (y + g), rtol=1e-13, atol=1e-15)
    assert np.all(np.abs(ns) <= np.abs(y) + 1e-15) and np.all(np.abs(ns) >= 0.5 * np.abs(y) - 1e-15)


def test_silu_of_the_output():
    X, Q, K, V, _ = _inputs(seed=6)
    y = _none(X, Q, K, V, True)
    got = oracle.gated_sdpa_variant(X, Q, K, V, None, gate="none", gate_fn="silu_self")[0]
    np.testing.assert_allclose(got, y * _sig(y), rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("with_gamma", [False, True])
def test_rmsnorm_per_head(with_gamma):
    X, Q, K, V, rng = _inputs(seed=7)
    Hq, dk = Q.shape[2], Q.shape[3]
    gamma = rng.standard_normal((Hq, dk)) if with_gamma else None
    eps = 1e-6
    y = _none(X, Q, K, V, True)
    got = oracle.gated_sdpa_variant(X, Q, K, V, gamma, gate="none", gate_fn="rmsnorm", eps=eps)[0]
    ref = y / np.sqrt((y * y).mean(axis=-1, keepdims=True) + eps)
    if with_gamma:
        ref = ref * gamma
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)
    if not with_gamma:
        # eps = 0: every head's row has unit mean square
        z = oracle.gated_sdpa_variant(X, Q, K, V, None, gate="none", gate_fn="rmsnorm", eps=0.0)[0]
        np.testing.assert_allclose((z * z).mean(axis=-1), 1.0, rtol=1e-12)


def test_variant_rejects_mismatched_function_and_gate():
    X, Q, K, V, rng = _inputs(seed=8)
    W = rng.standard_normal((X.shape[-1], Q.shape[2] * Q.shape[3]))
    with pytest.raises(ValueError):
        oracle.gated_sdpa_variant(X, Q, K, V, W, gate="elementwise", gate_fn="rmsnorm")
    with pytest.raises(ValueError):
        oracle.gated_sdpa_variant(X, Q, K, V, None, gate="none", gate_fn="silu_add")


def test_default_variant_matches_the_layer():
    X, Q, K, V, rng = _inputs(seed=9)
    for gate, G in (("elementwise", Q.shape[2] * Q.shape[3]), ("headwise", Q.shape[2])):
        W = rng.standard_normal((X.shape[-1], G))
        a = oracle.gated_sdpa_variant(X, Q, K, V, W, gate=gate)[0]
        b = oracle.gated_sdpa(X, Q, K, V, W, gate=gate)[0]
        np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------------ head-shared gates read as averages

@pytest.mark.parametrize("gate", ["elementwise_averaged", "headwise_averaged"])
@pytest.mark.parametrize("fn", ["sigmoid_mul", "ns_sigmoid_mul", "sigmoid_add", "silu_add", "identity_add"])
def test_averaged_gate_is_the_mean_of_the_heads_values(gate, fn):
    # "GatedAttention [2025]" sec. 1.3.2 (ii): the scores of the q heads averaged
    # into one score every head uses. numpy: each head's value of its own logit
    # (scipy-free: 1/(1+e^-x)), the mean over the heads, combined with the
    # pinned ungated output.
    X, Q, K, V, rng = _inputs(seed=11)
    B, Lq, Hq, dk = Q.shape
    G = Hq * dk if gate == "elementwise_averaged" else Hq
    W = rng.standard_normal((X.shape[-1], G))
    y = _none(X, Q, K, V, True)
    gl = X @ W
    gl = gl.reshape(B, Lq, Hq, dk) if gate == "elementwise_averaged" else np.broadcast_to(gl[..., None], (B, Lq, Hq, dk))
    v = {"sigmoid_mul": _sig(gl), "ns_sigmoid_mul": 0.5 + 0.5 * _sig(gl), "sigmoid_add": _sig(gl),
         "silu_add": gl * _sig(gl), "identity_add": gl}[fn]
    vbar = v.mean(axis=2, keepdims=True)              # [B, Lq, 1, dk]: every head the same
    ref = y + vbar if fn in ("sigmoid_add", "silu_add", "identity_add") else y * vbar
    got = oracle.gated_sdpa_variant(X, Q, K, V, W, gate=gate, gate_fn=fn)[0]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_averaged_gate_with_equal_heads_is_the_head_specific_gate():
    # when every head has the same gate columns, the average is each head's own value
    X, Q, K, V, rng = _inputs(seed=12)
    Hq, dk = Q.shape[2], Q.shape[3]
    Wc = rng.standard_normal((X.shape[-1], dk))
    We = np.tile(Wc, (1, Hq))
    got = oracle.gated_sdpa_variant(X, Q, K, V, We, gate="elementwise_averaged")[0]
    ref = oracle.gated_sdpa(X, Q, K, V, We, gate="elementwise")[0]
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)
    Wh = np.tile(rng.standard_normal((X.shape[-1], 1)), (1, Hq))
    got = oracle.gated_sdpa_variant(X, Q, K, V, Wh, gate="headwise_averaged")[0]
    ref = oracle.gated_sdpa(X, Q, K, V, Wh, gate="headwise")[0]
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)


def test_averaged_gate_with_one_head_is_the_head_specific_gate():
    X, Q, K, V, rng = _inputs(Hq=1, Hkv=1, seed=13)
    dk = Q.shape[3]
    W = rng.standard_normal((X.shape[-1], dk))
    got = oracle.gated_sdpa_variant(X, Q, K, V, W, gate="elementwise_averaged")[0]
    ref = oracle.gated_sdpa(X, Q, K, V, W, gate="elementwise")[0]
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)
