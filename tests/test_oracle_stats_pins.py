"""Pins of the oracle's gate scores and the gate statistics ("GatedAttention
[2025]", sec. 1.4.2: mean gating score, score distribution, fraction below a
threshold): the scores against scipy's logistic function of a numpy matmul and
against the (pinned) layer's gated / ungated outputs; the statistics on a
hand-made example and by their invariants."""
import numpy as np
import pytest
from scipy.special import expit

import oracle


@pytest.mark.parametrize("gate", ["elementwise", "headwise"])
def test_gate_scores_equal_expit_of_matmul(gate):
    rng = np.random.default_rng(11)
    B, L, dm, Hq, dk = 2, 5, 7, 3, 4
    X = rng.standard_normal((B, L, dm))
    G = Hq * dk if gate == "elementwise" else Hq
    W = rng.standard_normal((dm, G))
    got = oracle.gate_scores(X, W, Hq, dk, gate=gate)
    np.testing.assert_allclose(got, expit(X.reshape(-1, dm) @ W), rtol=1e-14, atol=1e-15)


def test_gate_scores_are_the_layers_gate():
    # gated output / ungated output = the score (where the ungated output is not ~0)
    rng = np.random.default_rng(12)
    B, L, Hq, Hkv, dk, dm = 1, 6, 2, 1, 4, 5
    X = rng.standard_normal((B, L, dm))
    Q = rng.standard_normal((B, L, Hq, dk))
    K = rng.standard_normal((B, L, Hkv, dk))
    V = rng.standard_normal((B, L, Hkv, dk))
    W = rng.standard_normal((dm, Hq * dk))
    y = oracle.gated_sdpa(X, Q, K, V, None, gate="none")[0]
    o = oracle.gated_sdpa(X, Q, K, V, W, gate="elementwise")[0]
    s = oracle.gate_scores(X, W, Hq, dk).reshape(B, L, Hq, dk)
    m = np.abs(y) > 1e-3
    np.testing.assert_allclose((o / np.where(m, y, 1))[m], s[m], rtol=1e-10)


def test_gate_statistics_hand_example():
    st = oracle.gate_statistics([0.0, 0.05, 0.1, 0.5, 0.99, 1.0], 10, 0.1)
    assert st["count"] == 6
    assert st["below"] == 2                       # 0 and 0.05 (0.1 is not below 0.1)
    assert st["mean"] == pytest.approx((0.05 + 0.1 + 0.5 + 0.99 + 1.0) / 6, rel=1e-15)
    assert list(st["hist"]) == [2, 1, 0, 0, 0, 1, 0, 0, 0, 2]   # 1.0 falls in the last bin


def test_gate_statistics_invariants():
    rng = np.random.default_rng(13)
    s = expit(rng.standard_normal(1000) * 3)
    for n in (1, 7, 32):
        st = oracle.gate_statistics(s, n, 0.25)
        assert st["hist"].sum() == st["count"] == 1000
        assert st["below"] == np.count_nonzero(s < 0.25)
    assert oracle.gate_statistics(s, 4, 0.25)["hist"][0] == oracle.gate_statistics(s, 4, 0.25)["below"]
