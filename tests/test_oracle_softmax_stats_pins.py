"""Pins of the oracle's softmax statistics (oracle.softmax_stats): the weight
on key 0 (the first-token share, "10 . 门控" sec. 3.4) and the log of the
softmax denominator, per query row and head, without the values or the gate.

Each pin is independent of the oracle's code: closed forms (all scores equal;
a single visible key), torch's CPU float64 logsumexp of scores formed with a
torch matmul (a library routine), and the full oracle's statistics, which are
pinned on their own in test_oracle_pins.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(B, Lq, Lk, Hq, Hkv, dk, seed):
    g = torch.Generator().manual_seed(seed)
    Q = torch.randn((B, Lq, Hq, dk), generator=g, dtype=torch.float64)
    K = torch.randn((B, Lk, Hkv, dk), generator=g, dtype=torch.float64)
    return Q, K


def test_equal_scores_give_the_harmonic_share_and_log_of_the_key_count():
    # Q = 0: every visible score is 0, so p_0 = 1 / (a + 1) and lse = log(a + 1)
    # with a = L_k - L_q + i the row's absolute position (bottom-right alignment)
    B, Lq, Lk, Hq, Hkv, dk = 2, 13, 20, 4, 2, 8
    Q = torch.zeros((B, Lq, Hq, dk), dtype=torch.float64)
    _, K = _rand(B, Lq, Lk, Hq, Hkv, dk, 1)
    p0, lse = oracle.softmax_stats(Q, K, causal=True)
    a = np.arange(Lq) + (Lk - Lq)
    np.testing.assert_allclose(p0, np.broadcast_to((1.0 / (a + 1))[None, :, None], p0.shape), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(a + 1.0)[None, :, None], lse.shape), rtol=0, atol=1e-14)
    # square causal case: the share is the harmonic number over L
    Lsq = 17
    Q2 = torch.zeros((1, Lsq, 2, dk), dtype=torch.float64)
    _, K2 = _rand(1, Lsq, Lsq, 2, 1, dk, 2)
    p0s, _ = oracle.softmax_stats(Q2, K2, causal=True)
    harmonic = sum(1.0 / k for k in range(1, Lsq + 1)) / Lsq
    np.testing.assert_allclose(oracle.sink_share(p0s), harmonic, rtol=0, atol=1e-15)
    # without the mask every row sees all L_k keys
    p0n, lsen = oracle.softmax_stats(Q, K, causal=False)
    np.testing.assert_allclose(p0n, 1.0 / Lk, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lsen, math.log(Lk), rtol=0, atol=1e-14)


def test_one_visible_key_has_all_the_weight():
    # L_q = L_k = 1: p_0 = 1 and lse = s_0 = <q, k_0> / sqrt(d_k)
    Q, K = _rand(3, 1, 1, 4, 4, 16, 3)
    p0, lse = oracle.softmax_stats(Q, K, causal=True)
    s0 = (Q[:, 0] * K[:, 0]).sum(-1).numpy() / math.sqrt(16)
    np.testing.assert_allclose(p0, 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[:, 0], s0, rtol=0, atol=1e-13)


@pytest.mark.parametrize("B,Lq,Lk,Hq,Hkv,dk,causal", [
    (2, 9, 9, 4, 2, 8, True),
    (1, 5, 23, 6, 3, 4, True),      # bottom-right suffix, GQA
    (2, 7, 11, 2, 1, 1, False),     # no mask, d_k = 1
])
def test_matches_torch_logsumexp_of_library_scores(B, Lq, Lk, Hq, Hkv, dk, causal):
    Q, K = _rand(B, Lq, Lk, Hq, Hkv, dk, 10 + Lq)
    p0, lse = oracle.softmax_stats(Q, K, causal=causal)
    Kr = K.repeat_interleave(Hq // Hkv, dim=2)                       # [B, Lk, Hq, dk]
    S = torch.einsum("bihc,bjhc->bhij", Q, Kr) / math.sqrt(dk)       # [B, Hq, Lq, Lk]
    if causal:
        a = torch.arange(Lq)[:, None] + (Lk - Lq)
        S = S.masked_fill(torch.arange(Lk)[None, :] > a, float("-inf"))
    ref_lse = torch.logsumexp(S, dim=-1).permute(0, 2, 1).numpy()    # [B, Lq, Hq]
    ref_p0 = torch.softmax(S, dim=-1)[..., 0].permute(0, 2, 1).numpy()
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(p0, ref_p0, rtol=0, atol=1e-14)


def test_agrees_with_the_full_oracle():
    B, Lq, Lk, Hq, Hkv, dk = 1, 31, 40, 4, 1, 16
    Q, K = _rand(B, Lq, Lk, Hq, Hkv, dk, 7)
    V = torch.randn((B, Lk, Hkv, dk), generator=torch.Generator().manual_seed(8), dtype=torch.float64)
    _, p0_full, lse_full = oracle.gated_sdpa(None, Q, K, V, None, gate="none", causal=True, return_lse=True)
    p0, lse = oracle.softmax_stats(Q, K, causal=True)
    np.testing.assert_allclose(p0, p0_full, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, lse_full, rtol=0, atol=1e-13)
