"""GPU parity of the backward pass (bf16, d_k = 128) against the float64 oracle.

The GPU side runs the training forward (O and the per-row log-denominators)
and then the backward through the C ABI; the oracle computes the exact
gradients of the same bf16-rounded inputs.

Tolerance. Each gradient element is a float32-accumulated sum of products
whose factors passed through up to four bf16 roundings (P or dS, dY or the
gate gradient, the operand of the last product, and the forward's bf16
output in D = sum(dO O)), each 2^-9 relative. These errors are relative to
the terms, so a gradient's error scales with its magnitude, and magnitudes
grow with the fan-in: dK and dV sum over every query of a key, dW_g over every
token. The bar is therefore relative L1 <= 5e-3 (as for the forward) and
max-abs <= 2e-2 max(1, max|ref|): four roundings give 4 * 2^-9 = 7.8e-3 of
the tensor's scale, with a 2.5x margin, which is the forward's unscaled 2e-2
on any tensor of unit scale or less. An unscaled 2e-2 cannot hold beyond
unit scale whatever the arithmetic: the gradients are returned as bf16, and
a value in [8, 16) (dK and dV reach that) is stored within half a bf16 ulp,
2^-5 = 0.031, of itself. Measured max-abs / max|ref|: 2.6e-3 to
4.4e-3 (each case prints its numbers); at the full headline size the sampled
dQ rows reach max-abs 9.7e-3 (the bf16 rounding of O in D shifts every dS of
a row the same way, so it does not average out over the keys).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_softmax_attention_gb300 import binding as gb
from gated_softmax_attention_gb300 import build as gbuild
from gated_softmax_attention_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

BWD_REL_L1 = 5e-3
BWD_MAX_ABS = 2e-2   # times max(1, max|ref|)


@pytest.fixture(scope="module", autouse=True)
def lib():
    gbuild.build()
    gb.load()


def _w(name, **kw):
    base = dict(name=name, dtype="bf16", B=1, L_q=300, L_k=300, d_model=256, H_q=2, H_kv=2, d_k=128,
                gate="elementwise", causal=True, seed=31)
    base.update(kw)
    return Workload(**base)


CASES = [
    _w("mha_elementwise_ragged"),
    _w("gqa_headwise_b2", B=2, L_q=257, L_k=257, H_q=8, H_kv=2, gate="headwise", seed=32),
    _w("no_gate_full_mask", L_q=200, L_k=300, gate="none", causal=False, seed=33),
    _w("elementwise_bottom_right_suffix", L_q=77, L_k=300, H_q=4, H_kv=1, seed=34),
    # a wide gate: dW_g [2560 x 2048] takes 256 x 512 tiles (K = 72 rows: a full chunk and a ragged one)
    _w("elementwise_wide_gate", L_q=72, L_k=72, d_model=2560, H_q=16, H_kv=4, seed=35),
    # a narrow gate over many rows: dW_g [256 x 8] has two 128 x 128 tiles and K = 1200 rows
    # (19 chunks of 64, the last ragged), so K is split in two, partials summed afterwards
    _w("headwise_split_k_dwg", B=4, L_q=300, L_k=300, H_q=8, H_kv=2, gate="headwise", seed=36),
]


def _dO(w):
    g = torch.Generator().manual_seed(1000 + w.seed)
    return torch.randn((w.B, w.L_q, w.H_q, w.d_k), generator=g).to(torch.bfloat16)


def _check(name, got, ref):
    err = np.abs(got - ref)
    rel = err.sum() / max(np.abs(ref).sum(), 1e-30)
    scale = max(1.0, float(np.abs(ref).max()))
    print(f"{name}: rel-L1 {rel:.2e}  max-abs {err.max():.2e}  max|ref| {np.abs(ref).max():.2e}  "
          f"ratio {err.max() / max(float(np.abs(ref).max()), 1e-30):.2e}")
    assert rel <= BWD_REL_L1, f"{name}: rel-L1 {rel:.3e}"
    assert err.max() <= BWD_MAX_ABS * scale, f"{name}: max-abs {err.max():.3e} vs bar {BWD_MAX_ABS * scale:.3e}"


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_backward_matches_oracle(w):
    t = make_inputs(w)
    dO = _dO(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    O, _, lse = gb.gated_sdpa_fwd_train(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=w.gate,
                                        causal=w.causal)
    g = gb.gated_sdpa_bwd(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], O, dO.cuda(), lse, gate=w.gate,
                          causal=w.causal)
    assert gb.check_device_error() == gb.OK
    ref = oracle.gated_sdpa_bwd(t["X"], t["Q"], t["K"], t["V"], t["W_g"], dO, gate=w.gate, causal=w.causal)
    assert set(g) == set(ref)
    for k in ref:
        _check(f"{w.name} {k}", g[k].double().cpu().numpy(), ref[k])


# ------------------------------------------------------------------ full size, the shape bench.py times

@pytest.mark.parametrize("name", ["bf16_mha_elementwise_L2048", "bf16_gqa_headwise_L4096"])
def test_full_size_backward_sampled_rows_and_properties(name):
    """A full-size workload's backward (the headline shape; GQA 32/4 headwise
    L4096, whose dK/dV units take four query heads each): dQ and dX on sampled
    query rows and dK, dV on sampled key rows against the oracle's row form; and
    two properties of the whole tensors: the values' gradients sum to the rows'
    dy = dO G (rows of p sum to one), and sum(dX X) = sum(dW_g W_g) (both equal
    sum(dGl (X W_g)))."""
    from gated_softmax_attention_gb300.workloads import WORKLOADS
    w = WORKLOADS[name]
    t = make_inputs(w)
    dO = _dO(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    O, _, lse = gb.gated_sdpa_fwd_train(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=w.gate,
                                        causal=w.causal)
    g = gb.gated_sdpa_bwd(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], O, dO.cuda(), lse, gate=w.gate,
                          causal=w.causal)
    assert gb.check_device_error() == gb.OK
    got = {k: v.double().cpu().numpy() for k, v in g.items()}
    rng = np.random.default_rng(5)
    fixed = [(0, 0), (0, 127), (0, 128), (w.B - 1, w.L_q - 1)]
    q_rows = sorted(set(fixed + [(int(rng.integers(w.B)), int(rng.integers(w.L_q))) for _ in range(12)]))
    k_rows = sorted(set(fixed + [(int(rng.integers(w.B)), int(rng.integers(w.L_k))) for _ in range(8)]))
    ref = oracle.gated_sdpa_bwd_rows(t["X"], t["Q"], t["K"], t["V"], t["W_g"], dO, q_rows, k_rows, gate=w.gate,
                                     causal=w.causal)
    _check("full dQ rows", np.stack([got["dQ"][b, i] for b, i in q_rows]), ref["dQ"])
    _check("full dK rows", np.stack([got["dK"][b, j] for b, j in k_rows]), ref["dK"])
    _check("full dV rows", np.stack([got["dV"][b, j] for b, j in k_rows]), ref["dV"])
    _check("full dX rows", np.stack([got["dX"][b, i] for b, i in q_rows]), ref["dX"])
    # properties of the whole tensors
    X = t["X"].double().numpy()
    W = t["W_g"].double().numpy()
    gate = 1.0 / (1.0 + np.exp(-(X @ W)))                                   # [B, L, H*d] or [B, L, H]
    if w.gate == "headwise":
        gate = np.repeat(gate, w.d_k, axis=-1)                              # one value per head, over d_k
    dy = dO.double().numpy().reshape(w.B, w.L_q, -1) * gate
    grp = w.H_q // w.H_kv
    dy_sum = dy.reshape(w.B, w.L_q, w.H_kv, grp, w.d_k).sum(axis=(1, 3))   # [B, H_kv, d]
    dv_sum = got["dV"].sum(axis=1)
    rel = np.abs(dv_sum - dy_sum).sum() / np.abs(dy_sum).sum()
    print(f"sum_j dV_j vs sum_i dy_i: rel-L1 {rel:.2e}")
    assert rel <= BWD_REL_L1
    a = float((got["dX"] * X).sum())
    c = float((got["dW_g"] * W).sum())
    print(f"sum(dX X) {a:.6e}  sum(dW_g W_g) {c:.6e}")
    assert abs(a - c) <= 1e-2 * max(abs(a), abs(c))


@pytest.mark.parametrize("w", [CASES[0], CASES[3]], ids=lambda w: w.name)
def test_saved_gate_backward_equals_recompute(w):
    # the training forward saves sigma(X W_g) as the attention multiplied by it;
    # the backward that takes those values gives the recomputing backward's bits
    t = make_inputs(w)
    d = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    O, _, lse, G = gb.gated_sdpa_fwd_train_save_gate(d["X"], d["Q"], d["K"], d["V"], d["W_g"], causal=w.causal)
    O2, _, lse2 = gb.gated_sdpa_fwd_train(d["X"], d["Q"], d["K"], d["V"], d["W_g"], gate=w.gate, causal=w.causal)
    assert torch.equal(O, O2) and torch.equal(lse, lse2)
    # the saved values are the gate scores: fp16 (2^-11 relative) of a
    # tanh-approximated sigmoid of a float32-accumulated product
    ref = oracle.gate_scores(t["X"], t["W_g"], w.H_q, w.d_k, gate="elementwise")
    assert G.shape == ref.shape and np.abs(G.double().cpu().numpy() - ref).max() <= 2e-3
    dO = _dO(w).cuda()
    a = gb.gated_sdpa_bwd(d["X"], d["Q"], d["K"], d["V"], d["W_g"], O, dO, lse, gate=w.gate, causal=w.causal)
    b = gb.gated_sdpa_bwd(d["X"], d["Q"], d["K"], d["V"], d["W_g"], O, dO, lse, gate=w.gate, causal=w.causal,
                          gate_saved=G)
    assert gb.check_device_error() == gb.OK
    assert a.keys() == b.keys()
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_backward_saturated_headwise_gates():
    """Headwise gate values of exactly 1 and 0 (logits +200 and -200, X = 1): the
    backward folds g into the row statistics (-lse log2 e + log2 g, -D / g), so
    g = 0 takes its own branch (p' = 0, the second statistic 0). The heads with
    g = 0 have zero gradients; those with g = 1 are plain attention's; all
    match the oracle."""
    w = _w("headwise_saturated", B=2, L_q=200, L_k=200, H_q=8, H_kv=2, gate="headwise", seed=38)
    t = make_inputs(w)
    t["X"] = torch.ones_like(t["X"])
    W = torch.empty((w.d_model, w.H_q), dtype=torch.float32)
    for h in range(w.H_q):
        W[:, h] = (200.0 if h % 2 == 0 else -200.0) / w.d_model
    t["W_g"] = W.to(torch.bfloat16)
    dO = _dO(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    O, _, lse = gb.gated_sdpa_fwd_train(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=w.gate,
                                        causal=w.causal)
    g = gb.gated_sdpa_bwd(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], O, dO.cuda(), lse, gate=w.gate,
                          causal=w.causal)
    assert gb.check_device_error() == gb.OK
    assert torch.all(g["dQ"][:, :, 1::2] == 0)   # the heads whose gate is 0
    ref = oracle.gated_sdpa_bwd(t["X"], t["Q"], t["K"], t["V"], t["W_g"], dO, gate=w.gate, causal=w.causal)
    for k in ref:
        got = g[k].double().cpu().numpy()
        if np.abs(ref[k]).max() < 1e-30:   # dX, dW_g: sigma(+-200) (1 - sigma) vanishes (1e-87 in float64)
            assert np.abs(got).max() < 1e-30, k
        else:
            _check(f"{w.name} {k}", got, ref[k])


@pytest.mark.parametrize("B", [8, 32], ids=["chunks_of_four_heads", "whole_groups"])
def test_gqa_backward_equals_repeated_heads(B):
    """GQA 16/2 (groups of 8), L 1024: the dK/dV units take several query heads
    each once the work is large enough (on 132 to 160 SMs: four heads per unit
    at B = 8, whose fp32 shares are then summed over two chunks; a kv head's
    whole group at B = 32, written directly). The gradients must equal the
    MHA backward on K, V repeated over each group (the same O and lse), with dK
    and dV summed over the group: dQ bit for bit (the same per-row arithmetic),
    dK and dV within the bf16 roundings. Bound: the GQA value is T rounded once
    and each MHA term t_h is rounded once, |error| <= 2^-8 |x| for each, so
    |gqa - sum_h mha_h| <= 2^-8 (|sum| + 2 sum_h |mha_h|), plus float32
    accumulation in different orders (1e-3 of the tensor's largest value).
    The mean error is about 2^-9 of a value per rounding (measured rel-L1
    2.2e-3 for dK at B = 8); the whole tensor takes the backward's 5e-3 bar."""
    H_q, H_kv, L = 16, 2, 1024
    group = H_q // H_kv
    w = Workload(name="gqa_units", dtype="bf16", B=B, L_q=L, L_k=L, d_model=128, H_q=H_q, H_kv=H_kv, d_k=128,
                 gate="none", causal=True, seed=37)
    t = make_inputs(w)
    Q, K, V = t["Q"].cuda(), t["K"].cuda(), t["V"].cuda()
    dO = _dO(w).cuda()
    O, _, lse = gb.gated_sdpa_fwd_train(None, Q, K, V, None, gate="none", causal=True)
    g = gb.gated_sdpa_bwd(None, Q, K, V, None, O, dO, lse, gate="none", causal=True)
    Kr = K.repeat_interleave(group, dim=2).contiguous()
    Vr = V.repeat_interleave(group, dim=2).contiguous()
    m = gb.gated_sdpa_bwd(None, Q, Kr, Vr, None, O, dO, lse, gate="none", causal=True)
    assert gb.check_device_error() == gb.OK
    assert torch.equal(g["dQ"], m["dQ"])
    for k in ("dK", "dV"):
        terms = m[k].double().view(B, L, H_kv, group, 128)
        ssum = terms.sum(dim=3)
        bound = 2.0 ** -8 * (ssum.abs() + 2 * terms.abs().sum(dim=3)) + 1e-3 * float(ssum.abs().max())
        err = (g[k].double() - ssum).abs()
        rel = float(err.sum() / ssum.abs().sum())
        print(f"B={B} {k}: max err / bound {float((err / bound).max()):.3f}  rel-L1 {rel:.2e}")
        assert bool((err <= bound).all()), k
        assert rel <= BWD_REL_L1, k
