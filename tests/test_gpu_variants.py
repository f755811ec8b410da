"""GPU parity of the gate variants (gated_sdpa_fwd_variant) against the float64
oracle: every gate shape (head-specific, head-shared, input-independent, and
the head-shared gate read as an average of the heads' values) with every
function of its logit, SiLU of the
output and the per-head RMSNorm (with and without its scale), on the float32
path, the bf16 single-CTA prefill kernel (d_k 128 and 64), the CTA-pair
prefill kernel (sampled rows of a 16384-key case) and the decode kernel.

Bars: the layer's (float32 max-abs <= 1e-4; bf16 max-abs <= 2e-2 and relative
L1 <= 5e-3). The bf16 path keeps the elementwise-family gate values as fp16
between the gate pass and the attention kernel (2^-11 relative), as for the
layer's own gate.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_softmax_attention_gb300 import binding as gb
from gated_softmax_attention_gb300 import build as gbuild
from gated_softmax_attention_gb300.workloads import Workload, make_inputs, variant_weight

pytestmark = pytest.mark.gpu

F32_MAX_ABS = 1e-4
BF16_MAX_ABS = 2e-2
BF16_REL_L1 = 5e-3

GATED_FNS = ["sigmoid_mul", "ns_sigmoid_mul", "sigmoid_add", "silu_add", "identity_add"]
SHAPES = ["elementwise", "headwise", "elementwise_shared", "headwise_shared", "static"]
COMBOS = [(g, f) for g in SHAPES for f in GATED_FNS] + [("none", "silu_self"), ("none", "rmsnorm"),
                                                         ("none", "rmsnorm_nogamma")]


@pytest.fixture(scope="module", autouse=True)
def lib():
    gbuild.build()
    gb.load()
    torch.cuda.init()


def _run(w, t, gate, fn):
    """GPU and oracle outputs of one variant on workload w's inputs t."""
    fn_call = "rmsnorm" if fn == "rmsnorm_nogamma" else fn
    base_gate = gate if gate in ("elementwise", "headwise") else "none"
    W = t["W_g"] if base_gate != "none" and gate == base_gate else variant_weight(w, gate, fn_call)
    if fn == "rmsnorm_nogamma":
        W = None
    X = t["X"]
    dev = lambda x: x.cuda() if x is not None else None
    O, _ = gb.gated_sdpa_fwd_variant(dev(X) if gate not in ("none", "static") else None, dev(t["Q"]), dev(t["K"]),
                                     dev(t["V"]), dev(W), gate=gate, gate_fn=fn_call, eps=1e-6, causal=w.causal)
    assert gb.check_device_error() == gb.OK
    return O.double().cpu().numpy(), X, W


def _check(w, got, ref, what):
    err = np.abs(got - ref)
    if w.dtype == "f32":
        assert err.max() <= F32_MAX_ABS, f"{what}: max-abs {err.max():.3e}"
    else:
        rel = err.sum() / max(np.abs(ref).sum(), 1e-30)
        print(f"{what}: rel-L1 {rel:.2e} max-abs {err.max():.2e}")
        assert err.max() <= BF16_MAX_ABS, f"{what}: max-abs {err.max():.3e} (rel-L1 {rel:.3e})"
        assert rel <= BF16_REL_L1, f"{what}: rel-L1 {rel:.3e} (max-abs {err.max():.3e})"


def _workload(dtype, gate, **kw):
    base = dict(name="variants", dtype=dtype, B=2, L_q=300, L_k=300, d_model=256, H_q=8, H_kv=2, d_k=128,
                gate=gate if gate in ("elementwise", "headwise") else "elementwise", causal=True, seed=41)
    base.update(kw)
    return Workload(**base)


def _full(w, gate, fn):
    t = make_inputs(w)
    got, X, W = _run(w, t, gate, fn)
    ref = oracle.gated_sdpa_variant(X, t["Q"], t["K"], t["V"], W, gate=gate,
                                    gate_fn="rmsnorm" if fn == "rmsnorm_nogamma" else fn, eps=1e-6,
                                    causal=w.causal)[0]
    _check(w, got, ref, f"{w.dtype} d{w.d_k} L{w.L_q}/{w.L_k} {gate}/{fn}")


@pytest.mark.parametrize("gate,fn", COMBOS, ids=[f"{g}-{f}" for g, f in COMBOS])
def test_f32(gate, fn):
    _full(_workload("f32", gate, B=1, L_q=70, L_k=90, d_model=64, H_q=4, H_kv=2, d_k=64), gate, fn)


@pytest.mark.parametrize("gate,fn", COMBOS, ids=[f"{g}-{f}" for g, f in COMBOS])
def test_bf16_prefill(gate, fn):
    _full(_workload("bf16", gate), gate, fn)


@pytest.mark.parametrize("gate,fn", [("elementwise_shared", "silu_add"), ("headwise_shared", "ns_sigmoid_mul"),
                                     ("static", "sigmoid_mul"), ("none", "rmsnorm"), ("none", "silu_self")])
def test_bf16_prefill_dk64(gate, fn):
    _full(_workload("bf16", gate, d_k=64, L_q=200, L_k=260), gate, fn)


# the head-shared gate read as an average over the heads' values
AVG_COMBOS = [(g, f) for g in ("elementwise_averaged", "headwise_averaged") for f in GATED_FNS]


@pytest.mark.parametrize("gate,fn", AVG_COMBOS, ids=[f"{g}-{f}" for g, f in AVG_COMBOS])
def test_averaged_f32(gate, fn):
    _full(_workload("f32", gate, B=1, L_q=70, L_k=90, d_model=64, H_q=4, H_kv=2, d_k=64), gate, fn)


@pytest.mark.parametrize("gate,fn", AVG_COMBOS, ids=[f"{g}-{f}" for g, f in AVG_COMBOS])
def test_averaged_bf16_prefill(gate, fn):
    _full(_workload("bf16", gate), gate, fn)


def test_averaged_bf16_decode_is_unsupported():
    w = _workload("bf16", "elementwise_averaged", B=4, L_q=1, L_k=700)
    t = make_inputs(w)
    W = variant_weight(w, "elementwise_averaged").cuda()
    with pytest.raises(gb.GsdpaError) as ei:
        gb.gated_sdpa_fwd_variant(t["X"].cuda(), t["Q"].cuda(), t["K"].cuda(), t["V"].cuda(), W,
                                  gate="elementwise_averaged", gate_fn="sigmoid_mul", causal=True)
    assert ei.value.status == gb.ERR_UNSUPPORTED
    assert gb.check_device_error() == gb.OK


@pytest.mark.parametrize("gate,fn", COMBOS, ids=[f"{g}-{f}" for g, f in COMBOS])
def test_bf16_decode(gate, fn):
    _full(_workload("bf16", gate, B=4, L_q=1, L_k=700), gate, fn)


PAIR_COMBOS = [("elementwise", "sigmoid_add"), ("elementwise_shared", "ns_sigmoid_mul"),
               ("headwise", "silu_add"), ("headwise_shared", "identity_add"), ("static", "sigmoid_mul"),
               ("none", "silu_self"), ("none", "rmsnorm"), ("elementwise_averaged", "sigmoid_mul"),
               ("headwise_averaged", "silu_add")]


@pytest.mark.parametrize("gate,fn", PAIR_COMBOS, ids=[f"{g}-{f}" for g, f in PAIR_COMBOS])
def test_bf16_pair_kernel_sampled_rows(gate, fn):
    # 16384 keys: the CTA-pair kernel; rows sampled (the oracle is row-exact)
    w = _workload("bf16", gate, B=1, L_q=16384, L_k=16384, H_q=8, H_kv=2, seed=43)
    t = make_inputs(w)
    got, X, W = _run(w, t, gate, fn)
    rng = np.random.default_rng(3)
    rows = sorted(set([(0, 0), (0, 127), (0, 128), (0, 255), (0, 16383)] +
                      [(0, int(i)) for i in rng.integers(0, w.L_q, 11)]))
    ref = oracle.gated_sdpa_variant(X, t["Q"], t["K"], t["V"], W, gate=gate, gate_fn=fn, eps=1e-6,
                                    causal=True, rows=rows)[0]
    _check(w, np.stack([got[b, i] for b, i in rows]), ref, f"pair {gate}/{fn}")


def test_variant_default_equals_the_layer():
    # gated_sdpa_fwd_variant with the sigmoid gate is gated_sdpa_fwd, bit for bit
    w = _workload("bf16", "elementwise")
    t = make_inputs(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    a, _ = gb.gated_sdpa_fwd(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate="elementwise")
    b, _ = gb.gated_sdpa_fwd_variant(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate="elementwise")
    assert torch.equal(a, b)
