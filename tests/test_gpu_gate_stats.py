"""GPU parity of the fused gate statistics (gated_sdpa_fwd_stats) against the
oracle's gate scores ("GatedAttention [2025]", sec. 1.4.2: mean gating score,
score distribution, fraction below a threshold).

What is unique is compared exactly: the number of scores and that the
histogram sums to it. The kernels bin their own values (bf16 path: the fp16
elementwise gate the attention multiplies by, 2^-11 relative; the headwise
gate in fp32 through tanh.approx, 2^-11 relative; float32 path: expf), so a
score within delta of a bin edge or of the threshold may land on either
side: each bin count (and the below-threshold count) must lie between the
oracle's count of scores surely inside and possibly inside. The mean is held
to delta.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_softmax_attention_gb300 import binding as gb
from gated_softmax_attention_gb300 import build as gbuild
from gated_softmax_attention_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    gbuild.build()
    gb.load()
    torch.cuda.init()


def _w(dtype, gate, **kw):
    base = dict(name="stats", dtype=dtype, B=2, L_q=300, L_k=300, d_model=256, H_q=8, H_kv=2, d_k=128, gate=gate,
                causal=True, seed=51, wg_std=0.15)
    base.update(kw)
    return Workload(**base)


CASES = [
    (_w("f32", "elementwise", B=1, L_q=70, L_k=90, d_model=64, H_q=4, H_kv=2, d_k=64), 10, 0.1, 1e-5),
    (_w("f32", "headwise", B=1, L_q=70, L_k=90, d_model=64, H_q=4, H_kv=2, d_k=64), 7, 0.3, 1e-5),
    (_w("bf16", "elementwise"), 20, 0.1, 2e-3),
    (_w("bf16", "headwise"), 16, 0.25, 2e-3),
    (_w("bf16", "elementwise", B=8, L_q=1, L_k=700), 20, 0.1, 2e-3),        # decode
    (_w("bf16", "headwise", B=8, L_q=1, L_k=700), 5, 0.5, 2e-3),            # decode
    (_w("bf16", "elementwise", B=1, L_q=16384, L_k=16384, H_q=2, H_kv=1), 64, 0.05, 2e-3),   # CTA pairs
    (_w("bf16", "headwise", B=1, L_q=16384, L_k=16384, H_q=8, H_kv=1), 10, 0.5, 2e-3),       # CTA pairs
]


@pytest.mark.parametrize("w,n_bins,thr,delta", CASES,
                         ids=[f"{w.dtype}-{w.gate}-B{w.B}-L{w.L_q}-{w.L_k}" for w, *_ in CASES])
def test_gate_statistics(w, n_bins, thr, delta):
    t = make_inputs(w)
    dev = {k: v.cuda() for k, v in t.items()}
    O, st = gb.gated_sdpa_fwd_stats(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=w.gate,
                                    causal=w.causal, n_bins=n_bins, threshold=thr)
    assert gb.check_device_error() == gb.OK
    s = oracle.gate_scores(t["X"], t["W_g"], w.H_q, w.d_k, gate=w.gate).ravel()
    ref = oracle.gate_statistics(s, n_bins, thr)
    print(f"count {st['count']} mean {st['mean']:.6f} (oracle {ref['mean']:.6f}) below {st['below']} "
          f"(oracle {ref['below']}) hist {st['hist'][:6]}... (oracle {list(ref['hist'][:6])}...)")
    assert st["count"] == ref["count"]
    assert sum(st["hist"]) == st["count"]
    assert abs(st["mean"] - ref["mean"]) <= delta
    # the threshold: scores within delta of it may fall on either side
    surely = np.count_nonzero(s < thr - delta)
    possibly = np.count_nonzero(s < thr + delta)
    assert surely <= st["below"] <= possibly
    for k in range(n_bins):
        lo, hi = k / n_bins, (k + 1) / n_bins
        lo_in = -np.inf if k == 0 else lo + delta
        hi_in = np.inf if k == n_bins - 1 else hi - delta
        lo_out = -np.inf if k == 0 else lo - delta
        hi_out = np.inf if k == n_bins - 1 else hi + delta
        surely = np.count_nonzero((s >= lo_in) & (s < hi_in))
        possibly = np.count_nonzero((s >= lo_out) & (s < hi_out))
        assert surely <= st["hist"][k] <= possibly, f"bin {k}: {st['hist'][k]} not in [{surely}, {possibly}]"
    # the output is gated_sdpa_fwd's
    O2, _ = gb.gated_sdpa_fwd(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=w.gate, causal=w.causal)
    assert torch.equal(O, O2)


def test_statistics_are_reproducible():
    # integer counters: two calls give the same bits
    w = _w("bf16", "elementwise")
    dev = {k: v.cuda() for k, v in make_inputs(w).items()}
    a = gb.gated_sdpa_fwd_stats(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], n_bins=32, threshold=0.2)[1]
    b = gb.gated_sdpa_fwd_stats(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], n_bins=32, threshold=0.2)[1]
    assert a == b
