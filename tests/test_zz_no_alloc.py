"""The decode entry point that allocates nothing (gated_sdpa_decode_noalloc).

Callers that cannot allocate device memory (code that must not make the
device synchronise, allocator-less plugin hooks, fixed memory budgets) use
this entry point: its scratch is a fixed array inside the library instead of
a caller-supplied workspace. These tests call it through the C ABI and hold
it to the same bf16 tolerance as the rest of the suite against the regular
entry point, on two calls in a row with different inputs (the shared scratch
keeps the previous call's contents). The file is named so that pytest
collects it last.
"""
import numpy as np
import pytest
import torch

from gated_softmax_attention_gb300 import binding as gb
from gated_softmax_attention_gb300 import build as gbuild
from gated_softmax_attention_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

BF16_MAX_ABS = 2e-2
BF16_REL_L1 = 5e-3
SINK_ABS = 2e-3


@pytest.fixture(scope="module", autouse=True)
def lib():
    gbuild.build()
    gb.load()


def _close(got, ref, what):
    g = got.double().cpu().numpy()
    r = ref.double().cpu().numpy()
    err = np.abs(g - r)
    rel = err.sum() / max(np.abs(r).sum(), 1e-30)
    assert err.max() <= BF16_MAX_ABS and rel <= BF16_REL_L1, f"{what}: max-abs {err.max():.3e} rel-L1 {rel:.3e}"


def _inputs(w):
    return {k: (v.cuda() if v is not None else None) for k, v in make_inputs(w).items()}


def test_noalloc_matches_the_workspace_entry_point_on_two_calls():
    w1 = Workload("noalloc_a", "bf16", B=8, L_q=1, L_k=1000, d_model=512, H_q=16, H_kv=4, d_k=128,
                  gate="elementwise", causal=True, seed=31)
    w2 = Workload("noalloc_b", "bf16", B=5, L_q=1, L_k=3000, d_model=256, H_q=32, H_kv=8, d_k=128,
                  gate="headwise", causal=True, seed=32)
    calls = []
    for w in (w1, w2):
        t = _inputs(w)
        ref, ref_sink = gb.gated_sdpa_fwd(t["X"], t["Q"], t["K"], t["V"], t["W_g"], gate=w.gate, causal=True,
                                          want_sink=True)
        calls.append((w, t, ref, ref_sink))
    torch.cuda.synchronize()
    # two no-alloc calls in a row, different shapes and gates: the second runs on
    # the scratch the first one left behind
    outs = [gb.decode_noalloc(t["X"], t["Q"], t["K"], t["V"], t["W_g"], gate=w.gate, want_sink=True)
            for (w, t, _, _) in calls]
    assert gb.check_device_error() == gb.OK
    for (w, _, ref, ref_sink), (o, sink) in zip(calls, outs):
        _close(o, ref, w.name)
        assert torch.allclose(sink, ref_sink, atol=SINK_ABS), w.name


def test_noalloc_rejects_problems_beyond_its_scratch():
    cap = gb.load().gsdpa_decode_noalloc_max_scratch()
    assert cap == 16 << 20
    B, L_k, d_model, H_q, H_kv, d_k = 256, 16384, 4096, 32, 8, 128
    need = gb.workspace_bytes(B, 1, L_k, d_model, H_q, H_kv, d_k, "elementwise", True, gb.BF16)
    assert need > cap
    # argument checks and the size check happen before any device work
    st = gb.load().gated_sdpa_decode_noalloc(256, 256, 256, 256, 256, 256, None, B, L_k, d_model, H_q, H_kv, d_k,
                                             gb.GATE_ELEMENTWISE, None)
    assert st == gb.ERR_WORKSPACE
