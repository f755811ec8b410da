"""The decode entry point that allocates nothing (gated_sdpa_decode_noalloc).

Callers that cannot allocate device memory (code that must not make the
device synchronise, allocator-less plugin hooks, fixed memory budgets) use
this entry point: its scratch is a fixed array inside the library instead of
a caller-supplied workspace. These tests call it through the C ABI and hold
its outputs to the suite's bf16 tolerance against the float64 oracle, on
calls in a row with different shapes and gates (the shared scratch keeps the
previous call's contents): a gate-free call after a headwise one checks that
the branch that clears the split counters with a memset (no gate kernel runs
first) starts from zero. The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle
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


def _check(got, ref, what):
    g = got.double().cpu().numpy()
    err = np.abs(g - ref)
    rel = err.sum() / max(np.abs(ref).sum(), 1e-30)
    assert err.max() <= BF16_MAX_ABS and rel <= BF16_REL_L1, f"{what}: max-abs {err.max():.3e} rel-L1 {rel:.3e}"


def test_noalloc_matches_the_oracle_on_calls_in_a_row():
    ws = [Workload("noalloc_a", "bf16", B=8, L_q=1, L_k=1000, d_model=512, H_q=16, H_kv=4, d_k=128,
                   gate="elementwise", causal=True, seed=31),
          Workload("noalloc_b", "bf16", B=5, L_q=1, L_k=3000, d_model=256, H_q=32, H_kv=8, d_k=128,
                   gate="headwise", causal=True, seed=32),
          Workload("noalloc_c", "bf16", B=6, L_q=1, L_k=2500, d_model=256, H_q=16, H_kv=4, d_k=128,
                   gate="none", causal=True, seed=33)]
    host = [make_inputs(w) for w in ws]
    dev = [{k: (v.cuda() if v is not None else None) for k, v in t.items()} for t in host]
    torch.cuda.synchronize()
    # calls in a row on the one shared scratch array, each leaving its contents to the next
    outs = [gb.decode_noalloc(d["X"], d["Q"], d["K"], d["V"], d["W_g"], gate=w.gate, want_sink=True)
            for w, d in zip(ws, dev)]
    assert gb.check_device_error() == gb.OK
    for w, t, (o, sink) in zip(ws, host, outs):
        ref, p0 = oracle.gated_sdpa(t["X"], t["Q"], t["K"], t["V"], t["W_g"], gate=w.gate, causal=True)
        _check(o, ref, w.name)
        sink_err = np.abs(sink.double().cpu().numpy() - oracle.sink_share(p0)).max()
        assert sink_err <= SINK_ABS, f"{w.name}: first-token share {sink_err:.3e}"


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


def test_noalloc_reports_gate_modes_it_does_not_cover():
    lib = gb.load()
    args = (256, 256, 256, 256, 256, 256, None, 2, 1024, 256, 8, 2, 128)
    # head-shared, input-independent and averaged gates: valid modes, not covered here
    for mode in (3, 4, 5, 6, 7):
        assert lib.gated_sdpa_decode_noalloc(*args, mode, None) == gb.ERR_UNSUPPORTED
    # values outside the gate-mode enumeration
    for mode in (-1, 8):
        assert lib.gated_sdpa_decode_noalloc(*args, mode, None) == gb.ERR_INVALID_ARG
