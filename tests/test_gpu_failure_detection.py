"""Failure detection on the GPU without a fault: bounded waits that run out.

Every wait inside the sm_103a kernels is bounded by a limit in nanoseconds
(gsdpa_set_wait_limit_ns sets it for the following launches). When a wait
runs out, the kernel records the timeout in a device error word, raises its
abort flag (both CTAs' flags on a CTA pair) so that the other roles give up
too, lets the copies and MMAs already in flight land, frees its tensor memory
and returns; the host reads the status with gsdpa_check_device_error. Nothing
here faults, traps or hangs the device: the first test waits on a barrier that
nothing completes, the second lets real waits of the real kernels run out.
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


@pytest.fixture(scope="module", autouse=True)
def lib():
    gbuild.build()
    gb.load()


@pytest.fixture(autouse=True)
def default_limit():
    gb.set_wait_limit_ns(0)
    yield
    gb.set_wait_limit_ns(0)


def _run(w, dev):
    O, _ = gb.gated_sdpa_fwd(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=w.gate, causal=w.causal)
    return O


def _check(w, t, O):
    ref, _ = oracle.gated_sdpa(t["X"], t["Q"], t["K"], t["V"], t["W_g"], gate=w.gate, causal=w.causal)
    got = O.double().cpu().numpy()
    err = np.abs(got - ref)
    rel = err.sum() / np.abs(ref).sum()
    assert err.max() <= BF16_MAX_ABS and rel <= BF16_REL_L1, f"{w.name}: max-abs {err.max():.3e} rel-L1 {rel:.3e}"


def _small(name, **kw):
    base = dict(name=name, dtype="bf16", B=1, L_q=300, L_k=300, d_model=256, H_q=4, H_kv=2, d_k=128,
                gate="elementwise", causal=True, seed=41)
    base.update(kw)
    return Workload(**base)


def test_a_wait_nothing_completes_reports_a_timeout():
    gb.set_wait_limit_ns(200_000)   # 200 us
    assert gb.wait_self_test() == gb.OK
    assert gb.check_device_error() == gb.ERR_DEVICE_TIMEOUT
    assert gb.check_device_error() == gb.OK   # the word is read and cleared
    gb.set_wait_limit_ns(0)
    # the context is still usable
    w = _small("after_self_test")
    t = make_inputs(w)
    dev = {k: v.cuda() for k, v in t.items()}
    O = _run(w, dev)
    assert gb.check_device_error() == gb.OK
    _check(w, t, O)


CASES = [
    _small("single_cta_elementwise"),
    _small("headwise", gate="headwise", H_q=8, H_kv=2),
    _small("pair_long_keys", L_q=256, L_k=16384, H_q=2, H_kv=1),
    _small("decode", B=4, L_q=1, L_k=1000, H_q=16, H_kv=4),
    # a long gate product: the gate GEMM's epilogue waits for 128 K chunks, far
    # longer than a wait that is checked against its limit every 32 tries
    _small("long_gate_product", d_model=8192),
]


def test_real_kernels_give_up_cleanly_with_a_tiny_limit():
    # Each real kernel (single-CTA prefill, headwise gate, CTA pair, decode, the
    # gate GEMM) runs once with a 1 ns wait limit, so that any wait not
    # satisfied within its first 32 tries runs out: it must report OK or a
    # timeout (never a fault), and the next call with the default limit must be
    # exact to the bar. Short waits are satisfied before the limit is checked,
    # so a single kernel may report OK; at least one case must report the
    # timeout, which shows that a real kernel's give-up path fired.
    statuses = {}
    for w in CASES:
        t = make_inputs(w)
        dev = {k: v.cuda() for k, v in t.items()}
        gb.set_wait_limit_ns(1)
        try:
            _run(w, dev)
            st = gb.check_device_error()
        finally:
            gb.set_wait_limit_ns(0)
        assert st in (gb.OK, gb.ERR_DEVICE_TIMEOUT), f"{w.name}: {gb.status_string(st)}"
        statuses[w.name] = st
        O = _run(w, dev)
        assert gb.check_device_error() == gb.OK
        _check(w, t, O)
    assert gb.ERR_DEVICE_TIMEOUT in statuses.values(), statuses
