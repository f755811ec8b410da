"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances (stated for this layer): float32 max-abs error <= 1e-4; bfloat16
max-abs error <= 2e-2 and relative L1 error sum|gpu - ref| / sum|ref| <= 5e-3.
The first-token share (float32 output on both paths) is held to 2e-3 absolute
for bf16 inputs (its weights come from bf16-rounded scores' softmax in fp32)
and 1e-5 for float32.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_softmax_attention_gb300 import binding as gb
from gated_softmax_attention_gb300 import build as gbuild
from gated_softmax_attention_gb300.workloads import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

F32_MAX_ABS = 1e-4
BF16_MAX_ABS = 2e-2
BF16_REL_L1 = 5e-3
# log of the softmax denominator (natural log): float32 scores of exact bf16
# inputs accumulate 128 products (2^-24 relative each, |s| <= ~40 with scaled
# keys: ~3e-4), the row sum float32 exponentials (2^-22 relative): 1e-3 absolute
LSE_ABS = 1e-3


@pytest.fixture(scope="module", autouse=True)
def lib():
    gbuild.build()
    gb.load()
    torch.cuda.init()


def run_gpu(w: Workload, t, want_sink=True):
    dev = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    O, sink = gb.gated_sdpa_fwd(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=w.gate, causal=w.causal,
                                want_sink=want_sink)
    assert gb.check_device_error() == gb.OK
    return O.double().cpu().numpy(), (sink.double().cpu().numpy() if sink is not None else None)


def run_oracle(w: Workload, t, rows=None):
    return oracle.gated_sdpa(t["X"], t["Q"], t["K"], t["V"], t["W_g"], gate=w.gate, causal=w.causal, rows=rows)


def assert_close(w: Workload, got, ref, what=""):
    err = np.abs(got - ref)
    if w.dtype == "f32":
        assert err.max() <= F32_MAX_ABS, f"{what} max-abs {err.max():.3e}"
    else:
        rel = err.sum() / max(np.abs(ref).sum(), 1e-30)
        assert err.max() <= BF16_MAX_ABS, f"{what} max-abs {err.max():.3e} (rel-L1 {rel:.3e})"
        assert rel <= BF16_REL_L1, f"{what} rel-L1 {rel:.3e} (max-abs {err.max():.3e})"


def sink_tol(w):
    return 1e-5 if w.dtype == "f32" else 2e-3


def small(dtype, **kw):
    base = dict(name="small", dtype=dtype, B=2, L_q=300, L_k=300, d_model=256, H_q=4, H_kv=2, d_k=128,
                gate="elementwise", causal=True, seed=21)
    base.update(kw)
    return Workload(**base)


# ------------------------------------------------------------------ full comparisons, small shapes

def test_f32_reference_workload():
    w = WORKLOADS["f32_mha_elementwise_L128"]
    t = make_inputs(w)
    O, sink = run_gpu(w, t)
    ref, p0 = run_oracle(w, t)
    assert_close(w, O, ref, "O")
    np.testing.assert_allclose(sink, oracle.sink_share(p0), atol=sink_tol(w))


CASES = [
    dict(),                                              # GQA 4/2, ragged 300, elementwise
    dict(gate="headwise", H_q=8, H_kv=2),                 # headwise (bf16 needs H_q % 8 == 0)
    dict(gate="none"),
    dict(causal=False),
    dict(d_k=64),
    dict(d_k=64, gate="headwise", H_q=8, H_kv=8, L_q=129, L_k=129),
    dict(L_q=77, L_k=300),                                # bottom-right causal, L_q < L_k
    dict(L_q=1, L_k=1, B=3),                              # single key
    dict(L_q=128, L_k=128, B=1, H_q=2, H_kv=1, d_model=64),
    dict(L_q=257, L_k=257, d_model=200, gate="elementwise"),  # ragged d_model (zero-filled K chunk tail)
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: ",".join(f"{k}={v}" for k, v in c.items()) or "base")
def test_small_shapes(dtype, case):
    w = small(dtype, **case)
    if dtype == "bf16" and w.d_model % 8:
        pytest.skip("bf16 needs d_model % 8 == 0")
    t = make_inputs(w)
    O, sink = run_gpu(w, t)
    ref, p0 = run_oracle(w, t)
    assert_close(w, O, ref, "O")
    np.testing.assert_allclose(sink, oracle.sink_share(p0), atol=sink_tol(w))


# Long key sequences (>= 16384 keys) run on the CTA-pair kernel: its units
# are four query tiles, two per CTA, and an MMA slot pairs tile 4u+2t of one
# CTA with tile 4u+2t+1 of the other. These cases cover a pair whose odd tile
# has no rows, a unit whose second slot has no rows, ragged L_k, GQA, both
# gates, no gate and no mask.
PAIR_CASES = [
    dict(L_q=300, L_k=16500),                                       # 3 tiles: odd tile of slot 1 empty
    dict(L_q=600, L_k=16384, gate="headwise", H_q=8, H_kv=2),       # 5 tiles: second unit has one tile
    dict(L_q=256, L_k=16448, gate="none", causal=False, H_q=2, H_kv=1),
    dict(L_q=512, L_k=16384, H_q=4, H_kv=4, d_model=512),
]


@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: ",".join(f"{k}={v}" for k, v in c.items()))
def test_pair_kernel_long_keys(case):
    w = small("bf16", B=1, **case)
    t = make_inputs(w)
    O, sink = run_gpu(w, t)
    ref, p0 = run_oracle(w, t)
    assert_close(w, O, ref, "O")
    np.testing.assert_allclose(sink, oracle.sink_share(p0), atol=sink_tol(w))


def test_pair_kernel_square_sampled():
    # L_q = L_k = 16384: many units per pair (phases carried across units), sampled rows
    w = small("bf16", B=1, L_q=16384, L_k=16384, H_q=2, H_kv=1, d_model=256, seed=23)
    t = make_inputs(w)
    O, sink = run_gpu(w, t)
    rows = sample_rows(w, 32)
    ref, p0 = run_oracle(w, t, rows=rows)
    got = np.stack([O[b, i] for b, i in rows])
    assert_close(w, got, ref, "O")
    assert np.isfinite(O).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("sign", [1.0, -1.0])
@pytest.mark.parametrize("gate", ["elementwise", "headwise"])
def test_gate_limits(dtype, sign, gate):
    """Logits of +200 give plain SDPA, logits of -200 give zero."""
    w = small(dtype, gate=gate, H_q=8, H_kv=4, d_model=64)
    t = make_inputs(w)
    t["X"] = torch.ones_like(t["X"])
    t["W_g"] = torch.full_like(t["W_g"], sign * 200.0 / w.d_model)
    O, _ = run_gpu(w, t, want_sink=False)
    if sign > 0:
        ref, _ = oracle.gated_sdpa(None, t["Q"], t["K"], t["V"], None, gate="none", causal=True)
        assert_close(w, O, ref, "O(+200)")
    else:
        assert np.abs(O).max() == 0.0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_v_ones_gives_the_gate(dtype):
    w = small(dtype, gate="elementwise")
    t = make_inputs(w)
    t["V"] = torch.ones_like(t["V"])
    O, _ = run_gpu(w, t, want_sink=False)
    ref, _ = run_oracle(w, t)
    assert_close(w, O, ref, "O")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_equal_scores_and_harmonic_sink(dtype):
    w = small(dtype, gate="none", L_q=200, L_k=200)
    t = make_inputs(w)
    t["Q"] = torch.zeros_like(t["Q"])
    O, sink = run_gpu(w, t)
    ref, p0 = run_oracle(w, t)
    assert_close(w, O, ref, "O")
    harmonic = sum(1.0 / i for i in range(1, 201)) / 200
    np.testing.assert_allclose(sink, harmonic, atol=sink_tol(w))


def test_empty_problem_is_a_no_op():
    w = small("bf16", B=1)
    t = make_inputs(w)
    dev = {k: v.cuda() for k, v in t.items()}
    O = torch.full_like(dev["Q"], 7.0)
    st = gb.fwd_raw(dev["X"].data_ptr(), dev["Q"].data_ptr(), dev["K"].data_ptr(), dev["V"].data_ptr(),
                    dev["W_g"].data_ptr(), O.data_ptr(), None, 0, w.L_q, w.L_k, w.d_model, w.H_q, w.H_kv, w.d_k,
                    2, 1, gb.BF16, None, 0, None)
    assert st == gb.OK
    torch.cuda.synchronize()
    assert bool((O == 7.0).all())


def test_workspace_too_small_is_rejected():
    w = small("bf16", gate="headwise", H_q=8, H_kv=2)
    t = {k: v.cuda() for k, v in make_inputs(w).items()}
    O = torch.empty_like(t["Q"])
    need = gb.workspace_bytes(w.B, w.L_q, w.L_k, w.d_model, w.H_q, w.H_kv, w.d_k, "headwise", False, gb.BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = gb.fwd_raw(t["X"].data_ptr(), t["Q"].data_ptr(), t["K"].data_ptr(), t["V"].data_ptr(),
                    t["W_g"].data_ptr(), O.data_ptr(), None, w.B, w.L_q, w.L_k, w.d_model, w.H_q, w.H_kv, w.d_k,
                    1, 1, gb.BF16, ws.data_ptr(), need - 256, None)
    assert st == gb.ERR_WORKSPACE


def test_binding_passes_the_real_workspace_size():
    # a caller's workspace tensor smaller than the problem needs is rejected by
    # the library (the binding passes the tensor's own size, not the size the
    # problem needs), before anything is enqueued
    w = small("bf16", gate="headwise", H_q=8, H_kv=2)
    t = make_inputs(w)
    dev = {k: v.cuda() for k, v in t.items()}
    need = gb.workspace_bytes(w.B, w.L_q, w.L_k, w.d_model, w.H_q, w.H_kv, w.d_k, w.gate, True, gb.BF16)
    short = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(gb.GsdpaError) as ei:
        gb.gated_sdpa_fwd(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=w.gate, causal=True,
                          want_sink=True, workspace=short)
    assert ei.value.status == gb.ERR_WORKSPACE
    assert gb.check_device_error() == gb.OK


@pytest.mark.parametrize("gate", ["none", "elementwise"])
def test_output_view_off_a_32_byte_boundary(gate):
    # The epilogue stores whole 32-byte sectors from registers when O is 32-byte
    # aligned; an output view that is only 16-byte aligned (what the ABI asks)
    # takes the staged bulk copies: same values either way.
    w = small("bf16", gate=gate, H_q=4, H_kv=2, L_q=300, L_k=300)
    t = {k: (v.cuda() if v is not None else None) for k, v in make_inputs(w).items()}
    O_ref, _ = gb.gated_sdpa_fwd(t["X"], t["Q"], t["K"], t["V"], t["W_g"], gate=gate, causal=True)
    n = t["Q"].numel()
    buf = torch.zeros(n + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(t["Q"].shape)   # 16 bytes past a 256-byte-aligned allocation
    assert out.data_ptr() % 32 == 16
    gb.gated_sdpa_fwd(t["X"], t["Q"], t["K"], t["V"], t["W_g"], gate=gate, causal=True, out=out)
    assert gb.check_device_error() == gb.OK
    assert torch.equal(out, O_ref)


BAD_ARGS = ["headwise_W_g_for_elementwise", "X_rows", "out_shape", "sink_size", "lse_size", "K_V_mismatch",
            "dtype", "gate_out_dtype", "bwd_dO_shape", "bwd_lse_size"]


@pytest.mark.parametrize("bad", BAD_ARGS)
def test_binding_rejects_wrong_sized_tensors(bad):
    # the library receives bare pointers: the binding checks each tensor against
    # the sizes the problem implies and raises before anything is enqueued (a
    # headwise W_g passed to the elementwise gate would otherwise be read far
    # past its end)
    w = small("bf16", gate="elementwise", H_q=4, H_kv=2, L_q=200, L_k=200)
    t = {k: v.cuda() for k, v in make_inputs(w).items()}
    X, Q, K, V, W_g = t["X"], t["Q"], t["K"], t["V"], t["W_g"]
    kw = {}
    if bad == "headwise_W_g_for_elementwise":
        W_g = W_g[:, :w.H_q].contiguous()
    elif bad == "X_rows":
        X = X[:, :-1].contiguous()
    elif bad == "out_shape":
        kw["out"] = torch.empty_like(Q[:, :-1])
    elif bad == "sink_size":
        kw["sink"] = torch.empty(w.B * w.H_q - 1, dtype=torch.float32, device="cuda")
    elif bad == "lse_size":
        kw["lse"] = torch.empty(w.B * w.H_q * w.L_q - 1, dtype=torch.float32, device="cuda")
    elif bad == "K_V_mismatch":
        V = V[:, :-1].contiguous()
    elif bad == "dtype":
        W_g = W_g.float()
    elif bad == "gate_out_dtype":
        kw["gate_out"] = torch.empty((w.B * w.L_q, w.H_q * w.d_k), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    with pytest.raises(ValueError):
        if bad.startswith("bwd_"):
            O, _, lse = gb.gated_sdpa_fwd_train(X, Q, K, V, W_g, gate=w.gate)
            dO = torch.randn_like(O)
            if bad == "bwd_dO_shape":
                dO = dO[:, :-1].contiguous()
            else:
                lse = lse[:, :, :-1].contiguous()
            gb.gated_sdpa_bwd(X, Q, K, V, W_g, O, dO, lse, gate=w.gate)
        elif bad in ("lse_size",):
            gb.gated_sdpa_fwd_train(X, Q, K, V, W_g, gate=w.gate, **kw)
        elif bad == "gate_out_dtype":
            gb.gated_sdpa_fwd_train_save_gate(X, Q, K, V, W_g, **kw)
        else:
            gb.gated_sdpa_fwd(X, Q, K, V, W_g, gate=w.gate, **kw)
    assert gb.check_device_error() == gb.OK


# ------------------------------------------------------------------ full-size workloads, sampled rows

def sample_rows(w: Workload, n, seed=0):
    rng = np.random.default_rng(seed)
    fixed = [(0, 0), (w.B - 1, w.L_q - 1), (0, min(127, w.L_q - 1)), (0, min(128, w.L_q - 1))]
    rnd = [(int(rng.integers(w.B)), int(rng.integers(w.L_q))) for _ in range(n)]
    return sorted(set(fixed + rnd))


@pytest.mark.parametrize("name", ["bf16_mha_elementwise_L2048", "bf16_gqa_headwise_L4096",
                                  "bf16_gqa_headwise_sink_L32768"])
def test_full_size_prefill_sampled(name):
    w = WORKLOADS[name]
    t = make_inputs(w)
    O, sink = run_gpu(w, t)
    rows = sample_rows(w, 24 if w.L_q > 8192 else 48)
    ref, p0 = run_oracle(w, t, rows=rows)
    got = np.stack([O[b, i] for b, i in rows])
    assert_close(w, got, ref, name)
    # properties that hold at any size
    assert np.isfinite(O).all()
    assert ((sink >= 0) & (sink <= 1)).all()
    if w.key0_scale != 1.0:
        # keys of token 0 scaled x8: rows attend to token 0 far more than uniformly
        assert sink.mean() > 2.0 * float(np.mean(1.0 / np.arange(1, w.L_q + 1)))


def test_long_context_first_token_share_matches_the_oracle():
    """The long-context workload's keys of token 0 are scaled x8 so that rows
    put sink-like mass on the first token ("10 . 门控" sec. 3.4 measures that
    share): every sink[b, h] of the call bench.py times against the oracle's
    mean over all 32768 rows of the weight on key 0 (softmax statistics only,
    no values: about a minute on the host's cores), and the training forward's
    log-denominators on sampled rows against the oracle's."""
    w = WORKLOADS["bf16_gqa_headwise_sink_L32768"]
    t = make_inputs(w)
    _, sink = run_gpu(w, t)
    p0, lse_ref = oracle.softmax_stats(t["Q"], t["K"], causal=w.causal)
    ref = oracle.sink_share(p0)
    err = np.abs(sink - ref)
    print(f"long-context sink: mean {ref.mean():.4f} (harmonic {np.mean(1.0 / np.arange(1, w.L_q + 1)):.4f}), "
          f"max-abs error {err.max():.2e}")
    assert err.max() <= sink_tol(w), f"sink max-abs {err.max():.3e}"
    # the log-denominators of the training forward ([B, H_q, L_q], natural log):
    # fp32 scores of exact bf16 inputs, |s| up to ~40 with the scaled keys
    dev = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    _, _, lse = gb.gated_sdpa_fwd_train(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=w.gate,
                                        causal=w.causal)
    assert gb.check_device_error() == gb.OK
    lse = lse.double().cpu().numpy()
    rows = sample_rows(w, 64, seed=3)
    got = np.stack([lse[b, :, i] for b, i in rows])
    want = np.stack([lse_ref[b, i, :] for b, i in rows])
    lerr = np.abs(got - want).max()
    print(f"long-context lse on {len(rows)} rows: max-abs error {lerr:.2e}")
    assert lerr <= LSE_ABS, f"lse max-abs {lerr:.3e}"


def test_full_size_decode_sampled():
    w = WORKLOADS["bf16_decode_gqa_elementwise_Lk8192"]
    t = make_inputs(w)
    O, sink = run_gpu(w, t)
    for b in (0, 17, 63):
        sl = {k: (v[b:b + 1] if k != "W_g" else v) for k, v in t.items()}
        ref, p0 = oracle.gated_sdpa(sl["X"], sl["Q"], sl["K"], sl["V"], sl["W_g"], gate=w.gate, causal=w.causal)
        assert_close(w, O[b:b + 1], ref, f"decode b={b}")
        np.testing.assert_allclose(sink[b], p0[0, 0], atol=sink_tol(w))


# ------------------------------------------------------------------ per-call state in a reused workspace

REUSE_CASES = [
    small("bf16", name="reuse_none", gate="none"),
    small("bf16", name="reuse_headwise", gate="headwise", H_q=8, H_kv=2),
    small("bf16", name="reuse_elementwise"),
    small("bf16", name="reuse_pair_long_keys", B=1, L_q=384, L_k=16384, H_q=2, H_kv=1, causal=False),
]


@pytest.mark.parametrize("w", REUSE_CASES, ids=lambda w: w.name)
def test_repeated_calls_on_one_workspace(w):
    """The unit counter and the first-token-share arrivals live in the
    workspace and are reset by every call (by the gate kernel that runs first,
    or by a memset without a gate): three calls on one workspace, with the
    outputs poisoned in between, give the same bits, and the oracle's values."""
    t = make_inputs(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    need = gb.workspace_bytes(w.B, w.L_q, w.L_k, w.d_model if w.gate != "none" else 0, w.H_q, w.H_kv, w.d_k, w.gate, True, gb.BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    O = torch.empty(w.B, w.L_q, w.H_q, w.d_k, dtype=torch.bfloat16, device="cuda")
    sink = torch.empty(w.B, w.H_q, dtype=torch.float32, device="cuda")
    runs = []
    for _ in range(3):
        O.fill_(float("nan"))
        sink.fill_(float("nan"))
        gb.gated_sdpa_fwd(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=w.gate, causal=w.causal,
                          out=O, sink=sink, workspace=ws)
        assert gb.check_device_error() == gb.OK
        runs.append((O.clone(), sink.clone()))
    for O_r, s_r in runs[1:]:
        assert torch.equal(O_r, runs[0][0]) and torch.equal(s_r, runs[0][1])
    ref, p0 = run_oracle(w, t)
    assert_close(w, runs[0][0].double().cpu().numpy(), ref, w.name)
    np.testing.assert_allclose(runs[0][1].double().cpu().numpy(), oracle.sink_share(p0), atol=sink_tol(w))


# ------------------------------------------------------------------ the training forward's log-sum-exp

# The LSE's error comes from the fp32 scores (exact bf16 products, fp32 sums
# of 128 terms: ~1e-5 relative to the score scale) and the fp32 sum of the
# exponentials (ex2.approx, ~1e-6 relative): 2e-3 absolute leaves a wide margin.
LSE_ATOL = 2e-3

LSE_CASES = [
    small("bf16", name="lse_elementwise"),
    small("bf16", name="lse_gqa_headwise", gate="headwise", H_q=8, H_kv=2),
    small("bf16", name="lse_no_gate_ragged_suffix", gate="none", L_q=77, L_k=300),
    small("bf16", name="lse_pair_long_keys", B=1, L_q=384, L_k=16384, H_q=2, H_kv=1),
]


@pytest.mark.parametrize("w", LSE_CASES, ids=lambda w: w.name)
def test_forward_train_writes_lse(w):
    t = make_inputs(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    O, _, lse = gb.gated_sdpa_fwd_train(dev["X"], dev["Q"], dev["K"], dev["V"], dev["W_g"], gate=w.gate,
                                        causal=w.causal)
    assert gb.check_device_error() == gb.OK
    ref, _, lse_ref = oracle.gated_sdpa(t["X"], t["Q"], t["K"], t["V"], t["W_g"], gate=w.gate, causal=w.causal,
                                        return_lse=True)
    assert_close(w, O.double().cpu().numpy(), ref, w.name)
    got = lse.double().cpu().numpy()                      # [B, H_q, L_q]
    np.testing.assert_allclose(got, lse_ref.transpose(0, 2, 1), atol=LSE_ATOL, rtol=0)
