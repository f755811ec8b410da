"""Host-only checks of the C ABI: the library builds, loads, exports every
symbol include/gsdpa.h declares, and rejects bad arguments before it touches
a device. No kernel is launched here."""
import ctypes
import os
import re

import pytest

from gated_softmax_attention_gb300 import binding as gb
from gated_softmax_attention_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gsdpa.h")


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gb.load()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"GSDPA_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_symbols())
    assert {"gated_sdpa_fwd", "gsdpa_workspace_bytes", "gsdpa_check_device_error",
            "gsdpa_status_string"} <= names


def test_library_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert names
    for n in names:
        assert hasattr(lib, n), n
        assert n in gb.SIGNATURES, f"binding lacks a signature for {n}"


def test_only_the_abi_is_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", gb.LIB_PATH], capture_output=True, text=True).stdout
    ours = {line.split()[-1] for line in out.splitlines()
            if line.split()[-1].startswith(("gsdpa", "gated_sdpa", "gated_attention"))}
    assert ours == set(declared_symbols())


def test_status_strings(lib):
    for code, name in [(0, "GSDPA_OK"), (-1, "GSDPA_ERR_INVALID_ARG"), (-2, "GSDPA_ERR_UNSUPPORTED"),
                       (-3, "GSDPA_ERR_ALIGNMENT"), (-4, "GSDPA_ERR_WORKSPACE"), (-5, "GSDPA_ERR_LAUNCH"),
                       (-6, "GSDPA_ERR_DEVICE_TIMEOUT")]:
        assert gb.status_string(code) == name
    assert gb.status_string(99) == "GSDPA_ERR_UNKNOWN"


def test_workspace_bytes(lib):
    # bf16 prefill: the per-call state, one 256-byte slot for the unit counter
    # of the dynamic schedule (8 bytes) ...
    counter = 256
    assert gb.workspace_bytes(2, 2048, 2048, 2048, 16, 16, 128, "none", False, gb.BF16) == counter
    # elementwise bf16 prefill: plus the gate sigma(X W_g) as fp16, [B*L_q, H_q*d_k]
    gate = 2 * 2 * 2048 * 16 * 128
    assert gb.workspace_bytes(2, 2048, 2048, 2048, 16, 16, 128, "elementwise", False, gb.BF16) == counter + gate
    # ... and, with the first-token share, one 64-bit word per (b, h) in the
    # same block: 8 + 2*16*8 bytes, 256-aligned
    n = gb.workspace_bytes(2, 2048, 2048, 2048, 16, 16, 128, "elementwise", True, gb.BF16)
    assert n == 512 + gate
    # the float32 path keeps per-tile partial sums: B*H_q*ceil(L/32) floats
    n = gb.workspace_bytes(2, 2048, 2048, 2048, 16, 16, 128, "elementwise", True, gb.F32)
    assert n >= 2 * 16 * 64 * 4 and n % 256 == 0
    # headwise bf16: split-K gate logits [splits, B*L, H_q]
    n = gb.workspace_bytes(1, 4096, 4096, 4096, 32, 4, 128, "headwise", False, gb.BF16)
    assert n >= 4096 * 32 * 4 and n % 256 == 0
    # empty problems need nothing
    assert gb.workspace_bytes(0, 16, 16, 64, 4, 4, 64, "elementwise", True, gb.BF16) == 0
    # rejected shapes
    for args in [(1, 8, 4, 64, 4, 4, 64), (1, 8, 8, 64, 3, 2, 64), (1, 8, 8, 64, 4, 4, 96)]:
        with pytest.raises(gb.GsdpaError):
            gb.workspace_bytes(*args, "elementwise", False, gb.BF16)
    with pytest.raises(gb.GsdpaError):  # bf16 headwise needs H_q % 8 == 0
        gb.workspace_bytes(1, 8, 8, 64, 4, 4, 64, "headwise", False, gb.BF16)
    assert gb.workspace_bytes(1, 8, 8, 64, 4, 4, 64, "headwise", False, gb.F32) == 0


def call(**kw):
    base = dict(X=16, Q=16, K=16, V=16, W_g=16, O=16, sink=None, B=1, L_q=8, L_k=8, d_model=64, H_q=4, H_kv=4,
                d_k=64, gate_mode=2, causal=1, dtype=0, workspace=None, workspace_bytes=0, stream=None)
    base.update(kw)
    return gb.fwd_raw(**base)


def test_argument_validation_before_any_device_work(lib):
    assert call(L_q=9, L_k=8) == gb.ERR_INVALID_ARG        # L_q > L_k
    assert call(L_k=0, L_q=0) == gb.ERR_INVALID_ARG        # no keys
    assert call(H_q=6, H_kv=4) == gb.ERR_INVALID_ARG       # H_q % H_kv
    assert call(gate_mode=3) == gb.ERR_INVALID_ARG
    assert call(dtype=7) == gb.ERR_INVALID_ARG
    assert call(d_k=96) == gb.ERR_UNSUPPORTED
    assert call(Q=None) == gb.ERR_INVALID_ARG
    assert call(W_g=None) == gb.ERR_INVALID_ARG            # gated without W_g
    assert call(X=24) == gb.ERR_ALIGNMENT
    assert call(O=8) == gb.ERR_ALIGNMENT
    assert call(B=0) == gb.OK                              # empty problem: nothing enqueued
    assert call(L_q=0) == gb.OK
    assert call(dtype=1, d_model=60) == gb.ERR_UNSUPPORTED  # bf16 rows must start on 16 bytes
    # bf16 prefill adds the first-token share in a fixed-point word whose count
    # field holds 4 arrivals per 128-row tile: L_q up to 2^24 with a share
    big = 1 << 24
    assert call(dtype=1, sink=4, L_q=big + 1, L_k=big + 1) == gb.ERR_UNSUPPORTED


def test_fwd_signature_matches_header(lib):
    # 7 pointers, 10 ints, workspace pointer, size, stream
    res, args = gb.SIGNATURES["gated_sdpa_fwd"]
    assert len(args) == 20 and res is ctypes.c_int


def test_bwd_workspace_and_validation(lib):
    # bf16, d_k = 128: gate recompute buffers + dY + D, lse (padded to 128 rows) + dGl
    n = gb.bwd_workspace_bytes(2, 300, 300, 256, 4, 2, 128, "elementwise")
    assert n >= 2 * 300 * 4 * 128 * 2 + 2 * (2 * 4 * 384 * 4) + 2 * 300 * 512 * 2 and n % 256 == 0
    assert gb.bwd_workspace_bytes(0, 16, 16, 64, 4, 4, 128, "none") == 0
    with pytest.raises(gb.GsdpaError):   # d_k = 64 is not covered
        gb.bwd_workspace_bytes(1, 8, 8, 64, 4, 4, 64, "elementwise")
    # argument checks happen before any device work (fake pointers)
    lib_ = gb.load()
    args = [16] * 13 + [1, 8, 8, 64, 4, 4, 128, 2, 1, gb.BF16, None, 0, None]
    bad = list(args)
    bad[13 + 6] = 64                      # d_k 64
    assert lib_.gated_sdpa_bwd(*bad) == gb.ERR_UNSUPPORTED
    bad = list(args)
    bad[6] = None                         # no dO
    assert lib_.gated_sdpa_bwd(*bad) == gb.ERR_INVALID_ARG
    bad = list(args)
    bad[8] = 24                           # dQ misaligned
    assert lib_.gated_sdpa_bwd(*bad) == gb.ERR_ALIGNMENT


def call_variant(**kw):
    base = dict(X=16, Q=16, K=16, V=16, W_g=16, O=16, sink=None, B=1, L_q=8, L_k=8, d_model=64, H_q=4, H_kv=4,
                d_k=64, gate_mode=2, gate_fn=0, eps=1e-6, causal=1, dtype=0, workspace=None, workspace_bytes=0,
                stream=None)
    base.update(kw)
    return int(gb.load().gated_sdpa_fwd_variant(*base.values()))


def test_variant_validation_before_any_device_work(lib):
    # a gate with a function of the output alone, or no gate with a function of a logit
    assert call_variant(gate_mode=2, gate_fn=5) == gb.ERR_INVALID_ARG
    assert call_variant(gate_mode=1, gate_fn=6) == gb.ERR_INVALID_ARG
    assert call_variant(gate_mode=0, gate_fn=3) == gb.ERR_INVALID_ARG
    assert call_variant(gate_mode=8) == gb.ERR_INVALID_ARG
    assert call_variant(gate_mode=7, X=None) == gb.ERR_INVALID_ARG   # the averaged gates read X
    assert call_variant(gate_fn=7) == gb.ERR_INVALID_ARG
    assert call_variant(gate_mode=0, gate_fn=6, eps=-1.0) == gb.ERR_INVALID_ARG
    # the input-independent gate reads no X; RMSNorm's gamma may be absent; a shared gate reads X
    assert call_variant(gate_mode=5, X=None, B=0) == gb.OK
    assert call_variant(gate_mode=0, gate_fn=6, W_g=None, X=None, B=0) == gb.OK
    assert call_variant(gate_mode=4, X=None) == gb.ERR_INVALID_ARG
    assert call_variant(gate_mode=5, W_g=None) == gb.ERR_INVALID_ARG
    assert call_variant(gate_mode=3, W_g=8) == gb.ERR_ALIGNMENT
    # gated_sdpa_fwd keeps to the three base shapes
    assert call(gate_mode=4) == gb.ERR_INVALID_ARG


def test_variant_workspace_bytes(lib):
    w = gb.workspace_bytes_variant
    # the default variant needs what gated_sdpa_fwd needs
    assert w(2, 300, 300, 256, 8, 2, 128, "elementwise", "sigmoid_mul", True, gb.BF16) == \
        gb.workspace_bytes(2, 300, 300, 256, 8, 2, 128, "elementwise", True, gb.BF16)
    # head-shared elementwise: fp16 values [B*L_q, d_k]; input-independent: [H_q * d_k]
    n_sh = w(2, 300, 300, 256, 8, 2, 128, "elementwise_shared", "silu_add", False, gb.BF16)
    n_st = w(2, 300, 300, 256, 8, 2, 128, "static", "sigmoid_mul", False, gb.BF16)
    n_no = w(2, 300, 300, 256, 8, 2, 128, "none", "rmsnorm", False, gb.BF16)
    assert n_sh >= n_no + 2 * 600 * 128 and n_st >= n_no + 2 * 8 * 128
    # head-shared headwise: one split of [B*L_q, 1] logits (any H_q: no tensor map over W_g)
    assert w(2, 300, 300, 256, 6, 2, 128, "headwise_shared", "sigmoid_mul", False, gb.BF16) >= n_no + 4 * 600
    with pytest.raises(gb.GsdpaError):
        w(2, 300, 300, 256, 8, 2, 128, "elementwise", "rmsnorm", False, gb.BF16)


def test_stats_validation_before_any_device_work(lib):
    def c(**kw):
        base = dict(X=16, Q=16, K=16, V=16, W_g=16, O=16, sink=None, stats=16, n_bins=10, threshold=0.1, B=1, L_q=8,
                    L_k=8, d_model=64, H_q=4, H_kv=4, d_k=64, gate_mode=2, causal=1, dtype=0, workspace=None,
                    workspace_bytes=0, stream=None)
        base.update(kw)
        return int(gb.load().gated_sdpa_fwd_stats(*base.values()))
    assert c(gate_mode=0) == gb.ERR_INVALID_ARG       # statistics of a gate
    assert c(gate_mode=4) == gb.ERR_INVALID_ARG
    assert c(stats=None) == gb.ERR_INVALID_ARG
    assert c(n_bins=0) == gb.ERR_INVALID_ARG
    assert c(n_bins=65) == gb.ERR_INVALID_ARG
    assert c(threshold=1.5) == gb.ERR_INVALID_ARG
    assert c(threshold=float("nan")) == gb.ERR_INVALID_ARG
    assert c(stats=12) == gb.ERR_ALIGNMENT
    assert c(B=0) == gb.OK


def test_layer_workspace_and_validation(lib):
    n = gb.layer_workspace_bytes(2, 300, 256, 4, 2, 128, "elementwise")
    rows = 600
    # the attention's plan (state, fp16 gate) + Q, K, V, O in bf16
    assert n >= rows * (4 + 2 + 2 + 4) * 128 * 2 + rows * 4 * 128 * 2 and n % 256 == 0
    assert gb.layer_workspace_bytes(0, 300, 256, 4, 2, 128, "elementwise") == 0
    for args in [(2, 300, 128, 4, 2, 128, "elementwise"),   # d_model < 256
                 (2, 300, 256, 4, 2, 64, "elementwise"),    # d_k 64
                 (2, 1, 256, 4, 2, 128, "elementwise"),     # one token
                 (2, 300, 256, 4, 2, 128, "headwise")]:
        with pytest.raises(gb.GsdpaError):
            gb.layer_workspace_bytes(*args)
    L = gb.load()
    st = L.gated_attention_layer(16, 16, 16, 16, 2, 300, 256, 4, 2, 128, 2, 1, None, 0, None)
    assert st == gb.ERR_WORKSPACE or st == gb.ERR_LAUNCH or st == gb.ERR_UNSUPPORTED   # (no device here)
    assert L.gated_attention_layer(8, 16, 16, 16, 2, 300, 256, 4, 2, 128, 2, 1, None, 0, None) == gb.ERR_ALIGNMENT
    assert L.gated_attention_layer(None, 16, 16, 16, 2, 300, 256, 4, 2, 128, 2, 1, None, 0, None) == gb.ERR_INVALID_ARG


def test_saved_gate_validation_before_any_device_work(lib):
    # gated_sdpa_fwd_train_save_gate / gated_sdpa_bwd_saved_gate: elementwise
    # gate and a 16-byte aligned gate buffer, checked before any device work
    lib_ = gb.load()
    ints = [1, 8, 8, 64, 4, 4, 128, 2, 1, gb.BF16]
    fwd = [16] * 9 + ints + [None, 0, None]     # X, Q, K, V, W_g, O, sink, lse, gate_out
    bad = list(fwd)
    bad[9 + 7] = 1                                # headwise
    assert lib_.gated_sdpa_fwd_train_save_gate(*bad) == gb.ERR_INVALID_ARG
    bad = list(fwd)
    bad[8] = None
    assert lib_.gated_sdpa_fwd_train_save_gate(*bad) == gb.ERR_INVALID_ARG
    bad = list(fwd)
    bad[8] = 24
    assert lib_.gated_sdpa_fwd_train_save_gate(*bad) == gb.ERR_ALIGNMENT
    bad = list(fwd)
    bad[9 + 9] = gb.F32                           # the training forward is bf16 only
    assert lib_.gated_sdpa_fwd_train_save_gate(*bad) == gb.ERR_UNSUPPORTED
    bwd = [16] * 14 + ints + [None, 0, None]    # X .. lse, gate_saved, dX, dQ, dK, dV, dW_g
    bad = list(bwd)
    bad[14 + 7] = 0                               # no gate
    assert lib_.gated_sdpa_bwd_saved_gate(*bad) == gb.ERR_INVALID_ARG
    bad = list(bwd)
    bad[8] = None
    assert lib_.gated_sdpa_bwd_saved_gate(*bad) == gb.ERR_INVALID_ARG
    bad = list(bwd)
    bad[8] = 40
    assert lib_.gated_sdpa_bwd_saved_gate(*bad) == gb.ERR_ALIGNMENT
    bad = list(bwd)
    bad[10] = 24                                  # dQ misaligned
    assert lib_.gated_sdpa_bwd_saved_gate(*bad) == gb.ERR_ALIGNMENT
    bad = list(bwd)
    bad[14 + 6] = 64                              # d_k 64 has no backward
    assert lib_.gated_sdpa_bwd_saved_gate(*bad) == gb.ERR_UNSUPPORTED


def test_binding_signatures_match_the_header():
    # every declaration's parameter count is the binding's argument count
    text = open(HEADER).read()
    decls = dict(re.findall(r"GSDPA_API\s+[\w\s\*]+?\b(\w+)\s*\(([^)]*)\)\s*;", text))
    assert decls.keys() == gb.SIGNATURES.keys()
    for name, params in decls.items():
        params = params.strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert len(gb.SIGNATURES[name][1]) == n, name


def test_binding_shape_helpers():
    # the sizes the binding derives from the tensors and checks every buffer against
    import torch
    Q = torch.empty(2, 5, 8, 16)
    K = torch.empty(2, 7, 4, 16)
    assert gb._attn_dims(Q, K, K.clone()) == (2, 5, 7, 8, 4, 16)
    with pytest.raises(ValueError):
        gb._attn_dims(Q, K, torch.empty(2, 6, 4, 16))        # V unlike K
    with pytest.raises(ValueError):
        gb._attn_dims(Q, torch.empty(2, 7, 4, 8), torch.empty(2, 7, 4, 8))   # d_k unlike Q's
    with pytest.raises(ValueError):
        gb._attn_dims(Q, torch.empty(3, 7, 4, 16), torch.empty(3, 7, 4, 16))  # batch unlike Q's
    assert gb._x_dim(torch.empty(2, 5, 32), 2, 5) == 32
    assert gb._x_dim(torch.empty(10, 32), 2, 5) == 32
    with pytest.raises(ValueError):
        gb._x_dim(torch.empty(2, 4, 32), 2, 5)
    assert gb._gate_cols(gb.GATE_ELEMENTWISE, 8, 16) == 128
    assert gb._gate_cols(gb.GATE_HEADWISE, 8, 16) == 8
    assert [gb._gate_cols(m, 8, 16) for m in (3, 4, 6, 7)] == [1, 16, 8, 128]


def test_binding_rejects_host_tensors_before_the_library():
    # a host tensor is refused by the binding's own checks, before any pointer
    # reaches the library
    import torch
    Q = torch.empty(1, 4, 2, 64, dtype=torch.bfloat16)
    K = torch.empty(1, 4, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        gb.gated_sdpa_fwd(None, Q, K, K.clone(), None, gate="none")
    with pytest.raises(ValueError, match="CUDA"):
        gb.decode_noalloc(None, Q[:, :1].contiguous(), K, K.clone(), None, gate="none")
