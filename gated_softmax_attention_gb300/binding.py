"""ctypes binding of libgsdpa.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels. Torch is
used here for device memory (output and workspace tensors when the caller
does not pass them) and for the current stream. If the library has not been
built, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgsdpa.so")

GATE_NONE, GATE_HEADWISE, GATE_ELEMENTWISE = 0, 1, 2
GATE_CODES = {"none": GATE_NONE, "headwise": GATE_HEADWISE, "elementwise": GATE_ELEMENTWISE}
F32, BF16 = 0, 1

OK = 0
ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_WORKSPACE, ERR_LAUNCH, ERR_DEVICE_TIMEOUT = -1, -2, -3, -4, -5, -6

# Every entry point the header declares, with its ctypes signature.
_VP, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "gsdpa_workspace_bytes": (_SZ, [_I] * 10),
    "gated_sdpa_fwd": (_I, [_VP] * 7 + [_I] * 10 + [_VP, _SZ, _VP]),
    "gated_sdpa_fwd_train": (_I, [_VP] * 8 + [_I] * 10 + [_VP, _SZ, _VP]),
    "gated_sdpa_fwd_train_save_gate": (_I, [_VP] * 9 + [_I] * 10 + [_VP, _SZ, _VP]),
    "gsdpa_workspace_bytes_variant": (_SZ, [_I] * 11),
    "gated_sdpa_fwd_stats": (_I, [_VP] * 8 + [_I, ctypes.c_float] + [_I] * 10 + [_VP, _SZ, _VP]),
    "gsdpa_layer_workspace_bytes": (_SZ, [_I] * 7),
    "gated_attention_layer": (_I, [_VP] * 4 + [_I] * 8 + [_VP, _SZ, _VP]),
    "gated_sdpa_fwd_variant": (_I, [_VP] * 7 + [_I] * 9 + [ctypes.c_float, _I, _I, _VP, _SZ, _VP]),
    "gsdpa_bwd_workspace_bytes": (_SZ, [_I] * 8),
    "gated_sdpa_bwd": (_I, [_VP] * 13 + [_I] * 10 + [_VP, _SZ, _VP]),
    "gated_sdpa_bwd_saved_gate": (_I, [_VP] * 14 + [_I] * 10 + [_VP, _SZ, _VP]),
    "gsdpa_check_device_error": (_I, [_VP]),
    "gsdpa_status_string": (ctypes.c_char_p, [_I]),
    "gsdpa_set_wait_limit_ns": (_I, [ctypes.c_ulonglong]),
    "gsdpa_wait_self_test": (_I, [_VP]),
    "gated_sdpa_decode_noalloc": (_I, [_VP] * 7 + [_I] * 7 + [_VP]),
    "gsdpa_decode_noalloc_max_scratch": (_SZ, []),
}

_lock = threading.Lock()
_lib = None


class GsdpaError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def load(path: str = LIB_PATH):
    """Load libgsdpa.so (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with "
                                   "`python -m gated_softmax_attention_gb300.build`")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().gsdpa_status_string(int(status)).decode()


def workspace_bytes(B, L_q, L_k, d_model, H_q, H_kv, d_k, gate="elementwise", want_sink=False, dtype=BF16) -> int:
    n = load().gsdpa_workspace_bytes(B, L_q, L_k, d_model, H_q, H_kv, d_k, GATE_CODES[gate], int(bool(want_sink)),
                                     dtype)
    if n == ctypes.c_size_t(-1).value:
        raise GsdpaError(ERR_INVALID_ARG, "gsdpa_workspace_bytes")
    return int(n)


def set_wait_limit_ns(ns: int) -> None:
    load().gsdpa_set_wait_limit_ns(int(ns))


def wait_self_test(stream=None) -> int:
    """Enqueue the bounded-wait diagnostic (a wait nothing completes); returns the launch status."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(load().gsdpa_wait_self_test(ctypes.c_void_p(s.cuda_stream)))


def check_device_error(stream=None) -> int:
    """Synchronise the stream and return the device error status (0 = none)."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(load().gsdpa_check_device_error(ctypes.c_void_p(s.cuda_stream)))


def fwd_raw(X, Q, K, V, W_g, O, sink, B, L_q, L_k, d_model, H_q, H_kv, d_k, gate_mode, causal, dtype,
            workspace, workspace_bytes, stream) -> int:
    """Direct call of gated_sdpa_fwd with integer pointers; returns the status."""
    return int(load().gated_sdpa_fwd(X, Q, K, V, W_g, O, sink, B, L_q, L_k, d_model, H_q, H_kv, d_k, gate_mode,
                                     int(bool(causal)), dtype, workspace, workspace_bytes, stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# The library receives bare pointers and sizes: it cannot see how large a
# buffer is. Every tensor is therefore checked here against the sizes the
# problem implies (dtype, element count, device, contiguity) before its
# pointer is passed, so that a wrong-shaped argument raises instead of being
# read or written past its end.
def _expect(t, name, numel, dtype, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, not {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, the call's tensors on {device}")
    if t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements (shape {tuple(t.shape)}), the problem needs {numel}")


def _stream(stream, device):
    """The stream to launch on: the caller's, else the current stream of the
    device that holds the tensors (which must then be the current device)."""
    import torch
    if stream is None:
        if device.index != torch.cuda.current_device():
            raise ValueError(f"the tensors are on {device} but the current device is "
                             f"cuda:{torch.cuda.current_device()}: pass a stream of {device}")
        return torch.cuda.current_stream()
    if stream.device != device:
        raise ValueError(f"the stream belongs to {stream.device}, the tensors to {device}")
    return stream


def _attn_dims(Q, K, V):
    """(B, L_q, L_k, H_q, H_kv, d_k) from Q [B, L_q, H_q, d_k] and K, V [B, L_k, H_kv, d_k]."""
    if Q.dim() != 4 or K.dim() != 4 or V.dim() != 4:
        raise ValueError("Q, K and V must be 4-D: [B, L, H, d_k]")
    B, L_q, H_q, d_k = Q.shape
    if tuple(K.shape) != tuple(V.shape) or K.shape[0] != B or K.shape[3] != d_k:
        raise ValueError(f"K {tuple(K.shape)} and V {tuple(V.shape)} must be [B={B}, L_k, H_kv, d_k={d_k}]")
    return B, L_q, K.shape[1], H_q, K.shape[2], d_k


def _x_dim(X, B, L_q):
    """d_model of X [B, L_q, d_model] (any shape with that element count and last dimension)."""
    if X is None or X.dim() == 0:
        raise ValueError("X is required")
    d_model = X.shape[-1]
    if X.numel() != B * L_q * d_model:
        raise ValueError(f"X {tuple(X.shape)} must hold B * L_q = {B * L_q} rows of d_model = {d_model}")
    return d_model


# columns of W_g [d_model, G] (or the rows x columns of a table that does not read X)
def _gate_cols(gate_mode, H_q, d_k):
    return {GATE_HEADWISE: H_q, GATE_ELEMENTWISE: H_q * d_k, 3: 1, 4: d_k, 6: H_q, 7: H_q * d_k}[gate_mode]


def gated_sdpa_fwd(X, Q, K, V, W_g=None, *, gate="elementwise", causal=True, out=None, sink=None,
                   want_sink=False, workspace=None, stream=None):
    """Gated attention forward through the C ABI on torch CUDA tensors.

    X [B, L_q, d_model], Q [B, L_q, H_q, d_k], K/V [B, L_k, H_kv, d_k],
    W_g [d_model, H_q*d_k | H_q] (None for gate="none"). All contiguous, on
    the current CUDA device, float32 or bfloat16 (all the same dtype).
    Returns (O, sink) where sink is None unless requested.
    """
    O, sink, _ = _fwd(X, Q, K, V, W_g, gate, causal, out, sink, want_sink, None, workspace, stream)
    return O, sink


def gated_sdpa_fwd_train(X, Q, K, V, W_g=None, *, gate="elementwise", causal=True, out=None, sink=None,
                         want_sink=False, lse=None, workspace=None, stream=None):
    """gated_sdpa_fwd that also returns lse [B, H_q, L_q] float32, the natural
    log of each row's softmax denominator (bf16 prefill). Returns (O, sink, lse)."""
    import torch
    B, L_q, H_q, _ = Q.shape
    if lse is None:
        lse = torch.empty((B, H_q, L_q), dtype=torch.float32, device=Q.device)
    return _fwd(X, Q, K, V, W_g, gate, causal, out, sink, want_sink, lse, workspace, stream)


def gated_sdpa_fwd_train_save_gate(X, Q, K, V, W_g, *, causal=True, out=None, sink=None, want_sink=False, lse=None,
                                   gate_out=None, workspace=None, stream=None):
    """gated_sdpa_fwd_train for the elementwise gate that also returns the gate's
    fp16 values [B * L_q, H_q * d_k] for gated_sdpa_bwd_saved_gate. Returns
    (O, sink, lse, gate_out)."""
    import torch
    B, L_q, H_q, d_k = Q.shape
    if lse is None:
        lse = torch.empty((B, H_q, L_q), dtype=torch.float32, device=Q.device)
    if gate_out is None:
        gate_out = torch.empty((B * L_q, H_q * d_k), dtype=torch.float16, device=Q.device)
    O, sink, lse = _fwd(X, Q, K, V, W_g, "elementwise", causal, out, sink, want_sink, lse, workspace, stream,
                        gate_out=gate_out)
    return O, sink, lse, gate_out


def _workspace(workspace, need, device):
    """(pointer, size in bytes) of the call's workspace: the caller's tensor,
    whose real size is passed so that the library can reject one too small,
    or a new one of the size the problem needs."""
    import torch
    if workspace is None:
        if need <= 0:
            return None, 0
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("the workspace must be a contiguous CUDA tensor")
    if workspace.device != device:
        raise ValueError(f"the workspace is on {workspace.device}, the call's tensors on {device}")
    return workspace, workspace.numel() * workspace.element_size()


def _fwd(X, Q, K, V, W_g, gate, causal, out, sink, want_sink, lse, workspace, stream, gate_out=None):
    import torch
    if Q.dtype == torch.bfloat16:
        dtype = BF16
    elif Q.dtype == torch.float32:
        dtype = F32
    else:
        raise TypeError(f"unsupported dtype {Q.dtype}")
    gm = GATE_CODES[gate]
    B, L_q, L_k, H_q, H_kv, d_k = _attn_dims(Q, K, V)
    dev = Q.device
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        _expect(t, name, t.numel(), Q.dtype, dev)
    d_model = 0
    if gm != GATE_NONE:
        d_model = _x_dim(X, B, L_q)
        _expect(X, "X", B * L_q * d_model, Q.dtype, dev)
        _expect(W_g, "W_g", d_model * _gate_cols(gm, H_q, d_k), Q.dtype, dev)
    if out is None:
        out = torch.empty_like(Q)
    _expect(out, "out", Q.numel(), Q.dtype, dev)
    if sink is None and want_sink:
        sink = torch.empty((B, H_q), dtype=torch.float32, device=dev)
    if sink is not None:
        _expect(sink, "sink", B * H_q, torch.float32, dev)
    if lse is not None:
        _expect(lse, "lse", B * H_q * L_q, torch.float32, dev)
    if gate_out is not None:
        _expect(gate_out, "gate_out", B * L_q * H_q * d_k, torch.float16, dev)
    need = workspace_bytes(B, L_q, L_k, d_model, H_q, H_kv, d_k, gate, sink is not None, dtype)
    workspace, ws_bytes = _workspace(workspace, need, dev)
    s = _stream(stream, dev)
    args = [_ptr(X) if gm != GATE_NONE else None, _ptr(Q), _ptr(K), _ptr(V),
            _ptr(W_g) if gm != GATE_NONE else None, _ptr(out), _ptr(sink)]
    tail = [B, L_q, L_k, d_model, H_q, H_kv, d_k, gm, int(bool(causal)), dtype,
            _ptr(workspace), ws_bytes, ctypes.c_void_p(s.cuda_stream)]
    if gate_out is not None:
        st = int(load().gated_sdpa_fwd_train_save_gate(*args, _ptr(lse), _ptr(gate_out), *tail))
        where = "gated_sdpa_fwd_train_save_gate"
    elif lse is None:
        st = int(load().gated_sdpa_fwd(*args, *tail))
        where = "gated_sdpa_fwd"
    else:
        st = int(load().gated_sdpa_fwd_train(*args, _ptr(lse), *tail))
        where = "gated_sdpa_fwd_train"
    if st != OK:
        raise GsdpaError(st, where)
    return out, sink, lse


# gate shapes and gate functions of gated_sdpa_fwd_variant (gsdpa.h)
VARIANT_GATE_CODES = dict(GATE_CODES, headwise_shared=3, elementwise_shared=4, static=5, headwise_averaged=6,
                          elementwise_averaged=7)
GATE_FNS = {"sigmoid_mul": 0, "ns_sigmoid_mul": 1, "sigmoid_add": 2, "silu_add": 3, "identity_add": 4,
            "silu_self": 5, "rmsnorm": 6}


def workspace_bytes_variant(B, L_q, L_k, d_model, H_q, H_kv, d_k, gate="elementwise", gate_fn="sigmoid_mul",
                            want_sink=False, dtype=BF16) -> int:
    n = load().gsdpa_workspace_bytes_variant(B, L_q, L_k, d_model, H_q, H_kv, d_k, VARIANT_GATE_CODES[gate],
                                             GATE_FNS[gate_fn], int(bool(want_sink)), dtype)
    if n == ctypes.c_size_t(-1).value:
        raise GsdpaError(ERR_INVALID_ARG, "gsdpa_workspace_bytes_variant")
    return int(n)


def gated_sdpa_fwd_variant(X, Q, K, V, W_g=None, *, gate="elementwise", gate_fn="sigmoid_mul", eps=1e-6,
                           causal=True, out=None, sink=None, want_sink=False, workspace=None, stream=None):
    """The forward with a gate variant (gated_sdpa_fwd_variant): ``gate`` one of
    none, headwise, elementwise, headwise_shared (W_g [d_model, 1]),
    elementwise_shared (W_g [d_model, d_k]), static (W_g = theta [H_q, d_k],
    X unused); ``gate_fn`` one of GATE_FNS (rmsnorm: W_g = gamma [H_q, d_k] or
    None). Returns (O, sink)."""
    import torch
    if Q.dtype == torch.bfloat16:
        dtype = BF16
    elif Q.dtype == torch.float32:
        dtype = F32
    else:
        raise TypeError(f"unsupported dtype {Q.dtype}")
    gm, fn = VARIANT_GATE_CODES[gate], GATE_FNS[gate_fn]
    reads_x = gm not in (GATE_NONE, 5)
    B, L_q, L_k, H_q, H_kv, d_k = _attn_dims(Q, K, V)
    dev = Q.device
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        _expect(t, name, t.numel(), Q.dtype, dev)
    d_model = 0
    if reads_x:
        d_model = _x_dim(X, B, L_q)
        _expect(X, "X", B * L_q * d_model, Q.dtype, dev)
        _expect(W_g, "W_g", d_model * _gate_cols(gm, H_q, d_k), Q.dtype, dev)
    elif gm == 5:
        _expect(W_g, "W_g (theta)", H_q * d_k, Q.dtype, dev)
    elif fn == GATE_FNS["rmsnorm"] and W_g is not None:
        _expect(W_g, "W_g (gamma)", H_q * d_k, Q.dtype, dev)
    if out is None:
        out = torch.empty_like(Q)
    _expect(out, "out", Q.numel(), Q.dtype, dev)
    if sink is None and want_sink:
        sink = torch.empty((B, H_q), dtype=torch.float32, device=dev)
    if sink is not None:
        _expect(sink, "sink", B * H_q, torch.float32, dev)
    need = workspace_bytes_variant(B, L_q, L_k, d_model, H_q, H_kv, d_k, gate, gate_fn, sink is not None, dtype)
    workspace, ws_bytes = _workspace(workspace, need, dev)
    s = _stream(stream, dev)
    st = int(load().gated_sdpa_fwd_variant(
        _ptr(X) if reads_x else None, _ptr(Q), _ptr(K), _ptr(V), _ptr(W_g), _ptr(out), _ptr(sink),
        B, L_q, L_k, d_model, H_q, H_kv, d_k, gm, fn, float(eps), int(bool(causal)), dtype,
        _ptr(workspace), ws_bytes, ctypes.c_void_p(s.cuda_stream)))
    if st != OK:
        raise GsdpaError(st, "gated_sdpa_fwd_variant")
    return out, sink


def gated_sdpa_fwd_stats(X, Q, K, V, W_g, *, gate="elementwise", causal=True, n_bins=20, threshold=0.1, out=None,
                         workspace=None, stream=None):
    """gated_sdpa_fwd with the gate statistics: returns (O, stats) where stats is
    a dict with count, mean (sum / 2^32 / count), below, hist (n_bins counts)."""
    import torch
    dtype = BF16 if Q.dtype == torch.bfloat16 else F32
    gm = GATE_CODES[gate]
    B, L_q, L_k, H_q, H_kv, d_k = _attn_dims(Q, K, V)
    dev = Q.device
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        _expect(t, name, t.numel(), Q.dtype, dev)
    d_model = _x_dim(X, B, L_q)
    _expect(X, "X", B * L_q * d_model, Q.dtype, dev)
    if gm != GATE_NONE:   # (without a gate the library rejects the call)
        _expect(W_g, "W_g", d_model * _gate_cols(gm, H_q, d_k), Q.dtype, dev)
    if out is None:
        out = torch.empty_like(Q)
    _expect(out, "out", Q.numel(), Q.dtype, dev)
    st = torch.empty(3 + n_bins, dtype=torch.int64, device=dev)
    need = workspace_bytes(B, L_q, L_k, d_model, H_q, H_kv, d_k, gate, False, dtype)
    workspace, ws_bytes = _workspace(workspace, need, dev)
    s = _stream(stream, dev)
    status = int(load().gated_sdpa_fwd_stats(
        _ptr(X), _ptr(Q), _ptr(K), _ptr(V), _ptr(W_g), _ptr(out), None, _ptr(st), int(n_bins), float(threshold),
        B, L_q, L_k, d_model, H_q, H_kv, d_k, gm, int(bool(causal)), dtype,
        _ptr(workspace), ws_bytes, ctypes.c_void_p(s.cuda_stream)))
    if status != OK:
        raise GsdpaError(status, "gated_sdpa_fwd_stats")
    h = st.cpu().tolist()
    count = h[0]
    return out, {"count": count, "sum_fixed": h[1], "mean": (h[1] / 2.0 ** 32 / count) if count else 0.0,
                 "below": h[2], "hist": h[3:]}


def layer_workspace_bytes(B, L, d_model, H_q, H_kv, d_k, gate="elementwise") -> int:
    n = load().gsdpa_layer_workspace_bytes(B, L, d_model, H_q, H_kv, d_k, GATE_CODES[gate])
    if n == ctypes.c_size_t(-1).value:
        raise GsdpaError(ERR_UNSUPPORTED, "gsdpa_layer_workspace_bytes")
    return int(n)


def gated_attention_layer(X, W_in, W_O, *, H_q, H_kv, d_k=128, gate="elementwise", causal=True, out=None,
                          workspace=None, stream=None):
    """The whole layer (gated_attention_layer): X [B, L, d_model] bf16, W_in
    [d_model, (H_q + 2 H_kv) d_k + G] (G = H_q d_k elementwise, H_q headwise,
    0 without a gate), W_O [H_q d_k, d_model]. Returns Y."""
    import torch
    if X.dim() != 3:
        raise ValueError("X must be [B, L, d_model]")
    B, L, d_model = X.shape
    dev = X.device
    gm = GATE_CODES[gate]
    G = 0 if gm == GATE_NONE else _gate_cols(gm, H_q, d_k)
    _expect(X, "X", X.numel(), torch.bfloat16, dev)
    _expect(W_in, "W_in", d_model * ((H_q + 2 * H_kv) * d_k + G), torch.bfloat16, dev)
    _expect(W_O, "W_O", H_q * d_k * d_model, torch.bfloat16, dev)
    if out is None:
        out = torch.empty_like(X)
    _expect(out, "out", X.numel(), torch.bfloat16, dev)
    need = layer_workspace_bytes(B, L, d_model, H_q, H_kv, d_k, gate)
    workspace, ws_bytes = _workspace(workspace, need, dev)
    s = _stream(stream, dev)
    st = int(load().gated_attention_layer(_ptr(X), _ptr(W_in), _ptr(W_O), _ptr(out), B, L, d_model, H_q, H_kv, d_k,
                                          GATE_CODES[gate], int(bool(causal)),
                                          _ptr(workspace), ws_bytes,
                                          ctypes.c_void_p(s.cuda_stream)))
    if st != OK:
        raise GsdpaError(st, "gated_attention_layer")
    return out


def bwd_workspace_bytes(B, L_q, L_k, d_model, H_q, H_kv, d_k, gate="elementwise") -> int:
    n = load().gsdpa_bwd_workspace_bytes(B, L_q, L_k, d_model, H_q, H_kv, d_k, GATE_CODES[gate])
    if n == ctypes.c_size_t(-1).value:
        raise GsdpaError(ERR_UNSUPPORTED, "gsdpa_bwd_workspace_bytes")
    return int(n)


def gated_sdpa_bwd(X, Q, K, V, W_g, O, dO, lse, *, gate="elementwise", causal=True, workspace=None, stream=None,
                   gate_saved=None):
    """Backward through the C ABI (bf16, d_k = 128): returns a dict with dQ, dK,
    dV and, with a gate, dX (the gate path's share) and dW_g. gate_saved (the
    elementwise gate's values from gated_sdpa_fwd_train_save_gate) calls
    gated_sdpa_bwd_saved_gate, which does not recompute them."""
    import torch
    gm = GATE_CODES[gate]
    B, L_q, L_k, H_q, H_kv, d_k = _attn_dims(Q, K, V)
    dev = Q.device
    bf = torch.bfloat16
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        _expect(t, name, t.numel(), bf, dev)
    _expect(O, "O", Q.numel(), bf, dev)
    _expect(dO, "dO", Q.numel(), bf, dev)
    _expect(lse, "lse", B * H_q * L_q, torch.float32, dev)
    d_model = 0
    if gm != GATE_NONE:
        d_model = _x_dim(X, B, L_q)
        _expect(X, "X", B * L_q * d_model, bf, dev)
        _expect(W_g, "W_g", d_model * _gate_cols(gm, H_q, d_k), bf, dev)
    out = {"dQ": torch.empty_like(Q), "dK": torch.empty_like(K), "dV": torch.empty_like(V)}
    if gm != GATE_NONE:
        out["dX"] = torch.empty_like(X)
        out["dW_g"] = torch.empty_like(W_g)
    need = bwd_workspace_bytes(B, L_q, L_k, d_model, H_q, H_kv, d_k, gate)
    workspace, ws_bytes = _workspace(workspace, need, dev)
    s = _stream(stream, dev)
    head = [_ptr(X) if gm != GATE_NONE else None, _ptr(Q), _ptr(K), _ptr(V), _ptr(W_g) if gm != GATE_NONE else None,
            _ptr(O), _ptr(dO), _ptr(lse)]
    rest = [_ptr(out.get("dX")), _ptr(out["dQ"]), _ptr(out["dK"]), _ptr(out["dV"]), _ptr(out.get("dW_g")), B, L_q,
            L_k, d_model, H_q, H_kv, d_k, gm, int(bool(causal)), BF16, _ptr(workspace),
            ws_bytes, ctypes.c_void_p(s.cuda_stream)]
    if gate_saved is not None:
        _expect(gate_saved, "gate_saved", B * L_q * H_q * d_k, torch.float16, dev)
        st, where = int(load().gated_sdpa_bwd_saved_gate(*head, _ptr(gate_saved), *rest)), "gated_sdpa_bwd_saved_gate"
    else:
        st, where = int(load().gated_sdpa_bwd(*head, *rest)), "gated_sdpa_bwd"
    if st != OK:
        raise GsdpaError(st, where)
    return out


def decode_noalloc(X, Q, K, V, W_g=None, *, gate="elementwise", out=None, sink=None, want_sink=False, stream=None):
    """The decode call (L_q == 1, bf16) without a workspace: the library's fixed
    scratch array is used instead (for callers that cannot allocate device
    memory). Same tensors as gated_sdpa_fwd with L_q == 1."""
    import torch
    gm = GATE_CODES[gate]
    B, L_q, L_k, H_q, H_kv, d_k = _attn_dims(Q, K, V)
    if L_q != 1:
        raise ValueError("decode_noalloc takes one query row per sequence")
    dev = Q.device
    bf = torch.bfloat16
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        _expect(t, name, t.numel(), bf, dev)
    d_model = 0
    if gm != GATE_NONE:
        d_model = _x_dim(X, B, L_q)
        _expect(X, "X", B * d_model, bf, dev)
        _expect(W_g, "W_g", d_model * _gate_cols(gm, H_q, d_k), bf, dev)
    if out is None:
        out = torch.empty_like(Q)
    _expect(out, "out", Q.numel(), bf, dev)
    if sink is None and want_sink:
        sink = torch.empty((B, H_q), dtype=torch.float32, device=dev)
    if sink is not None:
        _expect(sink, "sink", B * H_q, torch.float32, dev)
    s = _stream(stream, dev)
    st = int(load().gated_sdpa_decode_noalloc(
        _ptr(X) if gm != GATE_NONE else None, _ptr(Q), _ptr(K), _ptr(V), _ptr(W_g) if gm != GATE_NONE else None,
        _ptr(out), _ptr(sink), B, L_k, d_model, H_q, H_kv, d_k, gm, ctypes.c_void_p(s.cuda_stream)))
    if st != OK:
        raise GsdpaError(st, "gated_sdpa_decode_noalloc")
    return out, sink
