"""float64 CPU oracle for the G1 gated attention layer.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The GPU library never
imports this package, and this package imports nothing from the GPU library.

The arithmetic lives in ``gsdpa_oracle.c`` (plain C, double precision, the
layer's definition written out; its header lists the page and section each
step follows). This module compiles it with gcc on first use and exposes it
to numpy.

Every function here is pinned by ``tests/test_oracle_pins.py`` (and, for
the backward and the gate variants, ``tests/test_oracle_bwd_pins.py`` and
``tests/test_oracle_variant_pins.py``) against closed forms, invariants and
library routines (torch's CPU float64 SDPA and autograd, numpy matmul); no
function is left with parity unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gsdpa_oracle.c")
_LIB = os.path.join(_HERE, "libgsdpa_oracle.so")
_lock = threading.Lock()
_lib = None

GATE_NONE, GATE_HEADWISE, GATE_ELEMENTWISE = 0, 1, 2
GATE_HEADWISE_SHARED, GATE_ELEMENTWISE_SHARED, GATE_STATIC = 3, 4, 5
GATE_HEADWISE_AVERAGED, GATE_ELEMENTWISE_AVERAGED = 6, 7
_GATE_CODES = {"none": GATE_NONE, "headwise": GATE_HEADWISE, "elementwise": GATE_ELEMENTWISE}
_VARIANT_GATE_CODES = dict(_GATE_CODES, headwise_shared=GATE_HEADWISE_SHARED,
                           elementwise_shared=GATE_ELEMENTWISE_SHARED, static=GATE_STATIC,
                           headwise_averaged=GATE_HEADWISE_AVERAGED, elementwise_averaged=GATE_ELEMENTWISE_AVERAGED)
# the gate's function of its logit and its combination with the SDPA output y,
# or (without a gate) a function of y alone
GATE_FNS = {"sigmoid_mul": 0, "ns_sigmoid_mul": 1, "sigmoid_add": 2, "silu_add": 3, "identity_add": 4,
            "silu_self": 5, "rmsnorm": 6}


def build(force: bool = False) -> str:
    """Compile the oracle into a shared object next to its source."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)  # serial build without OpenMP
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int)
            lib.gsdpa_oracle_fwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp] + [ctypes.c_int] * 9 + [
                ip, ip, ctypes.c_long, ctypes.c_int]
            lib.gsdpa_oracle_fwd.restype = ctypes.c_int
            lib.gsdpa_oracle_fwd_variant.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp] + [ctypes.c_int] * 9 + [
                ctypes.c_double, ctypes.c_int, ip, ip, ctypes.c_long, ctypes.c_int]
            lib.gsdpa_oracle_fwd_variant.restype = ctypes.c_int
            lib.gsdpa_oracle_gate_scores.argtypes = [dp, dp, dp, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_int]
            lib.gsdpa_oracle_gate_scores.restype = ctypes.c_int
            lib.gsdpa_oracle_bwd.argtypes = [dp] * 11 + [ctypes.c_int] * 9
            lib.gsdpa_oracle_bwd.restype = ctypes.c_int
            lib.gsdpa_oracle_bwd_rows.argtypes = [dp] * 6 + [ctypes.c_int] * 9 + [ip, ip, ctypes.c_long, ip, ip,
                                                                                   ctypes.c_long, dp, dp, dp, dp,
                                                                                   ctypes.c_int]
            lib.gsdpa_oracle_bwd_rows.restype = ctypes.c_int
            lib.gsdpa_oracle_softmax_stats.argtypes = [dp, dp, dp, dp] + [ctypes.c_int] * 8
            lib.gsdpa_oracle_softmax_stats.restype = ctypes.c_int
            lib.gsdpa_oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().gsdpa_oracle_max_threads())


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor -> exact float64 upcast on the host
        a = a.detach().to("cpu")
        import torch
        a = a.to(torch.float64).numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a, t=ctypes.c_double):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(t))


def gated_sdpa(X, Q, K, V, W_g, *, gate="elementwise", causal=True, rows=None, n_threads=0, return_lse=False):
    """Gated SDPA in float64.

    Shapes: X [B, L_q, d_model], Q [B, L_q, H_q, d_k], K/V [B, L_k, H_kv, d_k],
    W_g [d_model, H_q*d_k] (elementwise) or [d_model, H_q] (headwise), or None
    when ``gate == "none"``.

    ``rows``: None for every row, else a list/array of (b, i) pairs.
    Returns (O, p0): O [B, L_q, H_q, d_k] (or [n_rows, H_q, d_k]) and the
    attention weight on key 0 per row and head, [B, L_q, H_q] (or [n_rows, H_q]);
    with ``return_lse``, also the natural-log softmax denominator per row and
    head (max score + log of the sum of exp(score - max)), shaped like p0.
    """
    gm = _GATE_CODES[gate]
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, Lq, Hq, dk = Q.shape
    _, Lk, Hkv, _ = K.shape
    if gm == GATE_NONE:
        Xd, Wd, d_model = None, None, 0
    else:
        Xd, Wd = _f64(X), _f64(W_g)
        d_model = Xd.shape[-1]
        expect = Hq * dk if gm == GATE_ELEMENTWISE else Hq
        if Wd.shape != (d_model, expect):
            raise ValueError(f"W_g shape {Wd.shape} != {(d_model, expect)}")
    if rows is None:
        O = np.empty((B, Lq, Hq, dk), np.float64)
        p0 = np.empty((B, Lq, Hq), np.float64)
        lse = np.empty((B, Lq, Hq), np.float64) if return_lse else None
        rb = ri = None
        n = -1
    else:
        rows = np.asarray(rows, dtype=np.int32).reshape(-1, 2)
        rb = np.ascontiguousarray(rows[:, 0])
        ri = np.ascontiguousarray(rows[:, 1])
        n = rows.shape[0]
        O = np.empty((n, Hq, dk), np.float64)
        p0 = np.empty((n, Hq), np.float64)
        lse = np.empty((n, Hq), np.float64) if return_lse else None
    rc = _load().gsdpa_oracle_fwd(
        _ptr(Xd), _ptr(Q), _ptr(K), _ptr(V), _ptr(Wd), _ptr(O), _ptr(p0), _ptr(lse),
        B, Lq, Lk, d_model, Hq, Hkv, dk, gm, int(bool(causal)),
        _ptr(rb, ctypes.c_int), _ptr(ri, ctypes.c_int), n, int(n_threads))
    if rc != 0:
        raise ValueError("oracle rejected the shapes or rows")
    return (O, p0, lse) if return_lse else (O, p0)


def gated_sdpa_variant(X, Q, K, V, W_g, *, gate="elementwise", gate_fn="sigmoid_mul", eps=1e-6, causal=True,
                       rows=None, n_threads=0):
    """The layer with one of the gate variants, in float64 (see the header of
    ``gsdpa_oracle.c`` for the definitions and their sources).

    ``gate``: "none", "headwise" (W_g [d_model, H_q]), "elementwise"
    ([d_model, H_q*d_k]), "headwise_shared" ([d_model, 1]), "elementwise_shared"
    ([d_model, d_k]), "static" (W_g holds theta [H_q, d_k]; X is not read), or
    "headwise_averaged" / "elementwise_averaged" (W_g as for "headwise" /
    "elementwise"; every head uses the mean over the heads of their values).
    ``gate_fn``: "sigmoid_mul", "ns_sigmoid_mul", "sigmoid_add", "silu_add" or
    "identity_add" with a gate; "silu_self" or "rmsnorm" (W_g holds gamma
    [H_q, d_k], or None for 1) with ``gate == "none"``.
    Returns (O, p0) shaped as :func:`gated_sdpa`'s.
    """
    gm = _VARIANT_GATE_CODES[gate]
    fn = GATE_FNS[gate_fn]
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, Lq, Hq, dk = Q.shape
    _, Lk, Hkv, _ = K.shape
    Xd = _f64(X) if (X is not None and gm not in (GATE_NONE, GATE_STATIC)) else None
    Wd = _f64(W_g) if W_g is not None else None
    d_model = Xd.shape[-1] if Xd is not None else 0
    if rows is None:
        O = np.empty((B, Lq, Hq, dk), np.float64)
        p0 = np.empty((B, Lq, Hq), np.float64)
        rb = ri = None
        n = -1
    else:
        rows = np.asarray(rows, dtype=np.int32).reshape(-1, 2)
        rb = np.ascontiguousarray(rows[:, 0])
        ri = np.ascontiguousarray(rows[:, 1])
        n = rows.shape[0]
        O = np.empty((n, Hq, dk), np.float64)
        p0 = np.empty((n, Hq), np.float64)
    rc = _load().gsdpa_oracle_fwd_variant(
        _ptr(Xd), _ptr(Q), _ptr(K), _ptr(V), _ptr(Wd), _ptr(O), _ptr(p0), None,
        B, Lq, Lk, d_model, Hq, Hkv, dk, gm, fn, float(eps), int(bool(causal)),
        _ptr(rb, ctypes.c_int), _ptr(ri, ctypes.c_int), n, int(n_threads))
    if rc != 0:
        raise ValueError("oracle rejected the shapes, the gate variant or the rows")
    return O, p0


def gate_scores(X, W_g, H_q, d_k, *, gate="elementwise"):
    """sigma(X W_g) in float64 for every row and gate column: [B*L_q, H_q*d_k]
    (elementwise) or [B*L_q, H_q] (headwise)."""
    gm = _GATE_CODES[gate]
    Xd, Wd = _f64(X), _f64(W_g)
    d_model = Xd.shape[-1]
    rows = Xd.size // d_model
    G = H_q * d_k if gm == GATE_ELEMENTWISE else H_q
    out = np.empty((rows, G), np.float64)
    rc = _load().gsdpa_oracle_gate_scores(_ptr(Xd), _ptr(Wd), _ptr(out), rows, d_model, H_q, d_k, gm)
    if rc != 0:
        raise ValueError("oracle rejected the gate")
    return out


def gate_statistics(scores, n_bins, threshold):
    """The gate statistics of "GatedAttention [2025]" sec. 1.4.2 (Table 4: the
    mean gating score; Figure 3: the distribution; appendix: the fraction of
    scores below a threshold) of an array of scores in [0, 1]: a dict with
    count, mean, below (how many scores are < threshold) and hist (n_bins
    equal bins over [0, 1]; bin k holds k/n <= s < (k+1)/n, 1 in the last)."""
    s = np.asarray(scores, np.float64).ravel()
    idx = np.minimum(np.floor(s * n_bins).astype(np.int64), n_bins - 1)
    hist = np.bincount(idx, minlength=n_bins)
    return {"count": int(s.size), "mean": float(s.mean()) if s.size else 0.0,
            "below": int(np.count_nonzero(s < threshold)), "hist": hist}


def gated_attention_layer(X, W_in, W_O, H_q, H_kv, d_k, *, gate="elementwise", causal=True, rows=None):
    """The layer around the attention, in float64 ("GatedAttention [2025]",
    sec. 1.2.1: Q = X W_Q, K = X W_K, V = X W_V; sec. 1.2.2: the gate
    sigma(X W_g); the gated heads concatenated and projected by W_O):
    W_in = [W_Q | W_K | W_V | W_g] [d_model, (H_q + 2 H_kv) d_k (+ H_q d_k)],
    W_O [H_q d_k, d_model]. The projections are matrix products (numpy), the
    attention is :func:`gated_sdpa`. Returns Y [B, L, d_model], or
    [n_rows, d_model] for the (b, i) pairs in ``rows``."""
    Xd, Wi, Wo = _f64(X), _f64(W_in), _f64(W_O)
    B, L, dm = Xd.shape
    qc, kc = H_q * d_k, H_kv * d_k
    P = Xd @ Wi
    Q = np.ascontiguousarray(P[..., :qc]).reshape(B, L, H_q, d_k)
    K = np.ascontiguousarray(P[..., qc:qc + kc]).reshape(B, L, H_kv, d_k)
    V = np.ascontiguousarray(P[..., qc + kc:qc + 2 * kc]).reshape(B, L, H_kv, d_k)
    Wg = np.ascontiguousarray(Wi[:, qc + 2 * kc:]) if gate != "none" else None
    O, _ = gated_sdpa(Xd if gate != "none" else None, Q, K, V, Wg, gate=gate, causal=causal, rows=rows)
    return O.reshape(O.shape[0], L, qc) @ Wo if rows is None else O.reshape(-1, qc) @ Wo


def gated_sdpa_bwd(X, Q, K, V, W_g, dO, *, gate="elementwise", causal=True):
    """Backward of :func:`gated_sdpa` in float64, given dO = dL/dO [B, L_q, H_q, d_k].

    Returns a dict with dQ, dK, dV and, with a gate, dX (the gate path's share)
    and dW_g, each shaped like its input.
    """
    gm = _GATE_CODES[gate]
    Q, K, V, dOd = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, Lq, Hq, dk = Q.shape
    _, Lk, Hkv, _ = K.shape
    if dOd.shape != Q.shape:
        raise ValueError(f"dO shape {dOd.shape} != {Q.shape}")
    if gm == GATE_NONE:
        Xd = Wd = dX = dW = None
        d_model = 0
    else:
        Xd, Wd = _f64(X), _f64(W_g)
        d_model = Xd.shape[-1]
        dX = np.empty_like(Xd)
        dW = np.empty_like(Wd)
    dQ = np.empty_like(Q)
    dK = np.empty_like(K)
    dV = np.empty_like(V)
    rc = _load().gsdpa_oracle_bwd(
        _ptr(Xd), _ptr(Q), _ptr(K), _ptr(V), _ptr(Wd), _ptr(dOd),
        _ptr(dX), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(dW),
        B, Lq, Lk, d_model, Hq, Hkv, dk, gm, int(bool(causal)))
    if rc != 0:
        raise ValueError("oracle rejected the shapes")
    out = {"dQ": dQ, "dK": dK, "dV": dV}
    if gm != GATE_NONE:
        out["dX"] = dX
        out["dW_g"] = dW
    return out


def softmax_stats(Q, K, *, causal=True, n_threads=0):
    """The softmax statistics of every query row and head in float64, without
    the values or the gate (half the cost of the full layer): p0 [B, L_q, H_q],
    the attention weight on key 0, and lse [B, L_q, H_q], the natural log of
    the softmax denominator (max score + log of the sum of exp(score - max))."""
    Q, K = _f64(Q), _f64(K)
    B, Lq, Hq, dk = Q.shape
    _, Lk, Hkv, _ = K.shape
    p0 = np.empty((B, Lq, Hq), np.float64)
    lse = np.empty((B, Lq, Hq), np.float64)
    rc = _load().gsdpa_oracle_softmax_stats(_ptr(Q), _ptr(K), _ptr(p0), _ptr(lse), B, Lq, Lk, Hq, Hkv, dk,
                                            int(bool(causal)), int(n_threads))
    if rc != 0:
        raise ValueError("oracle rejected the shapes")
    return p0, lse


def sink_share(p0):
    """First-token attention share per (b, h): the mean over query rows of p0.

    p0 is the [B, L_q, H_q] output of :func:`gated_sdpa` over all rows.
    """
    return np.asarray(p0).mean(axis=1)


def gated_sdpa_bwd_rows(X, Q, K, V, W_g, dO, q_rows, k_rows, *, gate="elementwise", causal=True, n_threads=0):
    """The backward's outputs on sampled rows: dQ for the (b, i) pairs in
    ``q_rows`` ([nq, H_q, d_k]), dK, dV for the (b, j) pairs in ``k_rows``
    ([nk, H_kv, d_k] each) and, with a gate, the gate path's input gradient
    dX for the rows of ``q_rows`` ([nq, d_model]). Same definition as
    :func:`gated_sdpa_bwd`."""
    gm = _GATE_CODES[gate]
    Q, K, V, dOd = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, Lq, Hq, dk = Q.shape
    _, Lk, Hkv, _ = K.shape
    if gm == GATE_NONE:
        Xd = Wd = None
        d_model = 0
    else:
        Xd, Wd = _f64(X), _f64(W_g)
        d_model = Xd.shape[-1]
    qr = np.asarray(q_rows, dtype=np.int32).reshape(-1, 2)
    kr = np.asarray(k_rows, dtype=np.int32).reshape(-1, 2)
    qb, qi = np.ascontiguousarray(qr[:, 0]), np.ascontiguousarray(qr[:, 1])
    kb, kj = np.ascontiguousarray(kr[:, 0]), np.ascontiguousarray(kr[:, 1])
    dQ = np.empty((qr.shape[0], Hq, dk), np.float64)
    dK = np.empty((kr.shape[0], Hkv, dk), np.float64)
    dV = np.empty((kr.shape[0], Hkv, dk), np.float64)
    dX = np.empty((qr.shape[0], d_model), np.float64) if gm != GATE_NONE else None
    ip = ctypes.c_int
    rc = _load().gsdpa_oracle_bwd_rows(
        _ptr(Xd), _ptr(Q), _ptr(K), _ptr(V), _ptr(Wd), _ptr(dOd), B, Lq, Lk, d_model, Hq, Hkv, dk, gm,
        int(bool(causal)), _ptr(qb, ip), _ptr(qi, ip), qr.shape[0], _ptr(kb, ip), _ptr(kj, ip), kr.shape[0],
        _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(dX), int(n_threads))
    if rc != 0:
        raise ValueError("oracle rejected the shapes or rows")
    out = {"dQ": dQ, "dK": dK, "dV": dV}
    if dX is not None:
        out["dX"] = dX
    return out
