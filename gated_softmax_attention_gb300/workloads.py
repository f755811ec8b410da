"""Seeded synthetic inputs for the gated attention layer.

This module holds no arithmetic of the layer itself: it only draws random
numbers, applies the input recipe and rounds to the storage dtype. Both the
GPU tests/benchmark and the float64 oracle take their inputs from here.

Recipe (the same on every machine):
  * a CPU ``torch.Generator`` seeded with the workload's seed draws float32
    standard normals in the order X, Q, K, V, W_g;
  * W_g is scaled by 0.02 (so W_g ~ N(0, 0.02^2));
  * the long-context workload multiplies every key of token 0 by 8 (all K/V
    heads, K only) to create sink-like score mass;
  * bf16 workloads round each tensor once to bf16 (round to nearest even);
    the GPU path and the oracle both see exactly those values.

Gate variants (``variant_weight``): a second generator seeded with
``seed + 7919`` draws the variant's parameter as float32 standard normals:
  * head-shared gates, W_g [d_model, 1] or [d_model, d_k], scaled by
    1/sqrt(d_model) (so the logits X W_g are about N(0, 1));
  * the input-independent gate, theta [H_q, d_k], unscaled;
  * the RMSNorm scale, gamma [H_q, d_k] = 1 + 0.1 N(0, 1);
then rounded once to the workload's dtype, like the other inputs.

The whole layer (``layer_weights``): a generator seeded with ``seed + 104729``
draws W_in [d_model, (H_q + 2 H_kv) d_k (+ H_q d_k gated)] ~ N(0, 1/d_model)
(so Q, K, V and the gate logits are about N(0, 1)) and W_O [H_q d_k, d_model]
~ N(0, 1/(H_q d_k)); X is the workload's own.

Layouts: X [B, L_q, d_model]; Q [B, L_q, H_q, d_k]; K, V [B, L_k, H_kv, d_k];
W_g [d_model, H_q*d_k] (elementwise, head-major columns) or [d_model, H_q]
(headwise). The model shapes follow the pages' settings: context 4096 for
training and 32k for the long-context stage ("GatedAttention [2025]",
sec. 1.3.1 and sec. 1.4.4).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str          # "f32" or "bf16"
    B: int
    L_q: int
    L_k: int
    d_model: int
    H_q: int
    H_kv: int
    d_k: int
    gate: str           # "none" | "headwise" | "elementwise"
    causal: bool
    seed: int
    key0_scale: float = 1.0
    wg_std: float = 0.02

    @property
    def gate_cols(self) -> int:
        if self.gate == "elementwise":
            return self.H_q * self.d_k
        if self.gate == "headwise":
            return self.H_q
        return 0

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    # -- algorithmic work per call (what one forward must read, write and compute) --
    def causal_pairs(self) -> int:
        """(query, key) pairs that enter the softmax, summed over one (b, h)."""
        if not self.causal:
            return self.L_q * self.L_k
        off = self.L_k - self.L_q
        # query i sees keys 0..off+i
        return self.L_q * (off + 1) + self.L_q * (self.L_q - 1) // 2

    def attn_flops(self) -> int:
        return 4 * self.B * self.H_q * self.d_k * self.causal_pairs()

    def gate_flops(self) -> int:
        return 2 * self.B * self.L_q * self.d_model * self.gate_cols

    def flops(self) -> int:
        return self.attn_flops() + self.gate_flops()

    def algorithmic_bytes(self) -> int:
        es = 4 if self.dtype == "f32" else 2
        n = 0
        if self.gate != "none":
            n += self.B * self.L_q * self.d_model + self.d_model * self.gate_cols
        n += self.B * self.L_q * self.H_q * self.d_k            # Q
        n += 2 * self.B * self.L_k * self.H_kv * self.d_k       # K, V
        n += self.B * self.L_q * self.H_q * self.d_k            # O
        return n * es


# The named workloads: shapes and gates of the pages' model settings.
WORKLOADS = {
    w.name: w for w in [
        # small fp32 case the oracle finishes instantly
        Workload("f32_mha_elementwise_L128", "f32", B=1, L_q=128, L_k=128, d_model=256,
                 H_q=4, H_kv=4, d_k=64, gate="elementwise", causal=True, seed=0),
        # bf16 causal prefill, MHA, elementwise gate (the headline prefill case)
        Workload("bf16_mha_elementwise_L2048", "bf16", B=2, L_q=2048, L_k=2048, d_model=2048,
                 H_q=16, H_kv=16, d_k=128, gate="elementwise", causal=True, seed=1),
        # bf16 causal prefill, GQA 32/4, headwise gate, context 4096
        Workload("bf16_gqa_headwise_L4096", "bf16", B=1, L_q=4096, L_k=4096, d_model=4096,
                 H_q=32, H_kv=4, d_k=128, gate="headwise", causal=True, seed=2),
        # bf16 long context 32k, GQA 16/2, headwise gate, token-0 keys x8
        Workload("bf16_gqa_headwise_sink_L32768", "bf16", B=1, L_q=32768, L_k=32768, d_model=2048,
                 H_q=16, H_kv=2, d_k=128, gate="headwise", causal=True, seed=3, key0_scale=8.0),
        # bf16 decode: 64 single-query rows against an 8192-token cache
        Workload("bf16_decode_gqa_elementwise_Lk8192", "bf16", B=64, L_q=1, L_k=8192, d_model=4096,
                 H_q=32, H_kv=8, d_k=128, gate="elementwise", causal=True, seed=4),
    ]
}

PREFILL_HEADLINE = "bf16_mha_elementwise_L2048"
DECODE_HEADLINE = "bf16_decode_gqa_elementwise_Lk8192"


def torch_dtype(w: Workload):
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def make_inputs(w: Workload, device="cpu"):
    """Return dict(X, Q, K, V, W_g) for workload ``w`` on ``device``.

    Values are drawn on the CPU (so every machine gets the same numbers) and
    then moved. X and W_g are None when the gate is "none".
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed))
    f = torch.float32
    X = torch.randn((w.B, w.L_q, w.d_model), generator=g, dtype=f) if w.d_model > 0 else None
    Q = torch.randn((w.B, w.L_q, w.H_q, w.d_k), generator=g, dtype=f)
    K = torch.randn((w.B, w.L_k, w.H_kv, w.d_k), generator=g, dtype=f)
    V = torch.randn((w.B, w.L_k, w.H_kv, w.d_k), generator=g, dtype=f)
    W = None
    if w.gate != "none":
        W = torch.randn((w.d_model, w.gate_cols), generator=g, dtype=f) * w.wg_std
    if w.key0_scale != 1.0:
        K[:, 0, :, :] *= w.key0_scale
    td = torch_dtype(w)
    out = {}
    for k, t in (("X", X), ("Q", Q), ("K", K), ("V", V), ("W_g", W)):
        if t is None or (k == "X" and w.gate == "none"):
            out[k] = None
            continue
        out[k] = t.to(td).contiguous().to(device)
    return out


def variant_weight(w: Workload, gate: str, gate_fn: str = "sigmoid_mul", device="cpu"):
    """The parameter a gate variant reads in place of W_g: the head-shared
    and averaged gates' W_g (scaled so that the logits are about N(0, 1)), the
    input-independent gate's theta, or the RMSNorm scale gamma
    (None for the gates that use the workload's own W_g, and for a variant
    without a parameter)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed) + 7919)
    f = torch.float32
    if gate == "headwise_shared":
        t = torch.randn((w.d_model, 1), generator=g, dtype=f) / w.d_model ** 0.5
    elif gate == "headwise_averaged":
        t = torch.randn((w.d_model, w.H_q), generator=g, dtype=f) / w.d_model ** 0.5
    elif gate == "elementwise_averaged":
        t = torch.randn((w.d_model, w.H_q * w.d_k), generator=g, dtype=f) / w.d_model ** 0.5
    elif gate == "elementwise_shared":
        t = torch.randn((w.d_model, w.d_k), generator=g, dtype=f) / w.d_model ** 0.5
    elif gate == "static":
        t = torch.randn((w.H_q, w.d_k), generator=g, dtype=f)
    elif gate == "none" and gate_fn == "rmsnorm":
        t = 1.0 + 0.1 * torch.randn((w.H_q, w.d_k), generator=g, dtype=f)
    else:
        return None
    return t.to(torch_dtype(w)).contiguous().to(device)


def layer_weights(w: Workload, device="cpu"):
    """(W_in, W_O) of the whole layer for workload ``w`` (see the recipe above)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed) + 104729)
    f = torch.float32
    n_in = (w.H_q + 2 * w.H_kv) * w.d_k + w.gate_cols   # the gate's columns: H_q d_k, H_q or none
    W_in = torch.randn((w.d_model, n_in), generator=g, dtype=f) / w.d_model ** 0.5
    W_O = torch.randn((w.H_q * w.d_k, w.d_model), generator=g, dtype=f) / (w.H_q * w.d_k) ** 0.5
    td = torch_dtype(w)
    return W_in.to(td).contiguous().to(device), W_O.to(td).contiguous().to(device)
