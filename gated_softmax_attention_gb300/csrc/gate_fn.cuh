// gate_fn.cuh -- the gate functions of the attention epilogues and the gate
// passes: how a gate logit gl becomes the gate's value, and how that value
// acts on the SDPA output y ("GatedAttention [2025]", sec. 1.2.2 items (4),
// (5); sec. 1.4.2 (iv) for NS-sigmoid). Codes are gsdpa_gate_fn's.
#pragma once
#include <cstdint>

#include "gsdpa_internal.h"

namespace gsdpa {

// sigma(x) = 1/2 + tanh(x/2)/2 with one MUFU operation (tanh.approx, relative
// error about 2^-11).
__device__ __forceinline__ float sigmoid_tanh(float x) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
    return fmaf(0.5f, t, 0.5f);
}

// The gate's value for gate functions 0..4: sigma, NS-sigmoid, sigma, SiLU, identity.
__device__ __forceinline__ float gate_value(float gl, int fn) {
    switch (fn) {
    case 1: return fmaf(0.5f, sigmoid_tanh(gl), 0.5f);
    case 3: return gl * sigmoid_tanh(gl);
    case 4: return gl;
    default: return sigmoid_tanh(gl);
    }
}

// Gate functions 2..4 add the gate's value to y, 0 and 1 multiply.
__device__ __forceinline__ bool gate_adds(int fn) { return fn >= 2 && fn <= 4; }

__device__ __forceinline__ float gate_combine(float y, float g, bool add) { return add ? y + g : y * g; }

}  // namespace gsdpa

namespace gsdpa {

// Gate statistics ("GatedAttention [2025]", sec. 1.4.2: the mean gating score,
// the distribution of the scores, the fraction below a threshold), as
// integers so that the result does not depend on the order of the additions:
//   stats[0] number of scores, stats[1] sum of round(score * 2^32),
//   stats[2] number of scores < threshold, stats[3 + k] scores in bin k of
//   n_bins equal bins over [0, 1] (bin min(floor(score * n_bins), n_bins - 1)).

__device__ __forceinline__ int gate_bin(float s, int n_bins) {
    int k = __float2int_rd(s * (float)n_bins);
    return k < 0 ? 0 : (k >= n_bins ? n_bins - 1 : k);
}

__device__ __forceinline__ unsigned long long gate_fixed(float s) {
    return (unsigned long long)__float2ull_rn(s * 4294967296.0f);
}

// Adds the scores s of the lanes with `valid` set (every lane of the warp
// calls this, converged): the warp's totals in one atomic each, its
// histogram with one atomic per distinct bin.
__device__ __forceinline__ void gate_stats_warp(const GateStats& st, float s, bool valid) {
    const unsigned m = __ballot_sync(0xffffffffu, valid);
    if (m == 0) return;
    unsigned long long fx = valid ? gate_fixed(s) : 0ull;
    unsigned below = (valid && s < st.threshold) ? 1u : 0u;
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) {
        fx += __shfl_xor_sync(0xffffffffu, fx, sh);
        below += __shfl_xor_sync(0xffffffffu, below, sh);
    }
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        atomicAdd(st.out, (unsigned long long)__popc(m));
        atomicAdd(st.out + 1, fx);
        if (below) atomicAdd(st.out + 2, (unsigned long long)below);
    }
    const int bin = valid ? gate_bin(s, st.n_bins) : -1;
    const unsigned same = __match_any_sync(0xffffffffu, bin);
    if (valid && lane == __ffs(same) - 1) atomicAdd(st.out + 3 + bin, (unsigned long long)__popc(same));
}

}  // namespace gsdpa
