// gate_fn.cuh -- the gate functions of the attention epilogues and the gate
// passes: how a gate logit gl becomes the gate's value, and how that value
// acts on the SDPA output y ("GatedAttention [2025]", sec. 1.2.2 items (4),
// (5); sec. 1.4.2 (iv) for NS-sigmoid). Codes are gsdpa_gate_fn's.
#pragma once
#include <cstdint>

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
