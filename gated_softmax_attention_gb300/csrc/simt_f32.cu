// simt_f32.cu -- float32 gated attention on the CUDA cores (FFMA).
//
// The float32 path exists for exact-precision callers: tf32 tensor cores
// cannot meet a 1e-4 max-abs error, so every product here is an fp32 FFMA.
// It covers every gate mode, GQA, causal or not, prefill and decode.
//
// Computes O = softmax(Q K^T / sqrt(d_k) + causal) V (.) sigmoid(X W_g)
// ("GatedAttention [2025]", sec. 1.2.1 and 1.2.2; "10 . 门控", sec. 3.2)
// with an online (running max / running sum) softmax over key tiles, and the
// gate variants of gated_sdpa_fwd_variant (shared and input-independent gate
// shapes, NS-sigmoid, additive gates, SiLU of the output, per-head RMSNorm;
// sec. 1.2.2 items (3)-(5), 1.4.1, 1.4.2).
//
// Block: 32 query rows of one (b, h); 4 threads per row, thread part p owns
// the head dimensions c = p + 4 t (interleaved so that the 4 threads of a row
// read 4 consecutive floats). Keys stream through shared memory 32 at a time.
#include "gsdpa_internal.h"
#include "gate_fn.cuh"

#include <cmath>

namespace gsdpa {
namespace {

constexpr int kRows = 32;      // query rows per block
constexpr int kParts = 4;      // threads per row
constexpr int kKeys = 32;      // keys per shared-memory tile
constexpr int kThreads = kRows * kParts;

template <int DK>
__global__ void __launch_bounds__(kThreads)
gated_attn_f32_kernel(const float* __restrict__ X, const float* __restrict__ Q, const float* __restrict__ K,
                      const float* __restrict__ V, const float* __restrict__ Wg, float* __restrict__ O,
                      float* __restrict__ sink_part, int B, int Lq, int Lk, int d_model, int Hq, int Hkv,
                      int gate_mode, int causal, int gate_fn, float eps, GateStats gs) {
    constexpr int DPT = DK / kParts;  // dims per thread
    __shared__ float sK[kKeys][DK];
    __shared__ float sV[kKeys][DK];
    __shared__ float sRed[kRows];

    const int tid = threadIdx.x;
    const int r = tid / kParts;
    const int part = tid % kParts;
    const int q0 = blockIdx.x * kRows;
    const int h = blockIdx.y;
    const int b = blockIdx.z;
    const int kvh = h / (Hq / Hkv);
    const int i = q0 + r;
    const bool row_valid = i < Lq;
    const int ic = row_valid ? i : (Lq - 1);  // clamp for loads; results of invalid rows are dropped
    const long off = (long)Lk - Lq;
    const long a = off + ic;                  // absolute position (bottom-right causal)
    const float scale = 1.0f / sqrtf((float)DK);

    float q[DPT], o[DPT], g[DPT];
    const float* qp = Q + (((long)b * Lq + ic) * Hq + h) * DK;
#pragma unroll
    for (int t = 0; t < DPT; ++t) {
        q[t] = qp[part + kParts * t] * scale;
        o[t] = 0.f;
        g[t] = 1.f;
    }

    // ---- the gate's logits for this row's columns (gsdpa_gate_mode): X W_g over
    // the columns the gate shape gives, or theta for the input-independent gate
    float gl[DPT];
#pragma unroll
    for (int t = 0; t < DPT; ++t) gl[t] = 0.f;
    const float* xp = X ? X + ((long)b * Lq + ic) * d_model : nullptr;
    if (gate_mode == 2 || gate_mode == 4) {
        // elementwise (W_g [d_model, H_q*DK], columns h*DK + c) or shared by the heads ([d_model, DK])
        const long cols = gate_mode == 2 ? (long)Hq * DK : DK;
        const long c0 = gate_mode == 2 ? (long)h * DK : 0;
        for (int m = 0; m < d_model; ++m) {
            const float xv = xp[m];
            const float* wrow = Wg + (long)m * cols + c0 + part;
#pragma unroll
            for (int t = 0; t < DPT; ++t) gl[t] = fmaf(xv, wrow[kParts * t], gl[t]);
        }
    } else if (gate_mode == 1 || gate_mode == 3) {
        // headwise (W_g [d_model, H_q], column h) or shared by the heads ([d_model, 1])
        const long cols = gate_mode == 1 ? Hq : 1;
        const long c0 = gate_mode == 1 ? h : 0;
        float acc = 0.f;
        for (int m = part; m < d_model; m += kParts) acc = fmaf(xp[m], Wg[(long)m * cols + c0], acc);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
#pragma unroll
        for (int t = 0; t < DPT; ++t) gl[t] = acc;
    } else if (gate_mode == 5) {
        // input-independent: theta [H_q, DK]
#pragma unroll
        for (int t = 0; t < DPT; ++t) gl[t] = Wg[(long)h * DK + part + kParts * t];
    }
    // the gate's value: sigma, NS-sigmoid, sigma, SiLU or identity of the logit
    auto value = [&](float x) {
        const float sg = 1.f / (1.f + expf(-x));
        return gate_fn == 1 ? 0.5f + 0.5f * sg : (gate_fn == 3 ? x * sg : (gate_fn == 4 ? x : sg));
    };
    if (gate_mode == 6 || gate_mode == 7) {
        // averaged over the heads: every head's value of its own logit (headwise
        // W_g [d_model, H_q] or elementwise [d_model, H_q*DK]), then their mean
        float acc[DPT];
#pragma unroll
        for (int t = 0; t < DPT; ++t) acc[t] = 0.f;
        for (int hh = 0; hh < Hq; ++hh) {
            if (gate_mode == 7) {
                float glh[DPT];
#pragma unroll
                for (int t = 0; t < DPT; ++t) glh[t] = 0.f;
                for (int m = 0; m < d_model; ++m) {
                    const float xv = xp[m];
                    const float* wrow = Wg + (long)m * Hq * DK + (long)hh * DK + part;
#pragma unroll
                    for (int t = 0; t < DPT; ++t) glh[t] = fmaf(xv, wrow[kParts * t], glh[t]);
                }
#pragma unroll
                for (int t = 0; t < DPT; ++t) acc[t] += value(glh[t]);
            } else {
                float a1 = 0.f;
                for (int m = part; m < d_model; m += kParts) a1 = fmaf(xp[m], Wg[(long)m * Hq + hh], a1);
                a1 += __shfl_xor_sync(0xffffffffu, a1, 1);
                a1 += __shfl_xor_sync(0xffffffffu, a1, 2);
                const float v = value(a1);
#pragma unroll
                for (int t = 0; t < DPT; ++t) acc[t] += v;
            }
        }
#pragma unroll
        for (int t = 0; t < DPT; ++t) g[t] = acc[t] / (float)Hq;
    } else {
#pragma unroll
        for (int t = 0; t < DPT; ++t) g[t] = value(gl[t]);
    }
    const bool gated = gate_mode != 0;
    const bool add = gate_fn >= 2 && gate_fn <= 4;
    if (gs.out) {
        // gate statistics: each score once (headwise: one per row, from part 0)
        const bool per_col = gate_mode == 2;
#pragma unroll
        for (int t = 0; t < DPT; ++t) gate_stats_warp(gs, g[t], row_valid && (per_col || (part == 0 && t == 0)));
    }

    // ---- online softmax over keys
    long key_end = Lk;
    if (causal) {
        const long last_row = (q0 + kRows - 1 < Lq) ? (q0 + kRows - 1) : (Lq - 1);
        key_end = off + last_row + 1;
        if (key_end > Lk) key_end = Lk;
    }
    float m_run = -INFINITY, l_run = 0.f, s0 = 0.f;
    const long row_limit = causal ? a : (long)Lk - 1;  // last visible key of this row

    for (long k0 = 0; k0 < key_end; k0 += kKeys) {
        __syncthreads();
        for (int e = tid; e < kKeys * DK / 4; e += kThreads) {
            const int kr = (e * 4) / DK;
            const int kc = (e * 4) % DK;
            const long key = k0 + kr;
            float4 kv4 = make_float4(0.f, 0.f, 0.f, 0.f), vv4 = kv4;
            if (key < Lk) {
                const long base = (((long)b * Lk + key) * Hkv + kvh) * DK + kc;
                kv4 = *reinterpret_cast<const float4*>(K + base);
                vv4 = *reinterpret_cast<const float4*>(V + base);
            }
            *reinterpret_cast<float4*>(&sK[kr][kc]) = kv4;
            *reinterpret_cast<float4*>(&sV[kr][kc]) = vv4;
        }
        __syncthreads();
        const int nk = (key_end - k0 < kKeys) ? (int)(key_end - k0) : kKeys;
        for (int j = 0; j < nk; ++j) {
            float s = 0.f;
#pragma unroll
            for (int t = 0; t < DPT; ++t) s = fmaf(q[t], sK[j][part + kParts * t], s);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            const long key = k0 + j;
            if (key == 0) s0 = s;
            if (key <= row_limit) {
                const float m_new = fmaxf(m_run, s);
                const float alpha = expf(m_run - m_new);
                const float pj = expf(s - m_new);
                l_run = l_run * alpha + pj;
#pragma unroll
                for (int t = 0; t < DPT; ++t) o[t] = fmaf(pj, sV[j][part + kParts * t], o[t] * alpha);
                m_run = m_new;
            }
        }
    }

    const float inv_l = 1.f / l_run;
    float y[DPT];
#pragma unroll
    for (int t = 0; t < DPT; ++t) {
        y[t] = o[t] * inv_l;
        if (gated) y[t] = add ? y[t] + g[t] : y[t] * g[t];
        else if (gate_fn == 5) y[t] = y[t] / (1.f + expf(-y[t]));   // SiLU of the output
    }
    if (gate_fn == 6) {
        // per-head RMSNorm: the row's mean square over its DK columns (4 threads), gamma or 1
        float ss = 0.f;
#pragma unroll
        for (int t = 0; t < DPT; ++t) ss = fmaf(y[t], y[t], ss);
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        const float rr = 1.f / sqrtf(ss / DK + eps);
#pragma unroll
        for (int t = 0; t < DPT; ++t) y[t] *= rr * (Wg ? Wg[(long)h * DK + part + kParts * t] : 1.f);
    }
    if (row_valid) {
        float* op = O + (((long)b * Lq + i) * Hq + h) * DK;
#pragma unroll
        for (int t = 0; t < DPT; ++t) op[part + kParts * t] = y[t];
    }
    if (sink_part) {
        if (part == 0) sRed[r] = row_valid ? expf(s0 - m_run) * inv_l : 0.f;
        __syncthreads();
        if (tid < 32) {
            float v = sRed[tid];
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) v += __shfl_xor_sync(0xffffffffu, v, sh);
            if (tid == 0) sink_part[((long)b * Hq + h) * gridDim.x + blockIdx.x] = v;
        }
    }
}

}  // namespace

cudaError_t launch_f32_simt(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime&, cudaStream_t s) {
    dim3 grid((p.Lq + kRows - 1) / kRows, p.Hq, p.B);
    float* sink_part = p.sink ? reinterpret_cast<float*>(ws + w.sink_part) : nullptr;
    const float* X = static_cast<const float*>(p.X);
    const float* Wg = static_cast<const float*>(p.Wg);
    if (p.dk == 64) {
        gated_attn_f32_kernel<64><<<grid, kThreads, 0, s>>>(
            X, static_cast<const float*>(p.Q), static_cast<const float*>(p.K), static_cast<const float*>(p.V), Wg,
            static_cast<float*>(p.O), sink_part, p.B, p.Lq, p.Lk, p.d_model, p.Hq, p.Hkv, p.gate_mode, p.causal,
            p.gate_fn, p.eps, p.stats);
    } else {
        gated_attn_f32_kernel<128><<<grid, kThreads, 0, s>>>(
            X, static_cast<const float*>(p.Q), static_cast<const float*>(p.K), static_cast<const float*>(p.V), Wg,
            static_cast<float*>(p.O), sink_part, p.B, p.Lq, p.Lk, p.d_model, p.Hq, p.Hkv, p.gate_mode, p.causal,
            p.gate_fn, p.eps, p.stats);
    }
    return cudaGetLastError();
}

}  // namespace gsdpa
