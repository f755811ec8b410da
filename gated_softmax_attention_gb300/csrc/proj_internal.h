// proj_internal.h -- host-side launch interfaces of the layer's neighbouring
// GEMMs (input projection, output projection). Not part of the public ABI.
#pragma once
#include "gsdpa_internal.h"

namespace gsdpa {

// X [rows, d_model] times W_in = [W_Q | W_K | W_V | W_g] [d_model, N] into Q
// [rows, H_q d_k], K and V [rows, H_kv d_k] (bf16) and, when gated, the
// elementwise gate sigma(X W_g) [rows, H_q d_k] (fp16): launch_pair_gemm_bf16
// with those four outputs. d_k a multiple of 128 (every output's width a
// multiple of 128 columns). W_in's
// rows hold w_ld elements (0: N; more when columns the kernel does not
// project follow, e.g. a headwise gate's). Runs first in a call: zeroes
// `zero`, then lets the next kernel start.
cudaError_t launch_proj_qkvg_bf16(const void* X, const void* W_in, void* Qo, void* Ko, void* Vo, void* Go, int rows,
                                  int d_model, int Hq, int Hkv, int dk, bool gated, ZeroJob zero, const Runtime& rt,
                                  cudaStream_t s, int w_ld = 0);

// One output of launch_pair_gemm_bf16: `cols` consecutive columns of the
// product, stored [rows, cols] at `ptr` as bf16, or, for the gate, as fp16
// values sigma(x).
struct GemmOut {
    void* ptr;
    int cols;
    bool gate;
};

// X [rows, d_model] (bf16) times W [d_model, N] (bf16, rows of w_ld elements)
// on CTA pairs, persistent over 256 x 256 tiles (proj_sm103.cu). The product's
// columns are the outputs `outs[0..n_outs)` side by side (at most four, at
// most one gate); every output but the last a multiple of 128 columns wide,
// the last a multiple of 64. Runs first in a call: zeroes `zero`, then lets
// the next kernel start.
cudaError_t launch_pair_gemm_bf16(const void* X, int rows, int d_model, const void* W, int w_ld, int N,
                                  const GemmOut* outs, int n_outs, ZeroJob zero, const Runtime& rt, cudaStream_t s);

// The bf16 prefill attention as an ordinary launch (not a programmatic
// dependent of the kernel before it): for callers whose previous kernel
// produces Q, K or V, which the attention kernel reads from its first step
// (prefill_sm103.cu, prefill_pair_sm103.cu). Sigmoid gate, none or elementwise.
cudaError_t launch_prefill_bf16_ordered(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                        cudaStream_t s);
cudaError_t launch_prefill_pair_bf16_ordered(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                             cudaStream_t s);

// C [M x N] (bf16) = A B on CTA pairs with A stored [M][K] and B stored [K][N]
// (bwd_gemm_sm103.cu), N >= 256: the output projection O W_O.
cudaError_t launch_gemm_pair_bf16_kn(const void* A, const void* Bm, void* C, int M, int N, int K, const Runtime& rt,
                                     cudaStream_t s);

// The backward pass with the elementwise gate's values sigma(X W_g) (fp16
// [B*L_q, H_q*d_k]) taken from `gate_saved`, where the training forward saved
// them, instead of recomputing them (bwd_sm103.cu); gate_saved NULL
// recomputes, as launch_bwd_bf16 does.
cudaError_t launch_bwd_bf16_saved(const Problem& p, const BwdArgs& g, const void* gate_saved, const BwdPlan& w,
                                  char* ws, const Runtime& rt, cudaStream_t s);

}  // namespace gsdpa
