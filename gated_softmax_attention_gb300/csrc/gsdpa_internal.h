// gsdpa_internal.h -- host-side launch interfaces shared by the .cu files of
// libgsdpa.so. Not part of the public ABI (include/gsdpa.h is).
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gsdpa {

// Gate statistics of a call (gated_sdpa_fwd_stats): the device array
// [3 + n_bins] of 64-bit counters, or null (not computed).
struct GateStats {
    unsigned long long* out = nullptr;
    int n_bins = 0;
    float threshold = 0.f;
};

struct Problem {
    const void* X;
    const void* Q;
    const void* K;
    const void* V;
    const void* Wg;
    void* O;
    float* sink;
    float* lse;      // [B, Hq, Lq] natural-log softmax denominators, or null
    int B, Lq, Lk, d_model, Hq, Hkv, dk;
    int gate_mode;   // 0 none, 1 headwise, 2 elementwise, 3 headwise shared, 4 elementwise shared, 5 static
    int causal;
    int dtype;       // 0 f32, 1 bf16
    int gate_fn = 0; // gsdpa_gate_fn
    int wg_ld = 0;   // W_g row length in elements (0: its own width; the layer's W_g is a column block of W_in)
    float eps = 0.f; // RMSNorm
    GateStats stats; // gate statistics, or none
};

struct Runtime {
    uint32_t* err;                 // device error word
    unsigned long long limit_ns;   // bounded-wait limit
    int num_sms;
};

// Workspace carve-up (byte offsets, all 256-aligned) for one problem.
struct WorkspacePlan {
    size_t total = 0;
    size_t sink_part = 0;   // float [B, Hq, n_tiles]          (sink partial sums)
    int sink_tiles = 0;
    size_t gate_part = 0;   // float [gate_splits, rows, cols] (gate logits, split-K partials)
    size_t gate_sig = 0;    // fp16  [B*L_q, H_q*d_k]          (elementwise prefill: sigma(X W_g))
    bool has_gate_sig = false;
    // bf16 prefill, per-call state (zero at the start of every call): int [0]
    // the next unit to claim; from byte 8, with the first-token share, one
    // 64-bit word per (b, h): the share in fixed point and its arrivals
    size_t state = 0;
    int state_ints = 0;
    int gate_splits = 0;
    int gate_rows = 0, gate_cols = 0;
    size_t dec_ml = 0;      // float [B, Hq, splits, 2]        (decode running max, sum)
    size_t dec_o = 0;       // float [B, Hq, splits, dk]       (decode partial outputs)
    size_t dec_x0 = 0;      // float [B, Hq]                   (decode: scaled score of key 0)
    size_t dec_cnt = 0;     // int   [B, Hkv * head_chunks]     (decode arrival counters)
    int dec_splits = 0;
    int dec_heads_per_cta = 0;
    size_t dec_cnt_bytes = 0;
};

WorkspacePlan plan_workspace(const Problem& p, int num_sms);
// columns of W_g: H_q * d_k (elementwise), H_q (headwise), 1 (headwise
// shared), d_k (elementwise shared), 0 (no gate; the static gate's theta
// [H_q, d_k] is not multiplied by X)
inline int gate_cols(const Problem& p) {
    switch (p.gate_mode) {
    case 1: case 6: return p.Hq;
    case 2: case 7: return p.Hq * p.dk;
    case 3: return 1;
    case 4: return p.dk;
    default: return 0;
    }
}
// Gate families of the bf16 kernels: one value per (row, head) from logits
// summed in the attention epilogue (headwise, headwise shared, headwise
// averaged), or one value per (row, head, column) computed ahead as fp16
// (elementwise, elementwise shared, static, elementwise averaged).
inline bool gate_headwise_family(const Problem& p) { return p.gate_mode == 1 || p.gate_mode == 3 || p.gate_mode == 6; }
inline bool gate_elementwise_family(const Problem& p) {
    return p.gate_mode == 2 || p.gate_mode == 4 || p.gate_mode == 5 || p.gate_mode == 7;
}
// The gate values of every head averaged over the heads (gate modes 6, 7): a
// pass after the gate kernel leaves the average where head 0's value was.
inline bool gate_averaged(const Problem& p) { return p.gate_mode == 6 || p.gate_mode == 7; }
// The attention kernels' view of the gate: the GATE template parameter
// (0 none, 1 headwise family, 2 elementwise family, 3 SiLU of the output,
// 4 per-head RMSNorm) and the runtime fields.
struct GateEpi {
    int fn = 0;            // gsdpa_gate_fn
    int g_rs = 0, g_hs = 0;   // elementwise family: value at row * g_rs + h * g_hs + c
    int l_cols = 0, l_hs = 0; // headwise family: logit partials at (split * rows + row) * l_cols + h * l_hs
    const void* gamma = nullptr;   // RMSNorm scale [H_q, d_k] (bf16) or null
    float eps = 0.f;
};
inline int gate_template(const Problem& p) {
    if (gate_headwise_family(p)) return 1;
    if (gate_elementwise_family(p)) return 2;
    return p.gate_fn == 5 ? 3 : (p.gate_fn == 6 ? 4 : 0);
}
inline GateEpi gate_epi(const Problem& p) {
    GateEpi g;
    g.fn = p.gate_fn;
    switch (p.gate_mode) {
    case 2: g.g_rs = p.Hq * p.dk; g.g_hs = p.dk; break;
    case 4: g.g_rs = p.dk; g.g_hs = 0; break;
    case 5: g.g_rs = 0; g.g_hs = p.dk; break;
    case 1: g.l_cols = p.Hq; g.l_hs = 1; break;
    case 3: g.l_cols = 1; g.l_hs = 0; break;
    // averaged: every head reads column 0 of its row, where the averaging pass
    // left the average of the heads' values (the headwise one as a value, so
    // the epilogue's function is the identity; multiplied or added as before)
    case 6: g.l_cols = p.Hq; g.l_hs = 0; g.fn = 4; break;
    case 7: g.g_rs = p.Hq * p.dk; g.g_hs = 0; break;
    default: break;
    }
    if (p.gate_fn == 6) g.gamma = p.Wg;
    g.eps = p.eps;
    return g;
}

// The dedicated decode kernel covers bf16, L_q == 1, d_k == 128 and query
// groups of a multiple of 4 heads; other decode shapes use the prefill kernel.
bool decode_supported(const Problem& p);
int decode_splits(const Problem& p, int num_sms);

// Current-device runtime facts (gsdpa_api.cu); the SM count workspace plans use.
bool current_runtime(Runtime* rt, int* cc_major, int* cc_minor);
int plan_sms();

// Driver entry point for tensor-map encoding (resolved once, no -lcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// Gate modes 6, 7: average the gate values of every head over the heads, in
// place (the average where head 0's value was), after the gate kernel and
// before the attention kernel, as a programmatic dependent between them
// (gate_sigmoid_sm103.cu).
cudaError_t launch_gate_average_bf16(const Problem& p, const WorkspacePlan& w, char* ws, cudaStream_t s);

// Launchers: return cudaSuccess or the launch error. `ws` is the workspace base.
cudaError_t launch_f32_simt(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                            cudaStream_t s);
// A kernel that runs first in a call and zeroes `n` ints at `p` (its CTA 0,
// before it lets the dependent kernel start); n = 0: nothing to zero.
struct ZeroJob {
    int* p = nullptr;
    int n = 0;
};
cudaError_t launch_gate_logits_bf16(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                    cudaStream_t s, bool* launched, ZeroJob zero = ZeroJob());
// Elementwise bf16 prefill: sigma(X W_g) as fp16 into the workspace (gate_sigmoid_sm103.cu).
cudaError_t launch_gate_sigmoid_bf16(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                     cudaStream_t s, ZeroJob zero);
cudaError_t launch_prefill_bf16(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                cudaStream_t s);
// d_k = 128 on CTA pairs (prefill_pair_sm103.cu); launch_prefill_bf16 routes
// problems with at least kPairMinKeys keys there.
constexpr long kPairMinKeys = 16384;
cudaError_t launch_prefill_pair_bf16(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                     cudaStream_t s);
// dependent: the gate-logit kernel just before it has zeroed the split
// counters and this launch is its programmatic dependent (the decode kernel
// waits for it only where it reads the logits); otherwise the counters are
// zeroed here and the launch is an ordinary one.
cudaError_t launch_decode_bf16(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                               cudaStream_t s, bool dependent);
cudaError_t launch_sink_finalize(const Problem& p, const WorkspacePlan& w, char* ws, cudaStream_t s);

// ---- backward (bwd_sm103.cu): bf16, d_k = 128
struct BwdArgs {
    const void* O;       // the training forward's output
    const void* dO;      // dL/dO
    const float* lse;    // [B, Hq, Lq] from the training forward
    void* dX;            // gate path's share, like X (gated only)
    void* dQ;
    void* dK;
    void* dV;
    void* dWg;           // like W_g (gated only)
};
struct BwdPlan {
    size_t total = 0;
    WorkspacePlan fwd;   // the gate recompute's buffers (the forward's plan)
    int Lq_pad = 0;      // rows of the per-(b, h) arrays, a multiple of 128
    size_t dY = 0;       // bf16 [B, Lq, Hq, 128]
    size_t Dv = 0;       // float [B, Hq, Lq_pad]
    size_t lse2 = 0;     // float [B, Hq, Lq_pad]
    size_t dGl = 0;      // bf16 [B*Lq, G]
    size_t part_dK = 0;  // GQA: float [B, Lk, Hq, 128], each query head's share
    size_t part_dV = 0;
    int dx_splits = 1, dwg_splits = 1;   // K splits of the gate-gradient GEMMs on the single-CTA kernel
    size_t gemm_part = 0;                // float [splits, M, N] partials of the split GEMM
};
bool bwd_supported(const Problem& p);
BwdPlan plan_bwd(const Problem& p, int num_sms);
cudaError_t launch_bwd_bf16(const Problem& p, const BwdArgs& g, const BwdPlan& w, char* ws, const Runtime& rt,
                            cudaStream_t s);
// C [M x N] (bf16, row-major) = A B on CTA pairs (bwd_gemm_sm103.cu), for N >= 256.
// ab_mn: A stored [K][M] and B stored [K][N]; else A stored [M][K] and B^T
// stored [N][K]. Every row stride a multiple of 16 bytes, every base 16-byte aligned.
cudaError_t launch_gemm_pair_bf16(const void* A, const void* Bm, void* C, int M, int N, int K, bool ab_mn,
                                  const Runtime& rt, cudaStream_t s);
// bf16 prefill kernels: where the first-token share accumulates (null without
// it), its fixed-point scale 2^F with F = 43 - ceil(log2(L_q + 1)), the factor
// 2^-F / L_q back to the mean, and the arrivals of a full set (4 per query tile).
constexpr long kSinkMaxLq = 1L << 24;   // keeps 4 x tiles below 2^20 (the count field)
void set_sink_args(const Problem& p, const WorkspacePlan& w, char* ws, int n_qtiles, unsigned long long** word,
                   float** sink, float* scale, double* inv, int* arrivals);

// Launch `kernel` as a programmatic dependent of the previous kernel on the
// stream: it may be scheduled once every CTA of that kernel has signalled
// (griddepcontrol.launch_dependents) or exited, and must itself wait
// (griddepcontrol.wait) before it relies on that kernel's memory.
// Devices one process can drive (indexes of the per-device tables).
constexpr int kMaxDevices = 64;

// One-time set-up of a kernel on each device: function attributes (dynamic
// shared memory size) and occupancy queries belong to one device's context,
// and one process may launch on several devices. `fn(int& value)` runs once
// per device under a mutex (so concurrent first calls from several host
// threads run it once) and may leave a result in `value` (e.g. the number of
// resident CTA pairs); later calls on that device return at once with the
// stored value. A failed set-up is retried on the next call.
struct PerDeviceSetup {
    std::mutex mu;
    std::atomic<bool> done[kMaxDevices] = {};
    int value[kMaxDevices] = {};
};
template <typename F>
cudaError_t setup_once_per_device(PerDeviceSetup& st, F&& fn, int* value = nullptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!st.done[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(st.mu);
        if (!st.done[dev].load(std::memory_order_relaxed)) {
            e = fn(st.value[dev]);
            if (e != cudaSuccess) return e;
            st.done[dev].store(true, std::memory_order_release);
        }
    }
    if (value) *value = st.value[dev];
    return cudaSuccess;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace gsdpa
