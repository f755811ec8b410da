// gsdpa_api.cu -- the C ABI of libgsdpa.so (declared in include/gsdpa.h):
// argument validation, workspace planning, dispatch to the kernels, and the
// device error word that bounded waits report into.
#include "gsdpa.h"
#include "gsdpa_internal.h"
#include "proj_internal.h"
#include "sm103_ptx.cuh"

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

namespace gsdpa {

// Set by a kernel's bounded wait when it runs out; read and cleared by
// gsdpa_check_device_error().
__device__ uint32_t g_error_word;

namespace {

constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;  // 2 s
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};

// Split-K factors are planned for a fixed SM count so that the workspace size
// is a pure function of the problem (152 SMs on GB300; a little headroom).
constexpr int kPlanSms = 160;

struct DeviceInfo {
    bool ready = false;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    uint32_t* err = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

const DeviceInfo* device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
        if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return nullptr;
        if (cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return nullptr;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
        d.err = static_cast<uint32_t*>(p);
        d.ready = true;
    }
    return &d;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side checks shared by gsdpa_workspace_bytes and gated_sdpa_fwd.
int validate_shape(const Problem& p) {
    if (p.B < 0 || p.Lq < 0 || p.Lk < 1 || p.Lq > p.Lk) return GSDPA_ERR_INVALID_ARG;
    if (p.Hq < 1 || p.Hkv < 1 || p.Hq % p.Hkv != 0) return GSDPA_ERR_INVALID_ARG;
    if (p.gate_mode < GSDPA_GATE_NONE || p.gate_mode > GSDPA_GATE_ELEMENTWISE_AVERAGED) return GSDPA_ERR_INVALID_ARG;
    if (p.gate_fn < GSDPA_FN_SIGMOID_MUL || p.gate_fn > GSDPA_FN_RMSNORM) return GSDPA_ERR_INVALID_ARG;
    // the functions of the output alone take no gate; a gate takes one of the five functions of its logit
    if (p.gate_mode == GSDPA_GATE_NONE && p.gate_fn != GSDPA_FN_SIGMOID_MUL && p.gate_fn < GSDPA_FN_SILU_SELF)
        return GSDPA_ERR_INVALID_ARG;
    if (p.gate_mode != GSDPA_GATE_NONE && p.gate_fn >= GSDPA_FN_SILU_SELF) return GSDPA_ERR_INVALID_ARG;
    if (p.gate_fn == GSDPA_FN_RMSNORM && !(p.eps >= 0.f)) return GSDPA_ERR_INVALID_ARG;
    if (p.dtype != GSDPA_F32 && p.dtype != GSDPA_BF16) return GSDPA_ERR_INVALID_ARG;
    if (gate_cols(p) > 0 && p.d_model < 1) return GSDPA_ERR_INVALID_ARG;
    if (p.dk != 64 && p.dk != 128) return GSDPA_ERR_UNSUPPORTED;
    if (p.dtype == GSDPA_BF16) {
        // TMA needs every row stride to be a multiple of 16 bytes.
        if (gate_cols(p) > 0 && p.d_model % 8 != 0) return GSDPA_ERR_UNSUPPORTED;
        if (p.gate_mode == GSDPA_GATE_HEADWISE && p.Hq % 8 != 0) return GSDPA_ERR_UNSUPPORTED;
    }
    const long long units = (long long)((p.Lq + 127) / 128) * p.Hq * p.B;
    if (units > 0x7fffffffLL) return GSDPA_ERR_UNSUPPORTED;
    return GSDPA_OK;
}

}  // namespace

int gate_col_tile(int cols);  // gate_gemm_sm103.cu

// Runtime facts of the current device (SM count, compute capability, the
// device address of the error word) for entry points defined in other files.
bool current_runtime(Runtime* rt, int* cc_major, int* cc_minor) {
    const DeviceInfo* d = device_info();
    if (!d) return false;
    rt->err = d->err;
    rt->limit_ns = g_wait_limit_ns.load();
    rt->num_sms = d->num_sms;
    *cc_major = d->cc_major;
    *cc_minor = d->cc_minor;
    return true;
}

int plan_sms() { return kPlanSms; }

WorkspacePlan plan_workspace(const Problem& p, int num_sms) {
    WorkspacePlan w;
    size_t off = 0;
    const bool bf16 = p.dtype == GSDPA_BF16;
    const bool decode = decode_supported(p);
    if (p.sink && !decode && !bf16) {
        w.sink_tiles = (p.Lq + 31) / 32;
        w.sink_part = off;
        off = align256(off + sizeof(float) * (size_t)p.B * p.Hq * w.sink_tiles);
    }
    // Gate logits computed ahead of the attention kernel: bf16 headwise (and
    // head-shared headwise) prefill and every bf16 decode gate that reads X
    // (the elementwise prefill gates are computed ahead as values, below).
    const bool gate_prepass = bf16 && gate_cols(p) > 0 && (decode || gate_headwise_family(p));
    if (gate_prepass) {
        w.gate_rows = p.B * p.Lq;
        w.gate_cols = gate_cols(p);
        // Prefill: no split (one CTA per 128 rows reads its rows of X once). The
        // attention kernel starts on the SMs these few CTAs leave free and reads
        // the logits only in its epilogues, so a long pre-pass on few SMs costs
        // less than a short one on all of them (measured on GQA 32/4 L4096:
        // 120.0 -> 113.8 us per call). Decode: the rows are few, and the
        // splits spread the W_g read over the SMs.
        int splits = 1;   // (head-shared headwise: one row-dot kernel, no split)
        if (p.gate_mode != GSDPA_GATE_HEADWISE_SHARED && decode) {
            const int nt = gate_col_tile(w.gate_cols);
            const int tiles = ((w.gate_rows + 127) / 128) * ((w.gate_cols + nt - 1) / nt);
            const int nkc = (p.d_model + 63) / 64;
            splits = (num_sms + tiles - 1) / tiles;
            int max_splits = nkc / 4 > 0 ? nkc / 4 : 1;
            if (splits > max_splits) splits = max_splits;
            if (splits < 1) splits = 1;
        }
        w.gate_splits = splits;
        w.gate_part = off;
        off = align256(off + sizeof(float) * (size_t)splits * w.gate_rows * w.gate_cols);
    }
    // bf16 prefill: the counter from which the CTAs of the attention kernel
    // claim their units (dynamic schedule) and, with the first-token share, one
    // 64-bit word per (b, h) in which the warps add their rows' shares; zeroed
    // at the start of every call.
    if (bf16 && !decode) {
        w.state = off;
        w.state_ints = 2 + (p.sink ? 2 * p.B * p.Hq : 0);
        off = align256(off + sizeof(int) * (size_t)w.state_ints);
    }
    // Elementwise bf16 prefill (and its head-shared and input-independent
    // forms): the gate's values computed ahead of the attention kernel, whose
    // epilogue applies them -- [B*L_q, gate columns], or [H_q * d_k] for the
    // input-independent gate.
    if (bf16 && !decode && gate_elementwise_family(p)) {
        w.has_gate_sig = true;
        w.gate_sig = off;
        const size_t n = p.gate_mode == GSDPA_GATE_STATIC ? (size_t)p.Hq * p.dk
                                                          : (size_t)p.B * p.Lq * gate_cols(p);
        off = align256(off + 2 * n);
    }
    if (decode) {
        const int chunks = (p.Hq / p.Hkv) / 4;
        w.dec_splits = decode_splits(p, num_sms);
        w.dec_heads_per_cta = 4;
        w.dec_ml = off;
        off = align256(off + sizeof(float) * 2 * (size_t)p.B * p.Hq * w.dec_splits);
        w.dec_o = off;
        off = align256(off + sizeof(float) * (size_t)p.B * p.Hq * w.dec_splits * p.dk);
        w.dec_x0 = off;
        off = align256(off + sizeof(float) * (size_t)p.B * p.Hq);
        w.dec_cnt = off;
        w.dec_cnt_bytes = sizeof(int) * (size_t)p.B * p.Hkv * chunks;
        off = align256(off + w.dec_cnt_bytes);
    }
    w.total = off;
    return w;
}

static std::once_flag g_encode_once;
static EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_tiled_fn() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

// sink[b,h] = (1 / L_q) * sum over query tiles of the per-tile sums of p(i -> key 0).
// Zeroes the call's statistics counters as a programmatic dependent of the
// kernel before it on the stream (a memset node there would end the overlap of
// consecutive calls' kernels). Its own dependent, the call's first gate kernel,
// may start its prologue at once: that kernel waits for this one to complete
// before it touches global memory, and every statistics update of the call
// comes after that wait, or after a wait on a kernel that made it.
__global__ void stats_zero_kernel(unsigned long long* __restrict__ out, int n) {
    pdl_trigger();
    pdl_wait();
    for (int k = threadIdx.x; k < n; k += blockDim.x) out[k] = 0;
}

// Zeroes the attention kernel's per-call state when no gate kernel runs first
// in the call (the gate kernels do it otherwise). A programmatic dependent of
// the kernel before it on the stream, which may be the previous call's
// attention kernel still using this state: it waits for that kernel to
// complete, zeroes, and only then lets its own dependent, the attention
// kernel, start (whose set-up thus overlaps this launch instead of following
// a memset node).
__global__ void state_zero_kernel(int* __restrict__ p, int n) {
    pdl_wait();
    for (int k = threadIdx.x; k < n; k += blockDim.x) p[k] = 0;
    __threadfence();
    __syncthreads();
    pdl_trigger();
}

__global__ void sink_finalize_kernel(const float* __restrict__ part, float* __restrict__ sink, int n, int tiles,
                                     float inv_lq) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n) return;
    float s = 0.f;
    for (int t = 0; t < tiles; ++t) s += part[(long)idx * tiles + t];
    sink[idx] = s * inv_lq;
}

// One thread waits on an mbarrier that nothing arrives on: the bounded wait
// gives up after the current limit and records ERR_WAIT_TIMEOUT.
__global__ void wait_self_test_kernel(WaitCtl ctl) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        mbar_fence_init();
        mbar_wait(&bar, 0, &abort_flag, ctl);
    }
}

void set_sink_args(const Problem& p, const WorkspacePlan& w, char* ws, int n_qtiles, unsigned long long** word,
                   float** sink, float* scale, double* inv, int* arrivals) {
    int lg = 0;
    while ((1L << lg) < (long)p.Lq + 1) ++lg;   // ceil(log2(L_q + 1))
    const int F = 43 - lg;
    *word = p.sink ? reinterpret_cast<unsigned long long*>(ws + w.state + 8) : nullptr;
    *sink = p.sink;
    *scale = std::ldexp(1.0f, F);
    *inv = std::ldexp(1.0, -F) / (double)p.Lq;
    *arrivals = 4 * n_qtiles;
}

cudaError_t launch_sink_finalize(const Problem& p, const WorkspacePlan& w, char* ws, cudaStream_t s) {
    const int n = p.B * p.Hq;
    sink_finalize_kernel<<<(n + 127) / 128, 128, 0, s>>>(reinterpret_cast<const float*>(ws + w.sink_part), p.sink, n,
                                                         w.sink_tiles, 1.0f / (float)p.Lq);
    return cudaGetLastError();
}

}  // namespace gsdpa

using namespace gsdpa;

extern "C" {

size_t gsdpa_workspace_bytes(int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k, int gate_mode,
                             int want_sink, int dtype) {
    Problem p{};
    p.B = B;
    p.Lq = L_q;
    p.Lk = L_k;
    p.d_model = d_model;
    p.Hq = H_q;
    p.Hkv = H_kv;
    p.dk = d_k;
    p.gate_mode = gate_mode;
    p.dtype = dtype;
    p.sink = want_sink ? reinterpret_cast<float*>(16) : nullptr;
    if (gate_mode > GSDPA_GATE_ELEMENTWISE || validate_shape(p) != GSDPA_OK) return (size_t)-1;
    if (B == 0 || L_q == 0) return 0;
    return plan_workspace(p, kPlanSms).total;
}

size_t gsdpa_bwd_workspace_bytes(int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k, int gate_mode) {
    Problem p{};
    p.B = B;
    p.Lq = L_q;
    p.Lk = L_k;
    p.d_model = d_model;
    p.Hq = H_q;
    p.Hkv = H_kv;
    p.dk = d_k;
    p.gate_mode = gate_mode;
    p.dtype = GSDPA_BF16;
    p.causal = 1;
    if (validate_shape(p) != GSDPA_OK || !bwd_supported(p)) return (size_t)-1;
    if (B == 0 || L_q == 0) return 0;
    return plan_bwd(p, kPlanSms).total;
}

namespace {
int bwd_impl(const void* X, const void* Q, const void* K, const void* V, const void* W_g, const void* O, const void* dO,
             const float* lse, const void* gate_saved, void* dX, void* dQ, void* dK, void* dV, void* dW_g, int B,
             int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k, int gate_mode, int causal, int dtype,
             void* workspace, size_t workspace_bytes, void* stream) {
    Problem p{};
    p.X = X;
    p.Q = Q;
    p.K = K;
    p.V = V;
    p.Wg = W_g;
    p.B = B;
    p.Lq = L_q;
    p.Lk = L_k;
    p.d_model = d_model;
    p.Hq = H_q;
    p.Hkv = H_kv;
    p.dk = d_k;
    p.gate_mode = gate_mode;
    p.causal = causal ? 1 : 0;
    p.dtype = dtype;
    int st = validate_shape(p);
    if (st != GSDPA_OK) return st;
    if (B == 0 || L_q == 0) return GSDPA_OK;
    if (!bwd_supported(p)) return GSDPA_ERR_UNSUPPORTED;
    const bool gated = gate_mode != GSDPA_GATE_NONE;
    if (!Q || !K || !V || !O || !dO || !lse || !dQ || !dK || !dV) return GSDPA_ERR_INVALID_ARG;
    if (gated && (!X || !W_g || !dX || !dW_g)) return GSDPA_ERR_INVALID_ARG;
    for (const void* t : {Q, K, V, O, dO, static_cast<const void*>(dQ), static_cast<const void*>(dK),
                          static_cast<const void*>(dV)})
        if (!aligned16(t)) return GSDPA_ERR_ALIGNMENT;
    if (gated && (!aligned16(X) || !aligned16(W_g) || !aligned16(dX) || !aligned16(dW_g))) return GSDPA_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(lse) & 3u) return GSDPA_ERR_ALIGNMENT;

    const DeviceInfo* dev = device_info();
    if (!dev) return GSDPA_ERR_LAUNCH;
    if (!(dev->cc_major == 10 && dev->cc_minor == 3) || !encode_tiled_fn()) return GSDPA_ERR_UNSUPPORTED;
    const BwdPlan w = plan_bwd(p, kPlanSms);
    if (!workspace || workspace_bytes < w.total) return GSDPA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return GSDPA_ERR_ALIGNMENT;
    Runtime rt;
    rt.err = dev->err;
    rt.limit_ns = g_wait_limit_ns.load();
    rt.num_sms = dev->num_sms;
    BwdArgs g;
    g.O = O;
    g.dO = dO;
    g.lse = lse;
    g.dX = dX;
    g.dQ = dQ;
    g.dK = dK;
    g.dV = dV;
    g.dWg = dW_g;
    const cudaError_t e = launch_bwd_bf16_saved(p, g, gate_saved, w, static_cast<char*>(workspace), rt,
                                                static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidValue) return GSDPA_ERR_INVALID_ARG;
    return e == cudaSuccess ? GSDPA_OK : GSDPA_ERR_LAUNCH;
}
}  // namespace

int gated_sdpa_bwd(const void* X, const void* Q, const void* K, const void* V, const void* W_g, const void* O,
                   const void* dO, const float* lse, void* dX, void* dQ, void* dK, void* dV, void* dW_g, int B,
                   int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k, int gate_mode, int causal, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream) {
    return bwd_impl(X, Q, K, V, W_g, O, dO, lse, nullptr, dX, dQ, dK, dV, dW_g, B, L_q, L_k, d_model, H_q, H_kv, d_k,
                    gate_mode, causal, dtype, workspace, workspace_bytes, stream);
}

int gated_sdpa_bwd_saved_gate(const void* X, const void* Q, const void* K, const void* V, const void* W_g,
                              const void* O, const void* dO, const float* lse, const void* gate_saved, void* dX,
                              void* dQ, void* dK, void* dV, void* dW_g, int B, int L_q, int L_k, int d_model, int H_q,
                              int H_kv, int d_k, int gate_mode, int causal, int dtype, void* workspace,
                              size_t workspace_bytes, void* stream) {
    if (gate_mode != GSDPA_GATE_ELEMENTWISE || !gate_saved) return GSDPA_ERR_INVALID_ARG;
    if (!aligned16(gate_saved)) return GSDPA_ERR_ALIGNMENT;
    return bwd_impl(X, Q, K, V, W_g, O, dO, lse, gate_saved, dX, dQ, dK, dV, dW_g, B, L_q, L_k, d_model, H_q, H_kv,
                    d_k, gate_mode, causal, dtype, workspace, workspace_bytes, stream);
}

namespace {
int fwd_impl(const void* X, const void* Q, const void* K, const void* V, const void* W_g, void* O, float* sink,
             float* lse, int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k, int gate_mode, int causal,
             int dtype, void* workspace, size_t workspace_bytes, void* stream, int gate_fn = 0, float eps = 0.f,
             GateStats stats = GateStats()) {
    Problem p{};
    p.gate_fn = gate_fn;
    p.eps = eps;
    p.stats = stats;
    p.lse = lse;
    p.X = X;
    p.Q = Q;
    p.K = K;
    p.V = V;
    p.Wg = W_g;
    p.O = O;
    p.sink = sink;
    p.B = B;
    p.Lq = L_q;
    p.Lk = L_k;
    p.d_model = d_model;
    p.Hq = H_q;
    p.Hkv = H_kv;
    p.dk = d_k;
    p.gate_mode = gate_mode;
    p.causal = causal ? 1 : 0;
    p.dtype = dtype;
    int st = validate_shape(p);
    if (st != GSDPA_OK) return st;
    if (B == 0 || L_q == 0) return GSDPA_OK;
    if (!Q || !K || !V || !O) return GSDPA_ERR_INVALID_ARG;
    const bool reads_x = gate_cols(p) > 0;
    if (reads_x && !X) return GSDPA_ERR_INVALID_ARG;
    if (gate_mode != GSDPA_GATE_NONE && !W_g) return GSDPA_ERR_INVALID_ARG;   // (RMSNorm: gamma may be NULL)
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return GSDPA_ERR_ALIGNMENT;
    if ((reads_x && !aligned16(X)) || (W_g && !aligned16(W_g))) return GSDPA_ERR_ALIGNMENT;
    if (sink && (reinterpret_cast<uintptr_t>(sink) & 3u)) return GSDPA_ERR_ALIGNMENT;
    if (sink && dtype == GSDPA_BF16 && !decode_supported(p) && (long)L_q > kSinkMaxLq) return GSDPA_ERR_UNSUPPORTED;
    // (the averaged gates are built for the prefill kernels and the float32 path)
    if (gate_averaged(p) && dtype == GSDPA_BF16 && decode_supported(p)) return GSDPA_ERR_UNSUPPORTED;

    const DeviceInfo* dev = device_info();
    if (!dev) return GSDPA_ERR_LAUNCH;
    if (dtype == GSDPA_BF16 && !(dev->cc_major == 10 && dev->cc_minor == 3)) return GSDPA_ERR_UNSUPPORTED;
    if (dtype == GSDPA_BF16 && !encode_tiled_fn()) return GSDPA_ERR_UNSUPPORTED;

    const WorkspacePlan w = plan_workspace(p, kPlanSms);
    if (w.total > 0) {
        if (!workspace || workspace_bytes < w.total) return GSDPA_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return GSDPA_ERR_ALIGNMENT;
    }
    char* ws = static_cast<char*>(workspace);
    Runtime rt;
    rt.err = dev->err;
    rt.limit_ns = g_wait_limit_ns.load();
    rt.num_sms = dev->num_sms;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    cudaError_t e = cudaSuccess;
    if (stats.out) {
        // (bf16: the call starts with a gate kernel that waits before touching memory;
        // the float32 kernel is an ordinary launch)
        const int n = 3 + stats.n_bins;
        e = dtype == GSDPA_F32 ? cudaMemsetAsync(stats.out, 0, sizeof(unsigned long long) * (size_t)n, s)
                               : launch_dependent(stats_zero_kernel, dim3(1), dim3(64), 0, s, stats.out, n);
    }
    if (e != cudaSuccess) return GSDPA_ERR_LAUNCH;
    if (dtype == GSDPA_F32) {
        e = launch_f32_simt(p, w, ws, rt, s);
        if (e == cudaSuccess && sink) e = launch_sink_finalize(p, w, ws, s);
    } else {
        // The per-call state of the attention kernel (the prefill kernel's unit
        // counter and share words, the decode kernel's split counters) is zeroed
        // by the gate kernel that runs first, before it lets the attention kernel
        // start; without a gate kernel, by state_zero_kernel in the same way.
        const bool decode = decode_supported(p);
        ZeroJob zero;
        if (decode) {
            zero.p = reinterpret_cast<int*>(ws + w.dec_cnt);
            zero.n = (int)(w.dec_cnt_bytes / sizeof(int));
        } else if (w.state_ints > 0) {
            zero.p = reinterpret_cast<int*>(ws + w.state);
            zero.n = w.state_ints;
        }
        bool gate_launched = false;
        if (w.has_gate_sig) {
            e = launch_gate_sigmoid_bf16(p, w, ws, rt, s, zero);
            gate_launched = true;
            zero.n = 0;
        }
        bool logits_launched = false;
        if (e == cudaSuccess) e = launch_gate_logits_bf16(p, w, ws, rt, s, &logits_launched, zero);
        if (logits_launched) {
            gate_launched = true;
            zero.n = 0;
        }
        // averaged gates: the heads' values averaged in place before the attention reads them
        if (e == cudaSuccess && gate_averaged(p)) e = launch_gate_average_bf16(p, w, ws, s);
        if (decode) {
            if (e == cudaSuccess) e = launch_decode_bf16(p, w, ws, rt, s, gate_launched);
        } else {
            if (e == cudaSuccess && zero.n > 0)
                e = launch_dependent(state_zero_kernel, dim3(1), dim3(256), 0, s, zero.p, zero.n);
            // (the prefill kernel also finishes the first-token share)
            if (e == cudaSuccess) e = launch_prefill_bf16(p, w, ws, rt, s);
        }
    }
    if (e == cudaErrorInvalidValue) return GSDPA_ERR_INVALID_ARG;
    return e == cudaSuccess ? GSDPA_OK : GSDPA_ERR_LAUNCH;
}
}  // namespace

int gated_sdpa_fwd(const void* X, const void* Q, const void* K, const void* V, const void* W_g, void* O, float* sink,
                   int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k, int gate_mode, int causal,
                   int dtype, void* workspace, size_t workspace_bytes, void* stream) {
    // (the other gate shapes go through gated_sdpa_fwd_variant)
    if (gate_mode < GSDPA_GATE_NONE || gate_mode > GSDPA_GATE_ELEMENTWISE) return GSDPA_ERR_INVALID_ARG;
    return fwd_impl(X, Q, K, V, W_g, O, sink, nullptr, B, L_q, L_k, d_model, H_q, H_kv, d_k, gate_mode, causal, dtype,
                    workspace, workspace_bytes, stream);
}

size_t gsdpa_workspace_bytes_variant(int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k,
                                     int gate_mode, int gate_fn, int want_sink, int dtype) {
    Problem p{};
    p.B = B;
    p.Lq = L_q;
    p.Lk = L_k;
    p.d_model = d_model;
    p.Hq = H_q;
    p.Hkv = H_kv;
    p.dk = d_k;
    p.gate_mode = gate_mode;
    p.gate_fn = gate_fn;
    p.dtype = dtype;
    p.sink = want_sink ? reinterpret_cast<float*>(16) : nullptr;
    if (validate_shape(p) != GSDPA_OK) return (size_t)-1;
    if (B == 0 || L_q == 0) return 0;
    return plan_workspace(p, kPlanSms).total;
}

int gated_sdpa_fwd_variant(const void* X, const void* Q, const void* K, const void* V, const void* W_g, void* O,
                           float* sink, int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k,
                           int gate_mode, int gate_fn, float eps, int causal, int dtype, void* workspace,
                           size_t workspace_bytes, void* stream) {
    return fwd_impl(X, Q, K, V, W_g, O, sink, nullptr, B, L_q, L_k, d_model, H_q, H_kv, d_k, gate_mode, causal, dtype,
                    workspace, workspace_bytes, stream, gate_fn, eps);
}

}  // extern "C"

namespace gsdpa {
namespace {
// The layer's problem and workspace: the attention's own plan, then Q, K, V
// and the attention output (bf16), each 256-byte aligned.
struct LayerPlan {
    Problem p{};
    WorkspacePlan w;
    size_t q = 0, k = 0, v = 0, o = 0, total = 0;
};
int plan_layer(int B, int L, int d_model, int H_q, int H_kv, int d_k, int gate_mode, int causal, LayerPlan* lp) {
    Problem& p = lp->p;
    p.B = B;
    p.Lq = L;
    p.Lk = L;
    p.d_model = d_model;
    p.Hq = H_q;
    p.Hkv = H_kv;
    p.dk = d_k;
    p.gate_mode = gate_mode;
    p.causal = causal ? 1 : 0;
    p.dtype = GSDPA_BF16;
    if (gate_mode < GSDPA_GATE_NONE || gate_mode > GSDPA_GATE_ELEMENTWISE) return GSDPA_ERR_INVALID_ARG;
    if (d_model < 1) return GSDPA_ERR_INVALID_ARG;
    const int st = validate_shape(p);
    if (st != GSDPA_OK) return st;
    if (d_k != 128 || d_model % 8 != 0 || d_model < 256 || (B > 0 && L < 2)) return GSDPA_ERR_UNSUPPORTED;
    // (headwise: W_in's rows hold (H_q + 2 H_kv) d_k + H_q elements, a multiple of 8 for the tensor maps)
    if (gate_mode == GSDPA_GATE_HEADWISE && H_q % 8 != 0) return GSDPA_ERR_UNSUPPORTED;
    lp->w = plan_workspace(p, kPlanSms);
    size_t off = lp->w.total;
    const size_t rows = (size_t)B * L;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align256(off + bytes);
        return at;
    };
    lp->q = take(rows * H_q * d_k * 2);
    lp->k = take(rows * H_kv * d_k * 2);
    lp->v = take(rows * H_kv * d_k * 2);
    lp->o = take(rows * H_q * d_k * 2);
    lp->total = off;
    return GSDPA_OK;
}
}  // namespace
}  // namespace gsdpa

extern "C" {

size_t gsdpa_layer_workspace_bytes(int B, int L, int d_model, int H_q, int H_kv, int d_k, int gate_mode) {
    LayerPlan lp;
    if (plan_layer(B, L, d_model, H_q, H_kv, d_k, gate_mode, 1, &lp) != GSDPA_OK) return (size_t)-1;
    if (B == 0 || L == 0) return 0;
    return lp.total;
}

int gated_attention_layer(const void* X, const void* W_in, const void* W_O, void* Y, int B, int L, int d_model,
                          int H_q, int H_kv, int d_k, int gate_mode, int causal, void* workspace,
                          size_t workspace_bytes, void* stream) {
    LayerPlan lp;
    const int st = plan_layer(B, L, d_model, H_q, H_kv, d_k, gate_mode, causal, &lp);
    if (st != GSDPA_OK) return st;
    if (B == 0 || L == 0) return GSDPA_OK;
    if (!X || !W_in || !W_O || !Y) return GSDPA_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W_in) || !aligned16(W_O) || !aligned16(Y)) return GSDPA_ERR_ALIGNMENT;
    const DeviceInfo* dev = device_info();
    if (!dev) return GSDPA_ERR_LAUNCH;
    if (!(dev->cc_major == 10 && dev->cc_minor == 3) || !encode_tiled_fn()) return GSDPA_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < lp.total) return GSDPA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return GSDPA_ERR_ALIGNMENT;
    char* ws = static_cast<char*>(workspace);
    Runtime rt;
    rt.err = dev->err;
    rt.limit_ns = g_wait_limit_ns.load();
    rt.num_sms = dev->num_sms;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Problem p = lp.p;
    p.X = X;
    p.Q = ws + lp.q;
    p.K = ws + lp.k;
    p.V = ws + lp.v;
    p.O = ws + lp.o;
    const bool gated = gate_mode == GSDPA_GATE_ELEMENTWISE;
    const int qkv_cols = (H_q + 2 * H_kv) * d_k;
    // 1. [Q | K | V | gate] = X W_in (zeroes the attention kernel's per-call state);
    // 2. the attention (its gate values already in place); 3. Y = O W_O.
    // Headwise gate: its H_q columns of W_in are not part of the projection;
    // the gate-logit pre-pass reads them (row length (H_q + 2 H_kv) d_k + H_q)
    // after the projection, and the attention kernel runs as its programmatic
    // dependent (it reads the logits only in its epilogues, after waiting for
    // the pre-pass, which itself started only once Q, K, V were written).
    ZeroJob zero;
    zero.p = reinterpret_cast<int*>(ws + lp.w.state);
    zero.n = lp.w.state_ints;
    const bool headwise = gate_mode == GSDPA_GATE_HEADWISE;
    cudaError_t e = launch_proj_qkvg_bf16(X, W_in, ws + lp.q, ws + lp.k, ws + lp.v, gated ? ws + lp.w.gate_sig : nullptr,
                                          B * L, d_model, H_q, H_kv, d_k, gated, zero, rt, s,
                                          headwise ? qkv_cols + H_q : 0);
    if (headwise) {
        p.Wg = static_cast<const char*>(W_in) + (size_t)qkv_cols * 2;
        p.wg_ld = qkv_cols + H_q;
        bool launched = false;
        if (e == cudaSuccess) e = launch_gate_logits_bf16(p, lp.w, ws, rt, s, &launched, ZeroJob());
        if (e == cudaSuccess) e = launch_prefill_bf16(p, lp.w, ws, rt, s);
    } else {
        // (an ordinary launch: the attention reads Q, K, V from its first step)
        if (e == cudaSuccess) e = launch_prefill_bf16_ordered(p, lp.w, ws, rt, s);
    }
    if (e == cudaSuccess) e = launch_gemm_pair_bf16_kn(ws + lp.o, W_O, Y, B * L, d_model, H_q * d_k, rt, s);
    if (e == cudaErrorInvalidValue) return GSDPA_ERR_INVALID_ARG;
    return e == cudaSuccess ? GSDPA_OK : GSDPA_ERR_LAUNCH;
}

int gated_sdpa_fwd_stats(const void* X, const void* Q, const void* K, const void* V, const void* W_g, void* O,
                         float* sink, unsigned long long* stats, int n_bins, float threshold, int B, int L_q, int L_k,
                         int d_model, int H_q, int H_kv, int d_k, int gate_mode, int causal, int dtype, void* workspace,
                         size_t workspace_bytes, void* stream) {
    if (gate_mode != GSDPA_GATE_HEADWISE && gate_mode != GSDPA_GATE_ELEMENTWISE) return GSDPA_ERR_INVALID_ARG;
    if (!stats || n_bins < 1 || n_bins > 64 || !(threshold >= 0.f && threshold <= 1.f)) return GSDPA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(stats) & 7u) return GSDPA_ERR_ALIGNMENT;
    GateStats st;
    st.out = stats;
    st.n_bins = n_bins;
    st.threshold = threshold;
    return fwd_impl(X, Q, K, V, W_g, O, sink, nullptr, B, L_q, L_k, d_model, H_q, H_kv, d_k, gate_mode, causal, dtype,
                    workspace, workspace_bytes, stream, 0, 0.f, st);
}

int gated_sdpa_fwd_train(const void* X, const void* Q, const void* K, const void* V, const void* W_g, void* O,
                         float* sink, float* lse, int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k,
                         int gate_mode, int causal, int dtype, void* workspace, size_t workspace_bytes,
                         void* stream) {
    if (!lse) return GSDPA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(lse) & 3u) return GSDPA_ERR_ALIGNMENT;
    if (dtype != GSDPA_BF16 || L_q == 1) return GSDPA_ERR_UNSUPPORTED;   // the bf16 prefill kernels write it
    if (gate_mode < GSDPA_GATE_NONE || gate_mode > GSDPA_GATE_ELEMENTWISE) return GSDPA_ERR_INVALID_ARG;
    return fwd_impl(X, Q, K, V, W_g, O, sink, lse, B, L_q, L_k, d_model, H_q, H_kv, d_k, gate_mode, causal, dtype,
                    workspace, workspace_bytes, stream);
}

int gated_sdpa_fwd_train_save_gate(const void* X, const void* Q, const void* K, const void* V, const void* W_g,
                                   void* O, float* sink, float* lse, void* gate_out, int B, int L_q, int L_k,
                                   int d_model, int H_q, int H_kv, int d_k, int gate_mode, int causal, int dtype,
                                   void* workspace, size_t workspace_bytes, void* stream) {
    if (gate_mode != GSDPA_GATE_ELEMENTWISE || !gate_out) return GSDPA_ERR_INVALID_ARG;
    if (!aligned16(gate_out)) return GSDPA_ERR_ALIGNMENT;
    const int st = gated_sdpa_fwd_train(X, Q, K, V, W_g, O, sink, lse, B, L_q, L_k, d_model, H_q, H_kv, d_k, gate_mode,
                                        causal, dtype, workspace, workspace_bytes, stream);
    if (st != GSDPA_OK || B == 0 || L_q == 0) return st;
    // the gate kernel's fp16 values, [B*L_q, H_q*d_k] at the start of their workspace region
    Problem p{};
    p.B = B;
    p.Lq = L_q;
    p.Lk = L_k;
    p.d_model = d_model;
    p.Hq = H_q;
    p.Hkv = H_kv;
    p.dk = d_k;
    p.gate_mode = gate_mode;
    p.causal = causal ? 1 : 0;
    p.dtype = dtype;
    p.sink = sink;
    const WorkspacePlan w = plan_workspace(p, kPlanSms);
    if (!w.has_gate_sig) return GSDPA_ERR_UNSUPPORTED;
    const size_t bytes = (size_t)B * L_q * H_q * d_k * sizeof(__half);
    const cudaError_t e = cudaMemcpyAsync(gate_out, static_cast<char*>(workspace) + w.gate_sig, bytes,
                                          cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GSDPA_OK : GSDPA_ERR_LAUNCH;
}

int gsdpa_check_device_error(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return GSDPA_ERR_LAUNCH;
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v)) != cudaSuccess) return GSDPA_ERR_LAUNCH;
    if (v != 0) {
        const uint32_t zero = 0;
        cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
        return GSDPA_ERR_DEVICE_TIMEOUT;
    }
    return GSDPA_OK;
}

const char* gsdpa_status_string(int status) {
    switch (status) {
        case GSDPA_OK: return "GSDPA_OK";
        case GSDPA_ERR_INVALID_ARG: return "GSDPA_ERR_INVALID_ARG";
        case GSDPA_ERR_UNSUPPORTED: return "GSDPA_ERR_UNSUPPORTED";
        case GSDPA_ERR_ALIGNMENT: return "GSDPA_ERR_ALIGNMENT";
        case GSDPA_ERR_WORKSPACE: return "GSDPA_ERR_WORKSPACE";
        case GSDPA_ERR_LAUNCH: return "GSDPA_ERR_LAUNCH";
        case GSDPA_ERR_DEVICE_TIMEOUT: return "GSDPA_ERR_DEVICE_TIMEOUT";
        default: return "GSDPA_ERR_UNKNOWN";
    }
}

int gsdpa_wait_self_test(void* stream) {
    const DeviceInfo* dev = device_info();
    if (!dev) return GSDPA_ERR_LAUNCH;
    WaitCtl ctl;
    ctl.err = dev->err;
    ctl.limit_ns = g_wait_limit_ns.load();
    wait_self_test_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(ctl);
    return cudaGetLastError() == cudaSuccess ? GSDPA_OK : GSDPA_ERR_LAUNCH;
}

int gsdpa_set_wait_limit_ns(unsigned long long ns) {
    g_wait_limit_ns.store(ns ? ns : kDefaultWaitLimitNs);
    return GSDPA_OK;
}

}  // extern "C"
