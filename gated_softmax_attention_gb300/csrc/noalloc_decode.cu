// noalloc_decode.cu -- the decode call for callers that cannot allocate
// device memory.
//
// Some callers of this library run where a device allocation is not allowed:
// code that must never make the device synchronise (cudaMalloc and cudaFree
// can), plugin or callback hooks that hand out no allocator, or processes
// whose device memory budget is fixed before they start. For them this file
// provides gated_sdpa_decode_noalloc(), which needs no workspace argument: the
// split-K scratch of the decode path lives in one file-scope device array that
// every GPU loading the library holds until the process exits.
//
// The array is shared by every call on a device and keeps the previous call's
// contents; the arrival counters that must start at zero are cleared at the
// start of every call. Calls that overlap on the device (two streams, or two
// threads) race on the array and must be serialised by the caller.
#include "gsdpa.h"
#include "gsdpa_internal.h"

#include <mutex>

namespace gsdpa {
namespace {

constexpr size_t kScratchBytes = 16u << 20;   // 16 MiB per device
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

char* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Host code must not use g_decode_scratch directly (that name is a host-side
// stand-in): resolve the device address once per device, with it current.
// The address is kept for the life of the process; a device or primary-context
// reset would leave it stale (the header says no call may follow one).
char* scratch_for_current_device(int* status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *status = GSDPA_ERR_LAUNCH;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) {
            *status = GSDPA_ERR_LAUNCH;
            return nullptr;
        }
        g_scratch_addr[dev] = static_cast<char*>(ptr);
    }
    return g_scratch_addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace gsdpa

using namespace gsdpa;

extern "C" GSDPA_API size_t gsdpa_decode_noalloc_max_scratch(void) { return kScratchBytes; }

extern "C" GSDPA_API int gated_sdpa_decode_noalloc(const void* X, const void* Q, const void* K, const void* V,
                                                   const void* W_g, void* O, float* sink, int B, int L_k,
                                                   int d_model, int H_q, int H_kv, int d_k, int gate_mode,
                                                   void* stream) {
    Problem p{};
    p.X = X;
    p.Q = Q;
    p.K = K;
    p.V = V;
    p.Wg = W_g;
    p.O = O;
    p.sink = sink;
    p.B = B;
    p.Lq = 1;
    p.Lk = L_k;
    p.d_model = d_model;
    p.Hq = H_q;
    p.Hkv = H_kv;
    p.dk = d_k;
    p.gate_mode = gate_mode;
    p.causal = 1;
    p.dtype = GSDPA_BF16;
    if (B < 0 || L_k < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0) return GSDPA_ERR_INVALID_ARG;
    if (gate_mode < GSDPA_GATE_NONE || gate_mode > GSDPA_GATE_ELEMENTWISE_AVERAGED) return GSDPA_ERR_INVALID_ARG;
    // (the head-shared, input-independent and averaged gates are valid modes of
    // gated_sdpa_fwd_variant that this entry point does not cover)
    if (gate_mode > GSDPA_GATE_ELEMENTWISE) return GSDPA_ERR_UNSUPPORTED;
    if (gate_mode != GSDPA_GATE_NONE && (d_model < 1 || !X || !W_g)) return GSDPA_ERR_INVALID_ARG;
    if (B == 0) return GSDPA_OK;
    if (!Q || !K || !V || !O) return GSDPA_ERR_INVALID_ARG;
    // this entry point covers the dedicated decode kernel only
    if (!decode_supported(p)) return GSDPA_ERR_UNSUPPORTED;
    if (gate_mode != GSDPA_GATE_NONE && d_model % 8 != 0) return GSDPA_ERR_UNSUPPORTED;
    if (gate_mode == GSDPA_GATE_HEADWISE && H_q % 8 != 0) return GSDPA_ERR_UNSUPPORTED;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return GSDPA_ERR_ALIGNMENT;
    if (gate_mode != GSDPA_GATE_NONE && (!aligned16(X) || !aligned16(W_g))) return GSDPA_ERR_ALIGNMENT;
    if (sink && (reinterpret_cast<uintptr_t>(sink) & 3u)) return GSDPA_ERR_ALIGNMENT;

    const WorkspacePlan w = plan_workspace(p, plan_sms());
    if (w.total > kScratchBytes) return GSDPA_ERR_WORKSPACE;   // problem too large for the fixed scratch

    Runtime rt;
    int ccM = 0, ccm = 0;
    if (!current_runtime(&rt, &ccM, &ccm)) return GSDPA_ERR_LAUNCH;
    if (!(ccM == 10 && ccm == 3) || !encode_tiled_fn()) return GSDPA_ERR_UNSUPPORTED;
    int st = GSDPA_OK;
    char* ws = scratch_for_current_device(&st);
    if (!ws) return st;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool gate_launched = false;
    ZeroJob zero;   // the split counters, zeroed by the gate kernel when there is one
    zero.p = reinterpret_cast<int*>(ws + w.dec_cnt);
    zero.n = (int)(w.dec_cnt_bytes / sizeof(int));
    cudaError_t e = launch_gate_logits_bf16(p, w, ws, rt, s, &gate_launched, zero);
    if (e == cudaSuccess) e = launch_decode_bf16(p, w, ws, rt, s, gate_launched);
    if (e == cudaErrorInvalidValue) return GSDPA_ERR_INVALID_ARG;
    return e == cudaSuccess ? GSDPA_OK : GSDPA_ERR_LAUNCH;
}
