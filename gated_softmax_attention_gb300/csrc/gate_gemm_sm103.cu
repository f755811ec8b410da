// gate_gemm_sm103.cu -- gate logits X W_g on sm_103a tensor cores.
//
// Computes the pre-sigmoid gate logits GL[r, c] = sum_m X[r, m] W_g[m, c]
// ("GatedAttention [2025]", sec. 1.2.2: the gate is sigma(X W_theta); no bias,
// "10 . 门控", sec. 3.2) for every row r of X viewed as [rows, d_model] and
// every column c of W_g [d_model, cols], as float32 split-K partials
// out[split, r, c]; the consumer (attention epilogue or decode combine) sums
// the splits and applies the sigmoid.
//
// Used where the gate cannot live inside the attention CTA without re-reading
// X once per head:
//   * headwise gate (cols = H_q): one 128-row tile computes the logits of
//     every head at once, so X is read from HBM once;
//   * decode (rows = batch): every column of W_g is read once for the whole
//     batch instead of once per batch row.
//
// CTA: 128 rows x NT columns (NT = 64 or 128) over one K-split. Warp 0 loads
// X [128 x 64] and W_g [64 x NT] chunks with TMA into a 4-stage ring, warp 1
// lane 0 issues tcgen05.mma (A = X, K-major; B = W_g, MN-major; both 128B
// swizzle) into a TMEM fp32 accumulator, warps 2..5 read it back and store.
// Rows past the end of X and columns past the end of W_g load as zeros (TMA
// out-of-bounds fill) and are not stored.
//
// The head-shared headwise gate (W_g [d_model, 1], one logit per row for
// every head) is a matrix-vector product whose single column cannot be a
// tensor-map operand (its rows are 2 bytes apart): gate_rowdot_kernel, one
// warp per row, 16-byte loads of X and W_g.
#include "gsdpa_internal.h"
#include "sm103_ptx.cuh"

namespace gsdpa {
namespace {

constexpr int kThreads = 192;
constexpr int NS = 4;

template <int NT>
struct GateCfg {
    static constexpr uint32_t X_BYTES = 128 * 64 * 2;
    static constexpr uint32_t W_BYTES = 64 * NT * 2;
    static constexpr uint32_t STAGE = X_BYTES + W_BYTES;
    static constexpr uint32_t OFF_BAR = NS * STAGE;
    static constexpr uint32_t OFF_MISC = OFF_BAR + (2 * NS + 2) * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
};

struct GateArgs {
    float* out;          // [splits, rows, cols]
    int rows, cols, d_model;
    int row_tiles, col_tiles, splits, nkc;
    ZeroJob zero;        // per-call state of the attention kernel, zeroed by CTA 0
    WaitCtl ctl;
};

template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
gate_logits_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const GateArgs args) {
    using C = GateCfg<NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* full = bars;
    uint64_t* empty = bars + NS;
    uint64_t* acc_full = bars + 2 * NS;
    uint64_t* drain = bars + 2 * NS + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int u = blockIdx.x;
    const int rt = u % args.row_tiles;
    const int ct = (u / args.row_tiles) % args.col_tiles;
    const int ks = u / (args.row_tiles * args.col_tiles);
    const int kc0 = (int)((long)ks * args.nkc / args.splits);
    const int kc1 = (int)((long)(ks + 1) * args.nkc / args.splits);
    const int r0 = rt * 128;
    const int c0 = ct * NT;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, NT);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // This kernel is a programmatic dependent of the previous kernel on the
    // stream, so the prologue above can overlap that kernel's tail. Nothing in
    // global memory is touched before it has completed: it may have produced
    // the inputs, or be the previous call's attention kernel, which still
    // reads this workspace.
    pdl_wait();
    if (blockIdx.x == 0 && args.zero.n > 0) {
        // the attention kernel's per-call state; visible before it can start
        for (int k = threadIdx.x; k < args.zero.n; k += blockDim.x) args.zero.p[k] = 0;
        __threadfence();
        __syncthreads();
    }
    pdl_trigger();   // the consumer (attention or decode) may start; it reads the logits late

    if (warp == 0) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            uint32_t armed_phase[NS];
            bool armed[NS];
            for (int s = 0; s < NS; ++s) armed[s] = false;
            bool ok = true;
            for (int kc = kc0; kc < kc1; ++kc) {
                if (!(ok = mbar_wait(&empty[stage], phase ^ 1u, abort_flag, args.ctl))) break;
                mbar_arrive_expect_tx(&full[stage], C::STAGE);
                armed[stage] = true;
                armed_phase[stage] = phase;
                uint8_t* st = smem + stage * C::STAGE;
                tma_load_2d(st, &tmX, kc * 64, r0, &full[stage]);
                for (int cb = 0; cb < NT / 64; ++cb)
                    tma_load_2d(st + C::X_BYTES + cb * 8192, &tmW, c0 + cb * 64, kc * 64, &full[stage]);
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                volatile int never = 0;
                for (int s = 0; s < NS; ++s)
                    if (armed[s]) mbar_wait(&full[s], armed_phase[s], &never, args.ctl);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            constexpr uint32_t idG = idesc_bf16_f32(128, NT, false, true);
            const uint32_t base = smem_u32(smem);
            for (int kc = kc0; kc < kc1; ++kc) {
                if (!(ok = mbar_wait(&full[stage], phase, abort_flag, args.ctl))) break;
                tc_fence_after();
                const uint32_t st = base + stage * C::STAGE;
                constexpr uint32_t HI = desc_sw128_hi(1024);
                const uint32_t x0 = desc_sw128_lo(st, 16), w0 = desc_sw128_lo(st + C::X_BYTES, 8192);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss_lohi(tmem, x0 + kk * (32 >> 4), HI, w0 + kk * (2048 >> 4), HI, idG,
                                (kc != kc0 || kk != 0) ? 1u : 0u);
                mma_commit(&empty[stage]);
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok) {
                mma_commit(acc_full);
            } else {
                volatile int never = 0;
                mma_commit(drain);
                mbar_wait(drain, 0, &never, args.ctl);
            }
        }
    } else {
        const int qd = warp & 3;
        const int row = qd * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        bool ok = (kc1 > kc0) ? __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, args.ctl)) : true;
        tc_fence_after();
        if (ok) {
            const int r = r0 + row;
            float* dst = args.out + ((long)ks * args.rows + r) * args.cols;
#pragma unroll
            for (int cb = 0; cb < NT / 32; ++cb) {
                uint32_t v[32];
                if (kc1 > kc0) {
                    tmem_ld32(tmem + lane_base + cb * 32, v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0u;
                }
                if (r < args.rows) {
                    const int cbase = c0 + cb * 32;
                    if (cbase + 32 <= args.cols) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4*>(dst + cbase + e) =
                                make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                                            __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
                    } else {
                        for (int e = 0; e < 32 && cbase + e < args.cols; ++e) dst[cbase + e] = __uint_as_float(v[e]);
                    }
                }
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, NT);
    }
}

// out[r] = sum_m X[r, m] w[m] (fp32), one warp per row; d_model a multiple of 8.
// Runs first in the call, like the gate GEMM (zeroes the attention kernel's
// per-call state, then lets it start).
__global__ void __launch_bounds__(256) gate_rowdot_kernel(const __nv_bfloat16* __restrict__ X,
                                                          const __nv_bfloat16* __restrict__ w, float* __restrict__ out,
                                                          int rows, int d_model, ZeroJob zero) {
    pdl_wait();
    if (blockIdx.x == 0 && zero.n > 0) {
        for (int k = threadIdx.x; k < zero.n; k += blockDim.x) zero.p[k] = 0;
        __threadfence();
        __syncthreads();
    }
    pdl_trigger();
    const long r = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const __nv_bfloat16* x = X + r * d_model;
    float acc = 0.f;
    for (int m = lane * 8; m < d_model; m += 32 * 8) {
        const uint4 xv = *reinterpret_cast<const uint4*>(x + m);
        const uint4 wv = *reinterpret_cast<const uint4*>(w + m);
        const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            acc = fmaf(__uint_as_float(xa[q] << 16), __uint_as_float(wa[q] << 16), acc);
            acc = fmaf(__uint_as_float(xa[q] & 0xffff0000u), __uint_as_float(wa[q] & 0xffff0000u), acc);
        }
    }
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
    if (lane == 0) out[r] = acc;
}

bool make_map2d(CUtensorMap* m, const void* base, cuuint64_t d0, cuuint64_t d1, cuuint64_t stride1_bytes,
                cuuint32_t b0, cuuint32_t b1) {
    cuuint64_t d[2] = {d0, d1};
    cuuint64_t st[1] = {stride1_bytes};
    cuuint32_t box[2] = {b0, b1};
    cuuint32_t es[2] = {1, 1};
    return encode_tiled_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), d, st, box, es,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NT>
cudaError_t launch_gate_t(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt, cudaStream_t s,
                          ZeroJob zero) {
    using C = GateCfg<NT>;
    alignas(64) CUtensorMap tmX, tmW;
    const int rows = w.gate_rows, cols = w.gate_cols;
    if (!make_map2d(&tmX, p.X, (cuuint64_t)p.d_model, (cuuint64_t)rows, (cuuint64_t)p.d_model * 2, 64, 128))
        return cudaErrorInvalidValue;
    const cuuint64_t ld = (cuuint64_t)(p.wg_ld > 0 ? p.wg_ld : cols);
    if (!make_map2d(&tmW, p.Wg, (cuuint64_t)cols, (cuuint64_t)p.d_model, ld * 2, 64, 64))
        return cudaErrorInvalidValue;
    GateArgs a;
    a.out = reinterpret_cast<float*>(ws + w.gate_part);
    a.rows = rows;
    a.cols = cols;
    a.d_model = p.d_model;
    a.row_tiles = (rows + 127) / 128;
    a.col_tiles = (cols + NT - 1) / NT;
    a.splits = w.gate_splits;
    a.nkc = (p.d_model + 63) / 64;
    a.zero = zero;
    a.ctl.err = rt.err;
    a.ctl.limit_ns = rt.limit_ns;
    static PerDeviceSetup setup;   // per template instance
    cudaError_t r = setup_once_per_device(setup, [](int&) {
        return cudaFuncSetAttribute(gate_logits_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)C::SMEM_BYTES);
    });
    if (r != cudaSuccess) return r;
    const unsigned grid = (unsigned)(a.row_tiles * a.col_tiles * a.splits);
    return launch_dependent(gate_logits_kernel<NT>, dim3(grid), dim3(kThreads), C::SMEM_BYTES, s, tmX, tmW, a);
}

}  // namespace

// Gate-logit column tile: 128 when the gate is wide (elementwise), 64 for the
// narrow headwise gate (H_q columns, zero-padded by TMA up to 64).
int gate_col_tile(int cols) { return cols > 64 ? 128 : 64; }

cudaError_t launch_gate_logits_bf16(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                    cudaStream_t s, bool* launched, ZeroJob zero) {
    *launched = false;
    if (w.gate_splits == 0) return cudaSuccess;
    *launched = true;
    if (p.gate_mode == 3) {   // head-shared headwise: one split of [rows, 1]
        const unsigned blocks = (unsigned)((w.gate_rows + 7) / 8);
        return launch_dependent(gate_rowdot_kernel, dim3(blocks), dim3(256), 0, s,
                                static_cast<const __nv_bfloat16*>(p.X), static_cast<const __nv_bfloat16*>(p.Wg),
                                reinterpret_cast<float*>(ws + w.gate_part), w.gate_rows, p.d_model, zero);
    }
    if (gate_col_tile(w.gate_cols) == 128) return launch_gate_t<128>(p, w, ws, rt, s, zero);
    return launch_gate_t<64>(p, w, ws, rt, s, zero);
}

}  // namespace gsdpa
