// proj_sm103.cu -- the layer's input projection as one GEMM on pairs of SMs:
// X [rows, d_model] times [W_Q | W_K | W_V | W_g] [d_model, N], writing
//   Q [rows, H_q d_k], K and V [rows, H_kv d_k] as bf16 (no activation) and
//   the elementwise gate sigma(X W_g) [rows, H_q d_k] as fp16
// ("GatedAttention [2025]", sec. 1.2.1: Q, K, V are projections of the same
// hidden state X; sec. 1.2.2: the gate sigma(X W_theta) reads X too, so the
// four products share every load of X). The attention kernel then reads Q, K,
// V and the gate values as it reads them from a caller.
//
// Same CTA-pair GEMM as the gate GEMM (gate_sigmoid_sm103.cu): a pair computes
// a 256 x 512 tile in the whole of tensor memory, per K chunk of 64 each CTA
// loading its 128 rows of X and 256 columns of W (MN-major). The epilogue
// converts 32 columns at a time; every 128-column group lies in one of the four
// outputs (their widths are multiples of 128), so a group is staged as bf16 or
// as fp16 sigma, and stored by TMA into its output at the group's column
// within it. Rows past the end of X, columns past N and the K tail load as
// zeros and are not stored.
#include "gsdpa_internal.h"
#include "proj_internal.h"
#include "sm103_pair.cuh"
#include "sm103_ptx.cuh"

#include <cuda_fp16.h>

namespace gsdpa {
namespace {

constexpr int kThreads = 320;
constexpr int kNS = 4;
constexpr uint32_t kXBytes = 128 * 64 * 2;
constexpr uint32_t kWBytes = 64 * 256 * 2;
constexpr uint32_t kStage = kXBytes + kWBytes;
constexpr uint32_t kOffBar = kNS * kStage;
constexpr uint32_t kOffMisc = kOffBar + (2 * kNS + 2 + 4) * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;

struct ProjArgs {
    int rows, N, d_model;
    int seg_end[4];       // cumulative column ends of Q, K, V, gate (the gate's equals V's without one)
    int row_tiles, nkc;
    ZeroJob zero;         // per-call state of the attention kernel, zeroed by CTA 0
    WaitCtl ctl;
};

// sigma of two values as fp16 (1/2 + tanh(x/2)/2, tanh.approx.f16x2: about 2^-11 relative)
__device__ __forceinline__ uint32_t sigmoid2_h(float x0, float x1) {
    const __half2 hx = __floats2half2_rn(0.5f * x0, 0.5f * x1);
    uint32_t t;
    asm("tanh.approx.f16x2 %0, %1;" : "=r"(t) : "r"(*reinterpret_cast<const uint32_t*>(&hx)));
    const __half2 half2v = __floats2half2_rn(0.5f, 0.5f);
    const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&t), half2v, half2v);
    return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ int segment_of(const ProjArgs& a, int col) {
    return col < a.seg_end[0] ? 0 : (col < a.seg_end[1] ? 1 : (col < a.seg_end[2] ? 2 : 3));
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
proj_qkvg_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                 const ProjArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* full = bars;
    uint64_t* empty = bars + kNS;
    uint64_t* acc_full = bars + 2 * kNS;
    uint64_t* drain = bars + 2 * kNS + 1;
    uint64_t* grp_ready = bars + 2 * kNS + 2;   // [4]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    int* abort_word = reinterpret_cast<int*>(smem + kOffMisc + 4);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = pair::cta_rank();
    const pair::PairAbort ab{abort_word, pair::map_to(abort_word, rank ^ 1u)};
    const int tile = (int)pair::cluster_id();
    const int r0 = (tile % args.row_tiles) * 256;
    const int c0 = (tile / args.row_tiles) * 512;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        for (int g = 0; g < 4; ++g) mbar_init(&grp_ready[g], 4);
        *abort_word = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        pair::tmem_alloc(tmem_slot, 512);
        tc_fence_before();
    }
    __syncthreads();
    pair::cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // a programmatic dependent of the previous kernel on the stream: nothing in
    // global memory is touched before it has completed
    pdl_wait();
    if (blockIdx.x == 0 && args.zero.n > 0) {
        for (int k = threadIdx.x; k < args.zero.n; k += blockDim.x) args.zero.p[k] = 0;
        __threadfence();
        __syncthreads();
    }
    pdl_trigger();   // the attention kernel may start; it reads Q, K, V only after this grid completes

    if (warp == 0) {
        if (lane == 0) {
            for (int kc = 0; kc < args.nkc; ++kc) {
                const int s = kc % kNS;
                const uint32_t ph = (kc / kNS) & 1;
                if (!pair::wait(&empty[s], ph ^ 1u, ab, args.ctl)) break;
                if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * kStage);
                const uint32_t fb = pair::map_to(&full[s], 0);
                uint8_t* st = smem + s * kStage;
                pair::tma_load_2d(st, &tmX, kc * 64, r0 + (int)rank * 128, fb);
                pair::tma_load_3d(st + kXBytes, &tmW, 0, kc * 64, (c0 + (int)rank * 256) / 64, fb);
            }
            // stores: each 128-column group into its output as soon as its 4 warps are done
            bool ok = true;
            for (int g = 0; g < 4 && ok; ++g) {
                if (!(ok = pair::wait(&grp_ready[g], 0, ab, args.ctl))) break;
                const int gc = c0 + 128 * g;
                if (gc >= args.N) continue;
                const int sg = segment_of(args, gc);
                const int col = gc - (sg ? args.seg_end[sg - 1] : 0);
                const CUtensorMap* m = sg == 0 ? &tmQ : (sg == 1 ? &tmK : (sg == 2 ? &tmV : &tmG));
                const int row = r0 + (int)rank * 128;
                tma_store_2d(m, smem + g * 32768, col, row);
                tma_store_2d(m, smem + g * 32768 + 16384, col + 64, row);
                tma_store_commit();
            }
            tma_store_wait_all();
        }
    } else if (warp == 1) {
        if (rank == 0) {
            constexpr uint32_t idG = idesc_bf16_f32(256, 256, false, true);
            constexpr uint32_t HI = desc_sw128_hi(1024);
            const uint32_t base = smem_u32(smem);
            bool ok = true;
            for (int kc = 0; kc < args.nkc && ok; ++kc) {
                const int s = kc % kNS;
                if (!(ok = __all_sync(0xffffffffu, pair::wait(&full[s], (kc / kNS) & 1, ab, args.ctl)))) break;
                tc_fence_after();
                const uint32_t st = base + s * kStage;
                const uint32_t x0 = desc_sw128_lo(st, 16), w0 = desc_sw128_lo(st + kXBytes, 8192);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
                        pair::mma_ss(tmem + hh * 256, x0 + kk * (32 >> 4), HI, w0 + ((hh * 16384 + kk * 2048) >> 4), HI,
                                     idG, (kc | kk) != 0);
                pair::commit_both(&empty[s]);
            }
            if (ok) {
                pair::commit_both(acc_full);
            } else {
                WaitCtl c2 = args.ctl;
                if (c2.limit_ns < 1000000000ull) c2.limit_ns = 1000000000ull;
                int never = 0;
                const pair::PairAbort quiet{&never, ab.peer};
                asm volatile(
                    "{\n\t.reg .pred e;\n\t"
                    "elect.sync _|e, 0xffffffff;\n\t"
                    "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
                        smem_u32(drain))
                    : "memory");
                pair::wait(drain, 0, quiet, c2);
                __syncwarp();
            }
        }
    } else {
        // ---- epilogue: 32 columns at a time, bf16 (Q, K, V) or fp16 sigma (gate)
        const int qd = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = qd * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const bool ok = __all_sync(0xffffffffu, pair::wait(acc_full, 0, ab, args.ctl));
        tc_fence_after();
        if (ok) {
            uint32_t buf[2][32];
            tmem_ld32(tmem + lane_base + half * 256, buf[0]);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                tmem_wait_ld_regs(buf[k & 1]);
                if (k + 1 < 8) tmem_ld32(tmem + lane_base + half * 256 + (k + 1) * 32, buf[(k + 1) & 1]);
                const uint32_t* v = buf[k & 1];
                const int c = half * 256 + k * 32;
                // accumulator column -> tile column (the gate GEMM's column order)
                const int tc = 256 * ((c & 255) >> 7) + 128 * (c >> 8) + (c & 127);
                const bool gate = segment_of(args, c0 + (tc & ~127)) == 3;
                uint32_t hv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float x0 = __uint_as_float(v[2 * e]), x1 = __uint_as_float(v[2 * e + 1]);
                    hv[e] = gate ? sigmoid2_h(x0, x1) : pack_bf16x2(x0, x1);
                }
                uint8_t* blk = smem + (tc >> 6) * 16384;
                const uint32_t chunk0 = (uint32_t)(tc & 63) >> 3;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4*>(blk + sw128_offset((uint32_t)row, chunk0 + q)) =
                        make_uint4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]);
                if ((k & 3) == 3) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&grp_ready[(k >> 2) * 2 + half]);
                }
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    pair::cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        pair::tmem_dealloc(tmem, 512);
    }
}

bool map2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, cuuint64_t cols, cuuint64_t rows) {
    const cuuint64_t d[2] = {cols, rows};
    const cuuint64_t st[1] = {cols * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t es[2] = {1, 1};
    return encode_tiled_fn()(m, dt, 2, const_cast<void*>(base), d, st, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_proj_qkvg_bf16(const void* X, const void* W_in, void* Qo, void* Ko, void* Vo, void* Go, int rows,
                                  int d_model, int Hq, int Hkv, int dk, bool gated, ZeroJob zero, const Runtime& rt,
                                  cudaStream_t s, int w_ld) {
    if (rows == 0) return cudaSuccess;
    const int q_cols = Hq * dk, kv_cols = Hkv * dk;
    const int N = q_cols + 2 * kv_cols + (gated ? q_cols : 0);
    if (w_ld <= 0) w_ld = N;   // W_in's row length (more than N when headwise gate columns follow)
    alignas(64) CUtensorMap tmX, tmW, tmQ, tmK, tmV, tmG;
    {
        const cuuint64_t d[2] = {(cuuint64_t)d_model, (cuuint64_t)rows};
        const cuuint64_t st[1] = {(cuuint64_t)d_model * 2};
        const cuuint32_t box[2] = {64, 128};
        const cuuint32_t es[2] = {1, 1};
        if (encode_tiled_fn()(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), d, st, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // W viewed as (64 columns, d_model rows, N/64 column blocks)
        const cuuint64_t d[3] = {64, (cuuint64_t)d_model, (cuuint64_t)N / 64};
        const cuuint64_t st[2] = {(cuuint64_t)w_ld * 2, 128};
        const cuuint32_t box[3] = {64, 64, 4};
        const cuuint32_t es[3] = {1, 1, 1};
        if (encode_tiled_fn()(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(W_in), d, st, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    if (!map2d(&tmQ, Qo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q_cols, rows) ||
        !map2d(&tmK, Ko, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kv_cols, rows) ||
        !map2d(&tmV, Vo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kv_cols, rows))
        return cudaErrorInvalidValue;
    if (gated) {
        if (!map2d(&tmG, Go, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, q_cols, rows)) return cudaErrorInvalidValue;
    } else {
        tmG = tmQ;   // (no gate columns: never stored through)
    }
    ProjArgs a;
    a.rows = rows;
    a.N = N;
    a.d_model = d_model;
    a.seg_end[0] = q_cols;
    a.seg_end[1] = q_cols + kv_cols;
    a.seg_end[2] = q_cols + 2 * kv_cols;
    a.seg_end[3] = N;
    a.row_tiles = (rows + 255) / 256;
    a.nkc = (d_model + 63) / 64;
    a.zero = zero;
    a.ctl.err = rt.err;
    a.ctl.limit_ns = rt.limit_ns;
    static PerDeviceSetup setup;
    cudaError_t r = setup_once_per_device(setup, [](int&) {
        return cudaFuncSetAttribute(proj_qkvg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    });
    if (r != cudaSuccess) return r;
    const long tiles = (long)a.row_tiles * ((N + 511) / 512);
    return launch_dependent(proj_qkvg_kernel, dim3((unsigned)(2 * tiles)), dim3(kThreads), kSmemBytes, s, tmX, tmW,
                            tmQ, tmK, tmV, tmG, a);
}

}  // namespace gsdpa
