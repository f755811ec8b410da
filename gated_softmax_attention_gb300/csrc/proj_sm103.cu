// proj_sm103.cu -- the layer's input projection as one persistent GEMM on
// pairs of SMs: X [rows, d_model] times W_in = [W_Q | W_K | W_V | W_g]
// [d_model, N], whose columns are up to four outputs side by side, Q [rows,
// H_q d_k], K and V [rows, H_kv d_k] stored as bf16 (no activation) and the
// elementwise gate sigma(X W_g) [rows, H_q d_k] stored as fp16
// ("GatedAttention [2025]", sec. 1.2.1: Q, K, V are projections of the same
// hidden state X; sec. 1.2.2: the gate sigma(X W_theta) reads X too, so the
// four products share every load of X). The attention kernel then reads Q,
// K, V and the gate values as it reads them from a caller.
//
// Tiles of 256 rows x 256 columns, one per pair of CTAs (a cluster of two,
// tcgen05.mma .cta_group::2, M = 256, N = 256): per K chunk of 64 each CTA
// loads its 128 rows of X (16 KB, K-major) and its 128 columns of W (16 KB,
// MN-major: the even CTA the tile's columns 0..127, the odd one 128..255, the
// halves of the MMA's B operand), so accumulator column c is tile column c.
// The grid is persistent: pair p computes tiles p, p + P, p + 2P, ... into
// two accumulators of 256 tensor-memory columns used in turn, so the
// epilogue of one tile runs while the MMAs of the next one fill the other
// accumulator. The number of pairs P is the smallest that keeps the number of
// tiles per pair at its minimum, ceil(tiles / (SMs / 2)): the SMs it leaves
// free run the next kernel of the call early. (The projection has many
// tiles: 256 x 512 tiles without overlap ran 3.4 waves. The elementwise gate
// alone, gate_sigmoid_sm103.cu, has one wave of 256 x 512 tiles: those load a
// third fewer bytes per flop through L2, which measured worth more there
// than the overlap.)
//
// Per CTA: warp 0 TMA producer (both CTAs), warp 1 TMEM allocation (both) and
// MMA issue (even CTA), warps 2..9 epilogue: two groups of four warps (one
// per TMEM lane quadrant), group h converting the tile's columns [128 h,
// 128 h + 128) of its 128 rows, 32 columns at a time (the tensor-memory load
// of the next 32 in flight while the current ones are converted), into a
// staging buffer of its own (two 64-column blocks, 128-byte rows, 128B
// swizzle) that one thread of the group writes with two bulk tensor stores.
// Every output's width is a multiple of 128 columns (or the only output), so
// a group's 128 columns lie in one output. Rows past the end of X, columns
// past N and the K tail load as zeros (TMA out-of-bounds fill) and are not
// stored.
#include "gsdpa_internal.h"
#include "proj_internal.h"
#include "sm103_pair.cuh"
#include "sm103_ptx.cuh"

#include <cuda_fp16.h>

namespace gsdpa {
namespace {

constexpr int kThreads = 320;
constexpr int kNS = 4;                                  // K-chunk ring stages
constexpr uint32_t kXBytes = 128 * 64 * 2;              // X chunk: this CTA's 128 rows x 64
constexpr uint32_t kWBytes = 64 * 128 * 2;              // W chunk: 64 x this CTA's 128 columns
constexpr uint32_t kStage = kXBytes + kWBytes;
constexpr uint32_t kOffStg = kNS * kStage;              // staging: 4 blocks of 128 rows x 64 columns
constexpr uint32_t kStgBytes = 4 * 16384;
constexpr uint32_t kOffBar = kOffStg + kStgBytes;
// barriers: full[NS], empty[NS], acc_full[2], acc_empty[2], drain
constexpr int kNBar = 2 * kNS + 5;
constexpr uint32_t kOffMisc = kOffBar + kNBar * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per block");

struct PGArgs {
    int rows, N, nkc;          // X rows, W columns, K chunks of 64
    int row_tiles, n_tiles;    // tiles of 256 rows; tiles in all
    int seg_end[4];            // cumulative column ends of the outputs (unused ones: N)
    int gate_seg;              // the output holding the gate (fp16 sigma(x)), or -1
    ZeroJob zero;              // per-call state of the attention kernel, zeroed by CTA 0
    WaitCtl ctl;
};

// sigma of two values as fp16: 1/2 + tanh(x/2)/2 with one tanh.approx.f16x2
// for both (relative error about 2^-11, the precision fp16 keeps anyway).
__device__ __forceinline__ uint32_t sigmoid2_h(float x0, float x1) {
    const __half2 hx = __floats2half2_rn(0.5f * x0, 0.5f * x1);
    uint32_t t;
    asm("tanh.approx.f16x2 %0, %1;" : "=r"(t) : "r"(*reinterpret_cast<const uint32_t*>(&hx)));
    const __half2 half2v = __floats2half2_rn(0.5f, 0.5f);
    const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&t), half2v, half2v);
    return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ int segment_of(const PGArgs& a, int col) {
    return col < a.seg_end[0] ? 0 : (col < a.seg_end[1] ? 1 : (col < a.seg_end[2] ? 2 : 3));
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
pair_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1,
                 const __grid_constant__ CUtensorMap tmO2, const __grid_constant__ CUtensorMap tmO3,
                 const PGArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* full = bars;                   // [NS] even CTA: both CTAs' halves of the chunk landed
    uint64_t* empty = bars + kNS;            // [NS] both: the MMAs reading the stage completed
    uint64_t* acc_full = bars + 2 * kNS;     // [2] both: accumulator a holds a finished tile
    uint64_t* acc_empty = bars + 2 * kNS + 2;   // [2] even: both CTAs' epilogues have read accumulator a
    uint64_t* drain = bars + 2 * kNS + 4;    // even
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    int* abort_word = reinterpret_cast<int*>(smem + kOffMisc + 4);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = pair::cta_rank();
    const pair::PairAbort ab{abort_word, pair::map_to(abort_word, rank ^ 1u)};
    const int pid = (int)pair::cluster_id();
    const int np = (int)pair::n_clusters();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 16);   // 8 epilogue warps in each CTA
        }
        mbar_init(drain, 1);
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
    // A programmatic dependent of the previous kernel on the stream, so the
    // prologue above can overlap that kernel's tail. Nothing in global memory
    // is touched before it has completed: it may have produced X, or be the
    // previous call's attention kernel, which still reads this workspace.
    pdl_wait();
    if (blockIdx.x == 0 && args.zero.n > 0) {
        // the attention kernel's per-call state; visible before it can start
        for (int k = threadIdx.x; k < args.zero.n; k += blockDim.x) args.zero.p[k] = 0;
        __threadfence();
        __syncthreads();
    }
    pdl_trigger();   // the next kernel may start; it waits for this grid before reading what it writes

    if (warp == 0) {
        // ---- TMA producer: this CTA's rows of X and its 128 columns of W, tile after tile
        if (lane == 0) {
            bool ok = true;
            uint32_t armed = 0, armed_phase = 0;   // (even CTA) stages armed, and the phase armed
            int item = 0;                          // running K-chunk count (phases carry over tiles)
            for (int tile = pid; tile < args.n_tiles && ok; tile += np) {
                const int r0 = (tile % args.row_tiles) * 256, c0 = (tile / args.row_tiles) * 256;
                for (int kc = 0; kc < args.nkc; ++kc, ++item) {
                    const int s = item % kNS;
                    const uint32_t ph = (item / kNS) & 1;
                    if (!(ok = pair::wait(&empty[s], ph ^ 1u, ab, args.ctl))) break;
                    if (rank == 0) {
                        mbar_arrive_expect_tx(&full[s], 2 * kStage);   // both CTAs' bytes
                        armed |= 1u << s;
                        armed_phase = (armed_phase & ~(1u << s)) | (ph << s);
                    }
                    const uint32_t fb = pair::map_to(&full[s], 0);
                    uint8_t* st = smem + s * kStage;
                    pair::tma_load_2d(st, &tmX, kc * 64, r0 + (int)rank * 128, fb);
                    // W viewed as (64 columns, d_model rows, N/64 blocks): two 64-column blocks
                    pair::tma_load_3d(st + kXBytes, &tmW, 0, kc * 64, (c0 + (int)rank * 128) / 64, fb);
                }
            }
            if (!ok && rank == 0) {
                // Gave up: let the copies of every armed stage land before the CTA exits.
                WaitCtl c2 = args.ctl;
                if (c2.limit_ns < 1000000000ull) c2.limit_ns = 1000000000ull;
                int never = 0;
                const pair::PairAbort quiet{&never, ab.peer};
                for (int s = 0; s < kNS; ++s)
                    if (armed & (1u << s)) pair::wait(&full[s], (armed_phase >> s) & 1u, quiet, c2);
            }
        }
    } else if (warp == 1) {
        // ---- MMA issue (even CTA): D_a[256 x 256] += X[256 x 64] W[64 x 256] per chunk
        if (rank == 0) {
            constexpr uint32_t idG = idesc_bf16_f32(256, 256, false, true);
            constexpr uint32_t HI = desc_sw128_hi(1024);
            const uint32_t base = smem_u32(smem);
            bool ok = true;
            int item = 0, it = 0;
            for (int tile = pid; tile < args.n_tiles && ok; tile += np, ++it) {
                const int a = it & 1;
                // both CTAs' epilogues have read accumulator a (tile it - 2)
                if (!(ok = __all_sync(0xffffffffu, pair::wait(&acc_empty[a], ((it >> 1) & 1) ^ 1u, ab, args.ctl))))
                    break;
                tc_fence_after();
                for (int kc = 0; kc < args.nkc; ++kc, ++item) {
                    const int s = item % kNS;
                    if (!(ok = __all_sync(0xffffffffu, pair::wait(&full[s], (item / kNS) & 1, ab, args.ctl)))) break;
                    tc_fence_after();
                    const uint32_t st = base + s * kStage;
                    // X: K-major, one 64-column box; W: MN-major, 64-column blocks 8 KB apart
                    const uint32_t x0 = desc_sw128_lo(st, 16), w0 = desc_sw128_lo(st + kXBytes, 8192);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        pair::mma_ss(tmem + a * 256, x0 + kk * (32 >> 4), HI, w0 + ((kk * 2048) >> 4), HI, idG,
                                     (kc | kk) != 0);
                    pair::commit_both(&empty[s]);
                }
                if (ok) pair::commit_both(&acc_full[a]);
            }
            if (!ok) {
                // Gave up: let every MMA issued so far complete before TMEM is freed.
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
        // ---- epilogue: group h converts tile columns [128 h, 128 h + 128) of this CTA's rows
        const int qd = warp & 3;
        const int h = (warp - 2) >> 2;
        const int row = qd * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const bool storer = warp == 2 + 4 * h && lane == 0;   // issues the group's stores
        uint8_t* stg = smem + kOffStg + h * 32768;
        int it = 0;
        for (int tile = pid; tile < args.n_tiles; tile += np, ++it) {
            const int a = it & 1;
            bool ok = __all_sync(0xffffffffu, pair::wait(&acc_full[a], (it >> 1) & 1, ab, args.ctl));
            if (storer) tma_store_wait_read0();   // the previous tile's stores have read the staging blocks
            // (the group leaves together or not at all: it shares named barriers; the
            // barrier also tells the group that the staging blocks are free)
            ok = named_bar_and(1 + h, 128, ok);
            if (!ok) break;
            tc_fence_after();
            const int r0 = (tile % args.row_tiles) * 256, c0 = (tile / args.row_tiles) * 256;
            const int gc = c0 + 128 * h;   // the group's first column of W
            const int sg = segment_of(args, gc);
            const bool gate = sg == args.gate_seg;
            const uint32_t tb = tmem + lane_base + a * 256 + h * 128;
            uint32_t buf[2][32];
            tmem_ld32(tb, buf[0]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                tmem_wait_ld_regs(buf[k & 1]);
                if (k + 1 < 4) {
                    tmem_ld32(tb + (k + 1) * 32, buf[(k + 1) & 1]);
                } else {
                    // this warp's part of accumulator a is in registers: the MMAs of tile it + 2 may overwrite it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) pair::arrive_remote(pair::map_to(&acc_empty[a], 0));
                }
                const uint32_t* v = buf[k & 1];
                uint32_t hv[16];
                if (gate) {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        hv[e] = sigmoid2_h(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        hv[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                }
                // staging: [2 blocks of 64 columns][128 rows], 128-byte rows, 128B swizzle
                uint8_t* blk = stg + (k >> 1) * 16384;
                const uint32_t chunk0 = static_cast<uint32_t>(k & 1) * 4;   // 16-byte chunk of the 128-byte row
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4*>(blk + sw128_offset((uint32_t)row, chunk0 + q)) =
                        make_uint4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]);
            }
            // the group's 128 rows x 128 columns are staged: visible to the bulk copies
            fence_proxy_async_smem();
            named_bar_sync(1 + h, 128);
            if (storer && gc < args.N) {
                // (selected, not indexed: the arguments stay in the parameter space)
                const int start = sg == 0 ? 0 : (sg == 1 ? args.seg_end[0] : (sg == 2 ? args.seg_end[1] : args.seg_end[2]));
                const int end = sg == 0 ? args.seg_end[0]
                                        : (sg == 1 ? args.seg_end[1] : (sg == 2 ? args.seg_end[2] : args.seg_end[3]));
                const int col = gc - start, width = end - start;
                const CUtensorMap* m = sg == 0 ? &tmO0 : (sg == 1 ? &tmO1 : (sg == 2 ? &tmO2 : &tmO3));
                const int orow = r0 + (int)rank * 128;
                if (orow < args.rows) {
                    // (rows past the end of the output are clipped by the copy)
                    tma_store_2d(m, stg, col, orow);
                    if (col + 64 < width) tma_store_2d(m, stg + 16384, col + 64, orow);
                    tma_store_commit();
                }
            }
        }
        if (storer) tma_store_wait_all();
        tc_fence_before();
    }

    __syncthreads();
    pair::cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        pair::tmem_dealloc(tmem, 512);
    }
}

bool map2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, cuuint64_t cols, cuuint64_t rows,
           cuuint64_t ld) {
    const cuuint64_t d[2] = {cols, rows};
    const cuuint64_t st[1] = {ld * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t es[2] = {1, 1};
    return encode_tiled_fn()(m, dt, 2, const_cast<void*>(base), d, st, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_pair_gemm_bf16(const void* X, int rows, int d_model, const void* W, int w_ld, int N,
                                  const GemmOut* outs, int n_outs, ZeroJob zero, const Runtime& rt, cudaStream_t s) {
    if (rows == 0 || N == 0) return cudaSuccess;
    if (n_outs < 1 || n_outs > 4 || d_model <= 0 || N % 64 != 0 || w_ld < N || w_ld % 8 != 0 || d_model % 8 != 0)
        return cudaErrorInvalidValue;
    alignas(64) CUtensorMap tmX, tmW, tmO[4];
    if (!map2d(&tmX, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint64_t)d_model, (cuuint64_t)rows, (cuuint64_t)d_model))
        return cudaErrorInvalidValue;
    {
        // W viewed as (64 columns, d_model rows, N/64 column blocks; the blocks 128 bytes apart)
        const cuuint64_t d[3] = {64, (cuuint64_t)d_model, (cuuint64_t)N / 64};
        const cuuint64_t st[2] = {(cuuint64_t)w_ld * 2, 128};
        const cuuint32_t box[3] = {64, 64, 2};
        const cuuint32_t es[3] = {1, 1, 1};
        if (encode_tiled_fn()(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(W), d, st, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    PGArgs a;
    a.rows = rows;
    a.N = N;
    a.nkc = (d_model + 63) / 64;
    a.row_tiles = (rows + 255) / 256;
    a.n_tiles = a.row_tiles * ((N + 255) / 256);
    a.gate_seg = -1;
    int end = 0;
    for (int k = 0; k < 4; ++k) {
        if (k < n_outs) {
            const GemmOut& o = outs[k];
            // every output but the last starts and ends on a 128-column group
            if (o.cols <= 0 || o.cols % 64 != 0 || (k + 1 < n_outs && o.cols % 128 != 0)) return cudaErrorInvalidValue;
            if (!map2d(&tmO[k], o.ptr, o.gate ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                       (cuuint64_t)o.cols, (cuuint64_t)rows, (cuuint64_t)o.cols))
                return cudaErrorInvalidValue;
            if (o.gate) {
                if (a.gate_seg >= 0) return cudaErrorInvalidValue;   // one gate output
                a.gate_seg = k;
            }
            end += o.cols;
        } else {
            tmO[k] = tmO[0];   // (no columns: never stored through)
        }
        a.seg_end[k] = end;
    }
    if (end != N) return cudaErrorInvalidValue;
    a.zero = zero;
    a.ctl.err = rt.err;
    a.ctl.limit_ns = rt.limit_ns;
    static PerDeviceSetup setup;
    cudaError_t r = setup_once_per_device(setup, [](int&) {
        return cudaFuncSetAttribute(pair_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    });
    if (r != cudaSuccess) return r;
    // as few pairs as keep the tiles per pair at their minimum
    const long max_pairs = rt.num_sms / 2 > 0 ? rt.num_sms / 2 : 1;
    const long waves = (a.n_tiles + max_pairs - 1) / max_pairs;
    const long pairs = (a.n_tiles + waves - 1) / waves;
    return launch_dependent(pair_gemm_kernel, dim3((unsigned)(2 * pairs)), dim3(kThreads), kSmemBytes, s, tmX, tmW,
                            tmO[0], tmO[1], tmO[2], tmO[3], a);
}

cudaError_t launch_proj_qkvg_bf16(const void* X, const void* W_in, void* Qo, void* Ko, void* Vo, void* Go, int rows,
                                  int d_model, int Hq, int Hkv, int dk, bool gated, ZeroJob zero, const Runtime& rt,
                                  cudaStream_t s, int w_ld) {
    const int q_cols = Hq * dk, kv_cols = Hkv * dk;
    const int N = q_cols + 2 * kv_cols + (gated ? q_cols : 0);
    if (w_ld <= 0) w_ld = N;   // W_in's row length (more than N when headwise gate columns follow)
    const GemmOut outs[4] = {{Qo, q_cols, false}, {Ko, kv_cols, false}, {Vo, kv_cols, false}, {Go, q_cols, true}};
    return launch_pair_gemm_bf16(X, rows, d_model, W_in, w_ld, N, outs, gated ? 4 : 3, zero, rt, s);
}

}  // namespace gsdpa
