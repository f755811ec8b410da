// bwd_gemm_sm103.cu -- the gate's gradient GEMMs on pairs of SMs.
//
// The gate's weight and input gradients ("解密NeurIPS最佳论文：Gated Attention…",
// sec. 2.2: the gradient on the gate's input is the upstream gradient times
// the context times sigma (1 - sigma), here dGl per gate column) are plain
// products: dX = dGl W_g^T and dW_g = X^T dGl, each C [M x N] = A B with bf16
// operands, fp32 accumulation and a bf16 result. Both are large (at 4096
// rows, d_model 2048 and 16 heads of 128, 34 GFLOP each) and read their
// operands in place: dGl is [rows][G] and W_g is [d_model][G], so dX has both
// operands K-major, dW_g both MN-major.
//
// A pair of CTAs (cluster of two, tcgen05.mma .cta_group::2) computes a
// 256 x (256 NH) tile of C in tensor memory (NH = 1 or 2 MMAs of N = 256 per
// K step): per K chunk of 64 each CTA loads its 128 rows of A (16 KB) and
// 128 columns of each 256-column half of B (16 KB per half), for 512 NH MMA
// cycles -- half the L2 traffic per flop of 128 x 128 tiles on one SM.
//
// Column order. A pair MMA takes the first 128 of its 256 columns from the
// even CTA and the rest from the odd one, at the same shared-memory offset;
// CTA rho loads tile columns [256 h + 128 rho, 256 h + 128 rho + 128) of half
// h, so accumulator column c is tile column c.
//
// Per CTA: warp 0 TMA producer (both CTAs) and, once the accumulator is
// complete, the bulk stores of the result; warp 1 TMEM allocation (both) and
// MMA issue (even CTA); warps 2..9 epilogue, two per TMEM lane quadrant, each
// converting half of the columns to bf16 into the idle K-chunk ring (64-column
// blocks of 128-byte rows, 128B swizzle). Each 128-column group is stored as
// soon as its four warps have staged it. Rows and columns past the end of C
// and the K tail load as zeros (TMA out-of-bounds fill) and are not stored.
#include "gsdpa_internal.h"
#include "proj_internal.h"
#include "sm103_pair.cuh"
#include "sm103_ptx.cuh"

namespace gsdpa {
namespace {

constexpr int kThreads = 320;
constexpr uint32_t kABytes = 128 * 64 * 2;   // this CTA's 128 rows of A x 64 of K
constexpr uint32_t kBBytes = 128 * 64 * 2;   // this CTA's 128 columns of one half of B x 64 of K

template <int NH>
struct PairGemmCfg {
    static constexpr int NS = NH == 2 ? 4 : 6;                // K-chunk ring stages
    static constexpr uint32_t STAGE = kABytes + NH * kBBytes;
    static constexpr uint32_t OFF_BAR = NS * STAGE;
    static constexpr int NGRP = 2 * NH;                       // 128-column output groups
    static constexpr uint32_t OFF_MISC = OFF_BAR + (2 * NS + 2 + NGRP) * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;   // + alignment slack
    static_assert(NGRP * 2 * 16384 <= NS * STAGE, "the staged tile fits in the ring");
    static_assert(SMEM_BYTES <= 232448, "shared memory per block");
};

struct PairGemmArgs {
    int m_tiles, nkc;   // tiles of 256 rows; K chunks of 64
    WaitCtl ctl;
};

template <bool A_MN, bool B_MN, int NH>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmC, const PairGemmArgs args) {
    using C = PairGemmCfg<NH>;
    constexpr int NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* full = bars;                   // [NS] even CTA: both CTAs' halves of the chunk landed
    uint64_t* empty = bars + NS;             // [NS] both: the MMAs reading the stage completed
    uint64_t* acc_full = bars + 2 * NS;      // both: the accumulator is complete
    uint64_t* drain = bars + 2 * NS + 1;     // even
    uint64_t* grp_ready = bars + 2 * NS + 2; // [NGRP] the 4 warps staging group g are done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    int* abort_word = reinterpret_cast<int*>(smem + C::OFF_MISC + 4);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = pair::cta_rank();
    const pair::PairAbort ab{abort_word, pair::map_to(abort_word, rank ^ 1u)};
    const int tile = (int)pair::cluster_id();
    const int m0 = (tile % args.m_tiles) * 256;          // the pair's first row
    const int n0 = (tile / args.m_tiles) * (256 * NH);   // the pair's first column
    const int my_m = m0 + (int)rank * 128;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        for (int g = 0; g < C::NGRP; ++g) mbar_init(&grp_ready[g], 4);
        *abort_word = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        pair::tmem_alloc(tmem_slot, 256 * NH);
        tc_fence_before();
    }
    __syncthreads();
    pair::cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a programmatic dependent (the backward's gate-gradient GEMMs),
    // it reads only what kernels that completed before its predecessor started
    // wrote; it lets the next kernel start at once, and its last CTA leaves only
    // after the predecessor has completed, so that the grid completes after it.
    pdl_trigger();

    if (warp == 0) {
        // ---- TMA producer: this CTA's rows of A and its columns of B
        if (lane == 0) {
            for (int kc = 0; kc < args.nkc; ++kc) {
                const int s = kc % NS;
                const uint32_t ph = (kc / NS) & 1;
                if (!pair::wait(&empty[s], ph ^ 1u, ab, args.ctl)) break;
                if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * C::STAGE);   // both CTAs' bytes
                const uint32_t fb = pair::map_to(&full[s], 0);
                uint8_t* st = smem + s * C::STAGE;
                if (A_MN) {   // A stored [K][M]: two 64-wide M blocks
                    pair::tma_load_2d(st, &tmA, my_m, kc * 64, fb);
                    pair::tma_load_2d(st + 8192, &tmA, my_m + 64, kc * 64, fb);
                } else {      // A stored [M][K]
                    pair::tma_load_2d(st, &tmA, kc * 64, my_m, fb);
                }
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    const int nb = n0 + 256 * h + 128 * (int)rank;
                    uint8_t* sb = st + kABytes + h * kBBytes;
                    if (B_MN) {   // B stored [K][N]: two 64-wide N blocks
                        pair::tma_load_2d(sb, &tmB, nb, kc * 64, fb);
                        pair::tma_load_2d(sb + 8192, &tmB, nb + 64, kc * 64, fb);
                    } else {      // B^T stored [N][K]
                        pair::tma_load_2d(sb, &tmB, kc * 64, nb, fb);
                    }
                }
            }
            // ---- then the stores, one 128-column group at a time as it is staged
            // (rows / columns past the end of C are clipped by the copy)
            bool ok = true;
            for (int g = 0; g < C::NGRP && ok; ++g) {
                if (!(ok = pair::wait(&grp_ready[g], 0, ab, args.ctl))) break;
                tma_store_2d(&tmC, smem + g * 32768, n0 + 128 * g, my_m);
                tma_store_2d(&tmC, smem + g * 32768 + 16384, n0 + 128 * g + 64, my_m);
                tma_store_commit();
            }
            tma_store_wait_all();
        }
    } else if (warp == 1) {
        // ---- MMA issue (even CTA): D[256 x 256 NH] += A[256 x 64] B[64 x 256 NH] per chunk
        if (rank == 0) {
            constexpr uint32_t idG = idesc_bf16_f32(256, 256, A_MN, B_MN);
            constexpr uint32_t HI = desc_sw128_hi(1024);
            // K-major: 128-byte K rows, K advances 32 bytes per MMA;
            // MN-major: 64-wide blocks 8 KB apart, K advances 16 rows (2 KB)
            constexpr uint32_t A_STEP = A_MN ? (2048 >> 4) : (32 >> 4);
            constexpr uint32_t B_STEP = B_MN ? (2048 >> 4) : (32 >> 4);
            const uint32_t base = smem_u32(smem);
            bool ok = true;
            for (int kc = 0; kc < args.nkc && ok; ++kc) {
                const int s = kc % NS;
                if (!(ok = __all_sync(0xffffffffu, pair::wait(&full[s], (kc / NS) & 1, ab, args.ctl)))) break;
                tc_fence_after();
                const uint32_t st = base + s * C::STAGE;
                const uint32_t a0 = desc_sw128_lo(st, A_MN ? 8192 : 16);
                const uint32_t b0 = desc_sw128_lo(st + kABytes, B_MN ? 8192 : 16);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                    for (int h = 0; h < NH; ++h)
                        pair::mma_ss(tmem + h * 256, a0 + kk * A_STEP, HI, b0 + ((h * kBBytes) >> 4) + kk * B_STEP,
                                     HI, idG, (kc | kk) != 0);
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
        // ---- epilogue: bf16, 32 columns of one row per thread and step
        const int qd = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = qd * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const bool ok = __all_sync(0xffffffffu, pair::wait(acc_full, 0, ab, args.ctl));
        tc_fence_after();
        if (ok) {
            // (every MMA has completed, so the ring is idle; this warp stages
            // groups half, 2 + half, ... : columns 128 (half + 2 (k / 4)) + 32 (k % 4))
            constexpr int NK = 4 * NH;
            uint32_t buf[2][32];
            tmem_ld32(tmem + lane_base + 128 * half, buf[0]);
#pragma unroll
            for (int k = 0; k < NK; ++k) {
                tmem_wait_ld_regs(buf[k & 1]);
                if (k + 1 < NK)
                    tmem_ld32(tmem + lane_base + 128 * (half + 2 * ((k + 1) >> 2)) + 32 * ((k + 1) & 3),
                              buf[(k + 1) & 1]);
                const uint32_t* v = buf[k & 1];
                const int c = 128 * (half + 2 * (k >> 2)) + 32 * (k & 3);
                uint8_t* blk = smem + (c >> 6) * 16384;
                const uint32_t chunk0 = (uint32_t)(c & 63) >> 3;   // 16-byte chunk of the 128-byte row
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4*>(blk + sw128_offset((uint32_t)row, chunk0 + q)) = make_uint4(
                        pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                        pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                        pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                        pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
                if ((k & 3) == 3) {
                    // this warp's rows of group half + 2 (k / 4) are staged: make them
                    // visible to the bulk copy and tell the storing thread
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&grp_ready[half + 2 * (k >> 2)]);
                }
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    pair::cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        pair::tmem_dealloc(tmem, 256 * NH);
    }
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) pdl_wait();
}

// bf16 [rows][cols] (cols contiguous) as boxes of 64 columns x box_rows rows, 128B swizzle
bool map_bf16(CUtensorMap* m, const void* base, int rows, int cols, cuuint32_t box_rows) {
    const cuuint64_t d[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t st[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return encode_tiled_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), d, st, box, es,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool A_MN, bool B_MN, int NH>
cudaError_t launch_t(const void* A, const void* Bm, void* Cm, int M, int N, int K, const Runtime& rt,
                     cudaStream_t s, bool pdl) {
    using C = PairGemmCfg<NH>;
    alignas(64) CUtensorMap tmA, tmB, tmC;
    if (!(A_MN ? map_bf16(&tmA, A, K, M, 64) : map_bf16(&tmA, A, M, K, 128))) return cudaErrorInvalidValue;
    if (!(B_MN ? map_bf16(&tmB, Bm, K, N, 64) : map_bf16(&tmB, Bm, N, K, 128))) return cudaErrorInvalidValue;
    if (!map_bf16(&tmC, Cm, M, N, 128)) return cudaErrorInvalidValue;
    static PerDeviceSetup setup;   // per template instance
    cudaError_t r = setup_once_per_device(setup, [](int&) {
        return cudaFuncSetAttribute(gemm_pair_kernel<A_MN, B_MN, NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)C::SMEM_BYTES);
    });
    if (r != cudaSuccess) return r;
    PairGemmArgs a;
    a.m_tiles = (M + 255) / 256;
    a.nkc = (K + 63) / 64;
    a.ctl.err = rt.err;
    a.ctl.limit_ns = rt.limit_ns;
    const long tiles = (long)a.m_tiles * ((N + 256 * NH - 1) / (256 * NH));
    if (pdl)
        return launch_dependent(gemm_pair_kernel<A_MN, B_MN, NH>, dim3((unsigned)(2 * tiles)), dim3(kThreads),
                                C::SMEM_BYTES, s, tmA, tmB, tmC, a);
    gemm_pair_kernel<A_MN, B_MN, NH><<<(unsigned)(2 * tiles), kThreads, C::SMEM_BYTES, s>>>(tmA, tmB, tmC, a);
    return cudaGetLastError();
}

}  // namespace

// Tile width: 256 x 512 tiles (two MMAs per K step, the least L2 traffic per
// flop) unless that leaves most pairs idle where 256 x 256 tiles would not:
// cost ~ waves x (MMAs per step + one for the fixed per-tile costs).
int gemm_pair_nh(int M, int N, int num_sms) {
    const long pairs = num_sms / 2 > 0 ? num_sms / 2 : 1;
    const long m_tiles = (M + 255) / 256;
    const long t2 = m_tiles * ((N + 511) / 512), t1 = m_tiles * ((N + 255) / 256);
    const long cost2 = (t2 + pairs - 1) / pairs * 5, cost1 = (t1 + pairs - 1) / pairs * 3;   // x2: 2.5, 1.5
    return cost2 <= cost1 ? 2 : 1;
}

cudaError_t launch_gemm_pair_bf16_kn(const void* A, const void* Bm, void* C, int M, int N, int K, const Runtime& rt,
                                     cudaStream_t s) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    if (K <= 0) return cudaErrorInvalidValue;
    return gemm_pair_nh(M, N, rt.num_sms) == 2 ? launch_t<false, true, 2>(A, Bm, C, M, N, K, rt, s, false)
                                               : launch_t<false, true, 1>(A, Bm, C, M, N, K, rt, s, false);
}

cudaError_t launch_gemm_pair_bf16(const void* A, const void* Bm, void* C, int M, int N, int K, bool ab_mn,
                                  const Runtime& rt, cudaStream_t s) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    if (K <= 0) return cudaErrorInvalidValue;
    const int nh = gemm_pair_nh(M, N, rt.num_sms);
    if (ab_mn) return nh == 2 ? launch_t<true, true, 2>(A, Bm, C, M, N, K, rt, s, true)
                              : launch_t<true, true, 1>(A, Bm, C, M, N, K, rt, s, true);
    return nh == 2 ? launch_t<false, false, 2>(A, Bm, C, M, N, K, rt, s, true)
                   : launch_t<false, false, 1>(A, Bm, C, M, N, K, rt, s, true);
}

}  // namespace gsdpa
