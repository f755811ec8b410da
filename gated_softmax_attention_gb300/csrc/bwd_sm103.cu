// bwd_sm103.cu -- the backward pass of the gated attention layer (bf16,
// d_k = 128) on sm_103a.
//
// Given dO = dL/dO for O = Y (.) G, Y = softmax(Q K^T / sqrt(d_k) + mask) V,
// G = sigma(X W_g) ("GatedAttention [2025]", sec. 1.2.1 and 1.2.2), the chain
// rule gives (the gate's part: "解密NeurIPS最佳论文：Gated Attention…", sec.
// 2.2, gradient on the gate's input = upstream gradient x context x
// sigma (1 - sigma)):
//   dY   = dO (.) G                        the attention's upstream gradient
//   dGl  = dO (.) Y (.) G (1 - G) = dO (.) O (.) (1 - G)       (Y G = O)
//   D_i  = sum_c dY_ic Y_ic = sum_c dO_ic O_ic                  per row, head
//   p_ij = exp(s_ij - lse_i)               lse from the training forward
//   dS   = p (.) (dY V^T - D) / sqrt(d_k)
//   dQ   = dS K,   dK = dS^T Q,   dV = p^T dY   (summed over a GQA group)
//   dW_g = X^T dGl,   dX (gate path) = dGl W_g^T
// Headwise gates broadcast G over d_k, so dGl sums over the head's columns.
// Only the elementwise gate needs dY as a tensor (a bf16 operand of dP and
// dV). A headwise gate is one value g_i per row and head (without a gate,
// g_i = 1): then dY V^T = g_i (dO V^T) and p^T dY = (p g)^T dO, and with
//   p'_ij = p_ij g_i = exp2(s_ij log2(e)/sqrt(d_k) - lse_i log2(e) + log2 g_i)
//   dS_ij = p_ij (g_i dP'_ij - D_i) = p'_ij (dP'_ij - D_i / g_i),  dP' = dO V^T,
// the kernels read dO itself and run unchanged on the row statistics
// -lse log2(e) + log2 g and -D / g (g = 0: p' = 0 and the second one 0): no
// bf16 rounding of dY, and no dY tensor written and read back.
//
// Kernels (all tcgen05, accumulators in TMEM, operands staged by TMA):
//   bwd_prep_kernel    four (row, head) rows per warp: dY (elementwise gate), D,
//                      dGl and lse in log2 (both folded with g, headwise)
//                      units into padded per-(b, h) arrays (whole 128-row
//                      tiles are 512-byte bulk copies);
//   bwd_dq_kernel      per (b, h, 128-row query tile): S = Q K^T and
//                      dP = dY V^T (shared-memory operands), dS into TMEM,
//                      dQ += dS K (dS read from TMEM);
//   bwd_dkdv_kernel    per (b, kv head, 128-key tile): the key tile stays in
//                      shared memory while (Q, dY, lse, D) of every query tile
//                      of every head of the group stream through a ring;
//                      S^T = K Q^T, dP^T = V dY^T, then dV += P^T dY and
//                      dK += dS^T Q, so the group's sum needs no atomics;
//   gemm_bf16_kernel   dX = dGl W_g^T (both operands K-major) and
//                      dW_g = X^T dGl (both MN-major), read in place, where
//                      the product has fewer than 256 columns (else the CTA-pair
//                      GEMM of bwd_gemm_sm103.cu).
// dQ and dK/dV recompute S and dP each (two passes instead of atomics: the
// result does not depend on the order of the CTAs, and each pass keeps its
// accumulators in tensor memory). Every kernel after the prep kernel is a
// programmatic dependent of the one before it: dQ waits for the prep kernel
// before it reads; dK/dV and the gate-gradient GEMMs read nothing their
// predecessor writes, so each starts on the SMs that its predecessor's last
// CTAs leave free, and the last CTA of each waits for its predecessor before
// it exits, so that the call completes after all of them.
#include "gsdpa_internal.h"
#include "proj_internal.h"
#include "sm103_ptx.cuh"

#include <cuda_fp16.h>

namespace gsdpa {
namespace {

constexpr int HD = 128;
constexpr int kTile = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t TILE_BYTES = kTile * HD * 2;     // one [128 x 128] bf16 tile (two 64-column blocks)
constexpr uint32_t STG_BYTES = kTile * 32 * 2;      // one 32-column output chunk (64-byte rows)

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) into
// shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void unpack_bf16x4(uint2 w, float (&f)[4]) {
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xffff0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xffff0000u);
}

// ------------------------------------------------------------------ prep

struct PrepArgs {
    const __nv_bfloat16* dO;   // [B, Lq, Hq, HD]
    const __nv_bfloat16* O;    // [B, Lq, Hq, HD]
    const float* lse;          // [B, Hq, Lq] natural log
    const __half* gate_sig;    // elementwise: sigma(X W_g) [B*Lq, Hq*HD] fp16, else null
    const float* gate_part;    // headwise: logit partials [splits, B*Lq, Hq], else null
    int gate_splits;
    __nv_bfloat16* dY;         // elementwise gate: [B, Lq, Hq, HD], else null
    __nv_bfloat16* dGl;        // [B*Lq, G] (G = Hq*HD | Hq) or null
    float* Dv;                 // [B, Hq, Lq_pad]: -D (negated: added as is by the kernels); headwise -D / g
    float* lse2;               // [B, Hq, Lq_pad]: -lse * log2(e), headwise + log2 g; padding rows -inf
    int B, Lq, Hq, Lq_pad, gate_mode;
};

// Rows are taken in memory order, r = (b L_q + i) H_q + h (so one warp's rows
// are consecutive 256-byte rows of dO, O and the gate), kPrepRows per warp,
// with every load of a warp's rows issued before any is used: each warp keeps
// kPrepRows x 768 bytes in flight. Lane c holds columns 4c .. 4c + 3 of each
// row. The warps past the real rows write the padding rows' D (0) and lse2
// (+inf: no weight), one entry per lane.
constexpr int kPrepRows = 4;

__global__ void __launch_bounds__(256, 4) bwd_prep_kernel(const PrepArgs a) {
    pdl_trigger();   // the dQ kernel may start its set-up; it waits for this grid before reading
    const long wid = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long n_rows = (long)a.B * a.Lq * a.Hq;
    const long real_warps = (n_rows + kPrepRows - 1) / kPrepRows;
    if (wid >= real_warps) {
        // padding rows i in [L_q, L_q_pad) of every (b, h)
        const int pad = a.Lq_pad - a.Lq;
        const long k = (wid - real_warps) * 32 + lane;
        if (pad > 0 && k < (long)a.B * a.Hq * pad) {
            const long at = (k / pad) * a.Lq_pad + a.Lq + k % pad;
            a.Dv[at] = 0.f;
            a.lse2[at] = -INFINITY;
        }
        return;
    }
    const long r0 = wid * kPrepRows;
    uint2 dow[kPrepRows], ow[kPrepRows], gw[kPrepRows];
    float glv[kPrepRows];   // headwise: the row's logit, summed over the split-K partials
    float lse_l = 0.f;
#pragma unroll
    for (int k = 0; k < kPrepRows; ++k) {
        const long r = r0 + k;
        glv[k] = 0.f;
        if (r < n_rows) {
            const long base = r * HD + lane * 4;
            dow[k] = *reinterpret_cast<const uint2*>(a.dO + base);
            ow[k] = *reinterpret_cast<const uint2*>(a.O + base);
            if (a.gate_mode == 2) gw[k] = *reinterpret_cast<const uint2*>(a.gate_sig + base);
        }
    }
    if (a.gate_mode == 1) {
        // the rows' logits: lane 8 k + j adds row k's split-K partials j, j + 8, ...
        // (all of them loaded at once), then the eight lanes of a row add theirs
        static_assert(kPrepRows * 8 == 32, "eight lanes per row");
        const int kk = lane >> 3, jj = lane & 7;
        float part = 0.f;
        if (r0 + kk < n_rows)
            for (int s = jj; s < a.gate_splits; s += 8) part += a.gate_part[s * n_rows + r0 + kk];
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        part += __shfl_xor_sync(0xffffffffu, part, 4);
#pragma unroll
        for (int k = 0; k < kPrepRows; ++k) glv[k] = __shfl_sync(0xffffffffu, part, 8 * k);
    }
    // lane k < kPrepRows fetches row k's lse (natural log, [B, H_q, L_q]); its
    // (b, h, i), decoded once (32-bit divisions while the rows fit in 32 bits:
    // a 64-bit division costs the warp as much as the rest of the row's work)
    long bh = 0, i_row = 0;   // b H_q + h and i of the row of this lane
    if (lane < kPrepRows && r0 + lane < n_rows) {
        const long r = r0 + lane;
        long h, bi;
        if (n_rows <= 0xffffffffL) {
            const uint32_t r32 = (uint32_t)r, hq = (uint32_t)a.Hq, lq = (uint32_t)a.Lq;
            const uint32_t bi32 = r32 / hq, b32 = bi32 / lq;
            h = r32 - bi32 * hq;
            bi = bi32;
            i_row = bi32 - b32 * lq;
            bh = (long)b32 * a.Hq + h;
        } else {
            h = r % a.Hq;
            bi = r / a.Hq;   // b L_q + i
            i_row = bi % a.Lq;
            bh = (bi / a.Lq) * a.Hq + h;
        }
        lse_l = a.lse[bh * a.Lq + i_row];
    }
    float dsum[kPrepRows], gsum[kPrepRows], ghv[kPrepRows];
#pragma unroll
    for (int k = 0; k < kPrepRows; ++k) {
        const long r = r0 + k;
        dsum[k] = gsum[k] = 0.f;
        ghv[k] = 1.f;
        if (r >= n_rows) continue;
        const long base = r * HD + lane * 4;
        float dof[4], of[4];
        unpack_bf16x4(dow[k], dof);
        unpack_bf16x4(ow[k], of);
        float g[4] = {1.f, 1.f, 1.f, 1.f};
        if (a.gate_mode == 2) {
            const float2 g01 = __half22float2(*reinterpret_cast<const __half2*>(&gw[k].x));
            const float2 g23 = __half22float2(*reinterpret_cast<const __half2*>(&gw[k].y));
            g[0] = g01.x;
            g[1] = g01.y;
            g[2] = g23.x;
            g[3] = g23.y;
        } else if (a.gate_mode == 1) {
            ghv[k] = 1.0f / (1.0f + exp2f(-glv[k] * kLog2e));
            g[0] = g[1] = g[2] = g[3] = ghv[k];
        }
        float dgl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            dsum[k] = fmaf(dof[e], of[e], dsum[k]);
            dgl[e] = dof[e] * of[e] * (1.0f - g[e]);
            gsum[k] += dgl[e];
        }
        if (a.gate_mode == 2) {
            *reinterpret_cast<uint2*>(a.dY + base) =
                make_uint2(pack_bf16x2(dof[0] * g[0], dof[1] * g[1]), pack_bf16x2(dof[2] * g[2], dof[3] * g[3]));
            *reinterpret_cast<uint2*>(a.dGl + base) =
                make_uint2(pack_bf16x2(dgl[0], dgl[1]), pack_bf16x2(dgl[2], dgl[3]));
        }
    }
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) {
#pragma unroll
        for (int k = 0; k < kPrepRows; ++k) {
            dsum[k] += __shfl_xor_sync(0xffffffffu, dsum[k], sh);
            gsum[k] += __shfl_xor_sync(0xffffffffu, gsum[k], sh);
        }
    }
    // lane k < kPrepRows writes row k's D, lse2 and (headwise) dGl
    float d_me = dsum[0], g_me = gsum[0], gh_me = ghv[0];
#pragma unroll
    for (int k = 1; k < kPrepRows; ++k)
        if (lane == k) {
            d_me = dsum[k];
            g_me = gsum[k];
            gh_me = ghv[k];
        }
    if (lane < kPrepRows && r0 + lane < n_rows) {
        const long r = r0 + lane;
        const long at = bh * a.Lq_pad + i_row;
        if (a.gate_mode == 1) {
            // g folded into the row statistics (the kernels then read dO for dY)
            a.Dv[at] = gh_me > 0.f ? -d_me / gh_me : 0.f;
            a.lse2[at] = gh_me > 0.f ? log2f(gh_me) - lse_l * kLog2e : -INFINITY;
            a.dGl[r] = __float2bfloat16_rn(g_me);
        } else {
            a.Dv[at] = -d_me;
            a.lse2[at] = -(lse_l * kLog2e);
        }
    }
}

// ------------------------------------------------------------------ GEMM

// C [M x N] (bf16, row-major, ldc) = A B with fp32 accumulation in TMEM.
// A_MN: A stored as [K][M] (M contiguous), else [M][K]; B_MN: B stored as
// [K][N], else B^T stored as [N][K]. 128 x 128 tiles, K chunks of 64. When
// the tiles are too few to occupy the GPU (the narrow headwise dW_g), K is
// split: split s writes its fp32 partial to part[s], summed into C afterwards.
constexpr int kGemmThreads = 192;
constexpr int kGemmNS = 4;
constexpr uint32_t kGemmOpBytes = 128 * 64 * 2;   // 16 KB per operand per chunk
constexpr uint32_t kGemmStage = 2 * kGemmOpBytes;
constexpr uint32_t kGemmOffBar = kGemmNS * kGemmStage;
constexpr uint32_t kGemmOffMisc = kGemmOffBar + (2 * kGemmNS + 2) * 8;
constexpr uint32_t kGemmSmem = kGemmOffMisc + 16 + 1024;

struct GemmArgs {
    __nv_bfloat16* C;
    int M, N, K, ldc;
    int m_tiles, nkc;
    int tiles, splits;   // split s of tile t is CTA s * tiles + t
    float* part;         // splits > 1: fp32 [splits, M, N]
    WaitCtl ctl;
};

template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const GemmArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kGemmOffBar);
    uint64_t* full = bars;
    uint64_t* empty = bars + kGemmNS;
    uint64_t* acc_full = bars + 2 * kGemmNS;
    uint64_t* drain = bars + 2 * kGemmNS + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kGemmOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kGemmOffMisc + 4);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int tile = (int)blockIdx.x % args.tiles, split = (int)blockIdx.x / args.tiles;
    const int m0 = (tile % args.m_tiles) * 128;
    const int n0 = (tile / args.m_tiles) * 128;
    // this CTA's K chunks [kc0, kc1) (possibly none: it then writes zeros)
    const int per = (args.nkc + args.splits - 1) / args.splits;
    const int kc0 = split * per;
    const int kc1 = kc0 + per < args.nkc ? kc0 + per : args.nkc;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGemmNS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 128);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, armed = 0, armed_phase = 0;
            bool ok = true;
            for (int kc = kc0; kc < kc1; ++kc) {
                if (!(ok = mbar_wait(&empty[stage], phase ^ 1u, abort_flag, args.ctl))) break;
                mbar_arrive_expect_tx(&full[stage], kGemmStage);
                armed |= 1u << stage;
                armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
                uint8_t* st = smem + stage * kGemmStage;
                if (A_MN) {
                    for (int cb = 0; cb < 2; ++cb) tma_load_2d(st + cb * 8192, &tmA, m0 + cb * 64, kc * 64, &full[stage]);
                } else {
                    tma_load_2d(st, &tmA, kc * 64, m0, &full[stage]);
                }
                if (B_MN) {
                    for (int cb = 0; cb < 2; ++cb)
                        tma_load_2d(st + kGemmOpBytes + cb * 8192, &tmB, n0 + cb * 64, kc * 64, &full[stage]);
                } else {
                    tma_load_2d(st + kGemmOpBytes, &tmB, kc * 64, n0, &full[stage]);
                }
                if (++stage == kGemmNS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                volatile int never = 0;
                for (int s = 0; s < kGemmNS; ++s)
                    if (armed & (1u << s)) mbar_wait(&full[s], (armed_phase >> s) & 1u, &never, args.ctl);
            }
        }
    } else if (warp == 1) {
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        constexpr uint32_t idG = idesc_bf16_f32(128, 128, A_MN, B_MN);
        constexpr uint32_t HI = desc_sw128_hi(1024);
        const uint32_t base = smem_u32(smem);
        for (int kc = kc0; kc < kc1; ++kc) {
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase, abort_flag, args.ctl)))) break;
            tc_fence_after();
            const uint32_t st = base + stage * kGemmStage;
            // K-major: 64-element K rows of 128 B, K advances 32 B per MMA;
            // MN-major: 64-wide M/N blocks 8 KB apart, K advances 16 rows (2 KB)
            const uint32_t a0 = desc_sw128_lo(st, A_MN ? 8192 : 16);
            const uint32_t b0 = desc_sw128_lo(st + kGemmOpBytes, B_MN ? 8192 : 16);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_ss_elect(tmem, a0 + kk * (A_MN ? (2048 >> 4) : (32 >> 4)), HI,
                             b0 + kk * (B_MN ? (2048 >> 4) : (32 >> 4)), HI, idG, ((kc - kc0) | kk) != 0 ? 1u : 0u);
            mma_commit_elect(&empty[stage]);
            if (++stage == kGemmNS) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (ok) {
            mma_commit_elect(acc_full);
        } else {
            volatile int never = 0;
            mma_commit_elect(drain);
            mbar_wait(drain, 0, &never, args.ctl);
        }
    } else {
        const int qd = warp & 3;
        const int row = qd * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const bool ok = kc1 > kc0 && __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, args.ctl));
        tc_fence_after();
        const int r = m0 + row;
        __nv_bfloat16* dst = args.C + (long)r * args.ldc;
        float* pdst = args.splits > 1 ? args.part + ((long)split * args.M + r) * args.N : nullptr;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
            uint32_t v[32];
            if (ok) {   // (warp-uniform: every lane loads, only rows < M store)
                tmem_ld32(tmem + lane_base + cb * 32, v);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0u;
            }
            const int c = n0 + cb * 32;
            if (r >= args.M) continue;
            if (pdst) {
                if (c + 32 <= args.N && (args.N & 3) == 0) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<uint4*>(pdst + c + e) = make_uint4(v[e], v[e + 1], v[e + 2], v[e + 3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (c + e < args.N) pdst[c + e] = __uint_as_float(v[e]);
                }
            } else if (c + 32 <= args.N && (args.ldc & 7) == 0) {
#pragma unroll
                for (int e = 0; e < 32; e += 8)
                    *reinterpret_cast<uint4*>(dst + c + e) = make_uint4(
                        pack_bf16x2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                        pack_bf16x2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])),
                        pack_bf16x2(__uint_as_float(v[e + 4]), __uint_as_float(v[e + 5])),
                        pack_bf16x2(__uint_as_float(v[e + 6]), __uint_as_float(v[e + 7])));
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (c + e < args.N) dst[c + e] = __float2bfloat16_rn(__uint_as_float(v[e]));
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

// C = sum over the K splits of their fp32 partials, rounded once to bf16.
__global__ void __launch_bounds__(256) gemm_split_sum_kernel(const float* __restrict__ part,
                                                            __nv_bfloat16* __restrict__ C, long mn, int splits) {
    for (long k = (long)blockIdx.x * blockDim.x + threadIdx.x; k < mn; k += (long)gridDim.x * blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < splits; ++s) acc += part[s * mn + k];
        C[k] = __float2bfloat16_rn(acc);
    }
}

// ------------------------------------------------------------------ shared by dQ and dK/dV

// warp 0 copies, warp 1 MMAs, warps 4..7 and 8..11: two warpgroups, one row
// per thread each, splitting the 128 columns of a tile (64 each)
constexpr int kAttnThreads = 384;
// Register split: warpgroup 0 (copies, MMAs, two idle warps) gives registers
// to the two row warpgroups; the launch must provide 384 x kRegsLaunchMin.
constexpr int kRegsLow = 64;
constexpr int kRegsHigh = 216;
constexpr int kRegsLaunchMin = (kRegsLow * 128 + kRegsHigh * 256 + 383) / 384;
constexpr int kKNS = 3;             // dQ: K tile ring (K_j is read until dQ += dS_j K_j)
constexpr int kVNS = 2;             // dQ: V tile ring (V_j is read by dP_j only)
constexpr int kRingNS = kKNS + kVNS;
constexpr int kQNS = 2;             // dK/dV: (Q, dY, lse, D) ring
constexpr uint32_t VEC_BYTES = kTile * 4;   // 128 floats

struct AttnArgs {
    int B, Lq, Lk, Hq, Hkv, causal, n_qtiles, n_ktiles, Lq_pad;
    int hpu;             // dK/dV: query heads per unit; below the group size (GQA), each
                         // unit writes its heads' fp32 share, summed afterwards
    const float* lse2;   // [B, Hq, Lq_pad] -lse in log2 units
    const float* Dv;     // [B, Hq, Lq_pad] -D
    WaitCtl ctl;
};

// Let every MMA this warp issued complete (after a wait gave up), so that
// tensor memory can be freed.
__device__ __forceinline__ void drain_mmas(uint64_t* drain, const WaitCtl& ctl) {
    volatile int never = 0;
    WaitCtl c2 = ctl;
    if (c2.limit_ns < 1000000000ull) c2.limit_ns = 1000000000ull;
    mma_commit_elect(drain);
    mbar_wait(drain, 0, &never, c2);
    __syncwarp();
}

// 32 fp32 columns -> bf16 -> a 64-byte-swizzled [128 x 32] staging chunk
__device__ __forceinline__ void stage_chunk32(uint8_t* chunk, int row, const uint32_t (&v)[32]) {
    const int sw = (row >> 1) & 3;
    uint8_t* dst = chunk + row * 64;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(dst + ((q ^ sw) << 4)) = make_uint4(
            pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
            pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
            pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
            pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
}

// ------------------------------------------------------------------ dQ

struct DqCfg {
    static constexpr uint32_t OFF_Q = 0;                        // Q tile
    static constexpr uint32_t OFF_DY = TILE_BYTES;              // dY tile
    static constexpr uint32_t OFF_RING = 2 * TILE_BYTES;        // K slots 0..kKNS-1, then V slots
    static constexpr uint32_t OFF_STG = OFF_Q;                  // dQ output, 4 chunks (Q, dY are dead by then)
    static constexpr uint32_t OFF_BAR = OFF_RING + kRingNS * TILE_BYTES;
    // full, empty, q_full, s_full, p_full, g_full, drain, s_read, dq_done
    static constexpr int NBAR = 2 * kRingNS + 7;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
    static_assert(SMEM_BYTES <= 232448, "shared memory per block");
};

// Ring slot and phase of copy `item` (K_j = item 2j, V_j = item 2j + 1): K and V
// have rings of their own, so that K_j + kKNS can load while K_j still waits for
// dQ += dS_j K_j.
__device__ __forceinline__ void dq_slot(int item, int& slot, uint32_t& phase) {
    const int j = item >> 1;
    if ((item & 1) == 0) {
        slot = j % kKNS;
        phase = (uint32_t)(j / kKNS) & 1u;
    } else {
        slot = kKNS + j % kVNS;
        phase = (uint32_t)(j / kVNS) & 1u;
    }
}

// Unit = (b, h, 128-row query tile), heaviest first (last tiles first when causal).
// TMEM: S [0, 128), dP [128, 256), dQ [256, 384), dS (packed bf16) [384, 448):
// apart from S and dP, so that each warpgroup writes its half while the other
// still reads.
__global__ void __launch_bounds__(kAttnThreads, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdY,
              const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const __grid_constant__ CUtensorMap tmdQ, const AttnArgs args) {
    using C = DqCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* full = bars;
    uint64_t* empty = bars + kRingNS;
    uint64_t* q_full = bars + 2 * kRingNS;
    uint64_t* s_full = q_full + 1;    // S_j, dP_j in tensor memory
    uint64_t* p_full = q_full + 2;    // dS_j written (256 row threads)
    uint64_t* g_full = q_full + 3;    // every MMA done
    uint64_t* drain = q_full + 4;
    uint64_t* s_read = q_full + 5;    // the rows have loaded S_j, dP_j (256 row threads)
    uint64_t* dq_done = q_full + 6;   // dQ += dS_j K_j done: dS may be overwritten
    static_assert(2 * kRingNS + 7 == C::NBAR, "barrier layout");
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    const int per_tile = args.B * args.Hq;
    const int qt = args.causal ? args.n_qtiles - 1 - (int)blockIdx.x / per_tile : (int)blockIdx.x / per_tile;
    const int h = ((int)blockIdx.x % per_tile) % args.Hq;
    const int b = ((int)blockIdx.x % per_tile) / args.Hq;
    const int kvh = h / (args.Hq / args.Hkv);
    const int q0 = qt * kTile;
    const long off = (long)args.Lk - args.Lq;
    long kend = args.Lk;
    if (args.causal && off + q0 + kTile < kend) kend = off + q0 + kTile;
    const int nkv = (int)((kend + kTile - 1) / kTile);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRingNS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(s_full, 1);
        mbar_init(p_full, 256);
        mbar_init(g_full, 1);
        mbar_init(drain, 1);
        mbar_init(s_read, 256);
        mbar_init(dq_done, 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmdY);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdQ);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // a programmatic dependent of the prep kernel: its outputs are read only
    // after it has completed; then the dK/dV kernel may start
    pdl_wait();
    pdl_trigger();
    if (warp < 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));

    if (warp == 0) {
        if (lane == 0) {
            // ---- copies: Q, dY once; then K_0, V_0, K_1, V_1, ... through the ring
            mbar_arrive_expect_tx(q_full, 2 * TILE_BYTES);
            tma_load_5d(smem + C::OFF_Q, &tmQ, 0, h, q0, b, 0, q_full);
            tma_load_5d(smem + C::OFF_DY, &tmdY, 0, h, q0, b, 0, q_full);
            uint32_t armed = 0, armed_phase = 0;
            bool ok = true;
            for (int item = 0; item < 2 * nkv && ok; ++item) {
                int s;
                uint32_t ph;
                dq_slot(item, s, ph);
                if (!(ok = mbar_wait(&empty[s], ph ^ 1u, abort_flag, args.ctl))) break;
                mbar_arrive_expect_tx(&full[s], TILE_BYTES);
                armed |= 1u << s;
                armed_phase = (armed_phase & ~(1u << s)) | (ph << s);
                tma_load_5d(smem + C::OFF_RING + s * TILE_BYTES, (item & 1) ? &tmV : &tmK, 0, kvh, (item >> 1) * kTile,
                            b, 0, &full[s]);
            }
            if (!ok) {
                volatile int never = 0;
                for (int s = 0; s < kRingNS; ++s)
                    if (armed & (1u << s)) mbar_wait(&full[s], (armed_phase >> s) & 1u, &never, args.ctl);
            }
        }
    } else if (warp == 1) {
        // ---- MMAs: S_j = Q K_j^T, dP_j = dY V_j^T; S_{j+1}, dP_{j+1} as soon as the
        // rows have loaded S_j, dP_j (dS has its own columns), then dQ += dS_j K_j
        constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
        constexpr uint32_t idO = idesc_bf16_f32(128, 128, false, true);
        constexpr uint32_t HI = desc_sw128_hi(1024);
        const uint32_t base = smem_u32(smem);
        bool ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0, abort_flag, args.ctl));
        tc_fence_after();
        const uint32_t q_lo = desc_sw128_lo(base + C::OFF_Q, 16);
        const uint32_t dy_lo = desc_sw128_lo(base + C::OFF_DY, 16);
        // wait for copy `item`; its ring slot
        auto ring_ready = [&](int item, int& sl) -> bool {
            uint32_t ph;
            dq_slot(item, sl, ph);
            const bool r = __all_sync(0xffffffffu, mbar_wait(&full[sl], ph, abort_flag, args.ctl));
            tc_fence_after();
            return r;
        };
        auto issue_S_dP = [&](int j) -> bool {
            int sk, sv;
            if (!ring_ready(2 * j, sk)) return false;
            mma_ss_k128<16384, 16384>(tmem + 0, q_lo, desc_sw128_lo(base + C::OFF_RING + sk * TILE_BYTES, 16), HI, idS,
                                      0);
            if (!ring_ready(2 * j + 1, sv)) return false;
            mma_ss_k128<16384, 16384>(tmem + 128, dy_lo, desc_sw128_lo(base + C::OFF_RING + sv * TILE_BYTES, 16), HI,
                                      idS, 0);
            mma_commit_elect(&empty[sv]);   // V_j: read once
            mma_commit_elect(s_full);
            return true;
        };
        if (ok && nkv > 0) ok = issue_S_dP(0);
        for (int j = 0; j < nkv && ok; ++j) {
            if (j + 1 < nkv) {
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(s_read, j & 1, abort_flag, args.ctl)))) break;
                tc_fence_after();
                if (!(ok = issue_S_dP(j + 1))) break;
            }
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(p_full, j & 1, abort_flag, args.ctl)))) break;
            tc_fence_after();
            // dQ += dS_j K_j: dS (packed bf16) from TMEM, K_j as the MN-major B operand
            int sk;
            uint32_t phk;
            dq_slot(2 * j, sk, phk);
            mma_ts_k128(tmem + 256, tmem + 384, desc_sw128_lo(base + C::OFF_RING + sk * TILE_BYTES, 16384), HI, idO,
                        j != 0);
            mma_commit_elect(dq_done);
            mma_commit_elect(&empty[sk]);
        }
        if (ok) {
            mma_commit_elect(g_full);
        } else {
            drain_mmas(drain, args.ctl);
        }
    } else if (warp >= 4) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        // ---- one query row per thread, columns [64 wg, 64 wg + 64) of every key tile:
        // dS = p (dP - D) / sqrt(d_k); then the dQ epilogue
        const int wg = (warp - 4) >> 2;
        const int qd = warp & 3;
        const int row = qd * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const long i = (long)q0 + row;
        const long pidx = ((long)b * args.Hq + h) * args.Lq_pad + i;
        const float nlse2 = args.lse2[pidx];   // (both stored negated)
        const float nDv = args.Dv[pidx];
        const float sl2 = kLog2e / sqrtf((float)HD);
        const float isq = 1.0f / sqrtf((float)HD);
        bool ok = true;
        for (int j = 0; j < nkv && ok; ++j) {
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(s_full, j & 1, abort_flag, args.ctl)))) break;
            tc_fence_after();
            const long kv0 = (long)j * kTile;
            long lim_l = (long)args.Lk - 1 - kv0;   // last visible column of this row in this tile
            if (args.causal && off + i - kv0 < lim_l) lim_l = off + i - kv0;
            const int lim = lim_l > 127 ? 127 : (int)lim_l;
            uint32_t sv[2][32], dp[2][32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                tmem_ld32(tmem + lane_base + (2 * wg + cc) * 32, sv[cc]);
                tmem_ld32(tmem + lane_base + 128 + (2 * wg + cc) * 32, dp[cc]);
            }
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(s_read);   // S_{j+1}, dP_{j+1} may now overwrite S_j, dP_j
            // dS = p (dP - D), two columns per packed fp32 instruction (the 1/sqrt(d_k)
            // is applied to dQ in the epilogue); masks only where the tile needs them
            uint32_t pk[2][16];
            const float2 sl2x2 = make_float2(sl2, sl2), nl2 = make_float2(nlse2, nlse2), nD = make_float2(nDv, nDv);
            if (lim < 127) {   // masked scores become -inf (p = 0), outside the main loop
#pragma unroll
                for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if ((2 * wg + cc) * 32 + e > lim) sv[cc][e] = __float_as_uint(-INFINITY);
            }
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[cc][e]), __uint_as_float(sv[cc][e + 1])),
                                                sl2x2, nl2);
                    const float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    const float2 ds = __fmul2_rn(pr, __fadd2_rn(make_float2(__uint_as_float(dp[cc][e]),
                                                                            __uint_as_float(dp[cc][e + 1])), nD));
                    pk[cc][e >> 1] = pack_bf16x2(ds.x, ds.y);
                }
            }
            // dQ_{j-1} has read dS_{j-1}
            if (j > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(dq_done, (j - 1) & 1, abort_flag, args.ctl)))) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) tmem_st16(tmem + lane_base + 384 + (2 * wg + cc) * 16, pk[cc]);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(p_full);
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(g_full, 0, abort_flag, args.ctl));
        tc_fence_after();
        // (both warpgroups take the same branch: the epilogue has a 256-thread barrier)
        const bool ok_epi = named_bar_and(1, 256, ok);
        if (ok_epi) {
            uint8_t* stg = smem + C::OFF_STG;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * wg + cc;
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + 256 + c * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * isq);
                stage_chunk32(stg + c * STG_BYTES, row, v);
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 256);
            if (threadIdx.x == 128) {
                for (int c = 0; c < 4; ++c) tma_store_4d(&tmdQ, stg + c * STG_BYTES, c * 32, h, q0, b);
                tma_store_commit();
                tma_store_wait_all();
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ dK, dV

struct DkvCfg {
    static constexpr uint32_t OFF_K = 0;                        // K_j
    static constexpr uint32_t OFF_V = TILE_BYTES;               // V_j
    static constexpr uint32_t OFF_RING = 2 * TILE_BYTES;        // [Q_i | dY_i | lse2_i | D_i] per stage
    static constexpr uint32_t STAGE = 2 * TILE_BYTES + 2 * VEC_BYTES;
    static_assert(STAGE % 1024 == 0 && TILE_BYTES % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
    static constexpr uint32_t OFF_BAR = OFF_RING + kQNS * STAGE;
    static constexpr int NBAR = 2 * kQNS + 7;   // full, empty, kv_full, s_full[2], p_full[2], g_full, drain
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
    static_assert(SMEM_BYTES <= 232448, "shared memory per block");
    static_assert(16 * STG_BYTES <= kQNS * STAGE, "the output staging (fp32 partials) reuses the ring");
};

// Unit = (b, kv head, 128-key tile), key tile 0 first (the most query tiles when causal).
// Per step (query head h of the group, query tile t) two half steps u, one per
// 64 queries of the tile: S^T = K Q_u^T, dP^T = V dY_u^T into buffer u % 2;
// one key row per thread: P^T and dS^T (packed bf16) over the columns each
// warpgroup read; then dV += P^T dY_u, dK += dS^T Q_u. With two buffers the
// MMAs of half step u + 1 run while the rows of half step u are computed.
// TMEM: buffer 0 S^T [0, 64), dP^T [64, 128); buffer 1 [128, 192), [192, 256);
// dV [256, 384), dK [384, 512).
__global__ void __launch_bounds__(kAttnThreads, 1)
bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdY,
                const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                const AttnArgs args) {
    using C = DkvCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* full = bars;
    uint64_t* empty = bars + kQNS;
    uint64_t* kv_full = bars + 2 * kQNS;
    uint64_t* s_full = kv_full + 1;   // [2] S^T, dP^T of buffer u % 2 in tensor memory
    uint64_t* p_full = kv_full + 3;   // [2] P^T, dS^T of buffer u % 2 written (256 row threads)
    uint64_t* g_full = kv_full + 5;
    uint64_t* drain = kv_full + 6;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    // unit: (b, chunk of hpu query heads, key tile) summing over its heads; with
    // hpu = the group size a chunk is a kv head's whole group and the unit writes
    // dK, dV, else it writes the chunk's share (fp32)
    const int group = args.Hq / args.Hkv;
    const int chunks = args.Hq / args.hpu;
    const bool partial = args.hpu < group;
    const int per_tile = args.B * chunks;
    const int kt = (int)blockIdx.x / per_tile;
    const int hu = ((int)blockIdx.x % per_tile) % chunks;
    const int b = ((int)blockIdx.x % per_tile) / chunks;
    const int h_first = hu * args.hpu;   // query heads of the unit: h_first ..
    const int kvh = h_first / group;
    const int n_heads = args.hpu;
    const int k0 = kt * kTile;
    const long off = (long)args.Lk - args.Lq;
    // query tiles that see any key of this tile: query i sees key k0 when off + i >= k0
    int t0 = 0;
    if (args.causal && k0 - off > 0) t0 = (int)((k0 - off) / kTile);
    const int nqt = args.n_qtiles - t0;
    const int steps = n_heads * nqt;   // (head, query tile), head-major
    const int subs = 2 * steps;        // half steps

    if (threadIdx.x == 0) {
        for (int s = 0; s < kQNS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(kv_full, 1);
        for (int u = 0; u < 2; ++u) {
            mbar_init(&s_full[u], 1);
            mbar_init(&p_full[u], 256);
        }
        mbar_init(g_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmdY);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdK);
        tma_prefetch_desc(&tmdV);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // A programmatic dependent of the dQ kernel, whose output it does not read:
    // its inputs come from kernels that completed before the dQ kernel's CTAs
    // let it start. It lets the next kernel start at once; its last CTA leaves
    // only after the dQ kernel has completed, so that this grid completes after it.
    pdl_trigger();
    if (warp < 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));

    if (warp == 0) {
        if (lane == 0) {
            mbar_arrive_expect_tx(kv_full, 2 * TILE_BYTES);
            tma_load_5d(smem + C::OFF_K, &tmK, 0, kvh, k0, b, 0, kv_full);
            tma_load_5d(smem + C::OFF_V, &tmV, 0, kvh, k0, b, 0, kv_full);
            uint32_t armed = 0, armed_phase = 0;
            bool ok = true;
            for (int it = 0; it < steps && ok; ++it) {
                const int s = it % kQNS;
                const uint32_t ph = (it / kQNS) & 1;
                const int h = h_first + it / nqt;
                const int q0 = (t0 + it % nqt) * kTile;
                if (!(ok = mbar_wait(&empty[s], ph ^ 1u, abort_flag, args.ctl))) break;
                mbar_arrive_expect_tx(&full[s], 2 * TILE_BYTES + 2 * VEC_BYTES);
                armed |= 1u << s;
                armed_phase = (armed_phase & ~(1u << s)) | (ph << s);
                uint8_t* st = smem + C::OFF_RING + s * C::STAGE;
                tma_load_5d(st, &tmQ, 0, h, q0, b, 0, &full[s]);
                tma_load_5d(st + TILE_BYTES, &tmdY, 0, h, q0, b, 0, &full[s]);
                const long vidx = ((long)b * args.Hq + h) * args.Lq_pad + q0;
                bulk_load_1d(st + 2 * TILE_BYTES, args.lse2 + vidx, VEC_BYTES, &full[s]);
                bulk_load_1d(st + 2 * TILE_BYTES + VEC_BYTES, args.Dv + vidx, VEC_BYTES, &full[s]);
            }
            if (!ok) {
                volatile int never = 0;
                for (int s = 0; s < kQNS; ++s)
                    if (armed & (1u << s)) mbar_wait(&full[s], (armed_phase >> s) & 1u, &never, args.ctl);
            }
        }
    } else if (warp == 1) {
        constexpr uint32_t idS = idesc_bf16_f32(128, 64, false, false);   // 128 keys x 64 queries
        constexpr uint32_t idO = idesc_bf16_f32(128, 128, false, true);
        constexpr uint32_t HI = desc_sw128_hi(1024);
        const uint32_t base = smem_u32(smem);
        bool ok = __all_sync(0xffffffffu, mbar_wait(kv_full, 0, abort_flag, args.ctl));
        tc_fence_after();
        const uint32_t k_lo = desc_sw128_lo(base + C::OFF_K, 16);
        const uint32_t v_lo = desc_sw128_lo(base + C::OFF_V, 16);
        // S^T, dP^T of half step u: queries [64 (u % 2), 64 (u % 2) + 64) of the stage's
        // tile (8 KB into each 64-column block), into buffer u % 2
        auto issue_S = [&](int u) -> bool {
            const int it = u >> 1, s = it % kQNS;
            if ((u & 1) == 0) {
                if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (it / kQNS) & 1, abort_flag, args.ctl)))
                    return false;
                tc_fence_after();
            }
            const uint32_t st = base + C::OFF_RING + s * C::STAGE + (u & 1) * 8192;
            const uint32_t buf = tmem + (u & 1) * 128;
            mma_ss_k128<16384, 16384>(buf, k_lo, desc_sw128_lo(st, 16), HI, idS, 0);                 // S^T
            mma_ss_k128<16384, 16384>(buf + 64, v_lo, desc_sw128_lo(st + TILE_BYTES, 16), HI, idS, 0);  // dP^T
            mma_commit_elect(&s_full[u & 1]);
            return true;
        };
        if (ok) ok = issue_S(0);
        if (ok) ok = issue_S(1);
        for (int u = 0; u < subs && ok; ++u) {
            const int s = (u >> 1) % kQNS, hq = u & 1;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&p_full[hq], (u >> 1) & 1, abort_flag, args.ctl)))) break;
            tc_fence_after();
            // dV += P^T dY_u, dK += dS^T Q_u: A from TMEM (each warpgroup's 32 queries packed
            // over the first 16 of its 32 columns), B (dY_u, Q_u) MN-major
            const uint32_t st = base + C::OFF_RING + s * C::STAGE + hq * 8192;
            const uint32_t buf = tmem + hq * 128;
            mma_ts_k64_split<32>(tmem + 256, buf, desc_sw128_lo(st + TILE_BYTES, 16384), HI, idO, u != 0);
            mma_ts_k64_split<32>(tmem + 384, buf + 64, desc_sw128_lo(st, 16384), HI, idO, u != 0);
            if (hq == 1) mma_commit_elect(&empty[s]);
            // (the MMAs run in issue order: S^T of u + 2 overwrites this buffer after these read it)
            if (u + 2 < subs && !(ok = issue_S(u + 2))) break;
        }
        if (ok) {
            mma_commit_elect(g_full);
        } else {
            drain_mmas(drain, args.ctl);
        }
    } else if (warp >= 4) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        // ---- one key row per thread, query columns [32 wg, 32 wg + 32) of every half step
        const int wg = (warp - 4) >> 2;
        const int qd = warp & 3;
        const int row = qd * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const long kj = (long)k0 + row;   // this thread's key
        const float sl2 = kLog2e / sqrtf((float)HD);
        const float isq = 1.0f / sqrtf((float)HD);
        bool ok = true;
        for (int u = 0; u < subs && ok; ++u) {
            const int it = u >> 1, s = it % kQNS, hq = u & 1;
            const long qc = (long)(t0 + it % nqt) * kTile + 64 * hq + 32 * wg;   // this thread's first query
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&s_full[hq], (u >> 1) & 1, abort_flag, args.ctl)))) break;
            tc_fence_after();
            const float* L2 = reinterpret_cast<const float*>(smem + C::OFF_RING + s * C::STAGE + 2 * TILE_BYTES) +
                              64 * hq + 32 * wg;
            const float* Dd = L2 + kTile;
            // query column c (query qc + c) sees this key when off + qc + c >= kj
            const long cmin_l = args.causal ? kj - off - qc : 0;
            const int cmin = cmin_l < 0 ? 0 : (cmin_l > 32 ? 32 : (int)cmin_l);
            const uint32_t buf = tmem + lane_base + hq * 128 + 32 * wg;
            uint32_t sv[32], dp[32], ppk[16], dpk[16];
            tmem_ld32(buf, sv);
            tmem_ld32(buf + 64, dp);
            tmem_wait_ld();
            // p = exp2(s sl2 - lse2), dS = p (dP - D) (the 1/sqrt(d_k) is applied to
            // dK in the epilogue), two columns per packed fp32 instruction
            const float2 sl2x2 = make_float2(sl2, sl2);
            if (cmin > 0) {   // masked scores become -inf (p = 0), outside the main loop
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (e < cmin) sv[e] = __float_as_uint(-INFINITY);
            }
#pragma unroll
            for (int g4 = 0; g4 < 8; ++g4) {
                const float4 l4 = *reinterpret_cast<const float4*>(L2 + 4 * g4);
                const float4 d4 = *reinterpret_cast<const float4*>(Dd + 4 * g4);
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int e = 4 * g4 + 2 * h2;
                    const float2 nl = h2 ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y);   // (stored negated)
                    const float2 nd = h2 ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y);
                    const float2 x =
                        __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sl2x2, nl);
                    const float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    const float2 ds = __fmul2_rn(
                        pr, __fadd2_rn(make_float2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), nd));
                    ppk[2 * g4 + h2] = pack_bf16x2(pr.x, pr.y);
                    dpk[2 * g4 + h2] = pack_bf16x2(ds.x, ds.y);
                }
            }
            // packed P^T and dS^T over the first 16 of the 32 columns this warpgroup read
            tmem_st16(buf, ppk);
            tmem_st16(buf + 64, dpk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_full[hq]);
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(g_full, 0, abort_flag, args.ctl));
        tc_fence_after();
        const bool ok_epi = named_bar_and(1, 256, ok);
        if (ok_epi && !partial) {
            // every MMA has completed and every copy landed: stage dV, dK (bf16) in the ring
            uint8_t* stg = smem + C::OFF_RING;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * wg + cc;
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + 256 + c * 32, v);   // dV
                tmem_wait_ld();
                stage_chunk32(stg + c * STG_BYTES, row, v);
                tmem_ld32(tmem + lane_base + 384 + c * 32, v);   // dK (times 1/sqrt(d_k))
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * isq);
                stage_chunk32(stg + (4 + c) * STG_BYTES, row, v);
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 256);
            if (threadIdx.x == 128) {
                for (int c = 0; c < 4; ++c) tma_store_4d(&tmdV, stg + c * STG_BYTES, c * 32, kvh, k0, b);
                for (int c = 0; c < 4; ++c) tma_store_4d(&tmdK, stg + (4 + c) * STG_BYTES, c * 32, kvh, k0, b);
                tma_store_commit();
                tma_store_wait_all();
            }
        } else if (ok_epi) {
            // this head's share as fp32: [128 rows x 32 columns] chunks of 128-byte rows
            // (128-byte swizzle), summed over the group by the reduction kernel
            uint8_t* stg = smem + C::OFF_RING;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * wg + cc;
#pragma unroll
                for (int t = 0; t < 2; ++t) {   // t = 0: dV, 1: dK
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_base + 256 + t * 128 + c * 32, v);
                    tmem_wait_ld();
                    if (t == 1) {   // dK times 1/sqrt(d_k)
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * isq);
                    }
                    uint8_t* dst = stg + (t * 4 + c) * (2 * STG_BYTES) + row * 128;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        *reinterpret_cast<uint4*>(dst + ((q ^ (row & 7)) << 4)) =
                            make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 256);
            if (threadIdx.x == 128) {
                for (int c = 0; c < 4; ++c) tma_store_4d(&tmdV, stg + c * (2 * STG_BYTES), c * 32, hu, k0, b);
                for (int c = 0; c < 4; ++c) tma_store_4d(&tmdK, stg + (4 + c) * (2 * STG_BYTES), c * 32, hu, k0, b);
                tma_store_commit();
                tma_store_wait_all();
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) pdl_wait();
}

// ------------------------------------------------------------------ GQA: sum the heads' shares

// out[b, j, kvh, c] = bf16( sum over the group's heads h of part[b, j, h, c] ),
// the heads added in order (the same bits whatever order the units ran in).
// One thread per 4 columns.
__global__ void __launch_bounds__(256) bwd_group_sum_kernel(const float* __restrict__ part,
                                                            __nv_bfloat16* __restrict__ out, long rows_kv, int Hkv,
                                                            int group) {
    const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;   // over rows_kv * Hkv * 32
    if (idx >= rows_kv * Hkv * (HD / 4)) return;
    const int c4 = (int)(idx % (HD / 4));
    const long rk = idx / (HD / 4);          // (b, j, kvh)
    const int kvh = (int)(rk % Hkv);
    const long bj = rk / Hkv;
    const float* src = part + ((bj * Hkv + kvh) * group) * HD + c4 * 4;   // heads kvh*group .. contiguous
    float4 acc = *reinterpret_cast<const float4*>(src);
    for (int g = 1; g < group; ++g) {
        const float4 v = *reinterpret_cast<const float4*>(src + (long)g * HD);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    *reinterpret_cast<uint2*>(out + rk * HD + c4 * 4) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
}

// ------------------------------------------------------------------ host side

bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
              const cuuint32_t* box, CUtensorMapSwizzle sw,
              CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return encode_tiled_fn()(m, dt, rank, const_cast<void*>(base), dims, strides, box, es,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [B, L, H, 128] as (128, H, L, B) for stores of [128 rows x 32 columns]
bool map_out_f32(CUtensorMap* m, const void* base, int B, int L, int H) {
    const cuuint64_t e = 4;
    cuuint64_t d[4] = {HD, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B};
    cuuint64_t st[3] = {HD * e, (cuuint64_t)H * HD * e, (cuuint64_t)L * H * HD * e};
    cuuint32_t box[4] = {32, 1, 128, 1};
    return make_map(m, base, 4, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
}

// [B, L, H, 128] as (64 columns, H, L, B, 2 column blocks 128 B apart): one
// request loads a [128 rows x 128] tile as two 128B-swizzled 64-column blocks.
bool map_tile(CUtensorMap* m, const void* base, int B, int L, int H) {
    const cuuint64_t e = 2;
    cuuint64_t d[5] = {64, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B, 2};
    cuuint64_t st[4] = {HD * e, (cuuint64_t)H * HD * e, (cuuint64_t)L * H * HD * e, 128};
    cuuint32_t box[5] = {64, 1, 128, 1, 2};
    return make_map(m, base, 5, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// [B, L, H, 128] as (128, H, L, B) for stores of [128 rows x 32 columns]
bool map_out(CUtensorMap* m, const void* base, int B, int L, int H) {
    const cuuint64_t e = 2;
    cuuint64_t d[4] = {HD, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B};
    cuuint64_t st[3] = {HD * e, (cuuint64_t)H * HD * e, (cuuint64_t)L * H * HD * e};
    cuuint32_t box[4] = {32, 1, 128, 1};
    return make_map(m, base, 4, d, st, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

// GEMM operands: K-major [rows][K] (K contiguous) as 128 x 64 boxes; MN-major
// [K][cols] (cols contiguous) as 64 x 64 boxes (two per 128-wide tile).
bool map_kmajor(CUtensorMap* m, const void* base, int rows, int K) {
    cuuint64_t d[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t st[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {64, 128};
    return make_map(m, base, 2, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
bool map_mnmajor(CUtensorMap* m, const void* base, int K, int cols) {
    cuuint64_t d[2] = {(cuuint64_t)cols, (cuuint64_t)K};
    cuuint64_t st[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, 64};
    return make_map(m, base, 2, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <bool A_MN, bool B_MN>
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, __nv_bfloat16* C, int M, int N, int K,
                        int splits, float* part, const Runtime& rt, cudaStream_t s) {
    static PerDeviceSetup setup;   // per template instance
    cudaError_t r = setup_once_per_device(setup, [](int&) {
        return cudaFuncSetAttribute(gemm_bf16_kernel<A_MN, B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kGemmSmem);
    });
    if (r != cudaSuccess) return r;
    GemmArgs a;
    a.C = C;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ldc = N;
    a.m_tiles = (M + 127) / 128;
    a.nkc = (K + 63) / 64;
    a.tiles = a.m_tiles * ((N + 127) / 128);
    // (the plan sized the partials for up to `splits`; one wave on this device's SMs)
    const int fit = rt.num_sms / a.tiles;
    a.splits = splits > 1 && part ? (fit < splits ? fit : splits) : 1;
    if (a.splits < 1) a.splits = 1;
    a.part = part;
    a.ctl.err = rt.err;
    a.ctl.limit_ns = rt.limit_ns;
    gemm_bf16_kernel<A_MN, B_MN><<<(unsigned)((long)a.tiles * a.splits), kGemmThreads, kGemmSmem, s>>>(tmA, tmB, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || a.splits == 1) return e;
    const long mn = (long)M * N;
    const long blocks = (mn + 255) / 256 < 4096 ? (mn + 255) / 256 : 4096;
    gemm_split_sum_kernel<<<(unsigned)blocks, 256, 0, s>>>(part, C, mn, a.splits);
    return cudaGetLastError();
}

// Query heads per dK/dV unit under GQA: the largest divisor of the group size
// whose heaviest unit (the first key tile, every query tile of its heads) is
// at most 1.25 times one SM's average share of the work, so that the units,
// taken heaviest first, still spread about evenly. Larger units load each K,
// V tile for more heads and leave fewer fp32 shares to sum afterwards
// (measured on GQA 32/4 L4096: one head per unit 520 us, two 484, four 478).
int dkdv_heads_per_unit(const Problem& p, int num_sms) {
    const int group = p.Hq / p.Hkv;
    if (group <= 1) return 1;
    const long nq = (p.Lq + kTile - 1) / kTile, nk = (p.Lk + kTile - 1) / kTile;
    const long off = (long)p.Lk - p.Lq;
    long steps = 0, heaviest = 0;   // (query tile, key tile) pairs of one head
    for (long kt = 0; kt < nk; ++kt) {
        long t0 = 0;
        if (p.causal && kt * kTile - off > 0) t0 = (kt * kTile - off) / kTile;
        const long n = nq - t0 > 0 ? nq - t0 : 0;
        steps += n;
        if (n > heaviest) heaviest = n;
    }
    const double share = (double)steps * p.B * p.Hq / (num_sms > 0 ? num_sms : 1);
    int best = 1;
    for (int d = 2; d <= group; ++d)
        if (group % d == 0 && (double)d * heaviest <= 1.25 * share) best = d;
    return best;
}

// K splits for a [M x N x K] product on the single-CTA kernel when the
// 128 x 128 tiles are few: as many as fit in one wave, each split at least 8
// K chunks long (the launch lowers it to one wave of the device's own SMs).
int gemm_splits(int M, int N, int K, int num_sms) {
    const int tiles = ((M + 127) / 128) * ((N + 127) / 128);
    const int nkc = (K + 63) / 64;
    if (tiles >= num_sms / 2 || nkc < 16) return 1;
    int splits = num_sms / tiles;
    if (splits > nkc / 8) splits = nkc / 8;
    return splits > 1 ? splits : 1;
}

}  // namespace

// (the gate variants of gated_sdpa_fwd_variant have no backward here)
bool bwd_supported(const Problem& p) { return p.dtype == 1 && p.dk == HD && p.Lq >= 1 && p.gate_mode <= 2; }

int gate_col_tile(int cols);   // gate_gemm_sm103.cu

BwdPlan plan_bwd(const Problem& p, int num_sms) {
    BwdPlan w;
    Problem pf = p;
    pf.sink = nullptr;
    w.fwd = plan_workspace(pf, num_sms);   // the gate recompute uses the forward's gate buffers
    size_t off = w.fwd.total;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = (off + bytes + 255) & ~size_t(255);
        return at;
    };
    if (p.gate_mode == 1 && w.fwd.gate_splits > 0) {
        // The backward recomputes the headwise logits alone on the device (the
        // forward runs its pre-pass on a few SMs beside the attention kernel):
        // split K so that the pre-pass covers every SM, partials in their own buffer.
        const int nt = gate_col_tile(w.fwd.gate_cols);
        const int tiles = ((w.fwd.gate_rows + 127) / 128) * ((w.fwd.gate_cols + nt - 1) / nt);
        const int nkc = (p.d_model + 63) / 64;
        int splits = (num_sms + tiles - 1) / tiles;
        const int max_splits = nkc / 4 > 0 ? nkc / 4 : 1;
        if (splits > max_splits) splits = max_splits;
        if (splits > w.fwd.gate_splits) {
            w.fwd.gate_splits = splits;
            w.fwd.gate_part = take(sizeof(float) * (size_t)splits * w.fwd.gate_rows * w.fwd.gate_cols);
        }
    }
    w.Lq_pad = (p.Lq + kTile - 1) / kTile * kTile;
    if (p.gate_mode == 2) w.dY = take((size_t)p.B * p.Lq * p.Hq * HD * 2);   // (else the kernels read dO)
    w.Dv = take((size_t)p.B * p.Hq * w.Lq_pad * 4);
    w.lse2 = take((size_t)p.B * p.Hq * w.Lq_pad * 4);
    if (p.gate_mode != 0) w.dGl = take((size_t)p.B * p.Lq * gate_cols(p) * 2);
    if (p.gate_mode != 0) {   // the gate-gradient GEMMs that run on the single-CTA kernel
        const int rows = p.B * p.Lq, G = gate_cols(p);
        w.dx_splits = p.d_model >= 256 ? 1 : gemm_splits(rows, p.d_model, G, num_sms);
        w.dwg_splits = G >= 256 ? 1 : gemm_splits(p.d_model, G, rows, num_sms);
        size_t need = 0;
        if (w.dx_splits > 1) need = (size_t)w.dx_splits * rows * p.d_model;
        if (w.dwg_splits > 1 && (size_t)w.dwg_splits * p.d_model * G > need) need = (size_t)w.dwg_splits * p.d_model * G;
        if (need) w.gemm_part = take(need * 4);   // (the two GEMMs run one after the other)
    }
    if (p.Hq != p.Hkv) {   // GQA: dK, dV per query head, then summed over each group
        w.part_dK = take((size_t)p.B * p.Lk * p.Hq * HD * 4);
        w.part_dV = take((size_t)p.B * p.Lk * p.Hq * HD * 4);
    }
    w.total = off;
    return w;
}

cudaError_t launch_bwd_bf16(const Problem& p, const BwdArgs& g, const BwdPlan& w, char* ws, const Runtime& rt,
                            cudaStream_t s) {
    return launch_bwd_bf16_saved(p, g, nullptr, w, ws, rt, s);
}

cudaError_t launch_bwd_bf16_saved(const Problem& p, const BwdArgs& g, const void* gate_saved, const BwdPlan& w,
                                  char* ws, const Runtime& rt, cudaStream_t s) {
    // 1. the gate again (sigma(X W_g) as fp16, unless the forward saved it, or the headwise logits)
    if (p.gate_mode == 2 && !gate_saved) {
        cudaError_t e = launch_gate_sigmoid_bf16(p, w.fwd, ws, rt, s, ZeroJob());
        if (e != cudaSuccess) return e;
    } else if (p.gate_mode == 1) {
        bool launched = false;
        cudaError_t e = launch_gate_logits_bf16(p, w.fwd, ws, rt, s, &launched, ZeroJob());
        if (e != cudaSuccess) return e;
    }
    // 2. dY (elementwise gate), D, dGl, lse in log2 units (headwise: g folded into the last two)
    PrepArgs pa;
    pa.dO = static_cast<const __nv_bfloat16*>(g.dO);
    pa.O = static_cast<const __nv_bfloat16*>(g.O);
    pa.lse = g.lse;
    pa.gate_sig = p.gate_mode != 2 ? nullptr
                  : gate_saved     ? static_cast<const __half*>(gate_saved)
                                   : reinterpret_cast<const __half*>(ws + w.fwd.gate_sig);
    pa.gate_part = p.gate_mode == 1 ? reinterpret_cast<const float*>(ws + w.fwd.gate_part) : nullptr;
    pa.gate_splits = w.fwd.gate_splits;
    pa.dY = p.gate_mode == 2 ? reinterpret_cast<__nv_bfloat16*>(ws + w.dY) : nullptr;
    pa.dGl = p.gate_mode ? reinterpret_cast<__nv_bfloat16*>(ws + w.dGl) : nullptr;
    pa.Dv = reinterpret_cast<float*>(ws + w.Dv);
    pa.lse2 = reinterpret_cast<float*>(ws + w.lse2);
    pa.B = p.B;
    pa.Lq = p.Lq;
    pa.Hq = p.Hq;
    pa.Lq_pad = w.Lq_pad;
    pa.gate_mode = p.gate_mode;
    const long n_rows = (long)p.B * p.Lq * p.Hq;
    const long pad_entries = (long)p.B * p.Hq * (w.Lq_pad - p.Lq);
    const long warps = (n_rows + kPrepRows - 1) / kPrepRows + (pad_entries + 31) / 32;
    bwd_prep_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(pa);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // 3. dQ, then dK and dV
    alignas(64) CUtensorMap tmQ, tmdY, tmK, tmV, tmdQ, tmdK, tmdV;
    const int hpu = dkdv_heads_per_unit(p, rt.num_sms);
    const bool per_head = hpu < p.Hq / p.Hkv;
    const int chunks = p.Hq / hpu;
    // the dP / dV operand: dY with an elementwise gate, else dO itself (g folded into the row statistics)
    const void* dy_op = p.gate_mode == 2 ? static_cast<const void*>(ws + w.dY) : g.dO;
    if (!map_tile(&tmQ, p.Q, p.B, p.Lq, p.Hq) || !map_tile(&tmdY, dy_op, p.B, p.Lq, p.Hq) ||
        !map_tile(&tmK, p.K, p.B, p.Lk, p.Hkv) || !map_tile(&tmV, p.V, p.B, p.Lk, p.Hkv) ||
        !map_out(&tmdQ, g.dQ, p.B, p.Lq, p.Hq))
        return cudaErrorInvalidValue;
    if (per_head ? !(map_out_f32(&tmdK, ws + w.part_dK, p.B, p.Lk, chunks) &&
                     map_out_f32(&tmdV, ws + w.part_dV, p.B, p.Lk, chunks))
                 : !(map_out(&tmdK, g.dK, p.B, p.Lk, p.Hkv) && map_out(&tmdV, g.dV, p.B, p.Lk, p.Hkv)))
        return cudaErrorInvalidValue;
    AttnArgs aa;
    aa.B = p.B;
    aa.Lq = p.Lq;
    aa.Lk = p.Lk;
    aa.Hq = p.Hq;
    aa.Hkv = p.Hkv;
    aa.causal = p.causal;
    aa.n_qtiles = (p.Lq + kTile - 1) / kTile;
    aa.n_ktiles = (p.Lk + kTile - 1) / kTile;
    aa.Lq_pad = w.Lq_pad;
    aa.hpu = hpu;
    aa.lse2 = reinterpret_cast<const float*>(ws + w.lse2);
    aa.Dv = reinterpret_cast<const float*>(ws + w.Dv);
    aa.ctl.err = rt.err;
    aa.ctl.limit_ns = rt.limit_ns;
    static PerDeviceSetup setup;
    e = setup_once_per_device(setup, [](int&) {
        // The register split only fits if the launch allocates enough registers
        // per thread; refuse to launch otherwise (it would not finish).
        for (const void* k : {reinterpret_cast<const void*>(bwd_dq_kernel),
                              reinterpret_cast<const void*>(bwd_dkdv_kernel)}) {
            cudaFuncAttributes fa;
            cudaError_t r = cudaFuncGetAttributes(&fa, k);
            if (r != cudaSuccess) return r;
            if (fa.numRegs < kRegsLaunchMin) return cudaErrorInvalidConfiguration;
        }
        cudaError_t r =
            cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DqCfg::SMEM_BYTES);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)DkvCfg::SMEM_BYTES);
        return r;
    });
    if (e != cudaSuccess) return e;
    // dQ overlaps the prep kernel's tail (it waits for it before reading); dK/dV
    // and the gate-gradient GEMMs read only what the prep kernel and the
    // caller wrote, so each starts on the SMs its predecessor's tail leaves free
    e = launch_dependent(bwd_dq_kernel, dim3((unsigned)((long)aa.n_qtiles * p.B * p.Hq)), dim3(kAttnThreads),
                         DqCfg::SMEM_BYTES, s, tmQ, tmdY, tmK, tmV, tmdQ, aa);
    if (e != cudaSuccess) return e;
    e = launch_dependent(bwd_dkdv_kernel, dim3((unsigned)((long)aa.n_ktiles * p.B * chunks)),
                         dim3(kAttnThreads), DkvCfg::SMEM_BYTES, s, tmQ, tmdY, tmK, tmV, tmdK, tmdV, aa);
    if (e != cudaSuccess) return e;
    if (per_head) {
        const long rows_kv = (long)p.B * p.Lk;
        const long threads = rows_kv * p.Hkv * (HD / 4);
        const unsigned blocks = (unsigned)((threads + 255) / 256);
        bwd_group_sum_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const float*>(ws + w.part_dK),
                                                    static_cast<__nv_bfloat16*>(g.dK), rows_kv, p.Hkv, chunks / p.Hkv);
        bwd_group_sum_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const float*>(ws + w.part_dV),
                                                    static_cast<__nv_bfloat16*>(g.dV), rows_kv, p.Hkv, chunks / p.Hkv);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (p.gate_mode == 0) return e;

    // 4. the gate's weight and input gradients (on CTA pairs where N fills a 256-column tile)
    const int rows = p.B * p.Lq, G = gate_cols(p);
    // dX [rows x d_model] = dGl [rows x G] W_g^T: A = dGl (K = G contiguous), B^T = W_g [d_model][G]
    if (p.d_model >= 256) {
        e = launch_gemm_pair_bf16(ws + w.dGl, p.Wg, g.dX, rows, p.d_model, G, false, rt, s);
    } else {
        alignas(64) CUtensorMap tA, tB;
        if (!map_kmajor(&tA, ws + w.dGl, rows, G) || !map_kmajor(&tB, p.Wg, p.d_model, G))
            return cudaErrorInvalidValue;
        e = launch_gemm<false, false>(tA, tB, static_cast<__nv_bfloat16*>(g.dX), rows, p.d_model, G, w.dx_splits,
                                      reinterpret_cast<float*>(ws + w.gemm_part), rt, s);
    }
    if (e != cudaSuccess) return e;
    // dW_g [d_model x G] = X^T dGl: A stored as X [rows][d_model], B as dGl [rows][G]
    if (G >= 256) return launch_gemm_pair_bf16(p.X, ws + w.dGl, g.dWg, p.d_model, G, rows, true, rt, s);
    alignas(64) CUtensorMap tA2, tB2;
    if (!map_mnmajor(&tA2, p.X, rows, p.d_model) || !map_mnmajor(&tB2, ws + w.dGl, rows, G))
        return cudaErrorInvalidValue;
    return launch_gemm<true, true>(tA2, tB2, static_cast<__nv_bfloat16*>(g.dWg), p.d_model, G, rows, w.dwg_splits,
                                   reinterpret_cast<float*>(ws + w.gemm_part), rt, s);
}

}  // namespace gsdpa
