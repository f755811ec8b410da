// prefill_sm103.cu -- bf16 gated attention forward on sm_103a tensor cores.
//
// One CTA computes one unit (b, h, 128-row query tile):
//   S_j = Q K_j^T                       tcgen05.mma, fp32 accumulator in TMEM
//   P_j = exp2(S_j * log2(e)/sqrt(d_k) - m)  online softmax in registers
//   O  += P_j V_j                       tcgen05.mma, fp32 accumulator in TMEM
//   G   = X_tile W_g[:, h*d_k : (h+1)*d_k]   (elementwise gate, same CTA, TMEM)
//   out = O / l (.) sigmoid(G)          epilogue, bf16, TMA store
// ("GatedAttention [2025]", sec. 1.2.1 SDPA and sec. 1.2.2 gate;
//  "10 . 门控", sec. 3.2: G1 sits on each head's SDPA output before concat.)
// The ungated SDPA output never leaves the SM.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q once, gate X/W_g chunks, then K_0, K_1, V_0,
//               K_2, V_1, ... through a ring of NS shared-memory stages;
//   warp 1      TMEM allocation; lane 0 issues every tcgen05.mma and commit;
//   warps 2..5  softmax + epilogue, one thread per query row (TMEM lane).
// S is double-buffered in TMEM so that S_{j+1} = Q K_{j+1}^T runs while the
// softmax warps work on S_j. P goes through shared memory (K-major, 128B
// swizzle) as the A operand of the PV MMA.
//
// TMEM columns: S0 [0,128)  S1 [128,256)  O [256,256+d_k)  G [384,384+d_k).
//
// The causal mask is aligned bottom-right (query i at absolute position
// L_k - L_q + i); key tiles entirely above the diagonal are never loaded.
// Units are numbered heaviest first (last query tiles first) so that the
// hardware block scheduler hands out the long causal units early.
#include "gsdpa_internal.h"
#include "sm103_ptx.cuh"

#include <cmath>

namespace gsdpa {
namespace {

constexpr int kTile = 128;           // query rows per unit, keys per K/V tile
constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

template <int HD, int GATE>
struct PrefillCfg {
    static constexpr uint32_t Q_BYTES = kTile * HD * 2;
    static constexpr uint32_t P_BYTES = kTile * kTile * 2;
    static constexpr uint32_t KV_BYTES = kTile * HD * 2;
    static constexpr uint32_t GX_BYTES = kTile * 64 * 2;
    static constexpr uint32_t GW_BYTES = 64 * HD * 2;
    static constexpr uint32_t STAGE_BYTES =
        (GATE == 2 && GX_BYTES + GW_BYTES > KV_BYTES) ? GX_BYTES + GW_BYTES : KV_BYTES;
    static constexpr int NS = (HD == 128) ? 4 : 6;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_P = OFF_Q + Q_BYTES;
    static constexpr uint32_t OFF_RING = OFF_P + P_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_RING + NS * STAGE_BYTES;
    static constexpr int NBAR = 2 * NS + 9;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
};

struct PrefillArgs {
    int B, Lq, Lk, Hq, Hkv, d_model, causal, n_qtiles;
    const float* gate_part;  // headwise: [splits, B*Lq, Hq]
    int gate_splits;
    float* sink_part;        // [B, Hq, n_qtiles] or null
    WaitCtl ctl;
};

__device__ __forceinline__ float sigmoidf_fast(float x) {
    return 1.0f / (1.0f + ex2_approx(-x * kLog2e));
}

template <int HD, int GATE>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmX,
               const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmO,
               const PrefillArgs args) {
    using C = PrefillCfg<HD, GATE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + C::OFF_Q;
    uint8_t* sP = smem + C::OFF_P;
    uint8_t* ring = smem + C::OFF_RING;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* full = bars;                 // [NS]
    uint64_t* empty = bars + C::NS;        // [NS]
    uint64_t* q_full = bars + 2 * C::NS;
    uint64_t* s_full = q_full + 1;         // [2]
    uint64_t* s_free = q_full + 3;         // [2]
    uint64_t* p_full = q_full + 5;
    uint64_t* o_done = q_full + 6;
    uint64_t* g_full = q_full + 7;
    uint64_t* drain = q_full + 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    float* sred = reinterpret_cast<float*>(smem + C::OFF_MISC + 16);  // [4]

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    // ---- unit (heaviest first when causal)
    const int per_tile = args.Hq * args.B;
    const int u = blockIdx.x;
    const int qt = args.causal ? (args.n_qtiles - 1 - u / per_tile) : (u / per_tile);
    const int rem = u % per_tile;
    const int h = rem % args.Hq;
    const int b = rem / args.Hq;
    const int kvh = h / (args.Hq / args.Hkv);
    const int q0 = qt * kTile;
    const long off = (long)args.Lk - args.Lq;
    long kend = args.Lk;
    if (args.causal) {
        const long last = off + q0 + kTile;  // keys 0 .. off+q0+127 can be visible
        kend = last < kend ? last : kend;
    }
    const int n_kv = (int)((kend + kTile - 1) / kTile);
    const int nkc = (args.d_model + 63) / 64;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(&s_free[0], 128);
        mbar_init(&s_free[1], 128);
        mbar_init(p_full, 128);
        mbar_init(o_done, 1);
        mbar_init(g_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
        if (GATE == 2) {
            tma_prefetch_desc(&tmX);
            tma_prefetch_desc(&tmW);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ================================================================ TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            uint32_t armed_phase[C::NS];
            bool armed[C::NS];
            for (int s = 0; s < C::NS; ++s) armed[s] = false;
            bool ok = true;
            mbar_arrive_expect_tx(q_full, C::Q_BYTES);
            for (int cb = 0; cb < HD / 64; ++cb) tma_load_4d(sQ + cb * 16384, &tmQ, cb * 64, h, q0, b, q_full);

            auto acquire = [&](uint32_t bytes) -> uint8_t* {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, args.ctl)) return nullptr;
                mbar_arrive_expect_tx(&full[stage], bytes);
                armed[stage] = true;
                armed_phase[stage] = phase;
                return ring + stage * C::STAGE_BYTES;
            };
            auto advance = [&]() {
                if (++stage == (uint32_t)C::NS) {
                    stage = 0;
                    phase ^= 1u;
                }
            };
            if (GATE == 2) {
                for (int kc = 0; kc < nkc && ok; ++kc) {
                    uint8_t* st = acquire(C::GX_BYTES + C::GW_BYTES);
                    if (!st) { ok = false; break; }
                    tma_load_3d(st, &tmX, kc * 64, q0, b, &full[stage]);
                    for (int cb = 0; cb < HD / 64; ++cb)
                        tma_load_2d(st + C::GX_BYTES + cb * 8192, &tmW, h * HD + cb * 64, kc * 64, &full[stage]);
                    advance();
                }
            }
            auto load_kv = [&](const CUtensorMap* m, int j) -> bool {
                uint8_t* st = acquire(C::KV_BYTES);
                if (!st) return false;
                for (int cb = 0; cb < HD / 64; ++cb)
                    tma_load_4d(st + cb * 16384, m, cb * 64, kvh, j * kTile, b, &full[stage]);
                advance();
                return true;
            };
            if (ok) ok = load_kv(&tmK, 0);
            for (int j = 1; j < n_kv && ok; ++j) {
                ok = load_kv(&tmK, j);
                if (ok) ok = load_kv(&tmV, j - 1);
            }
            if (ok) ok = load_kv(&tmV, n_kv - 1);
            if (!ok) {
                // Let every copy already issued land before the CTA can exit.
                WaitCtl c2 = args.ctl;
                volatile int never = 0;
                mbar_wait(q_full, 0, &never, c2);
                for (int s = 0; s < C::NS; ++s)
                    if (armed[s]) mbar_wait(&full[s], armed_phase[s], &never, c2);
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            const uint32_t tS0 = tmem, tO = tmem + 256, tG = tmem + 384;
            constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t idO = idesc_bf16_f32(128, HD, false, true);
            const uint32_t sQa = smem_u32(sQ), sPa = smem_u32(sP), ringa = smem_u32(ring);
            auto advance = [&]() {
                if (++stage == (uint32_t)C::NS) {
                    stage = 0;
                    phase ^= 1u;
                }
            };
            ok = mbar_wait(q_full, 0, abort_flag, args.ctl);
            tc_fence_after();
            if (GATE == 2) {
                for (int kc = 0; kc < nkc && ok; ++kc) {
                    if (!(ok = mbar_wait(&full[stage], phase, abort_flag, args.ctl))) break;
                    tc_fence_after();
                    const uint32_t st = ringa + stage * C::STAGE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = smem_desc_sw128(st + kk * 32, 16, 1024);
                        const uint64_t bd = smem_desc_sw128(st + C::GX_BYTES + kk * 2048, 8192, 1024);
                        mma_bf16_ss(tG, ad, bd, idO, (kc | kk) != 0);
                    }
                    mma_commit(&empty[stage]);
                    advance();
                }
                if (ok) mma_commit(g_full);
            }
            auto issue_S = [&](int j) -> bool {
                if (j >= 2 && !mbar_wait(&s_free[j & 1], ((j >> 1) - 1) & 1, abort_flag, args.ctl)) return false;
                if (!mbar_wait(&full[stage], phase, abort_flag, args.ctl)) return false;
                tc_fence_after();
                const uint32_t st = ringa + stage * C::STAGE_BYTES;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16_ss(tS0 + (j & 1) * 128, smem_desc_sw128(sQa + koff, 16, 1024),
                                smem_desc_sw128(st + koff, 16, 1024), idS, kk != 0);
                }
                mma_commit(&empty[stage]);
                mma_commit(&s_full[j & 1]);
                advance();
                return true;
            };
            auto issue_PV = [&](int t) -> bool {
                if (!mbar_wait(p_full, t & 1, abort_flag, args.ctl)) return false;
                tc_fence_after();
                if (!mbar_wait(&full[stage], phase, abort_flag, args.ctl)) return false;
                tc_fence_after();
                const uint32_t st = ringa + stage * C::STAGE_BYTES;
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    const uint32_t poff = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16_ss(tO, smem_desc_sw128(sPa + poff, 16, 1024),
                                smem_desc_sw128(st + kk * 2048, 16384, 1024), idO, (t | kk) != 0);
                }
                mma_commit(&empty[stage]);
                mma_commit(o_done);
                advance();
                return true;
            };
            if (ok) ok = issue_S(0);
            for (int j = 1; j < n_kv && ok; ++j) {
                ok = issue_S(j);
                if (ok) ok = issue_PV(j - 1);
            }
            if (ok) ok = issue_PV(n_kv - 1);
            if (!ok) {
                // Gave up: let every MMA issued so far complete before TMEM is freed.
                volatile int never = 0;
                mma_commit(drain);
                mbar_wait(drain, 0, &never, args.ctl);
            }
        }
    } else {
        // ================================================================ softmax + epilogue
        const int qd = warp & 3;
        const int row = qd * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const int i = q0 + row;
        const long a_pos = off + i;
        const float sl2 = kLog2e / sqrtf((float)HD);
        float m = -INFINITY, l = 0.f, x0 = 0.f;
        bool ok = true;

        for (int j = 0; j < n_kv; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag, args.ctl));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + (j & 1) * 128 + c * 32, sr[c]);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&s_free[j & 1]);

            const int kv0 = j * kTile;
            const bool need_mask = (args.causal && (long)kv0 + kTile - 1 > off + q0) || (kv0 + kTile > args.Lk);
            float tmax = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    float x = __uint_as_float(sr[c][e]) * sl2;
                    if (need_mask) {
                        const long key = kv0 + c * 32 + e;
                        if ((args.causal && key > a_pos) || key >= args.Lk) x = -INFINITY;
                    }
                    sr[c][e] = __float_as_uint(x);
                    tmax = fmaxf(tmax, x);
                }
            }
            if (j == 0) x0 = __uint_as_float(sr[0][0]);
            const float m_new = fmaxf(m, tmax);
            bool waited = false;
            if (j == 0) {
                m = m_new;
            } else if (__any_sync(0xffffffffu, m_new > m + kRescaleThreshold)) {
                ok = __all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, abort_flag, args.ctl));
                if (!ok) break;
                tc_fence_after();
                waited = true;
                const float alpha = ex2_approx(m - m_new);
#pragma unroll
                for (int cb = 0; cb < HD / 32; ++cb) {
                    uint32_t orr[32];
                    tmem_ld32(tmem + lane_base + 256 + cb * 32, orr);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                    tmem_st32(tmem + lane_base + 256 + cb * 32, orr);
                }
                tmem_wait_st();
                l *= alpha;
                m = m_new;
            }
            // P = exp2(x - m), packed to bf16 pairs
            uint32_t pk[64];
            float rs = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float p0 = ex2_approx(__uint_as_float(sr[c][e]) - m);
                    const float p1 = ex2_approx(__uint_as_float(sr[c][e + 1]) - m);
                    rs += p0 + p1;
                    pk[(c * 32 + e) / 2] = pack_bf16x2(p0, p1);
                }
            }
            l += rs;
            if (j > 0 && !waited) {
                ok = __all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, abort_flag, args.ctl));
                if (!ok) break;
            }
            // P row -> shared memory, K-major, 128B swizzle (keys 0..63 box, keys 64..127 box)
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                const uint32_t addr = smem_u32(sP) + (ch >> 3) * 16384 + sw128_offset(row, ch & 7);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[ch * 4]),
                             "r"(pk[ch * 4 + 1]), "r"(pk[ch * 4 + 2]), "r"(pk[ch * 4 + 3])
                             : "memory");
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_full);
        }

        if (ok) ok = mbar_wait(o_done, (n_kv - 1) & 1, abort_flag, args.ctl);
        if (ok && GATE == 2) ok = mbar_wait(g_full, 0, abort_flag, args.ctl);
        tc_fence_after();
        // Every softmax thread takes the same branch (the epilogue has named barriers).
        ok = named_bar_and(1, 128, ok);
        if (ok) {
            // ---- epilogue: out = O / l (.) sigmoid(gate) -> bf16 -> sQ (swizzled) -> TMA store
            const float inv_l = 1.0f / l;
            float g_head = 1.0f;
            if (GATE == 1) {
                float gl = 0.f;
                if (i < args.Lq) {
                    const long rows = (long)args.B * args.Lq;
                    const long idx = ((long)b * args.Lq + i) * args.Hq + h;
                    for (int s = 0; s < args.gate_splits; ++s) gl += args.gate_part[s * rows * args.Hq + idx];
                }
                g_head = sigmoidf_fast(gl);
            }
#pragma unroll
            for (int cb = 0; cb < HD / 32; ++cb) {
                uint32_t orr[32];
                tmem_ld32(tmem + lane_base + 256 + cb * 32, orr);
                uint32_t grr[32];
                if (GATE == 2) tmem_ld32(tmem + lane_base + 384 + cb * 32, grr);
                tmem_wait_ld();
                uint32_t packed[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float v0 = __uint_as_float(orr[e]) * inv_l;
                    float v1 = __uint_as_float(orr[e + 1]) * inv_l;
                    if (GATE == 2) {
                        v0 *= sigmoidf_fast(__uint_as_float(grr[e]));
                        v1 *= sigmoidf_fast(__uint_as_float(grr[e + 1]));
                    } else if (GATE == 1) {
                        v0 *= g_head;
                        v1 *= g_head;
                    }
                    packed[e / 2] = pack_bf16x2(v0, v1);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int chunk = (cb & 1) * 4 + q;
                    const uint32_t addr = smem_u32(sQ) + (cb >> 1) * 16384 + sw128_offset(row, chunk);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(packed[q * 4]),
                                 "r"(packed[q * 4 + 1]), "r"(packed[q * 4 + 2]), "r"(packed[q * 4 + 3])
                                 : "memory");
                }
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (row == 0) {
                for (int cb = 0; cb < HD / 64; ++cb) tma_store_4d(&tmO, sQ + cb * 16384, cb * 64, h, q0, b);
                tma_store_commit();
                tma_store_wait_read0();
            }
            if (args.sink_part) {
                float p0 = (i < args.Lq) ? ex2_approx(x0 - m) * inv_l : 0.f;
#pragma unroll
                for (int sh = 16; sh > 0; sh >>= 1) p0 += __shfl_xor_sync(0xffffffffu, p0, sh);
                if (lane == 0) sred[qd] = p0;
                named_bar_sync(1, 128);
                if (row == 0)
                    args.sink_part[((long)b * args.Hq + h) * args.n_qtiles + qt] = sred[0] + sred[1] + sred[2] + sred[3];
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

// ------------------------------------------------------------------ host side

bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
              const cuuint32_t* box, CUtensorMapSwizzle sw) {
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = encode_tiled_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                                   strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int HD, int GATE>
cudaError_t launch_prefill_t(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt, cudaStream_t s) {
    using C = PrefillCfg<HD, GATE>;
    alignas(64) CUtensorMap tmQ, tmK, tmV, tmX, tmW, tmO;
    const cuuint64_t e = 2;
    {
        cuuint64_t d[4] = {(cuuint64_t)HD, (cuuint64_t)p.Hq, (cuuint64_t)p.Lq, (cuuint64_t)p.B};
        cuuint64_t st[3] = {HD * e, (cuuint64_t)p.Hq * HD * e, (cuuint64_t)p.Lq * p.Hq * HD * e};
        cuuint32_t box[4] = {64, 1, 128, 1};
        if (!make_map(&tmQ, p.Q, 4, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        if (!make_map(&tmO, p.O, 4, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t d[4] = {(cuuint64_t)HD, (cuuint64_t)p.Hkv, (cuuint64_t)p.Lk, (cuuint64_t)p.B};
        cuuint64_t st[3] = {HD * e, (cuuint64_t)p.Hkv * HD * e, (cuuint64_t)p.Lk * p.Hkv * HD * e};
        cuuint32_t box[4] = {64, 1, 128, 1};
        if (!make_map(&tmK, p.K, 4, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        if (!make_map(&tmV, p.V, 4, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    if (GATE == 2) {
        cuuint64_t d[3] = {(cuuint64_t)p.d_model, (cuuint64_t)p.Lq, (cuuint64_t)p.B};
        cuuint64_t st[2] = {(cuuint64_t)p.d_model * e, (cuuint64_t)p.Lq * p.d_model * e};
        cuuint32_t box[3] = {64, 128, 1};
        if (!make_map(&tmX, p.X, 3, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        cuuint64_t dw[2] = {(cuuint64_t)p.Hq * HD, (cuuint64_t)p.d_model};
        cuuint64_t sw[1] = {(cuuint64_t)p.Hq * HD * e};
        cuuint32_t bw[2] = {64, 64};
        if (!make_map(&tmW, p.Wg, 2, dw, sw, bw, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    } else {
        tmX = tmQ;  // unused
        tmW = tmQ;
    }
    PrefillArgs a;
    a.B = p.B;
    a.Lq = p.Lq;
    a.Lk = p.Lk;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.d_model = p.d_model;
    a.causal = p.causal;
    a.n_qtiles = (p.Lq + kTile - 1) / kTile;
    a.gate_part = (GATE == 1) ? reinterpret_cast<const float*>(ws + w.gate_part) : nullptr;
    a.gate_splits = w.gate_splits;
    a.sink_part = p.sink ? reinterpret_cast<float*>(ws + w.sink_part) : nullptr;
    a.ctl.err = rt.err;
    a.ctl.limit_ns = rt.limit_ns;

    static bool attr_done = false;  // per template instance
    if (!attr_done) {
        cudaError_t r = cudaFuncSetAttribute(prefill_kernel<HD, GATE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::SMEM_BYTES);
        if (r != cudaSuccess) return r;
        attr_done = true;
    }
    const long units = (long)a.n_qtiles * p.Hq * p.B;
    prefill_kernel<HD, GATE><<<(unsigned)units, kThreads, C::SMEM_BYTES, s>>>(tmQ, tmK, tmV, tmX, tmW, tmO, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_bf16(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                cudaStream_t s) {
    if (p.dk == 128) {
        if (p.gate_mode == 2) return launch_prefill_t<128, 2>(p, w, ws, rt, s);
        if (p.gate_mode == 1) return launch_prefill_t<128, 1>(p, w, ws, rt, s);
        return launch_prefill_t<128, 0>(p, w, ws, rt, s);
    }
    if (p.gate_mode == 2) return launch_prefill_t<64, 2>(p, w, ws, rt, s);
    if (p.gate_mode == 1) return launch_prefill_t<64, 1>(p, w, ws, rt, s);
    return launch_prefill_t<64, 0>(p, w, ws, rt, s);
}

}  // namespace gsdpa
