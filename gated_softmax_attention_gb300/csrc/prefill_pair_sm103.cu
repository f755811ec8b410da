// prefill_pair_sm103.cu -- bf16 gated attention forward for d_k = 128 on pairs
// of SMs (clusters of two CTAs) sharing M = 256 tcgen05 MMAs.
//
// A pair computes one unit (b, h, four 128-row query tiles). MMA slot t
// (t = 0, 1) stacks query tile 4u+2t of the even CTA over tile 4u+2t+1 of
// the odd CTA into one 256-row operand:
//   S_t = Q_t K_j^T                      tcgen05.mma.cta_group::2, A and B in smem
//   P_t = exp2(S_t log2(e)/sqrt(d_k) - m_t)   online softmax, one thread per row,
//                                        each CTA on its own 128 rows
//   O_t += P_t V_j                       tcgen05.mma.cta_group::2, P read from TMEM
//   G_t = X_t W_g[:, h*d_k:(h+1)*d_k]    elementwise gate GEMM, same pair
//   out_t = O_t / l_t (.) sigmoid(G_t)   epilogue, bf16 rows straight to HBM
// ("GatedAttention [2025]", sec. 1.2.1 SDPA and sec. 1.2.2 the gate
//  Y' = Y (.) sigma(X W); "10 . 门控", sec. 3.2: G1 gates each head's SDPA
//  output before the heads are concatenated.)
//
// Why pairs: a single-CTA 128 x 128 x 16 MMA reads 8 KB of operands from
// shared memory in its 64 cycles, the whole shared-memory bandwidth of the
// SM, and the K/V copies arriving in the same memory then stall it. In a
// pair each SM reads its own 128 A rows and only half of B (6 KB per 64
// cycles), each CTA loads only half of every K, V and W_g tile, and one
// thread issues the MMAs of both SMs.
//
// Operand split. K_j [128 keys x 128]: the even CTA holds keys 0..63, the odd
// CTA keys 64..127 (the N half of the S MMA). V_j [128 keys x 128]: the even
// CTA holds columns 0..63, the odd one columns 64..127 (the N half of the PV
// MMA). W_g chunk [64 x 128]: split by columns the same way. Q_t, X_t and P_t
// (A operands) stay with the CTA whose rows they are.
//
// Warp roles (384 threads per CTA):
//   warp 0       TMA producer of this CTA's halves (both CTAs);
//   warp 1       TMEM allocation (both CTAs, collectively); in the even CTA it
//                also issues every MMA and commit of the pair;
//   warps 2, 3   spare;
//   warps 4..7   softmax + epilogue of this CTA's tile of slot 0;
//   warps 8..11  softmax + epilogue of this CTA's tile of slot 1.
// Barriers the issuing thread waits on (ring stages full, Q loaded, P
// written, TMEM free, gate stages full) live in the even CTA; the odd CTA
// reaches them through cluster addresses. The copies of both CTAs complete
// their bytes on the even CTA's barriers, and the even CTA alone arms them
// with the byte count of both halves (the odd CTA's bytes may land first: a
// barrier's pending byte count may go below zero until it is armed). MMA
// completions (S ready, ring stages free, gate done) are multicast to both
// CTAs.
//
// TMEM (512 columns, same layout in both CTAs): S_0 [0,128) S_1 [128,256)
// O_0 [256,384) O_1 [384,512); P_t packed bf16 in S_t [0,64); G_t reuses S_t.
//
// Causal mask aligned bottom-right (query i at absolute position
// L_k - L_q + i). A slot runs over the key tiles its later query tile can
// see; the even CTA's rows mask the extra tile. Persistent grid: units
// (heaviest first) are dealt to the pairs in snake order.
#include "gsdpa_internal.h"
#include "sm103_pair.cuh"
#include "sm103_ptx.cuh"

#include <cmath>

namespace gsdpa {
namespace {

constexpr int kTile = 128;           // query rows per CTA tile, keys per K/V tile
constexpr int kHD = 128;
constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
constexpr int kRegsLow = 64;
constexpr int kRegsHigh = 216;
constexpr int kRegsLaunchMin = (kRegsLow * 128 + kRegsHigh * 256 + 383) / 384;

struct PairCfg {
    static constexpr uint32_t Q_BYTES = kTile * kHD * 2;      // this CTA's query tile of one slot
    static constexpr uint32_t STAGE_BYTES = 64 * kHD * 2;     // K half (64 keys) or V half (64 columns)
    static constexpr int NS = 8;
    static constexpr uint32_t GX_BYTES = kTile * 64 * 2;      // X chunk of this CTA's rows
    static constexpr uint32_t GW_BYTES = 64 * 64 * 2;         // W_g chunk, this CTA's 64 columns
    static constexpr uint32_t OFF_Q = 0;                      // Q of slot 0, slot 1
    static constexpr uint32_t OFF_RING = 2 * Q_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_RING + NS * STAGE_BYTES;
    // Gate phase (after every attention MMA has completed): Q and the ring are
    // reused as GNS stages, each X_0 | X_1 | W_g half.
    static constexpr uint32_t GSTAGE_BYTES = 2 * GX_BYTES + GW_BYTES;
    static constexpr int GNS = 4;
    static_assert(GNS * GSTAGE_BYTES <= OFF_BAR, "gate ring must fit over Q and the K/V ring");
    static constexpr int NBAR = 2 * NS + 2 * GNS + 10;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
};

struct PairArgs {
    int B, Lq, Lk, Hq, Hkv, d_model, causal, n_qtiles, n_quads;
    const float* gate_part;  // headwise: [splits, B*Lq, Hq]
    int gate_splits;
    float* sink_part;        // [B, Hq, n_qtiles] or null
    __nv_bfloat16* O;        // [B, Lq, Hq, d_k]
    WaitCtl ctl;
};

// sigma(x) = 1/2 + tanh(x/2)/2: one MUFU operation (tanh.approx, relative
// error about 2^-11, i.e. at most ~2.5e-4 absolute on the gate value).
__device__ __forceinline__ float sigmoid_fast(float x) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
    return fmaf(0.5f, t, 0.5f);
}

template <int GATE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
prefill_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmW, const PairArgs args) {
    using C = PairCfg;
    extern __shared__ uint8_t smem_raw[];
    // (both CTAs run the same code, so this offset -- which the MMA
    // descriptors of the even CTA also use for the odd one -- is the same)
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + C::OFF_Q;
    uint8_t* ring = smem + C::OFF_RING;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* full = bars;                  // [NS] even CTA: both halves of a ring item landed (armed by the even CTA)
    uint64_t* empty = bars + C::NS;         // [NS] both: the MMAs reading the item completed
    uint64_t* q_full = bars + 2 * C::NS;    // even: both CTAs' query tiles landed
    uint64_t* s_full = q_full + 1;          // [2] both: S_t complete (and every earlier MMA)
    uint64_t* p_full = q_full + 3;          // [2] even: the 8 softmax warps of slot t wrote P_t
    uint64_t* g_full = q_full + 5;          // [2] both: every MMA of slot t, gate included, complete
    uint64_t* drain = q_full + 7;           // even
    uint64_t* attn_done = q_full + 8;       // both: every attention MMA of the unit complete
    uint64_t* tmem_free = q_full + 9;       // even: the four epilogues of the pair read TMEM out
    uint64_t* gfull = q_full + 10;          // [GNS] even
    uint64_t* gempty = gfull + C::GNS;      // [GNS] both
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    int* abort_word = reinterpret_cast<int*>(smem + C::OFF_MISC + 4);
    volatile int* abort_flag = abort_word;
    float* sred = reinterpret_cast<float*>(smem + C::OFF_MISC + 16);  // [2][4]

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = pair::cta_rank();
    const pair::PairAbort ab{abort_flag, pair::map_to(abort_word, rank ^ 1u)};

    // ---- persistent schedule: units numbered heaviest first (last query quad
    // first when causal), dealt to the pairs in snake order.
    const int per_quad = args.Hq * args.B;
    const int n_units = args.n_quads * per_quad;
    const long off = (long)args.Lk - args.Lq;
    const int nkc = (args.d_model + 63) / 64;
    const int G = (int)pair::n_clusters();
    const int cid = (int)pair::cluster_id();
    struct Unit {
        int qd, h, b, kvh, nj;
        int q0[2], nkv[2];   // q0: first row of this CTA's tile in slot t
        bool act[2];         // slot t has rows (in either CTA)
        bool mine[2];        // this CTA's tile of slot t has rows
    };
    auto unit_index = [&](int r) -> int { return (r & 1) ? (r + 1) * G - 1 - cid : r * G + cid; };
    auto decode_unit = [&](int u) -> Unit {
        Unit x;
        x.qd = args.causal ? (args.n_quads - 1 - u / per_quad) : (u / per_quad);
        const int rem = u % per_quad;
        x.h = rem % args.Hq;
        x.b = rem / args.Hq;
        x.kvh = x.h / (args.Hq / args.Hkv);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int lo = (4 * x.qd + 2 * t) * kTile;          // the even CTA's tile
            x.q0[t] = lo + (int)rank * kTile;
            x.act[t] = lo < args.Lq;
            x.mine[t] = x.q0[t] < args.Lq;
            const int last = (lo + kTile < args.Lq) ? lo + kTile : lo;   // the slot's last tile with rows
            long kend = args.Lk;
            if (args.causal) {
                const long e = off + last + kTile;   // keys 0 .. off+last+127 can be visible
                kend = e < kend ? e : kend;
            }
            x.nkv[t] = x.act[t] ? (int)((kend + kTile - 1) / kTile) : 0;
        }
        x.nj = x.nkv[0] > x.nkv[1] ? x.nkv[0] : x.nkv[1];
        return x;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(q_full, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], 8);
            mbar_init(&g_full[t], 1);
        }
        mbar_init(drain, 1);
        mbar_init(attn_done, 1);
        mbar_init(tmem_free, 4);
        for (int s = 0; s < C::GNS; ++s) {
            mbar_init(&gfull[s], 1);
            mbar_init(&gempty[s], 1);
        }
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        if (GATE == 2) {
            tma_prefetch_desc(&tmX);
            tma_prefetch_desc(&tmW);
        }
    }
    if (warp == 1) {
        pair::tmem_alloc(tmem_slot, 512);
        tc_fence_before();
    }
    __syncthreads();
    pair::cluster_sync();   // both CTAs' barriers exist before anything reaches them
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (warp < 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == 0) {
        // ================================================================ TMA producer (both CTAs)
        if (lane == 0) {
            bool ok = true;
            int item = 0, gitem = 0;   // running counts: phases carry over units
            const uint32_t q_full_e = pair::map_to(q_full, 0);
            for (int r = 0; ok; ++r) {
            const int uix = unit_index(r);
            if (uix >= n_units) break;
            const Unit U = decode_unit(uix);
            // every MMA of the previous unit is complete (its gate ring overlays Q and K/V)
            if (r > 0 && !(ok = pair::wait(&g_full[1], (r - 1) & 1, ab, args.ctl))) break;
            // tiles with rows, both CTAs (the odd CTA's tile of a slot starts one tile later)
            const uint32_t q_tiles = (U.act[0] ? 1u : 0u) + (U.act[1] ? 1u : 0u) +
                                     (U.act[0] && U.q0[0] - (int)rank * kTile + kTile < args.Lq ? 1u : 0u) +
                                     (U.act[1] && U.q0[1] - (int)rank * kTile + kTile < args.Lq ? 1u : 0u);
            if (rank == 0) mbar_arrive_expect_tx(q_full, q_tiles * C::Q_BYTES);
            for (int t = 0; t < 2; ++t)
                if (U.mine[t])
                    for (int cb = 0; cb < 2; ++cb)
                        pair::tma_load_4d(sQ + t * C::Q_BYTES + cb * 16384, &tmQ, cb * 64, U.h, U.q0[t], U.b,
                                          q_full_e);
            auto acquire = [&]() -> uint8_t* {
                const int s = item % C::NS;
                const uint32_t ph = (item / C::NS) & 1;
                if (!pair::wait(&empty[s], ph ^ 1u, ab, args.ctl)) return nullptr;
                if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * C::STAGE_BYTES);
                return ring + s * C::STAGE_BYTES;
            };
            for (int j = 0; j < U.nj && ok; ++j) {
                // K_j: keys [64 rank, 64 rank + 64) of the tile, all d_k columns (two 64-column boxes)
                uint8_t* st = acquire();
                if (!st) { ok = false; break; }
                const uint32_t fk = pair::map_to(&full[item % C::NS], 0);
                for (int cb = 0; cb < 2; ++cb)
                    pair::tma_load_4d(st + cb * 8192, &tmK, cb * 64, U.kvh, j * kTile + (int)rank * 64, U.b, fk);
                ++item;
                // V_j: all 128 keys, columns [64 rank, 64 rank + 64)
                st = acquire();
                if (!st) { ok = false; break; }
                pair::tma_load_4d(st, &tmV, (int)rank * 64, U.kvh, j * kTile, U.b, pair::map_to(&full[item % C::NS], 0));
                ++item;
            }
            if (GATE == 2 && ok) {
                // The gate ring overlays Q and the K/V ring: start once they are idle.
                ok = pair::wait(attn_done, r & 1, ab, args.ctl);
                for (int kc = 0; kc < nkc && ok; ++kc, ++gitem) {
                    const int gs = gitem % C::GNS;
                    const uint32_t ph = (gitem / C::GNS) & 1;
                    if (!(ok = pair::wait(&gempty[gs], ph ^ 1u, ab, args.ctl))) break;
                    const uint32_t gf = pair::map_to(&gfull[gs], 0);
                    if (rank == 0) mbar_arrive_expect_tx(&gfull[gs], (q_tiles * C::GX_BYTES) + 2 * C::GW_BYTES);
                    uint8_t* st = smem + gs * C::GSTAGE_BYTES;
                    for (int t = 0; t < 2; ++t)
                        if (U.mine[t]) pair::tma_load_3d(st + t * C::GX_BYTES, &tmX, kc * 64, U.q0[t], U.b, gf);
                    pair::tma_load_2d(st + 2 * C::GX_BYTES, &tmW, U.h * kHD + (int)rank * 64, kc * 64, gf);
                }
            }
            }   // units
            if (!ok) {
                // Gave up: the other CTA stops too (both abort flags are raised);
                // give copies already issued time to land before the CTA exits.
                const unsigned long long t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) {
                }
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer (even CTA)
        if (rank == 0) {   // the whole warp runs the loop (warp-uniform operands); one elected lane issues
            bool ok = true;
            constexpr uint32_t idS = idesc_bf16_f32(256, 128, false, false);
            constexpr uint32_t idO = idesc_bf16_f32(256, kHD, false, true);
            const uint32_t sQa = smem_u32(sQ), ringa = smem_u32(ring);
            int ibase = 0, gbase = 0;      // running ring-item / gate-chunk counts
            int sp_base[2] = {0, 0};       // completed s_full / p_full phases per slot
            auto stage_addr = [&](int it) { return ringa + ((ibase + it) % C::NS) * C::STAGE_BYTES; };
            auto wait_full = [&](int it) -> bool {
                const int x = ibase + it;
                if (!__all_sync(0xffffffffu, pair::wait(&full[x % C::NS], (x / C::NS) & 1, ab, args.ctl)))
                    return false;
                tc_fence_after();
                return true;
            };
            constexpr uint32_t HI = desc_sw128_hi(1024);   // every operand: 8-row groups 1024 B apart
            auto issue_S = [&](int t, int j) {
                const uint32_t a0 = desc_sw128_lo(sQa + t * C::Q_BYTES, 16);
                const uint32_t b0 = desc_sw128_lo(stage_addr(2 * j), 16);
#pragma unroll
                for (int kk = 0; kk < kHD / 16; ++kk) {
                    // K-major, 64-column boxes: Q boxes are 128 rows (16 KB), K halves 64 rows (8 KB)
                    const uint32_t ka = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                    const uint32_t kb = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
                    pair::mma_ss(tmem + t * 128, a0 + ka, HI, b0 + kb, HI, idS, kk != 0);
                }
                pair::commit_both(&s_full[t]);
            };
            auto issue_PV = [&](int t, int j) -> bool {
                if (!__all_sync(0xffffffffu, pair::wait(&p_full[t], (sp_base[t] + j) & 1, ab, args.ctl)))
                    return false;
                tc_fence_after();
                // V half: MN-major, one 64-column block; 16 keys = 2 KB per K step
                const uint32_t v0 = desc_sw128_lo(stage_addr(2 * j + 1), 8192);
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)
                    pair::mma_ts(tmem + 256 + t * 128, tmem + t * 128 + kk * 8, v0 + kk * (2048 >> 4), HI, idO,
                                 (j | kk) != 0);
                return true;
            };

            for (int r = 0; ok; ++r) {
            const int uix = unit_index(r);
            if (uix >= n_units) break;
            const Unit U = decode_unit(uix);
            const int nj = U.nj;
            const int* nkv = U.nkv;
            ok = __all_sync(0xffffffffu, pair::wait(q_full, r & 1, ab, args.ctl));
            // S_t and O_t of the previous unit must have been read by its epilogues
            if (ok && r > 0) ok = __all_sync(0xffffffffu, pair::wait(tmem_free, (r - 1) & 1, ab, args.ctl));
            tc_fence_after();
            if (ok) ok = wait_full(0);
            if (ok) {
                if (U.act[0]) issue_S(0, 0);
                if (U.act[1]) issue_S(1, 0);
                pair::commit_both(&empty[ibase % C::NS]);
            }
            for (int j = 0; j < nj && ok; ++j) {
                if (!(ok = wait_full(2 * j + 1))) break;   // V_j
                bool k_ready = false;
                if (j < nkv[0]) {
                    if (!(ok = issue_PV(0, j))) break;
                    if (j + 1 < nkv[0]) {
                        if (!(ok = wait_full(2 * j + 2))) break;
                        k_ready = true;
                        issue_S(0, j + 1);
                    }
                }
                if (j < nkv[1]) {
                    if (!(ok = issue_PV(1, j))) break;
                }
                pair::commit_both(&empty[(ibase + 2 * j + 1) % C::NS]);     // V_j done
                if (j + 1 < nkv[1]) {
                    if (!k_ready && !(ok = wait_full(2 * j + 2))) break;
                    k_ready = true;
                    issue_S(1, j + 1);
                }
                if (k_ready) pair::commit_both(&empty[(ibase + 2 * j + 2) % C::NS]);  // K_{j+1} done
            }
            // gate GEMM G_t = X_t W_g[:, cols(h)] into the S_t columns, then signal the epilogues
            if (ok) pair::commit_both(attn_done);
            if (GATE == 2) {
                constexpr uint32_t idG = idesc_bf16_f32(256, kHD, false, true);
                const uint32_t base = smem_u32(smem);
                for (int kc = 0; kc < nkc && ok; ++kc) {
                    const int gi = gbase + kc;
                    const int gs = gi % C::GNS;
                    if (!(ok = __all_sync(0xffffffffu, pair::wait(&gfull[gs], (gi / C::GNS) & 1, ab, args.ctl))))
                        break;
                    tc_fence_after();
                    const uint32_t st = base + gs * C::GSTAGE_BYTES;
                    const uint32_t w0 = desc_sw128_lo(st + 2 * C::GX_BYTES, 8192);
                    for (int t = 0; t < 2; ++t) {
                        if (!U.act[t]) continue;
                        const uint32_t x0 = desc_sw128_lo(st + t * C::GX_BYTES, 16);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            pair::mma_ss(tmem + t * 128, x0 + kk * (32 >> 4), HI, w0 + kk * (2048 >> 4), HI, idG,
                                         (kc | kk) != 0);
                    }
                    pair::commit_both(&gempty[gs]);
                }
            }
            if (ok) {
                pair::commit_both(&g_full[0]);
                pair::commit_both(&g_full[1]);
            }
            ibase += 2 * nj;
            if (GATE == 2) gbase += nkc;
            sp_base[0] += nkv[0];
            sp_base[1] += nkv[1];
            }   // units
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
    } else if (warp >= 4) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        // ================================================================ softmax + epilogue (both CTAs)
        const int t = (warp - 4) >> 2;        // slot
        const int qd = warp & 3;               // TMEM lane quadrant of this warp
        const int row = qd * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const uint32_t tS = tmem + lane_base + t * 128;
        const uint32_t tO = tmem + lane_base + 256 + t * 128;
        const uint32_t p_full_e = pair::map_to(&p_full[t], 0);
        const uint32_t tmem_free_e = pair::map_to(tmem_free, 0);
        const float sl2 = kLog2e / sqrtf((float)kHD);
        bool ok = true;
        int sp_base = 0;     // completed s_full / p_full phases of this slot
        int g_base = 0;      // completed g_full phases of this slot
        for (int r = 0; ok; ++r) {
        const int uix = unit_index(r);
        if (uix >= n_units) break;
        const Unit U = decode_unit(uix);
        const int h = U.h, b = U.b;
        const int nkv = U.nkv[t];
        const int i = U.q0[t] + row;
        const long a_pos = off + i;
        float m = -INFINITY, l = 0.f, x0 = 0.f;

        for (int j = 0; j < nkv; ++j) {
            ok = __all_sync(0xffffffffu, pair::wait(&s_full[t], (sp_base + j) & 1, ab, args.ctl));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
            tmem_wait_ld();

            const int kv0 = j * kTile;
            // last visible column of this row in this key tile (>= 127: no mask)
            long lim_l = (long)args.Lk - 1 - kv0;
            if (args.causal && a_pos - kv0 < lim_l) lim_l = a_pos - kv0;
            const int lim = lim_l > 127 ? 127 : (int)lim_l;
            // raw scores; masked ones become -inf (the 1/sqrt(d_k)*log2(e) scale is
            // folded into the exp2 argument below, max commutes with it)
            if (lim < 127) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (c * 32 + e > lim) sr[c][e] = __float_as_uint(-INFINITY);
            }
            float mx[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx[e] = fmaxf(__uint_as_float(sr[0][e]), __uint_as_float(sr[0][e + 8]));
#pragma unroll
            for (int k = 16; k < 128; k += 16) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    mx[e] = fmax3(mx[e], __uint_as_float(sr[k >> 5][(k & 31) + e]),
                                  __uint_as_float(sr[(k + 8) >> 5][((k + 8) & 31) + e]));
            }
            const float tmax = sl2 * fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
            if (j == 0) x0 = __uint_as_float(sr[0][0]) * sl2;
            // (a row with no visible key in this tile keeps m; -inf - -inf never reaches exp2)
            const float m_new = fmaxf(m, tmax);
            if (j == 0) {
                m = m_new;
            } else if (__any_sync(0xffffffffu, m_new > m + kRescaleThreshold)) {
                // PV_t(j-1) is complete (S_t(j)'s commit covers it): rescale O_t in place.
                const float alpha = ex2_approx(m - m_new);
#pragma unroll
                for (int cb = 0; cb < kHD / 32; ++cb) {
                    uint32_t orr[32];
                    tmem_ld32(tO + cb * 32, orr);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                    tmem_st32(tO + cb * 32, orr);
                }
                l *= alpha;
                m = m_new;
            }
            // P = exp2(s * scale - m): packed bf16 pairs written over S_t[0, 64) for the PV MMA
            const float neg_m = -m;
            float2 rs[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) rs[e] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c][e]), sl2, neg_m));
                    const float p1 = ex2_approx(fmaf(__uint_as_float(sr[c][e + 1]), sl2, neg_m));
                    rs[(e >> 1) & 3] = __fadd2_rn(rs[(e >> 1) & 3], make_float2(p0, p1));
                    pk[e >> 1] = pack_bf16x2(p0, p1);
                }
                tmem_st16(tS + c * 16, pk);
            }
            l += ((rs[0].x + rs[0].y) + (rs[1].x + rs[1].y)) + ((rs[2].x + rs[2].y) + (rs[3].x + rs[3].y));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) pair::arrive_remote(p_full_e);   // one arrival per warp, 8 per slot and step
        }

        if (ok && nkv > 0) ok = pair::wait(&g_full[t], g_base & 1, ab, args.ctl);
        tc_fence_after();
        // Every thread of this warpgroup takes the same branch (the epilogue has named barriers).
        const bool ok_epi = named_bar_and(1 + t, 128, ok && nkv > 0);
        ok = named_bar_and(1 + t, 128, ok);
        if (ok_epi) {
            // ---- epilogue: out = O / l (.) sigmoid(gate) -> bf16 -> global (one 2*d_k-byte row per thread)
            const float inv_l = 1.0f / l;
            float g_head = 1.0f;
            if (GATE == 1) {
                float gl = 0.f;
                if (i < args.Lq) {
                    const long rows = (long)args.B * args.Lq;
                    const long idx = ((long)b * args.Lq + i) * args.Hq + h;
                    for (int s = 0; s < args.gate_splits; ++s) gl += args.gate_part[s * rows * args.Hq + idx];
                }
                g_head = sigmoid_fast(gl);
            }
            const bool store = U.mine[t] && i < args.Lq;
            uint4* dst = reinterpret_cast<uint4*>(args.O + (((long)b * args.Lq + i) * args.Hq + h) * kHD);
#pragma unroll 1
            for (int cb = 0; cb < kHD / 32; ++cb) {
                uint32_t orr[32];
                tmem_ld32(tO + cb * 32, orr);
                uint32_t grr[32];
                if (GATE == 2) tmem_ld32(tS + cb * 32, grr);
                tmem_wait_ld();
                uint32_t packed[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float v0 = __uint_as_float(orr[e]) * inv_l;
                    float v1 = __uint_as_float(orr[e + 1]) * inv_l;
                    if (GATE == 2) {
                        v0 *= sigmoid_fast(__uint_as_float(grr[e]));
                        v1 *= sigmoid_fast(__uint_as_float(grr[e + 1]));
                    } else if (GATE == 1) {
                        v0 *= g_head;
                        v1 *= g_head;
                    }
                    packed[e / 2] = pack_bf16x2(v0, v1);
                }
                if (store) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[cb * 4 + q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                }
            }
            // TMEM is no longer needed by this tile: the pair's next unit may start
            tc_fence_before();
            named_bar_sync(1 + t, 128);
            if (row == 0) pair::arrive_remote(tmem_free_e);
            if (args.sink_part && U.mine[t]) {
                float p0 = (i < args.Lq) ? ex2_approx(x0 - m) * inv_l : 0.f;
#pragma unroll
                for (int sh = 16; sh > 0; sh >>= 1) p0 += __shfl_xor_sync(0xffffffffu, p0, sh);
                if (lane == 0) sred[t * 4 + qd] = p0;
                named_bar_sync(1 + t, 128);
                if (row == 0)
                    args.sink_part[((long)b * args.Hq + h) * args.n_qtiles + U.q0[t] / kTile] =
                        sred[t * 4] + sred[t * 4 + 1] + sred[t * 4 + 2] + sred[t * 4 + 3];
            }
        }
        if (!ok_epi) {   // no epilogue for this tile in this unit: nothing to read from TMEM
            named_bar_sync(1 + t, 128);
            if (row == 0) pair::arrive_remote(tmem_free_e);
        }
        sp_base += nkv;
        g_base += 1;
        }   // units
        tc_fence_before();
    }

    __syncthreads();
    pair::cluster_sync();   // no CTA leaves while the other may still reach its memory
    if (warp == 1) {
        tc_fence_after();
        pair::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host side

bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
              const cuuint32_t* box) {
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = encode_tiled_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                                   strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int GATE>
cudaError_t launch_pair_t(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt, cudaStream_t s) {
    using C = PairCfg;
    alignas(64) CUtensorMap tmQ, tmK, tmV, tmX, tmW;
    const cuuint64_t e = 2;
    {
        cuuint64_t d[4] = {(cuuint64_t)kHD, (cuuint64_t)p.Hq, (cuuint64_t)p.Lq, (cuuint64_t)p.B};
        cuuint64_t st[3] = {kHD * e, (cuuint64_t)p.Hq * kHD * e, (cuuint64_t)p.Lq * p.Hq * kHD * e};
        cuuint32_t box[4] = {64, 1, 128, 1};
        if (!make_map(&tmQ, p.Q, 4, d, st, box)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t d[4] = {(cuuint64_t)kHD, (cuuint64_t)p.Hkv, (cuuint64_t)p.Lk, (cuuint64_t)p.B};
        cuuint64_t st[3] = {kHD * e, (cuuint64_t)p.Hkv * kHD * e, (cuuint64_t)p.Lk * p.Hkv * kHD * e};
        cuuint32_t box_k[4] = {64, 1, 64, 1};     // half a key tile
        cuuint32_t box_v[4] = {64, 1, 128, 1};    // a key tile, half the columns
        if (!make_map(&tmK, p.K, 4, d, st, box_k)) return cudaErrorInvalidValue;
        if (!make_map(&tmV, p.V, 4, d, st, box_v)) return cudaErrorInvalidValue;
    }
    if (GATE == 2) {
        cuuint64_t d[3] = {(cuuint64_t)p.d_model, (cuuint64_t)p.Lq, (cuuint64_t)p.B};
        cuuint64_t st[2] = {(cuuint64_t)p.d_model * e, (cuuint64_t)p.Lq * p.d_model * e};
        cuuint32_t box[3] = {64, 128, 1};
        if (!make_map(&tmX, p.X, 3, d, st, box)) return cudaErrorInvalidValue;
        cuuint64_t dw[2] = {(cuuint64_t)p.Hq * kHD, (cuuint64_t)p.d_model};
        cuuint64_t sw[1] = {(cuuint64_t)p.Hq * kHD * e};
        cuuint32_t bw[2] = {64, 64};
        if (!make_map(&tmW, p.Wg, 2, dw, sw, bw)) return cudaErrorInvalidValue;
    } else {
        tmX = tmQ;  // unused
        tmW = tmQ;
    }
    PairArgs a;
    a.B = p.B;
    a.Lq = p.Lq;
    a.Lk = p.Lk;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.d_model = p.d_model;
    a.causal = p.causal;
    a.n_qtiles = (p.Lq + kTile - 1) / kTile;
    a.n_quads = (a.n_qtiles + 3) / 4;
    a.gate_part = (GATE == 1) ? reinterpret_cast<const float*>(ws + w.gate_part) : nullptr;
    a.gate_splits = w.gate_splits;
    a.sink_part = p.sink ? reinterpret_cast<float*>(ws + w.sink_part) : nullptr;
    a.O = static_cast<__nv_bfloat16*>(p.O);
    a.ctl.err = rt.err;
    a.ctl.limit_ns = rt.limit_ns;

    static int max_pairs = 0;  // per template instance: pairs that can be resident at once
    if (max_pairs == 0) {
        // The register split above only fits if the launch allocates enough
        // registers per thread; refuse to launch otherwise (it would not finish).
        cudaFuncAttributes fa;
        cudaError_t r = cudaFuncGetAttributes(&fa, prefill_pair_kernel<GATE>);
        if (r != cudaSuccess) return r;
        if (fa.numRegs < kRegsLaunchMin) return cudaErrorInvalidConfiguration;
        r = cudaFuncSetAttribute(prefill_pair_kernel<GATE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)C::SMEM_BYTES);
        if (r != cudaSuccess) return r;
        // A persistent grid must not exceed what is resident at once: pairs
        // need two SMs of one GPC, so this can be below half the SM count.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(rt.num_sms & ~1));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        int n = 0;
        r = cudaOccupancyMaxActiveClusters(&n, prefill_pair_kernel<GATE>, &cfg);
        if (r != cudaSuccess) return r;
        if (n < 1) return cudaErrorInvalidConfiguration;
        max_pairs = n;
    }
    const long units = (long)a.n_quads * p.Hq * p.B;
    const long pairs = units < max_pairs ? units : max_pairs;
    prefill_pair_kernel<GATE><<<(unsigned)(2 * pairs), kThreads, C::SMEM_BYTES, s>>>(tmQ, tmK, tmV, tmX, tmW, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_pair_bf16(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                     cudaStream_t s) {
    if (p.gate_mode == 2) return launch_pair_t<2>(p, w, ws, rt, s);
    if (p.gate_mode == 1) return launch_pair_t<1>(p, w, ws, rt, s);
    return launch_pair_t<0>(p, w, ws, rt, s);
}

}  // namespace gsdpa
