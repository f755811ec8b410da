// prefill_pair_sm103.cu -- bf16 gated attention forward for d_k = 128 on pairs
// of SMs (clusters of two CTAs) sharing M = 256 tcgen05 MMAs.
//
// A pair computes one unit (b, h, 256 query rows): query tile 2u sits in the
// even CTA and tile 2u+1 in the odd one, stacked into the 256-row A operand
// of every MMA. The key tiles j = 0, 1, 2, ... of the unit alternate between
// two softmax warpgroups (p = j mod 2), each with its own score buffer S_p,
// output accumulator O_p and running row max m_p / row sum l_p:
//   S_p  = Q K_j^T                          tcgen05.mma.cta_group::2, A and B in smem
//   P_p  = exp2(S_p log2(e)/sqrt(d_k) - m_p)  online softmax of warpgroup p
//   O_p += P_p V_j                          tcgen05.mma.cta_group::2, P read from TMEM
// and the epilogue merges the two halves of the key range (with m = max(m_0, m_1)),
//   O = (2^(m_0-m) O_0 + 2^(m_1-m) O_1) / (2^(m_0-m) l_0 + 2^(m_1-m) l_1),
// multiplies by the gate g and stores bf16 rows, where g = sigma(X W_g)
// (elementwise, fp16, computed ahead by the gate GEMM) or sigma(x_i . w_h)
// (headwise, logits computed ahead).
// ("GatedAttention [2025]", sec. 1.2.1 SDPA and sec. 1.2.2 the gate
//  Y' = Y (.) sigma(X W); "10 . 门控", sec. 3.2: G1 gates each head's SDPA
//  output before the heads are concatenated.) The ungated output never leaves
//  the SM. Splitting the key range and merging the partial results is exact
//  (the merge is the same rescaling the online softmax applies tile by tile).
//
// Why two warpgroups over alternating key tiles: the QK MMA of key tile j+2
// needs only S_p free (P_p(j) consumed by its PV MMA, queued before it), so it
// runs while the other warpgroup computes the softmax of tile j+1. Each
// softmax has the MMAs of two key tiles to hide behind, where one tile's
// worth (two query tiles sharing one S buffer each) left the tensor pipe idle
// whenever a softmax took longer than the other tile's MMAs.
//
// Why pairs: a single-CTA 128 x 128 x 16 MMA reads 8 KB of operands from
// shared memory in its 64 cycles, the whole shared-memory bandwidth of the
// SM, and the K/V copies arriving in the same memory then stall it. In a
// pair each SM reads its own 128 A rows and only half of B (6 KB per 64
// cycles), each CTA loads only half of every K and V tile, and one thread
// issues the MMAs of both SMs.
//
// Operand split. K_j [128 keys x 128]: the even CTA holds keys 0..63, the odd
// CTA keys 64..127 (the N half of the S MMA). V_j [128 keys x 128]: the even
// CTA holds columns 0..63, the odd one columns 64..127 (the N half of the PV
// MMA). Q and P (A operands) stay with the CTA whose rows they are.
//
// Warp roles (384 threads per CTA):
//   warp 0       TMA producer of this CTA's halves (both CTAs);
//   warp 1       TMEM allocation (both CTAs, collectively); in the even CTA it
//                also issues every MMA and commit of the pair;
//   warps 2, 3   spare;
//   warps 4..7   softmax of the even key tiles, epilogue of output columns 0..63;
//   warps 8..11  softmax of the odd key tiles, epilogue of output columns 64..127.
// Barriers the issuing thread waits on (ring stages full, Q loaded, P
// written) live in the even CTA; the odd CTA reaches them through cluster
// addresses. The copies of both CTAs complete their bytes on the even CTA's
// barriers, and the even CTA alone arms them with the byte count of both
// halves (the odd CTA's bytes may land first: a barrier's pending byte count
// may go below zero until it is armed). MMA completions (S ready, ring stages
// free, unit done) are multicast to both CTAs.
//
// TMEM (512 columns, same layout in both CTAs): S_0 [0,128) S_1 [128,256)
// O_0 [256,384) O_1 [384,512); P_p packed bf16 in S_p [0,64).
//
// Causal mask aligned bottom-right (query i at absolute position
// L_k - L_q + i). A unit runs over the key tiles its odd CTA's rows can see;
// the even CTA's rows mask the extra tile. Persistent grid: the even CTA's
// producer claims the next unit from a counter in global memory (units
// numbered heaviest first: a longest-first greedy schedule) and hands it to
// every role of both CTAs through a small ring in shared memory.
#include "gsdpa_internal.h"
#include "sm103_pair.cuh"
#include "sm103_ptx.cuh"
#include "gate_fn.cuh"
#include "proj_internal.h"

#include <cmath>
#include <cuda_fp16.h>

namespace gsdpa {
namespace {

constexpr int kTile = 128;           // query rows per CTA tile, keys per K/V tile
constexpr int kHD = 128;
constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
// Register split: warpgroup 0 (producer, MMA, spare) gives registers to the
// two softmax warpgroups. The launch must provide 384 x kRegsLaunchMin.
constexpr int kRegsLow = 64;
constexpr int kRegsHigh = 216;
constexpr int kRegsLaunchMin = (kRegsLow * 128 + kRegsHigh * 256 + 383) / 384;

struct PairCfg {
    static constexpr uint32_t Q_BYTES = kTile * kHD * 2;      // this CTA's query tile
    static constexpr uint32_t HALF_BYTES = 64 * kHD * 2;      // K half (64 keys) or V half (64 columns)
    // A ring stage holds what one step of the MMA issue consumes: V_j and K_{j+2}
    // (the first stage of a unit: K_0 and K_1), one barrier wait per key tile.
    static constexpr uint32_t STAGE_BYTES = 2 * HALF_BYTES;
    static constexpr int NS = 5;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_RING = Q_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_RING + NS * STAGE_BYTES;
    static constexpr int NBAR = 2 * NS + 11;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    // misc: TMEM address, abort flag, (unused), unit ring [4]; then the
    // row statistics (m, l) of both warpgroups [2][128] for the merge, and
    // their partial sums of squares [2][128] (per-head RMSNorm)
    static constexpr uint32_t OFF_STATS = OFF_MISC + 64;
    static constexpr uint32_t OFF_SQ = OFF_STATS + 2 * 128 * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_SQ + 2 * 128 * 4 + 1024;  // + alignment slack
};

struct PairArgs {
    int B, Lq, Lk, Hq, Hkv, d_model, causal, n_qtiles, n_blk;
    const float* gate_part;  // headwise family: logit partials [splits, B*Lq, ge.l_cols]
    int gate_splits;
    const __half* gate_sig;  // elementwise family: the gate's values (row stride ge.g_rs, head stride ge.g_hs)
    GateEpi ge;              // gate function and the gate's layout
    GateStats gs;            // gate statistics (headwise gate), or none
    int* sched_counter;      // next unit to claim (0 at launch)
    unsigned long long* sink_word;  // [B, Hq] first-token share, fixed point + arrivals (0 at launch), or null
    float* sink;                    // [B, Hq] out
    float sink_scale;               // 2^F
    double sink_inv;                // 2^-F / L_q
    int sink_arrivals;              // 4 warps per 128-row query tile
    float* lse;                     // [B, Hq, Lq] or null
    __nv_bfloat16* O;        // [B, Lq, Hq, d_k]
    WaitCtl ctl;
};


template <int GATE, bool ADD>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
prefill_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const PairArgs args) {
    using C = PairCfg;
    extern __shared__ uint8_t smem_raw[];
    // (both CTAs run the same code, so this offset -- which the MMA
    // descriptors of the even CTA also use for the odd one -- is the same)
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + C::OFF_Q;
    uint8_t* ring = smem + C::OFF_RING;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* full = bars;                  // [NS] even CTA: both halves of a ring item landed
    uint64_t* empty = bars + C::NS;         // [NS] both: the MMAs reading the item completed
    uint64_t* q_full = bars + 2 * C::NS;    // even: both CTAs' query tiles landed
    uint64_t* s_full = q_full + 1;          // [2] both: S_p complete (and every earlier MMA)
    uint64_t* p_full = q_full + 3;          // [2] even: the 8 warps of warpgroup p (both CTAs) wrote P_p
    uint64_t* g_full = q_full + 5;          // both: every MMA of the unit complete
    uint64_t* drain = q_full + 6;           // even
    uint64_t* sched_full = q_full + 7;      // [4] both: unit r published in sched[r % 4]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    int* abort_word = reinterpret_cast<int*>(smem + C::OFF_MISC + 4);
    volatile int* abort_flag = abort_word;
    volatile int* sched = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 48);  // [4]
    float2* stats = reinterpret_cast<float2*>(smem + C::OFF_STATS);                   // [2][128]
    float* sq = reinterpret_cast<float*>(smem + C::OFF_SQ);                           // [2][128]

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = pair::cta_rank();
    const pair::PairAbort ab{abort_flag, pair::map_to(abort_word, rank ^ 1u)};

    // ---- units (b, h, block of 256 query rows), numbered heaviest first
    // (last query block first when causal)
    const int per_blk = args.Hq * args.B;
    const int n_units = args.n_blk * per_blk;
    const long off = (long)args.Lk - args.Lq;
    struct Unit {
        int h, b, kvh, nkv;
        int q0;        // first row of this CTA's query tile
        bool mine;     // this CTA's tile has rows
        int tiles;     // query tiles with rows in the pair (1 or 2)
    };
    auto decode_unit = [&](int u) -> Unit {
        Unit x;
        const int blk = args.causal ? (args.n_blk - 1 - u / per_blk) : (u / per_blk);
        const int rem = u % per_blk;
        x.h = rem % args.Hq;
        x.b = rem / args.Hq;
        x.kvh = x.h / (args.Hq / args.Hkv);
        const int lo = blk * 2 * kTile;                       // the even CTA's tile
        x.q0 = lo + (int)rank * kTile;
        x.mine = x.q0 < args.Lq;
        x.tiles = (lo + kTile < args.Lq) ? 2 : 1;
        const int last = (x.tiles == 2) ? lo + kTile : lo;    // the pair's last tile with rows
        long kend = args.Lk;
        if (args.causal) {
            const long e = off + last + kTile;                // keys 0 .. off+last+127 can be visible
            kend = e < kend ? e : kend;
        }
        x.nkv = (int)((kend + kTile - 1) / kTile);
        return x;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(q_full, 1);
        for (int p = 0; p < 2; ++p) {
            mbar_init(&s_full[p], 1);
            mbar_init(&p_full[p], 8);
        }
        mbar_init(g_full, 1);
        mbar_init(drain, 1);
        for (int k = 0; k < 4; ++k) mbar_init(&sched_full[k], 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
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
            int item = 0;   // running count of ring items: phases carry over units
            const uint32_t q_full_e = pair::map_to(q_full, 0);
            for (int r = 0; ok; ++r) {
            // the even CTA claims the next unit and publishes it in both CTAs (the
            // slot's previous unit, r - 4, was read long ago: both producers have
            // seen every MMA of unit r - 2 complete); the odd CTA takes it from there
            int uix;
            if (rank == 0) {
                uix = atomicAdd(args.sched_counter, 1);
                sched[r & 3] = uix;
                pair::store_remote_u32(pair::map_to(const_cast<int*>(&sched[r & 3]), 1), (uint32_t)uix);
                mbar_arrive(&sched_full[r & 3]);
                pair::arrive_remote_release(pair::map_to(&sched_full[r & 3], 1));
            } else {
                if (!(ok = pair::wait_acquire_cluster(&sched_full[r & 3], (r >> 2) & 1, ab, args.ctl))) break;
                uix = sched[r & 3];
            }
            if (uix >= n_units) {
                // no unit left for this CTA: the next kernel on the stream may be
                // scheduled (it waits for this grid to complete before it touches memory)
                pdl_trigger();
                break;
            }
            const Unit U = decode_unit(uix);
            // the previous unit's QK MMAs have read Q (its g_full commit covers every MMA)
            if (r > 0 && !(ok = pair::wait(g_full, (r - 1) & 1, ab, args.ctl))) break;
            if (rank == 0) mbar_arrive_expect_tx(q_full, (uint32_t)U.tiles * C::Q_BYTES);
            if (U.mine) pair::tma_load_5d(sQ, &tmQ, 0, U.h, U.q0, U.b, 0, q_full_e);
            // ring stages in the order the MMAs consume them: [K_0 | K_1], then [V_j | K_{j+2}]
            // (halves: V_j all 128 keys x columns [64 rank, 64 rank + 64); K_j keys
            // [64 rank, 64 rank + 64) x all columns; a missing K_1 / K_{j+2} is not loaded)
            auto load = [&](int v, int k0, int k1) -> bool {
                const int s = item % C::NS;
                const uint32_t ph = (item / C::NS) & 1;
                if (!pair::wait(&empty[s], ph ^ 1u, ab, args.ctl)) return false;
                const int halves = (v >= 0) + (k0 >= 0) + (k1 >= 0);
                if (rank == 0) mbar_arrive_expect_tx(&full[s], 2u * halves * C::HALF_BYTES);   // both CTAs' bytes
                const uint32_t fb = pair::map_to(&full[s], 0);
                uint8_t* st = ring + s * C::STAGE_BYTES;
                if (v >= 0) pair::tma_load_4d(st, &tmV, (int)rank * 64, U.kvh, v * kTile, U.b, fb);
                if (k0 >= 0) pair::tma_load_5d(st, &tmK, 0, U.kvh, k0 * kTile + (int)rank * 64, U.b, 0, fb);
                if (k1 >= 0)
                    pair::tma_load_5d(st + C::HALF_BYTES, &tmK, 0, U.kvh, k1 * kTile + (int)rank * 64, U.b, 0, fb);
                ++item;
                return true;
            };
            // stage 0: K_0 in the first half, K_1 in the second; stage j + 1: V_j, K_{j+2}
            ok = load(-1, 0, U.nkv > 1 ? 1 : -1);
            for (int j = 0; j < U.nkv && ok; ++j) ok = load(j, -1, j + 2 < U.nkv ? j + 2 : -1);
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
            constexpr uint32_t HI = desc_sw128_hi(1024);   // every operand: 8-row groups 1024 B apart
            const uint32_t sQa = smem_u32(sQ), ringa = smem_u32(ring);
            int it = 0;                    // running ring-item count
            int sp[2] = {0, 0};            // completed s_full / p_full phases per buffer
            auto take = [&]() -> int {     // wait for the next ring item; returns its stage
                const int s = it % C::NS;
                if (!__all_sync(0xffffffffu, pair::wait(&full[s], (it / C::NS) & 1, ab, args.ctl))) return -1;
                tc_fence_after();
                return s;
            };
            auto release = [&](int s) {    // the MMAs just issued are the last readers of stage s
                pair::commit_both(&empty[s]);
                ++it;
            };
            auto issue_S = [&](int p, int s, uint32_t k_off) {
                const uint32_t a0 = desc_sw128_lo(sQa, 16);
                const uint32_t b0 = desc_sw128_lo(ringa + s * C::STAGE_BYTES + k_off, 16);
                // K-major, 64-column blocks: Q blocks are 128 rows (16 KB), K halves 64 rows (8 KB)
                pair::mma_ss_k128<16384, 8192>(tmem + p * 128, a0, b0, HI, idS, 0);
                pair::commit_both(&s_full[p]);
            };
            auto issue_PV = [&](int p, int s, bool acc) {
                // V half: MN-major, one 64-column block; 16 keys = 2 KB per K step
                const uint32_t v0 = desc_sw128_lo(ringa + s * C::STAGE_BYTES, 8192);
                pair::mma_ts_k128(tmem + 256 + p * 128, tmem + p * 128, v0, HI, idO, acc ? 1u : 0u);
            };

            for (int r = 0; ok; ++r) {
            if (!(ok = __all_sync(0xffffffffu, pair::wait(&sched_full[r & 3], (r >> 2) & 1, ab, args.ctl)))) break;
            const int uix = sched[r & 3];
            if (uix >= n_units) break;
            const Unit U = decode_unit(uix);
            const int nkv = U.nkv;
            // (S_0 / S_1 are free: the previous unit's last PV MMAs, queued before
            // these, have read its last P. O_p is not written before PV(p) of this
            // unit, which waits for P_p from threads that first finished the
            // previous unit's epilogue -- so these QK MMAs overlap that epilogue.)
            ok = __all_sync(0xffffffffu, pair::wait(q_full, r & 1, ab, args.ctl));
            tc_fence_after();
            int s;
            if (ok && (ok = (s = take()) >= 0)) {                               // [K_0 | K_1]
                issue_S(0, s, 0);
                if (nkv > 1) issue_S(1, s, C::HALF_BYTES);
                release(s);
            }
            for (int j = 0; j < nkv && ok; ++j) {
                const int p = j & 1;
                if (!(ok = (s = take()) >= 0)) break;                          // [V_j | K_{j+2}]
                if (!(ok = __all_sync(0xffffffffu,
                                      pair::wait(&p_full[p], (sp[p] + (j >> 1)) & 1, ab, args.ctl))))
                    break;
                tc_fence_after();
                issue_PV(p, s, j >= 2);
                if (j + 2 < nkv) issue_S(p, s, C::HALF_BYTES);
                release(s);
            }
            if (ok) pair::commit_both(g_full);   // every MMA of the unit issued: signal on completion
            sp[0] += (nkv + 1) >> 1;
            sp[1] += nkv >> 1;
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
        const int p = (warp - 4) >> 2;         // key-tile parity of this warpgroup
        const int qd = warp & 3;               // TMEM lane quadrant of this warp
        const int row = qd * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const uint32_t tS = tmem + lane_base + p * 128;
        const uint32_t tOp = tmem + lane_base + 256 + p * 128;   // this warpgroup's accumulator
        const uint32_t tO0 = tmem + lane_base + 256;
        const uint32_t tO1 = tmem + lane_base + 384;
        const uint32_t p_full_e = pair::map_to(&p_full[p], 0);
        const float sl2 = kLog2e / sqrtf((float)kHD);
        bool ok = true;
        int sp = 0;          // completed s_full[p] / p_full[p] phases
        for (int r = 0; ok; ++r) {
        // (both warpgroups leave together or not at all: the merge has named barriers)
        ok = named_bar_and(1, 256, pair::wait_acquire_cluster(&sched_full[r & 3], (r >> 2) & 1, ab, args.ctl));
        if (!ok) break;
        const int uix = sched[r & 3];
        if (uix >= n_units) break;
        const int nkv = decode_unit(uix).nkv;
        const long a_pos = off + decode_unit(uix).q0 + row;
        float m = -INFINITY, l = 0.f, x0 = 0.f;

        int c = 0;   // key tiles of this warpgroup processed in this unit
        for (int jj = p; jj < nkv; jj += 2, ++c) {
            ok = __all_sync(0xffffffffu, pair::wait(&s_full[p], (sp + c) & 1, ab, args.ctl));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, sr[q]);
            tmem_wait_ld();

            const int kv0 = jj * kTile;
            // last visible column of this row in this key tile (>= 127: no mask)
            long lim_l = (long)args.Lk - 1 - kv0;
            if (args.causal && a_pos - kv0 < lim_l) lim_l = a_pos - kv0;
            const int lim = lim_l > 127 ? 127 : (lim_l < -1 ? -1 : (int)lim_l);
            // raw scores; masked ones become -inf (the 1/sqrt(d_k)*log2(e) scale is
            // folded into the exp2 argument below, max commutes with it)
            if (lim < 127) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (q * 32 + e > lim) sr[q][e] = __float_as_uint(-INFINITY);
            }
            // tile row max (scaled to log2 units; the scale is folded into the exp2 argument)
            auto tile_max = [&]() -> float {
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
                return sl2 * fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
            };
            // P = exp2(s * scale - mref): packed bf16 pairs written over S_p[0, 64) for
            // the PV MMA; returns the row sum of P (a row with no visible key so far,
            // mref = -inf, has all scores -inf and P = 0)
            auto exps = [&](float mref) -> float {
                const float neg_m = (mref == -INFINITY) ? 0.f : -mref;
                // (both exponent arguments of a column pair in one packed fused multiply-add)
                const float2 sl2x2 = make_float2(sl2, sl2), nm2 = make_float2(neg_m, neg_m);
                float2 rs[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) rs[e] = make_float2(0.f, 0.f);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float2 x = __ffma2_rn(
                            make_float2(__uint_as_float(sr[q][e]), __uint_as_float(sr[q][e + 1])), sl2x2, nm2);
                        const float p0 = ex2_approx(x.x);
                        const float p1 = ex2_approx(x.y);
                        rs[(e >> 1) & 3] = __fadd2_rn(rs[(e >> 1) & 3], make_float2(p0, p1));
                        pk[e >> 1] = pack_bf16x2(p0, p1);
                    }
                    tmem_st16(tS + q * 16, pk);
                }
                return ((rs[0].x + rs[0].y) + (rs[1].x + rs[1].y)) + ((rs[2].x + rs[2].y) + (rs[3].x + rs[3].y));
            };
            if (jj == 0) x0 = __uint_as_float(sr[0][0]) * sl2;
            float rsum;
            if (c == 0) {
                m = tile_max();
                rsum = exps(m);
            } else {
                // The running max m is raised only when a tile's max exceeds it by more
                // than 2^8 (log2 units), so the exponentials usually need only m: compute
                // them against it while the tile max is reduced alongside, and redo them
                // in the rare case that the max must move (before P is released).
                rsum = exps(m);
                const float tmax = tile_max();
                if (__any_sync(0xffffffffu, tmax > m + kRescaleThreshold)) {
                    const float m_new = fmaxf(m, tmax);
                    // PV(jj-2) is complete (S_p(jj)'s commit covers it): rescale O_p in place.
                    const float alpha = ex2_approx(m - m_new);
#pragma unroll
                    for (int cb = 0; cb < kHD / 32; ++cb) {
                        uint32_t orr[32];
                        tmem_ld32(tOp + cb * 32, orr);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                        tmem_st32(tOp + cb * 32, orr);
                    }
                    l *= alpha;
                    m = m_new;
                    rsum = exps(m);
                }
            }
            l += rsum;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) pair::arrive_remote(p_full_e);   // one arrival per warp, 8 per phase
        }
        sp += (nkv + 1 - p) >> 1;
        // (the unit is decoded again from its ring slot, valid until unit r + 4 is
        // claimed, so that none of its fields stays live through the loop above)
        const Unit U = decode_unit(sched[r & 3]);
        const int h = U.h, b = U.b;
        const int i = U.q0 + row;

        // elementwise gate: this row's 64 values of sigma(X W_g) for this warpgroup's
        // output columns, loaded before the last MMAs complete (hides the L2 latency)
        uint4 gq[GATE == 2 ? 8 : 1];
        if ((GATE == 1 || GATE == 2) && r == 0) pdl_wait();   // the gate kernel has completed (once per thread)
        if (GATE == 2) {
            if (U.mine && i < args.Lq) {
                const uint4* gsrc = reinterpret_cast<const uint4*>(
                    args.gate_sig + ((long)b * args.Lq + i) * args.ge.g_rs + (long)h * args.ge.g_hs + p * 64);
#pragma unroll
                for (int q = 0; q < 8; ++q) gq[q] = __ldg(gsrc + q);
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) gq[q] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (ok) ok = pair::wait(g_full, r & 1, ab, args.ctl);
        tc_fence_after();
        stats[p * 128 + row] = make_float2(m, l);
        // Both warpgroups take the same branch (the merge reads both accumulators).
        ok = named_bar_and(1, 256, ok);
        if (ok) {
            // ---- merge the two key halves, gate, bf16, this warpgroup's 64 output columns
            const float2 o = stats[(p ^ 1) * 128 + row];
            float mm = fmaxf(m, o.x);
            if (mm == -INFINITY) mm = 0.f;   // (rows past L_q only)
            const float a_me = (m == -INFINITY) ? 0.f : ex2_approx(m - mm);
            const float a_ot = (o.x == -INFINITY) ? 0.f : ex2_approx(o.x - mm);
            const float denom = l * a_me + o.y * a_ot;   // relative to 2^mm
            const float inv = 1.0f / denom;
            // log of the softmax denominator (natural log), from warpgroup 0
            if (args.lse && p == 0 && U.mine && i < args.Lq)
                args.lse[((long)b * args.Hq + h) * args.Lq + i] = (mm + log2f(denom)) * 0.6931471805599453f;
            const float s0 = (p == 0 ? a_me : a_ot) * inv;   // weight of O_0
            const float s1 = (p == 0 ? a_ot : a_me) * inv;   // weight of O_1
            const bool has1 = nkv > 1;                        // O_1 holds results only then
            // first-token share of this warp's 32 rows (key 0 lies in key tile 0, a tile of
            // warpgroup 0): added now, its result read after the stores
            unsigned long long sink_old = 0, sink_add = 0;
            const bool do_sink = args.sink_word && p == 0 && U.mine;
            if (do_sink) {
                float p0 = (i < args.Lq) ? ex2_approx(x0 - mm) * inv : 0.f;
#pragma unroll
                for (int sh = 16; sh > 0; sh >>= 1) p0 += __shfl_xor_sync(0xffffffffu, p0, sh);
                if (lane == 0) {
                    sink_add = sink_encode(p0, args.sink_scale);
                    sink_old = atomicAdd(args.sink_word + (long)b * args.Hq + h, sink_add);
                }
            }
            const int fn = args.ge.fn;
            constexpr bool add = ADD;   // the gate's value is added (else multiplied)
            float g_head = 1.0f;
            if (GATE == 1) {
                float gl = 0.f;
                if (U.mine && i < args.Lq) {
                    const long rows = (long)args.B * args.Lq;
                    const long idx = ((long)b * args.Lq + i) * args.ge.l_cols + (long)h * args.ge.l_hs;
                    for (int sg = 0; sg < args.gate_splits; ++sg)
                        gl += args.gate_part[sg * rows * args.ge.l_cols + idx];
                }
                g_head = gate_value(gl, fn);
                // (both warpgroups hold the row: warpgroup 0 counts it)
                if (args.gs.out) gate_stats_warp(args.gs, g_head, p == 0 && U.mine && i < args.Lq);
            }
            // per-head RMSNorm (no gate): this warpgroup's 64 columns' sum of squares,
            // exchanged with the other warpgroup's through shared memory
            float rr = 1.0f;
            const __nv_bfloat16* gamma = nullptr;
            if (GATE == 4) {
                float ss = 0.f;
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    const int col = p * 64 + cb * 16;
                    uint32_t r0[16], r1[16];
                    tmem_ld16(tO0 + col, r0);
                    if (has1) tmem_ld16(tO1 + col, r1);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float v = __uint_as_float(r0[e]) * s0;
                        if (has1) v = fmaf(__uint_as_float(r1[e]), s1, v);
                        ss = fmaf(v, v, ss);
                    }
                }
                sq[p * 128 + row] = ss;
                named_bar_sync(1, 256);
                rr = rsqrtf((ss + sq[(p ^ 1) * 128 + row]) / kHD + args.ge.eps);
                gamma = static_cast<const __nv_bfloat16*>(args.ge.gamma);
                if (gamma) gamma += (long)h * kHD + p * 64;
            }
            const bool store = U.mine && i < args.Lq;
            uint4* dst = reinterpret_cast<uint4*>(args.O + (((long)b * args.Lq + i) * args.Hq + h) * kHD + p * 64);
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                const int col = p * 64 + cb * 16;
                uint32_t r0[16], r1[16];
                tmem_ld16(tO0 + col, r0);
                if (has1) tmem_ld16(tO1 + col, r1);
                uint32_t gmw[8];   // RMSNorm scale of these 16 columns (bf16 pairs)
                if (GATE == 4) {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const uint4 w4 = gamma ? __ldg(reinterpret_cast<const uint4*>(gamma + cb * 16) + q)
                                               : make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
                        gmw[4 * q] = w4.x;
                        gmw[4 * q + 1] = w4.y;
                        gmw[4 * q + 2] = w4.z;
                        gmw[4 * q + 3] = w4.w;
                    }
                }
                tmem_wait_ld();
                uint32_t packed[8];
                const float2 s02 = make_float2(s0, s0), s12 = make_float2(s1, s1);
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    // column pairs in packed arithmetic (the same roundings as one at a time)
                    float2 v = __fmul2_rn(make_float2(__uint_as_float(r0[e]), __uint_as_float(r0[e + 1])), s02);
                    if (has1) v = __ffma2_rn(make_float2(__uint_as_float(r1[e]), __uint_as_float(r1[e + 1])), s12, v);
                    if (GATE == 2) {
                        // columns cb*16 + e, + 1 of this half: half2 number (e/2) % 4 of uint4 cb*2 + e/8
                        const uint32_t hw = (&gq[cb * 2 + (e >> 3)].x)[(e >> 1) & 3];
                        const float2 g2 = __half22float2(*reinterpret_cast<const __half2*>(&hw));
                        v = add ? __fadd2_rn(v, g2) : __fmul2_rn(v, g2);
                    } else if (GATE == 1) {
                        const float2 g2 = make_float2(g_head, g_head);
                        v = add ? __fadd2_rn(v, g2) : __fmul2_rn(v, g2);
                    }
                    float v0 = v.x, v1 = v.y;
                    if (GATE == 3) {   // SiLU of the output
                        v0 *= sigmoid_tanh(v0);
                        v1 *= sigmoid_tanh(v1);
                    } else if (GATE == 4) {
                        v0 *= rr * __uint_as_float(gmw[e >> 1] << 16);
                        v1 *= rr * __uint_as_float(gmw[e >> 1] & 0xffff0000u);
                    }
                    packed[e / 2] = pack_bf16x2(v0, v1);
                }
                if (store) {
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        dst[cb * 2 + q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                }
            }
            if (do_sink && lane == 0)
                sink_finish(sink_old, sink_add, args.sink_arrivals, args.sink_inv, args.sink + (long)b * args.Hq + h);
        }
        // both warpgroups have read O_0 and O_1 before either starts the next
        // unit (its first PV MMAs overwrite them)
        tc_fence_before();
        named_bar_sync(1, 256);
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

template <int GATE, bool ADD = false>
cudaError_t launch_pair_t(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt, cudaStream_t s,
                          bool pdl = true) {
    using C = PairCfg;
    alignas(64) CUtensorMap tmQ, tmK, tmV;
    const cuuint64_t e = 2;
    // [B, L, H, d] viewed as (64 columns, H, L, B, 2 column blocks): one request
    // loads a tile with both 64-column swizzled blocks
    {
        cuuint64_t d[5] = {64, (cuuint64_t)p.Hq, (cuuint64_t)p.Lq, (cuuint64_t)p.B, 2};
        cuuint64_t st[4] = {kHD * e, (cuuint64_t)p.Hq * kHD * e, (cuuint64_t)p.Lq * p.Hq * kHD * e, 128};
        cuuint32_t box[5] = {64, 1, 128, 1, 2};
        if (!make_map(&tmQ, p.Q, 5, d, st, box)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t d[5] = {64, (cuuint64_t)p.Hkv, (cuuint64_t)p.Lk, (cuuint64_t)p.B, 2};
        cuuint64_t st[4] = {kHD * e, (cuuint64_t)p.Hkv * kHD * e, (cuuint64_t)p.Lk * p.Hkv * kHD * e, 128};
        cuuint32_t box_k[5] = {64, 1, 64, 1, 2};     // half a key tile, all columns
        if (!make_map(&tmK, p.K, 5, d, st, box_k)) return cudaErrorInvalidValue;
        cuuint64_t dv[4] = {(cuuint64_t)kHD, (cuuint64_t)p.Hkv, (cuuint64_t)p.Lk, (cuuint64_t)p.B};
        cuuint32_t box_v[4] = {64, 1, 128, 1};       // a key tile, half the columns
        if (!make_map(&tmV, p.V, 4, dv, st, box_v)) return cudaErrorInvalidValue;
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
    a.n_blk = (a.n_qtiles + 1) / 2;
    a.gate_part = (GATE == 1) ? reinterpret_cast<const float*>(ws + w.gate_part) : nullptr;
    a.gate_splits = w.gate_splits;
    a.gate_sig = (GATE == 2) ? reinterpret_cast<const __half*>(ws + w.gate_sig) : nullptr;
    a.ge = gate_epi(p);
    a.gs = p.gate_mode == 1 ? p.stats : GateStats();
    a.sched_counter = reinterpret_cast<int*>(ws + w.state);
    set_sink_args(p, w, ws, a.n_qtiles, &a.sink_word, &a.sink, &a.sink_scale, &a.sink_inv, &a.sink_arrivals);
    a.lse = p.lse;
    a.O = static_cast<__nv_bfloat16*>(p.O);
    a.ctl.err = rt.err;
    a.ctl.limit_ns = rt.limit_ns;

    static PerDeviceSetup setup;   // per template instance; the value: pairs that can be resident at once
    int max_pairs = 0;
    const int num_sms = rt.num_sms;
    cudaError_t r0 = setup_once_per_device(setup, [num_sms](int& resident) {
        // The register split above only fits if the launch allocates enough
        // registers per thread; refuse to launch otherwise (it would not finish).
        cudaFuncAttributes fa;
        cudaError_t r = cudaFuncGetAttributes(&fa, prefill_pair_kernel<GATE, ADD>);
        if (r != cudaSuccess) return r;
        if (fa.numRegs < kRegsLaunchMin) return cudaErrorInvalidConfiguration;
        r = cudaFuncSetAttribute(prefill_pair_kernel<GATE, ADD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)C::SMEM_BYTES);
        if (r != cudaSuccess) return r;
        // A persistent grid must not exceed what is resident at once: pairs
        // need two SMs of one GPC, so this can be below half the SM count.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(num_sms & ~1));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        int n = 0;
        r = cudaOccupancyMaxActiveClusters(&n, prefill_pair_kernel<GATE, ADD>, &cfg);
        if (r != cudaSuccess) return r;
        if (n < 1) return cudaErrorInvalidConfiguration;
        resident = n;
        return cudaSuccess;
    }, &max_pairs);
    if (r0 != cudaSuccess) return r0;
    const long units = (long)a.n_blk * p.Hq * p.B;
    const long pairs = units < max_pairs ? units : max_pairs;
    // The kernel just before this one in the call (a gate kernel, or the
    // state-zeroing kernel when there is no gate) zeroes the per-call state and
    // then lets this one start early (programmatic dependent launch); with a
    // gate, the epilogues wait for that kernel to complete before reading it.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, prefill_pair_kernel<GATE, ADD>, tmQ, tmK, tmV, a);
}

}  // namespace

cudaError_t launch_prefill_pair_bf16_ordered(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                             cudaStream_t s) {
    if (p.gate_mode != 0 && p.gate_mode != 2) return cudaErrorInvalidValue;
    return p.gate_mode == 2 ? launch_pair_t<2>(p, w, ws, rt, s, false) : launch_pair_t<0>(p, w, ws, rt, s, false);
}

cudaError_t launch_prefill_pair_bf16(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                     cudaStream_t s) {
    const bool add = gate_template(p) != 0 && (p.gate_fn >= 2 && p.gate_fn <= 4);   // additive gates
    switch (gate_template(p)) {
    case 1: return add ? launch_pair_t<1, true>(p, w, ws, rt, s) : launch_pair_t<1>(p, w, ws, rt, s);
    case 2: return add ? launch_pair_t<2, true>(p, w, ws, rt, s) : launch_pair_t<2>(p, w, ws, rt, s);
    case 3: return launch_pair_t<3>(p, w, ws, rt, s);
    case 4: return launch_pair_t<4>(p, w, ws, rt, s);
    default: return launch_pair_t<0>(p, w, ws, rt, s);
    }
}

}  // namespace gsdpa
