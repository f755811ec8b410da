// prefill_sm103.cu -- bf16 gated attention forward on sm_103a tensor cores.
//
// One CTA computes one unit (b, h, pair of 128-row query tiles t = 0, 1):
//   S_t = Q_t K_j^T                      tcgen05.mma (A, B in shared memory)
//   P_t = exp2(S_t log2(e)/sqrt(d_k) - m_t)   online softmax, one thread per row
//   O_t += P_t V_j                       tcgen05.mma with P read from TMEM
//   out_t = O_t / l_t (.) g_t            epilogue: bf16 rows straight to HBM
// where g = sigma(X W_g) (elementwise gate, fp16, computed ahead by the gate
// GEMM) or sigma(x_i . w_h) (headwise gate, logits computed ahead).
// ("GatedAttention [2025]", sec. 1.2.1 SDPA and sec. 1.2.2 the gate
//  Y' = Y (.) sigma(X W); "10 . 门控", sec. 3.2: G1 gates each head's SDPA
//  output before the heads are concatenated.) The ungated output never leaves
//  the SM.
//
// Warp roles (384 threads):
//   warp 0       TMA producer: Q_0, Q_1 once, then K_0, V_0, K_1, V_1, ...
//                through a ring of NS shared-memory stages;
//   warp 1       TMEM allocation; issues every tcgen05.mma / commit (the
//                whole warp runs the loop, one elected lane issues);
//   warps 2, 3   spare;
//   warps 4..7   softmax + epilogue of query tile 0 (one thread per row);
//   warps 8..11  softmax + epilogue of query tile 1.
// Both query tiles consume the same K_j / V_j tiles, so each K/V tile is
// loaded once per 256 query rows. The MMA warp issues, per key tile j,
//   PV_0(j), S_0(j+1), PV_1(j), S_1(j+1)
// so that the tensor pipe works on one tile while the other tile's softmax
// runs. tcgen05.commit tracks every earlier MMA of the issuing thread, so once
// S_t(j) is complete PV_t(j-1) is complete too: the softmax may rescale O_t
// and overwrite S_t with P_t without further waits.
//
// TMEM (512 columns): S_0 [0,128)  S_1 [128,256)  O_0 [256,256+d_k)
//                     O_1 [384,384+d_k); P_t is packed bf16 in S_t [0,64).
//
// The causal mask is aligned bottom-right (query i at absolute position
// L_k - L_q + i); key tiles entirely above the diagonal are never loaded.
// The grid is persistent (one CTA per SM): each CTA's producer claims the
// next unit from a counter in global memory (units numbered heaviest first,
// so the claims form a longest-first greedy schedule that keeps the SMs
// evenly loaded, also when some CTAs start late) and hands it to the other
// roles through a small ring in shared memory; barrier phases carry over
// from one unit to the next.
#include "gsdpa_internal.h"
#include "sm103_ptx.cuh"
#include "gate_fn.cuh"
#include "proj_internal.h"

#include <cmath>
#include <cuda_fp16.h>

namespace gsdpa {
namespace {

// tcgen05.ld of 32 columns that also returns their maximum (the .red.max form):
// the tile's row maximum comes with the load instead of a pass over the scores.
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32], float& mx) {
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, %32, [%33];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=f"(mx)
        : "r"(taddr));
}

constexpr int kTile = 128;           // query rows per tile, keys per K/V tile
constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
// Register split: warpgroup 0 (producer, MMA, spare) gives registers to the
// two softmax warpgroups. The launch must provide 384 x kRegsLaunchMin.
constexpr int kRegsLow = 64;
constexpr int kRegsHigh = 216;
constexpr int kRegsLaunchMin = (kRegsLow * 128 + kRegsHigh * 256 + 383) / 384;

template <int HD, int GATE>
struct PrefillCfg {
    static constexpr uint32_t Q_BYTES = kTile * HD * 2;   // one query tile
    static constexpr uint32_t KV_BYTES = kTile * HD * 2;
    static constexpr uint32_t STAGE_BYTES = KV_BYTES;
    static constexpr int NS = (HD == 128) ? 4 : 8;
    static constexpr uint32_t OFF_Q = 0;                  // Q_0, Q_1
    static constexpr uint32_t OFF_RING = 2 * Q_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_RING + NS * STAGE_BYTES;
    // mbarriers: full[NS], empty[NS], then q_full, s_full[2], p_full[2],
    // g_full[2], drain, sched_full[4]
    static constexpr int NBAR_AFTER_RING = 12;
    static constexpr int NBAR = 2 * NS + NBAR_AFTER_RING;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    // output staging: per warpgroup two 8 KB buffers of 128 rows x 32 columns
    // (64-byte rows, 64-byte swizzle) that the TMA stores read
    static constexpr uint32_t STG_BYTES = kTile * 32 * 2;
    static constexpr uint32_t OFF_STG = (OFF_MISC + 64 + 1023) / 1024 * 1024;
    static constexpr uint32_t SMEM_BYTES = OFF_STG + 4 * STG_BYTES + 1024;  // + alignment slack
    static_assert(SMEM_BYTES <= 232448, "shared memory per block");
};

struct PrefillArgs {
    int B, Lq, Lk, Hq, Hkv, d_model, causal, n_qtiles, n_pairs;
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
    int sink_arrivals;              // 4 warps per query tile
    float* lse;                     // [B, Hq, Lq] or null
    __nv_bfloat16* out;             // O [B, Lq, Hq, HD] (the epilogue's direct stores)
    WaitCtl ctl;
};


// DIRECT: the epilogue stores O from registers as whole 32-byte sectors (O
// 32-byte aligned, no gate or the elementwise gate); otherwise it stages each
// 32-column chunk in shared memory for a bulk tensor copy.
template <int HD, int GATE, bool ADD, bool DIRECT>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
               const PrefillArgs args) {
    using C = PrefillCfg<HD, GATE>;
    static_assert(!DIRECT || GATE == 0 || GATE == 2, "direct stores only without a gate or with the elementwise one");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + C::OFF_Q;
    uint8_t* ring = smem + C::OFF_RING;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* full = bars;                 // [NS]
    uint64_t* empty = bars + C::NS;        // [NS]
    uint64_t* q_full = bars + 2 * C::NS;
    uint64_t* s_full = q_full + 1;         // [2] per query tile
    uint64_t* p_full = q_full + 3;         // [2]
    uint64_t* g_full = q_full + 5;         // [2]: every MMA of the unit done
    uint64_t* drain = q_full + 7;
    uint64_t* sched_full = q_full + 8;     // [4] unit r published in sched[r % 4]
    static_assert(8 + 4 == C::NBAR_AFTER_RING, "barrier layout");
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* sched = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 48);  // [4]

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    // ---- units, numbered heaviest first (last query pair first when causal)
    const int per_pair = args.Hq * args.B;
    const int n_units = args.n_pairs * per_pair;
    const long off = (long)args.Lk - args.Lq;
    struct Unit {
        int pr, h, b, kvh, nj;
        int q0[2], nkv[2];
        bool act[2];
    };
    auto decode_unit = [&](int u) -> Unit {
        Unit x;
        x.pr = args.causal ? (args.n_pairs - 1 - u / per_pair) : (u / per_pair);
        const int rem = u % per_pair;
        x.h = rem % args.Hq;
        x.b = rem / args.Hq;
        x.kvh = x.h / (args.Hq / args.Hkv);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            x.q0[t] = (2 * x.pr + t) * kTile;
            x.act[t] = x.q0[t] < args.Lq;
            long kend = args.Lk;
            if (args.causal) {
                const long last = off + x.q0[t] + kTile;  // keys 0 .. off+q0+127 can be visible
                kend = last < kend ? last : kend;
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
            mbar_init(&p_full[t], 128);
            mbar_init(&g_full[t], 1);
        }
        mbar_init(drain, 1);
        for (int k = 0; k < 4; ++k) mbar_init(&sched_full[k], 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // (each setmaxnreg sits inside the branch of the role it serves, so that
    // the compiler can give each role its own register budget)
    if (warp < 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == 0) {
        // ================================================================ TMA producer
        if (lane == 0) {
            uint32_t armed = 0, armed_phase = 0;
            bool ok = true;
            int item = 0;   // running count of ring items (phases carry over units)
            for (int r = 0; ok; ++r) {
            // claim the next unit and publish it to the MMA and softmax roles (the
            // slot's previous unit, r - 4, was read long ago: this thread has seen
            // every MMA of unit r - 2 complete)
            const int uix = atomicAdd(args.sched_counter, 1);
            sched[r & 3] = uix;
            mbar_arrive(&sched_full[r & 3]);
            if (uix >= n_units) {
                // no unit left for this CTA: the next kernel on the stream may be
                // scheduled (it waits for this grid to complete before it touches memory)
                pdl_trigger();
                break;
            }
            const Unit U = decode_unit(uix);
            const int h = U.h, b = U.b, kvh = U.kvh, nj = U.nj;
            const int* q0 = U.q0;
            const bool* act = U.act;
            // the previous unit's S MMAs have read Q: its g_full[1] commit is the
            // last of the unit and covers all of them
            if (r > 0 && !(ok = mbar_wait(&g_full[1], (r - 1) & 1, abort_flag, args.ctl))) break;
            mbar_arrive_expect_tx(q_full, (act[1] ? 2 : 1) * C::Q_BYTES);
            for (int t = 0; t < 2; ++t)
                if (act[t]) tma_load_5d(sQ + t * C::Q_BYTES, &tmQ, 0, h, q0[t], b, 0, q_full);

            auto acquire = [&](uint32_t bytes) -> uint8_t* {
                const int s = item % C::NS;
                const uint32_t ph = (item / C::NS) & 1;
                if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, args.ctl)) return nullptr;
                mbar_arrive_expect_tx(&full[s], bytes);
                armed |= 1u << s;
                armed_phase = (armed_phase & ~(1u << s)) | (ph << s);
                return ring + s * C::STAGE_BYTES;
            };
            for (int j = 0; j < nj && ok; ++j) {
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    uint8_t* st = acquire(C::KV_BYTES);
                    if (!st) { ok = false; break; }
                    tma_load_5d(st, kv ? &tmV : &tmK, 0, kvh, j * kTile, b, 0, &full[item % C::NS]);
                    ++item;
                }
            }
            }   // units
            if (!ok) {
                // Let every copy already issued land before the CTA can exit.
                volatile int never = 0;
                WaitCtl c2 = args.ctl;
                if (c2.limit_ns < 1000000000ull) c2.limit_ns = 1000000000ull;
                for (int s = 0; s < C::NS; ++s)
                    if (armed & (1u << s)) mbar_wait(&full[s], (armed_phase >> s) & 1u, &never, c2);
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        {   // the whole warp runs the issue loop (warp-uniform operands); one elected lane issues
            bool ok = true;
            constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t idO = idesc_bf16_f32(128, HD, false, true);
            const uint32_t sQa = smem_u32(sQ), ringa = smem_u32(ring);
            int ibase = 0;                 // running ring-item count
            int sp_base[2] = {0, 0};       // completed s_full / p_full phases per tile
            auto stage_addr = [&](int item) { return ringa + ((ibase + item) % C::NS) * C::STAGE_BYTES; };
            auto wait_full = [&](int item) -> bool {
                const int it = ibase + item;
                if (!__all_sync(0xffffffffu, mbar_wait(&full[it % C::NS], (it / C::NS) & 1, abort_flag, args.ctl)))
                    return false;
                tc_fence_after();
                return true;
            };
            constexpr uint32_t HI = desc_sw128_hi(1024);   // every operand: 8-row groups 1024 B apart
            auto issue_S = [&](int t, int j) {
                const uint32_t a0 = desc_sw128_lo(sQa + t * C::Q_BYTES, 16);
                const uint32_t b0 = desc_sw128_lo(stage_addr(2 * j), 16);
                if (HD == 128) {
                    // 128-row tiles: the second 64-column block of K lies 16 KB on
                    mma_ss_k128<16384, 16384>(tmem + t * 128, a0, b0, HI, idS, 0);
                } else {
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk)
                        mma_ss_elect(tmem + t * 128, a0 + kk * (32 >> 4), HI, b0 + kk * (32 >> 4), HI, idS, kk != 0);
                }
                mma_commit_elect(&s_full[t]);
            };
            auto issue_PV = [&](int t, int j) -> bool {
                if (!__all_sync(0xffffffffu, mbar_wait(&p_full[t], (sp_base[t] + j) & 1, abort_flag, args.ctl)))
                    return false;
                tc_fence_after();
                const uint32_t v0 = desc_sw128_lo(stage_addr(2 * j + 1), 16384);
                // 128 keys: eight K = 16 steps, P 8 TMEM columns and V 2 KB apart
                mma_ts_k128(tmem + 256 + t * 128, tmem + t * 128, v0, HI, idO, j != 0);
                return true;
            };

            for (int r = 0; ok; ++r) {
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&sched_full[r & 3], (r >> 2) & 1, abort_flag, args.ctl))))
                break;
            const int uix = sched[r & 3];
            if (uix >= n_units) break;
            const Unit U = decode_unit(uix);
            const int nj = U.nj;
            const int* nkv = U.nkv;
            const bool* act = U.act;
            // (the S columns are free: the previous unit's last PV MMAs, queued before
            // these, have read its last P. O_t is not written before PV_t(0), which
            // waits for P_t(0) from the threads that first finish the epilogue of the
            // previous unit -- so this unit's QK MMAs overlap that epilogue.)
            ok = __all_sync(0xffffffffu, mbar_wait(q_full, r & 1, abort_flag, args.ctl));
            tc_fence_after();
            if (ok) ok = wait_full(0);
            if (ok) {
                if (act[0]) issue_S(0, 0);
                if (act[1]) issue_S(1, 0);
                mma_commit_elect(&empty[ibase % C::NS]);
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
                    } else if (nkv[0] < nj) {
                        // tile 0 has fewer key tiles (causal): its epilogue need not
                        // wait for tile 1's last step
                        mma_commit_elect(&g_full[0]);
                    }
                }
                if (j < nkv[1]) {
                    if (!(ok = issue_PV(1, j))) break;
                }
                mma_commit_elect(&empty[(ibase + 2 * j + 1) % C::NS]);     // V_j done
                if (j + 1 < nkv[1]) {
                    if (!k_ready && !(ok = wait_full(2 * j + 2))) break;
                    k_ready = true;
                    issue_S(1, j + 1);
                }
                if (k_ready) mma_commit_elect(&empty[(ibase + 2 * j + 2) % C::NS]);  // K_{j+1} done
            }
            // every MMA of the unit issued: signal the epilogues (and the producer) on completion
            if (ok) {
                if (nkv[0] == nj) mma_commit_elect(&g_full[0]);
                mma_commit_elect(&g_full[1]);
            }
            ibase += 2 * nj;
            sp_base[0] += nkv[0];
            sp_base[1] += nkv[1];
            }   // units
            if (!ok) {
                // Gave up: let every MMA issued so far complete before TMEM is freed.
                volatile int never = 0;
                WaitCtl c2 = args.ctl;
                if (c2.limit_ns < 1000000000ull) c2.limit_ns = 1000000000ull;
                mma_commit_elect(drain);
                mbar_wait(drain, 0, &never, c2);
                __syncwarp();
            }
        }
    } else if (warp >= 4) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        // ================================================================ softmax + epilogue
        const int t = (warp - 4) / 4;
        const int qd = warp & 3;
        const int row = qd * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const uint32_t tS = tmem + lane_base + t * 128;
        const uint32_t tO = tmem + lane_base + 256 + t * 128;
        const float sl2 = kLog2e / sqrtf((float)HD);
        bool ok = true;
        int sp_base = 0;     // completed s_full / p_full phases of this tile
        int g_base = 0;      // completed g_full phases of this tile
        for (int r = 0; ok; ++r) {
        // (the warpgroup leaves together or not at all: its epilogue has named barriers)
        ok = named_bar_and(1 + t, 128, mbar_wait(&sched_full[r & 3], (r >> 2) & 1, abort_flag, args.ctl));
        if (!ok) break;
        const int uix = sched[r & 3];
        if (uix >= n_units) break;
        const Unit U = decode_unit(uix);
        const int h = U.h, b = U.b;
        // this warpgroup's tile, selected (not indexed by t) so that the unit
        // stays in registers
        const int my_q0 = t ? U.q0[1] : U.q0[0];
        const int my_nkv = t ? U.nkv[1] : U.nkv[0];
        const int i = my_q0 + row;
        const long a_pos = off + i;
        float m = -INFINITY, l = 0.f, x0 = 0.f;

        for (int j = 0; j < my_nkv; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t], (sp_base + j) & 1, abort_flag, args.ctl));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[4][32];
            float pmx[4];   // each 32-column load's maximum
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32_max(tS + c * 32, sr[c], pmx[c]);
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
            // tile row max: from the loads, or over the masked scores on the diagonal tiles
            float rmax = fmaxf(fmaxf(pmx[0], pmx[1]), fmaxf(pmx[2], pmx[3]));
            if (lim < 127) {
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
                rmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
            }
            const float tmax = sl2 * rmax;
            if (j == 0) x0 = __uint_as_float(sr[0][0]) * sl2;
            const float m_new = fmaxf(m, tmax);
            if (j == 0) {
                m = m_new;
            } else if (__any_sync(0xffffffffu, m_new > m + kRescaleThreshold)) {
                // PV_t(j-1) is complete (S_t(j)'s commit covers it): rescale O_t in place.
                const float alpha = ex2_approx(m - m_new);
#pragma unroll
                for (int cb = 0; cb < HD / 32; ++cb) {
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
            // (the softmax is bound by the instructions it issues: both exponent
            // arguments of a column pair come from one packed fused multiply-add)
            const float2 sl2x2 = make_float2(sl2, sl2), nm2 = make_float2(-m, -m);
            float2 rs[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) rs[e] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])),
                                                sl2x2, nm2);
                    const float p0 = ex2_approx(x.x);
                    const float p1 = ex2_approx(x.y);
                    rs[(e >> 1) & 3] = __fadd2_rn(rs[(e >> 1) & 3], make_float2(p0, p1));
                    pk[e >> 1] = pack_bf16x2(p0, p1);
                }
                tmem_st16(tS + c * 16, pk);
            }
            l += ((rs[0].x + rs[0].y) + (rs[1].x + rs[1].y)) + ((rs[2].x + rs[2].y) + (rs[3].x + rs[3].y));
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_full[t]);
        }

        // elementwise gate: this row's d_k values of sigma(X W_g), loaded before the
        // last MMAs complete so that the L2 / HBM latency hides behind the wait
        uint4 gq[GATE == 2 ? HD / 8 : 1];
        if ((GATE == 1 || GATE == 2) && r == 0) pdl_wait();   // the gate kernel has completed (once per thread)
        if (GATE == 2) {
            if (i < args.Lq && my_nkv > 0) {
                const uint4* gsrc = reinterpret_cast<const uint4*>(
                    args.gate_sig + ((long)b * args.Lq + i) * args.ge.g_rs + (long)h * args.ge.g_hs);
#pragma unroll
                // 256-bit loads, whole 32-byte sectors: the values live in the
                // workspace (256-byte aligned) in rows of a multiple of d_k halves
                for (int q = 0; q < HD / 16; ++q)
                    asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                                 : "=r"(gq[2 * q].x), "=r"(gq[2 * q].y), "=r"(gq[2 * q].z), "=r"(gq[2 * q].w),
                                   "=r"(gq[2 * q + 1].x), "=r"(gq[2 * q + 1].y), "=r"(gq[2 * q + 1].z), "=r"(gq[2 * q + 1].w)
                                 : "l"(gsrc + 2 * q));
            } else {
#pragma unroll
                for (int q = 0; q < HD / 8; ++q) gq[q] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (ok && my_nkv > 0) ok = mbar_wait(&g_full[t], g_base & 1, abort_flag, args.ctl);
        tc_fence_after();
        // Every thread of this warpgroup takes the same branch (the epilogue has named barriers).
        const bool ok_epi = named_bar_and(1 + t, 128, ok && my_nkv > 0);
        ok = named_bar_and(1 + t, 128, ok);
        if (ok_epi) {
            // ---- epilogue: out = O / l (.) gate -> bf16 -> global (one 2*d_k-byte row per thread)
            const float inv_l = 1.0f / l;
            // log of the softmax denominator (natural log; m and l are in log2 units)
            if (args.lse && i < args.Lq)
                args.lse[((long)b * args.Hq + h) * args.Lq + i] = (m + log2f(l)) * kLn2;
            // first-token share of this warp's 32 rows: added now, its result read after the stores
            unsigned long long sink_old = 0, sink_add = 0;
            if (args.sink_word) {
                float p0 = (i < args.Lq) ? ex2_approx(x0 - m) * inv_l : 0.f;
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
                if (i < args.Lq) {
                    const long rows = (long)args.B * args.Lq;
                    const long idx = ((long)b * args.Lq + i) * args.ge.l_cols + (long)h * args.ge.l_hs;
                    for (int s = 0; s < args.gate_splits; ++s)
                        gl += args.gate_part[s * rows * args.ge.l_cols + idx];
                }
                g_head = gate_value(gl, fn);
                if (args.gs.out) gate_stats_warp(args.gs, g_head, i < args.Lq);
            }
            // per-head RMSNorm (no gate): the row's mean square over its d_k columns first
            float rr = 1.0f;
            const __nv_bfloat16* gamma = nullptr;
            if (GATE == 4) {
                float ss = 0.f;
#pragma unroll 1
                for (int cb = 0; cb < HD / 32; ++cb) {
                    uint32_t orr[32];
                    tmem_ld32(tO + cb * 32, orr);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float v = __uint_as_float(orr[e]) * inv_l;
                        ss = fmaf(v, v, ss);
                    }
                }
                rr = rsqrtf(ss / HD + args.ge.eps);
                gamma = static_cast<const __nv_bfloat16*>(args.ge.gamma);
                if (gamma) gamma += (long)h * HD;
            }
            // 32 columns at a time: TMEM -> registers -> bf16 in a staging buffer ->
            // one TMA store of the tile's 128 rows (rows past L_q are clipped by the
            // tensor map; without a gate or with the elementwise gate, stores from
            // registers instead, below, when O is 32-byte aligned). The issuing
            // thread has seen the store two chunks back finish reading its buffer
            // before the barrier of the chunk in between.
            uint8_t* stg = smem + C::OFF_STG + t * 2 * C::STG_BYTES;
            const int sw = (row >> 1) & 3;   // 64-byte swizzle of this row's 16-byte pieces
#pragma unroll
            for (int cb = 0; cb < HD / 32; ++cb) {
                uint32_t orr[32];
                tmem_ld32(tO + cb * 32, orr);
                uint32_t gmw[16];   // RMSNorm scale of these 32 columns (bf16 pairs)
                if (GATE == 4) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 w4 = gamma ? __ldg(reinterpret_cast<const uint4*>(gamma + cb * 32) + q)
                                               : make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
                        gmw[4 * q] = w4.x;
                        gmw[4 * q + 1] = w4.y;
                        gmw[4 * q + 2] = w4.z;
                        gmw[4 * q + 3] = w4.w;
                    }
                }
                tmem_wait_ld();
                uint32_t packed[16];
                const float2 inv2 = make_float2(inv_l, inv_l);
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    // column pairs in packed multiplies (the same roundings as one at a time)
                    float2 v = __fmul2_rn(make_float2(__uint_as_float(orr[e]), __uint_as_float(orr[e + 1])), inv2);
                    if (GATE == 2) {
                        // columns cb*32 + e, + 1: half2 number (e/2) % 4 of uint4 cb*4 + e/8
                        const uint32_t hw = (&gq[cb * 4 + (e >> 3)].x)[(e >> 1) & 3];
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
                if (DIRECT) {
                    // The row's 64 bytes go straight from registers, as two whole
                    // 32-byte sectors (256-bit stores; O is 32-byte aligned and a row
                    // is d_k halves): no fence, barrier or bulk copy per chunk. Without a
                    // gate: 36.22 -> 35.13 us per call on the headline shape (16-byte
                    // stores gained a third of that). The elementwise gate's values
                    // are read as whole sectors too (above); with both, the gated
                    // call went 58.10 -> 57.33 us (with 16-byte gate loads these
                    // stores cost time instead: the partial-sector traffic competes
                    // with the gate reads in L2). The headwise family keeps the bulk
                    // copies (measured no better direct).
                    if (i < args.Lq) {
                        const __nv_bfloat16* dstg = args.out + (((long)b * args.Lq + i) * args.Hq + h) * HD + cb * 32;
#pragma unroll
                        for (int q = 0; q < 2; ++q)
                            asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dstg + 16 * q),
                                         "r"(packed[8 * q]), "r"(packed[8 * q + 1]), "r"(packed[8 * q + 2]),
                                         "r"(packed[8 * q + 3]), "r"(packed[8 * q + 4]), "r"(packed[8 * q + 5]),
                                         "r"(packed[8 * q + 6]), "r"(packed[8 * q + 7])
                                         : "memory");
                    }
                } else {
                    uint8_t* dst = stg + (cb & 1) * C::STG_BYTES + row * 64;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(dst + ((q ^ sw) << 4)) =
                            make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                    fence_proxy_async_smem();
                    if (row == 0) tma_store_wait_read0();   // the previous chunk's store has read its buffer
                    named_bar_sync(1 + t, 128);
                    if (row == 0) {
                        tma_store_4d(&tmO, stg + (cb & 1) * C::STG_BYTES, cb * 32, h, my_q0, b);
                        tma_store_commit();
                    }
                }
            }
            if (args.sink_word && lane == 0)
                sink_finish(sink_old, sink_add, args.sink_arrivals, args.sink_inv, args.sink + (long)b * args.Hq + h);
        }
        sp_base += my_nkv;
        g_base += 1;
        }   // units
        if (row == 0) tma_store_wait_all();   // the output tiles have been written
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

template <int HD, int GATE, bool ADD = false>
cudaError_t launch_prefill_t(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt, cudaStream_t s,
                             bool pdl = true) {
    using C = PrefillCfg<HD, GATE>;
    alignas(64) CUtensorMap tmQ, tmK, tmV, tmO;
    const cuuint64_t e = 2;
    // [B, L, H, d] viewed as (64 columns, H, L, B, d/64 blocks): one request
    // loads a 128-row tile with all d_k columns as d_k/64 swizzled blocks
    {
        cuuint64_t d[5] = {64, (cuuint64_t)p.Hq, (cuuint64_t)p.Lq, (cuuint64_t)p.B, (cuuint64_t)(HD / 64)};
        cuuint64_t st[4] = {HD * e, (cuuint64_t)p.Hq * HD * e, (cuuint64_t)p.Lq * p.Hq * HD * e, 128};
        cuuint32_t box[5] = {64, 1, 128, 1, HD / 64};
        if (!make_map(&tmQ, p.Q, 5, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t d[5] = {64, (cuuint64_t)p.Hkv, (cuuint64_t)p.Lk, (cuuint64_t)p.B, (cuuint64_t)(HD / 64)};
        cuuint64_t st[4] = {HD * e, (cuuint64_t)p.Hkv * HD * e, (cuuint64_t)p.Lk * p.Hkv * HD * e, 128};
        cuuint32_t box[5] = {64, 1, 128, 1, HD / 64};
        if (!make_map(&tmK, p.K, 5, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        if (!make_map(&tmV, p.V, 5, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    // O [B, L_q, H_q, d] as (d, H_q, L_q, B): one store writes 32 columns of a 128-row tile
    {
        cuuint64_t d[4] = {(cuuint64_t)HD, (cuuint64_t)p.Hq, (cuuint64_t)p.Lq, (cuuint64_t)p.B};
        cuuint64_t st[3] = {HD * e, (cuuint64_t)p.Hq * HD * e, (cuuint64_t)p.Lq * p.Hq * HD * e};
        cuuint32_t box[4] = {32, 1, 128, 1};
        if (!make_map(&tmO, p.O, 4, d, st, box, CU_TENSOR_MAP_SWIZZLE_64B)) return cudaErrorInvalidValue;
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
    a.n_pairs = (a.n_qtiles + 1) / 2;
    a.gate_part = (GATE == 1) ? reinterpret_cast<const float*>(ws + w.gate_part) : nullptr;
    a.gate_splits = w.gate_splits;
    a.gate_sig = (GATE == 2) ? reinterpret_cast<const __half*>(ws + w.gate_sig) : nullptr;
    a.ge = gate_epi(p);
    a.gs = p.gate_mode == 1 ? p.stats : GateStats();
    a.sched_counter = reinterpret_cast<int*>(ws + w.state);
    set_sink_args(p, w, ws, a.n_qtiles, &a.sink_word, &a.sink, &a.sink_scale, &a.sink_inv, &a.sink_arrivals);
    a.lse = p.lse;
    a.out = static_cast<__nv_bfloat16*>(p.O);
    a.ctl.err = rt.err;
    a.ctl.limit_ns = rt.limit_ns;

    // The API asks 16-byte alignment of O; the 256-bit stores need 32, so a
    // view that starts mid-sector takes the staged bulk copies instead.
    constexpr bool kCanDirect = (GATE == 0 || GATE == 2);
    const bool direct = kCanDirect && (reinterpret_cast<uintptr_t>(p.O) & 31u) == 0;
    static PerDeviceSetup setup;   // per template instance
    cudaError_t r = setup_once_per_device(setup, [](int&) {
        // The register split above only fits if the launch allocates enough
        // registers per thread; refuse to launch otherwise (it would not finish).
        for (int k = 0; k < (kCanDirect ? 2 : 1); ++k) {
            const void* fn = k ? reinterpret_cast<const void*>(prefill_kernel<HD, GATE, ADD, kCanDirect>)
                               : reinterpret_cast<const void*>(prefill_kernel<HD, GATE, ADD, false>);
            cudaFuncAttributes fa;
            cudaError_t e = cudaFuncGetAttributes(&fa, fn);
            if (e != cudaSuccess) return e;
            if (fa.numRegs < kRegsLaunchMin) return cudaErrorInvalidConfiguration;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    });
    if (r != cudaSuccess) return r;
    const long units = (long)a.n_pairs * p.Hq * p.B;
    const long grid = units < rt.num_sms ? units : rt.num_sms;   // persistent: one CTA per SM
    // The kernel just before this one in the call (a gate kernel, or the
    // state-zeroing kernel when there is no gate) zeroes the per-call state and
    // then lets this one start early (programmatic dependent launch); with a
    // gate, the epilogues wait for that kernel to complete before reading it.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (direct) return cudaLaunchKernelEx(&cfg, prefill_kernel<HD, GATE, ADD, kCanDirect>, tmQ, tmK, tmV, tmO, a);
    return cudaLaunchKernelEx(&cfg, prefill_kernel<HD, GATE, ADD, false>, tmQ, tmK, tmV, tmO, a);
}

}  // namespace

cudaError_t launch_prefill_bf16_ordered(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                        cudaStream_t s) {
    if ((long)p.Lk >= kPairMinKeys) return launch_prefill_pair_bf16_ordered(p, w, ws, rt, s);
    if (p.dk != 128 || (p.gate_mode != 0 && p.gate_mode != 2) || p.gate_fn != 0) return cudaErrorInvalidValue;
    return p.gate_mode == 2 ? launch_prefill_t<128, 2>(p, w, ws, rt, s, false)
                            : launch_prefill_t<128, 0>(p, w, ws, rt, s, false);
}

cudaError_t launch_prefill_bf16(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                cudaStream_t s) {
    const bool add = gate_template(p) != 0 && (p.gate_fn >= 2 && p.gate_fn <= 4);   // additive gates
    if (p.dk == 128) {
        // Long key sequences: CTA pairs (M = 256 MMAs, half the operand
        // traffic per SM). Shorter ones keep single-CTA units, whose finer
        // granularity balances causal work better across the SMs.
        if ((long)p.Lk >= kPairMinKeys) return launch_prefill_pair_bf16(p, w, ws, rt, s);
        switch (gate_template(p)) {
        case 1: return add ? launch_prefill_t<128, 1, true>(p, w, ws, rt, s) : launch_prefill_t<128, 1>(p, w, ws, rt, s);
        case 2: return add ? launch_prefill_t<128, 2, true>(p, w, ws, rt, s) : launch_prefill_t<128, 2>(p, w, ws, rt, s);
        case 3: return launch_prefill_t<128, 3>(p, w, ws, rt, s);
        case 4: return launch_prefill_t<128, 4>(p, w, ws, rt, s);
        default: return launch_prefill_t<128, 0>(p, w, ws, rt, s);
        }
    }
    switch (gate_template(p)) {
    case 1: return add ? launch_prefill_t<64, 1, true>(p, w, ws, rt, s) : launch_prefill_t<64, 1>(p, w, ws, rt, s);
    case 2: return add ? launch_prefill_t<64, 2, true>(p, w, ws, rt, s) : launch_prefill_t<64, 2>(p, w, ws, rt, s);
    case 3: return launch_prefill_t<64, 3>(p, w, ws, rt, s);
    case 4: return launch_prefill_t<64, 4>(p, w, ws, rt, s);
    default: return launch_prefill_t<64, 0>(p, w, ws, rt, s);
    }
}

}  // namespace gsdpa
