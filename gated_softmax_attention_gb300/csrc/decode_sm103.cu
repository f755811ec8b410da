// decode_sm103.cu -- bf16 gated attention for one new query per sequence
// (L_q == 1) against a K/V cache, split over the cache length.
//
// The work is HBM-bound: every K/V byte is read once and used for the four
// query heads that share it (GQA), so the kernel streams K/V through shared
// memory with TMA and does the small dot products on the CUDA cores in fp32.
// ("GatedAttention [2025]", sec. 1.3.1: the KV cache of grouped-query
// attention is what decode reads; sec. 1.2.1 / 1.2.2: SDPA and the gate.)
//
// Unit = (b, kv head, chunk of 4 query heads, split of the cache). A CTA:
//   * keeps q (4 heads x 128, pre-scaled by log2(e)/sqrt(d_k)) in registers;
//   * streams its keys 64 at a time: K and V tiles [64 x 128] land in a
//     3-stage TMA ring (warp 0 lane 0 issues the copies);
//   * 8 warps = 32 key groups x 8 lanes; lane j of a group owns dims
//     {8j..8j+7, 64+8j..64+8j+7}; a group takes keys g and g+32 of each tile,
//     reduce-scatters its 8 partial dot products (2 keys x 4 heads) across its
//     8 lanes, keeps a running max / sum per head, and accumulates p * V;
//   * merges the 32 groups in shared memory (log-sum-exp) and writes the
//     split's (max, sum, unnormalised output) to the workspace;
//   * the last split of a (b, kv head, chunk) to arrive (atomic counter) merges
//     all splits, multiplies by sigmoid(gate logits) and stores bf16 O and the
//     first-token share. No CTA ever waits for another.
// The gate logits X W_g come from the tensor-core pre-pass (gate_gemm_sm103.cu),
// which reads each column of W_g once for the whole batch.
#include "gsdpa_internal.h"
#include "sm103_ptx.cuh"
#include "gate_fn.cuh"

#include <cmath>

namespace gsdpa {
namespace {

constexpr int HD = 128;
constexpr int HPC = 4;           // query heads per CTA
constexpr int KT = 64;           // keys per tile
constexpr int NS = 3;            // ring stages
constexpr int kThreads = 256;
constexpr uint32_t TILE_BYTES = KT * HD * 2;        // 16 KB
constexpr uint32_t STAGE_BYTES = 2 * TILE_BYTES;    // K + V
constexpr uint32_t OFF_BAR = NS * STAGE_BYTES;
constexpr uint32_t OFF_MISC = OFF_BAR + 2 * NS * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;

struct DecodeArgs {
    int B, Lk, Hq, Hkv, chunks, splits, n_tiles;
    const __nv_bfloat16* Q;       // [B, 1, Hq, HD]
    __nv_bfloat16* O;             // [B, 1, Hq, HD]
    float* sink;                  // [B, Hq] or null
    const float* gate_part;       // [gate_splits, B, gate_cols] or null
    int gate_splits, gate_mode, gate_cols;
    const __nv_bfloat16* theta;   // input-independent gate [Hq, HD], or RMSNorm gamma [Hq, HD] (or null)
    int gate_fn;                  // gsdpa_gate_fn
    float eps;
    GateStats gs;                 // gate statistics (sigmoid gate), or none
    float* part_ml;               // [B, Hq, splits, 2]  (max in log2 units, sum)
    float* part_o;                // [B, Hq, splits, HD]
    float* part_x0;               // [B, Hq]  scaled score of key 0
    int* counters;                // [B, Hkv, chunks]
    WaitCtl ctl;
};

// bf16 pairs -> float2 pairs (the low half of each 32-bit word is the even element)
__device__ __forceinline__ void unpack8x2(const uint4& w, float2 (&f)[4]) {
    f[0] = make_float2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
    f[1] = make_float2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
    f[2] = make_float2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u));
    f[3] = make_float2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xffff0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xffff0000u);
    f[4] = __uint_as_float(w.z << 16);
    f[5] = __uint_as_float(w.z & 0xffff0000u);
    f[6] = __uint_as_float(w.w << 16);
    f[7] = __uint_as_float(w.w & 0xffff0000u);
}

__global__ void __launch_bounds__(kThreads, 1)
decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const DecodeArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* empty = full + NS;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC);
    int* s_last = reinterpret_cast<int*>(smem + OFF_MISC + 4);

    const int tid = threadIdx.x;
    const int warp = tid / 32;
    const int lane = tid % 32;
    const int grp = warp * 4 + lane / 8;   // key group 0..31
    const int j = lane & 7;                // lane within the group
    const int gbase = lane & ~7;

    // unit: split fastest so that the splits of one (b, kv head) finish together
    int u = blockIdx.x;
    const int split = u % args.splits;
    u /= args.splits;
    const int chunk = u % args.chunks;
    u /= args.chunks;
    const int kvh = u % args.Hkv;
    const int b = u / args.Hkv;
    const int h0 = kvh * (args.Hq / args.Hkv) + chunk * HPC;
    const int t0 = (int)((long)split * args.n_tiles / args.splits);
    const int t1 = (int)((long)(split + 1) * args.n_tiles / args.splits);

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kThreads / 32);
        }
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    __syncthreads();

    // producer: thread 0 keeps up to NS tiles in flight ahead of the consumers
    uint32_t p_stage = 0, p_phase = 0;
    uint32_t armed = 0, armed_phase = 0;  // bit s: stage s was filled; its phase parity
    int next_tile = t0;
    auto produce = [&]() -> bool {
        if (!mbar_wait(&empty[p_stage], p_phase ^ 1u, abort_flag, args.ctl)) return false;
        mbar_arrive_expect_tx(&full[p_stage], STAGE_BYTES);
        armed |= 1u << p_stage;
        armed_phase = (armed_phase & ~(1u << p_stage)) | (p_phase << p_stage);
        uint8_t* st = smem + p_stage * STAGE_BYTES;
        tma_load_4d(st, &tmK, 0, kvh, next_tile * KT, b, &full[p_stage]);
        tma_load_4d(st + TILE_BYTES, &tmV, 0, kvh, next_tile * KT, b, &full[p_stage]);
        ++next_tile;
        if (++p_stage == NS) {
            p_stage = 0;
            p_phase ^= 1u;
        }
        return true;
    };
    if (tid == 0) {
        for (int k = 0; k < NS && next_tile < t1; ++k) produce();
    }

    // q for this lane's 16 dims and the 4 heads, scaled into log2 units
    const float qs = kLog2e / sqrtf((float)HD);
    float2 q[HPC][8];   // (dims 8j..8j+7, 64+8j..64+8j+7) as float pairs
#pragma unroll
    for (int h = 0; h < HPC; ++h) {
        const __nv_bfloat16* qp = args.Q + ((long)b * args.Hq + h0 + h) * HD;
        const uint4 w0 = *reinterpret_cast<const uint4*>(qp + 8 * j);
        const uint4 w1 = *reinterpret_cast<const uint4*>(qp + 64 + 8 * j);
        float f[8];
        unpack8(w0, f);
#pragma unroll
        for (int e = 0; e < 4; ++e) q[h][e] = make_float2(f[2 * e] * qs, f[2 * e + 1] * qs);
        unpack8(w1, f);
#pragma unroll
        for (int e = 0; e < 4; ++e) q[h][4 + e] = make_float2(f[2 * e] * qs, f[2 * e + 1] * qs);
    }

    float2 o[HPC][8];
#pragma unroll
    for (int h = 0; h < HPC; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) o[h][e] = make_float2(0.f, 0.f);
    float m_cur[HPC];
#pragma unroll
    for (int h = 0; h < HPC; ++h) m_cur[h] = -INFINITY;
    float l_lane = 0.f;       // running sum for head (j & 3), this lane's keys
    float x0_lane = -INFINITY;
    const int my_head = j & 3;
    const int my_slot = j >> 2;

    uint32_t c_stage = 0, c_phase = 0;
    bool ok = true;
    for (int t = t0; t < t1; ++t) {
        ok = __all_sync(0xffffffffu, mbar_wait(&full[c_stage], c_phase, abort_flag, args.ctl));
        if (!ok) break;
        const uint8_t* Kt = smem + c_stage * STAGE_BYTES;
        const uint8_t* Vt = Kt + TILE_BYTES;

        // ---- scores: partial dots over this lane's 16 dims, 2 keys x 4 heads
        float v[2 * HPC];
#pragma unroll
        for (int sl = 0; sl < 2; ++sl) {
            const int key = grp + 32 * sl;
            const uint4 w0 = *reinterpret_cast<const uint4*>(Kt + key * (HD * 2) + j * 16);
            const uint4 w1 = *reinterpret_cast<const uint4*>(Kt + key * (HD * 2) + 128 + j * 16);
            float2 k2[8];
            unpack8x2(w0, *reinterpret_cast<float2(*)[4]>(&k2[0]));
            unpack8x2(w1, *reinterpret_cast<float2(*)[4]>(&k2[4]));
#pragma unroll
            for (int h = 0; h < HPC; ++h) {
                float2 acc = __fmul2_rn(q[h][0], k2[0]);
#pragma unroll
                for (int e = 1; e < 8; ++e) acc = __ffma2_rn(q[h][e], k2[e], acc);
                v[sl * HPC + h] = acc.x + acc.y;
            }
        }
        // reduce-scatter over the 8 lanes: lane j ends with value index j = slot*4 + head
        float w4[4];
        const bool b2 = (j & 4) != 0, b1 = (j & 2) != 0, b0 = (j & 1) != 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float mine = b2 ? v[4 + e] : v[e];
            const float other = b2 ? v[e] : v[4 + e];
            w4[e] = mine + __shfl_xor_sync(0xffffffffu, other, 4);
        }
        float w2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float mine = b1 ? w4[2 + e] : w4[e];
            const float other = b1 ? w4[e] : w4[2 + e];
            w2[e] = mine + __shfl_xor_sync(0xffffffffu, other, 2);
        }
        float s = (b0 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b0 ? w2[0] : w2[1], 1);
        const long key_abs = (long)t * KT + grp + 32 * my_slot;
        if (key_abs >= args.Lk) s = -INFINITY;
        if (key_abs == 0) x0_lane = s;

        // ---- running max per head (lanes j and j^4 hold the same head)
        const float mc = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 4));
        const bool need = mc > m_cur[my_head] + kRescaleThreshold || m_cur[my_head] == -INFINITY;
        if (__any_sync(0xffffffffu, need)) {
            float alpha[HPC];
#pragma unroll
            for (int h = 0; h < HPC; ++h) {
                const float mh = __shfl_sync(0xffffffffu, mc, gbase + h);
                const float mn = fmaxf(m_cur[h], mh);
                alpha[h] = (m_cur[h] == -INFINITY) ? 0.f : ex2_approx(m_cur[h] - mn);
                m_cur[h] = mn;
            }
#pragma unroll
            for (int h = 0; h < HPC; ++h) {
                const float2 a2 = make_float2(alpha[h], alpha[h]);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[h][e] = __fmul2_rn(o[h][e], a2);
            }
            l_lane *= alpha[my_head];
        }
        const float p = (s == -INFINITY) ? 0.f : ex2_approx(s - m_cur[my_head]);
        l_lane += p;
        float pp[2 * HPC];
#pragma unroll
        for (int e = 0; e < 2 * HPC; ++e) pp[e] = __shfl_sync(0xffffffffu, p, gbase + e);

        // ---- o += p * V
#pragma unroll
        for (int sl = 0; sl < 2; ++sl) {
            const int key = grp + 32 * sl;
            const uint4 w0 = *reinterpret_cast<const uint4*>(Vt + key * (HD * 2) + j * 16);
            const uint4 w1 = *reinterpret_cast<const uint4*>(Vt + key * (HD * 2) + 128 + j * 16);
            float2 v2[8];
            unpack8x2(w0, *reinterpret_cast<float2(*)[4]>(&v2[0]));
            unpack8x2(w1, *reinterpret_cast<float2(*)[4]>(&v2[4]));
#pragma unroll
            for (int h = 0; h < HPC; ++h) {
                const float2 ph = make_float2(pp[sl * HPC + h], pp[sl * HPC + h]);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[h][e] = __ffma2_rn(ph, v2[e], o[h][e]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[c_stage]);
        if (++c_stage == NS) {
            c_stage = 0;
            c_phase ^= 1u;
        }
        if (tid == 0 && next_tile < t1) {
            if (!produce()) ok = false;
        }
    }

    // ---- merge the 32 key groups of this CTA (log-sum-exp), reusing the ring
    ok = __syncthreads_and(ok && !*abort_flag);
    if (!ok) {
        // let copies in flight land before the CTA exits
        if (tid == 0) {
            volatile int never = 0;
            WaitCtl c2 = args.ctl;
            if (c2.limit_ns < 1000000000ull) c2.limit_ns = 1000000000ull;
            for (int s = 0; s < NS; ++s)
                if (armed & (1u << s)) mbar_wait(&full[s], (armed_phase >> s) & 1u, &never, c2);
        }
        return;
    }
    float* red_o = reinterpret_cast<float*>(smem);                 // [32 groups][HPC][128]
    float* red_m = red_o + 32 * HPC * HD;                          // [32][HPC]
    float* red_l = red_m + 32 * HPC;                               // [32][8 lanes]
    float* red_x0 = red_l + 32 * 8;                                // [HPC]
#pragma unroll
    for (int h = 0; h < HPC; ++h) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            red_o[(grp * HPC + h) * HD + 8 * j + 2 * e] = o[h][e].x;
            red_o[(grp * HPC + h) * HD + 8 * j + 2 * e + 1] = o[h][e].y;
            red_o[(grp * HPC + h) * HD + 64 + 8 * j + 2 * e] = o[h][4 + e].x;
            red_o[(grp * HPC + h) * HD + 64 + 8 * j + 2 * e + 1] = o[h][4 + e].y;
        }
    }
    if (j < HPC) red_m[grp * HPC + j] = m_cur[j];
    red_l[grp * 8 + j] = l_lane;
    if (t0 == 0 && grp == 0 && my_slot == 0) red_x0[my_head] = x0_lane;  // key 0 is key 0 of tile 0, group 0
    __syncthreads();

    // thread -> (head, 2 dims): merge over groups
    const int hh = tid / 64;            // 0..3
    const int dd = (tid % 64) * 2;      // 0..126
    float M = -INFINITY;
    for (int g = 0; g < 32; ++g) M = fmaxf(M, red_m[g * HPC + hh]);
    float acc0 = 0.f, acc1 = 0.f, L = 0.f;
    for (int g = 0; g < 32; ++g) {
        const float mg = red_m[g * HPC + hh];
        const float sc = (mg == -INFINITY) ? 0.f : ex2_approx(mg - M);
        acc0 += red_o[(g * HPC + hh) * HD + dd] * sc;
        acc1 += red_o[(g * HPC + hh) * HD + dd + 1] * sc;
        L += (red_l[g * 8 + hh] + red_l[g * 8 + 4 + hh]) * sc;
    }
    const int head = h0 + hh;
    const long pidx = ((long)b * args.Hq + head) * args.splits + split;
    args.part_o[pidx * HD + dd] = acc0;
    args.part_o[pidx * HD + dd + 1] = acc1;
    if (dd == 0) {
        args.part_ml[pidx * 2] = M;
        args.part_ml[pidx * 2 + 1] = L;
        if (t0 == 0) args.part_x0[(long)b * args.Hq + head] = red_x0[hh];
    }

    // ---- last arriver combines the splits
    __threadfence();
    __syncthreads();
    int* cnt = args.counters + ((long)b * args.Hkv + kvh) * args.chunks + chunk;
    if (tid == 0) *s_last = (atomicAdd(cnt, 1) == args.splits - 1);
    __syncthreads();
    if (!*s_last) return;
    __threadfence();

    const long base = ((long)b * args.Hq + head) * args.splits;
    float Mt = -INFINITY;
    for (int s2 = 0; s2 < args.splits; ++s2) Mt = fmaxf(Mt, __ldcg(&args.part_ml[(base + s2) * 2]));
    float Lt = 0.f, r0 = 0.f, r1 = 0.f;
    for (int s2 = 0; s2 < args.splits; ++s2) {
        const float ms = __ldcg(&args.part_ml[(base + s2) * 2]);
        const float sc = (ms == -INFINITY) ? 0.f : ex2_approx(ms - Mt);
        Lt += __ldcg(&args.part_ml[(base + s2) * 2 + 1]) * sc;
        r0 += __ldcg(&args.part_o[(base + s2) * HD + dd]) * sc;
        r1 += __ldcg(&args.part_o[(base + s2) * HD + dd + 1]) * sc;
    }
    const float inv = 1.0f / Lt;
    // ---- the gate (gsdpa_gate_mode / gsdpa_gate_fn) on y = (r0, r1) * inv
    float y0 = r0 * inv, y1 = r1 * inv;
    const int fn = args.gate_fn;
    if (args.gate_mode != 0) {
        float gl0 = 0.f, gl1 = 0.f;
        if (args.gate_mode == 5) {   // input-independent: theta [Hq, HD]
            gl0 = __bfloat162float(args.theta[(long)head * HD + dd]);
            gl1 = __bfloat162float(args.theta[(long)head * HD + dd + 1]);
        } else {
            pdl_wait();   // the gate-logit kernel has completed (a no-op after an ordinary launch)
            // logit column of (head, dd): elementwise, headwise, headwise shared, elementwise shared
            const int m = args.gate_mode;
            const long c0 = m == 2 ? (long)head * HD + dd : (m == 1 ? head : (m == 3 ? 0 : dd));
            const bool per_col = m == 2 || m == 4;
            const long rowoff = (long)b * args.gate_cols;
            const long gsz = (long)args.B * args.gate_cols;
            for (int s2 = 0; s2 < args.gate_splits; ++s2) {
                gl0 += args.gate_part[s2 * gsz + rowoff + c0];
                if (per_col) gl1 += args.gate_part[s2 * gsz + rowoff + c0 + 1];
            }
            if (!per_col) gl1 = gl0;
        }
        const bool add = gate_adds(fn);
        const float gv0 = gate_value(gl0, fn), gv1 = gate_value(gl1, fn);
        y0 = gate_combine(y0, gv0, add);
        y1 = gate_combine(y1, gv1, add);
        if (args.gs.out) {   // every thread of the block is here (the last arriver's)
            const bool per_col = args.gate_mode == 2;
            gate_stats_warp(args.gs, gv0, per_col || dd == 0);
            gate_stats_warp(args.gs, gv1, per_col);
        }
    } else if (fn == 5) {   // SiLU of the output
        y0 *= sigmoid_tanh(y0);
        y1 *= sigmoid_tanh(y1);
    } else if (fn == 6) {
        // per-head RMSNorm: the head's 128 columns live in 64 threads (two warps)
        float ss = fmaf(y0, y0, y1 * y1);
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, sh);
        float* red = reinterpret_cast<float*>(smem);   // (the merge above has read its arrays)
        __syncthreads();
        if ((tid & 31) == 0) red[tid >> 5] = ss;
        __syncthreads();
        const float tot = red[(tid >> 6) * 2] + red[(tid >> 6) * 2 + 1];
        const float rr = rsqrtf(tot / HD + args.eps);
        const float ga0 = args.theta ? __bfloat162float(args.theta[(long)head * HD + dd]) : 1.f;
        const float ga1 = args.theta ? __bfloat162float(args.theta[(long)head * HD + dd + 1]) : 1.f;
        y0 *= rr * ga0;
        y1 *= rr * ga1;
    }
    __nv_bfloat162 outv = __floats2bfloat162_rn(y0, y1);
    *reinterpret_cast<__nv_bfloat162*>(args.O + ((long)b * args.Hq + head) * HD + dd) = outv;
    if (args.sink && dd == 0) {
        const float x0 = __ldcg(&args.part_x0[(long)b * args.Hq + head]);
        args.sink[(long)b * args.Hq + head] = ex2_approx(x0 - Mt) * inv;
    }
    if (tid == 0) *cnt = 0;  // leave the counter ready for the next call
}

}  // namespace

bool decode_supported(const Problem& p) {
    return p.dtype == 1 && p.Lq == 1 && p.dk == HD && (p.Hq / p.Hkv) % HPC == 0;
}

// Splits of the cache per (b, kv head, chunk). Every CTA pays a fixed cost
// of a few microseconds (its first copies' latency, the merge of its key
// groups, the split combine), so the cache is cut into as few splits as give
// about four CTAs per SM: enough for the SMs to stay busy to the end, few
// enough that the fixed cost stays small next to the streaming.
int decode_splits(const Problem& p, int num_sms) {
    const int chunks = (p.Hq / p.Hkv) / HPC;
    const long base = (long)p.B * p.Hkv * chunks;
    const int n_tiles = (p.Lk + KT - 1) / KT;
    long s = (4L * num_sms + base - 1) / base;
    long max_s = n_tiles / 4 > 0 ? n_tiles / 4 : 1;
    if (s > max_s) s = max_s;
    if (s < 1) s = 1;
    return (int)s;
}

cudaError_t launch_decode_bf16(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                               cudaStream_t s, bool dependent) {
    alignas(64) CUtensorMap tmK, tmV;
    cuuint64_t d[4] = {(cuuint64_t)HD, (cuuint64_t)p.Hkv, (cuuint64_t)p.Lk, (cuuint64_t)p.B};
    cuuint64_t st[3] = {HD * 2, (cuuint64_t)p.Hkv * HD * 2, (cuuint64_t)p.Lk * p.Hkv * HD * 2};
    cuuint32_t box[4] = {HD, 1, KT, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    for (int k = 0; k < 2; ++k) {
        CUresult r = encode_tiled_fn()(k == 0 ? &tmK : &tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                                       const_cast<void*>(k == 0 ? p.K : p.V), d, st, box, es,
                                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    DecodeArgs a;
    a.B = p.B;
    a.Lk = p.Lk;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.chunks = (p.Hq / p.Hkv) / HPC;
    a.splits = w.dec_splits;
    a.n_tiles = (p.Lk + KT - 1) / KT;
    a.Q = static_cast<const __nv_bfloat16*>(p.Q);
    a.O = static_cast<__nv_bfloat16*>(p.O);
    a.sink = p.sink;
    a.gate_part = w.gate_splits ? reinterpret_cast<const float*>(ws + w.gate_part) : nullptr;
    a.gate_splits = w.gate_splits;
    a.gate_mode = p.gate_mode;
    a.gate_cols = w.gate_cols;
    a.theta = (p.gate_mode == 5 || p.gate_fn == 6) ? static_cast<const __nv_bfloat16*>(p.Wg) : nullptr;
    a.gate_fn = p.gate_fn;
    a.eps = p.eps;
    a.gs = p.stats;
    a.part_ml = reinterpret_cast<float*>(ws + w.dec_ml);
    a.part_o = reinterpret_cast<float*>(ws + w.dec_o);
    a.part_x0 = reinterpret_cast<float*>(ws + w.dec_x0);
    a.counters = reinterpret_cast<int*>(ws + w.dec_cnt);
    a.ctl.err = rt.err;
    a.ctl.limit_ns = rt.limit_ns;
    cudaError_t e = cudaSuccess;
    if (!dependent) e = cudaMemsetAsync(a.counters, 0, w.dec_cnt_bytes, s);
    if (e != cudaSuccess) return e;
    static PerDeviceSetup setup;
    e = setup_once_per_device(setup, [](int&) {
        return cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    });
    if (e != cudaSuccess) return e;
    const long units = (long)p.B * p.Hkv * a.chunks * a.splits;
    if (dependent)
        return launch_dependent(decode_kernel, dim3((unsigned)units), dim3(kThreads), SMEM_BYTES, s, tmK, tmV, a);
    decode_kernel<<<(unsigned)units, kThreads, SMEM_BYTES, s>>>(tmK, tmV, a);
    return cudaGetLastError();
}

}  // namespace gsdpa
