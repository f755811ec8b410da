// gate_sigmoid_sm103.cu -- the elementwise gate sigma(X W_g) for the bf16
// prefill path, as fp16, on pairs of SMs.
//
// Also the gate's other functions of the logit (NS-sigmoid, SiLU, identity:
// the FN template parameter, gsdpa_gate_fn's codes 0..4), the head-shared
// elementwise gate (W_g [d_model, d_k]: the same kernel with d_k columns) and
// the input-independent gate (gate_static_kernel: the value of theta [H_q, d_k]
// with no product).
//
// Computes gate[r, c] = fp16( sigma( sum_m X[r, m] W_g[m, c] ) ) for every row
// r of X viewed as [rows = B*L_q, d_model] and every column c of W_g
// [d_model, cols = H_q*d_k] ("GatedAttention [2025]", sec. 1.2.2: the gate
// is sigma(X W_theta), applied elementwise to the SDPA output; no bias,
// "10 . 门控", sec. 3.2). The attention epilogue multiplies its output rows by
// these values, so the ungated SDPA output never leaves the SM; the gate
// values (values in (0, 1), where fp16 keeps 11 significant bits) make one
// round trip through L2 / HBM.
//
// This is a plain GEMM with a sigmoid epilogue, kept out of the attention
// kernel: there, one head's 128 gate columns per unit re-read X once per head
// from L2 and the tile shape (256 x 128) needs more L2 bandwidth per flop
// than the SMs get. Here a pair of CTAs (cluster of two, tcgen05.mma
// .cta_group::2) computes a 256 x 512 tile in the whole of tensor memory:
// per K chunk of 64, each CTA loads its 128 rows of X (16 KB) and a
// contiguous block of 256 columns of W_g (32 KB, one copy request) for 1024
// MMA cycles.
//
// Column order. A pair MMA takes the first half of its N columns from the
// even CTA and the second half from the odd one. CTA rho holds W_g columns
// [256 rho, 256 rho + 256) of the tile; MMA h (h = 0, 1) takes columns
// [128 h, 128 h + 128) of each CTA's block, so accumulator column c holds
// tile column 256 * ((c % 256) / 128) + 128 * (c / 256) + c % 128.
//
// Per CTA: warp 0 TMA producer (both CTAs), warp 1 TMEM allocation (both) and
// MMA issue (even CTA), warps 2..9 epilogue: two warps per TMEM lane quadrant,
// each converting half of the 512 accumulator columns of its 32 rows (the
// tensor-memory load of the next 32 columns in flight while the current ones
// are converted). The fp16 tile is staged in the idle K-chunk ring as 64-column
// 128B-swizzled blocks and written with four 32 KB bulk copies, each issued by
// the producer thread (idle by then) as soon as its 128 columns are staged, so
// that the stores overlap the conversion: one thread per row writing 16-byte
// pieces of its own row would cost one memory transaction per piece.
// Rows past the end of X, columns past the end of W_g and the K tail load as
// zeros (TMA out-of-bounds fill) and are not stored.
#include "gsdpa_internal.h"
#include "sm103_pair.cuh"
#include "sm103_ptx.cuh"
#include "gate_fn.cuh"

#include <cuda_fp16.h>

namespace gsdpa {
namespace {

constexpr int kThreads = 320;
constexpr int kNS = 4;                                  // K-chunk ring stages
constexpr uint32_t kXBytes = 128 * 64 * 2;              // X chunk: this CTA's 128 rows x 64
constexpr uint32_t kWBytes = 64 * 256 * 2;              // W_g chunk: 64 x this CTA's 256 columns
constexpr uint32_t kStage = kXBytes + kWBytes;
constexpr uint32_t kOffBar = kNS * kStage;
constexpr uint32_t kOffMisc = kOffBar + (2 * kNS + 2 + 4) * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack

struct SigArgs {
    __half* out;     // [rows, cols]
    int rows, cols, d_model;
    int row_tiles, nkc;   // tiles of 256 rows; K chunks of 64
    ZeroJob zero;         // per-call state of the attention kernel, zeroed by CTA 0
    GateStats st;         // gate statistics of the stored values (STATS instances)
    WaitCtl ctl;
};

// sigma of two values as fp16: 1/2 + tanh(x/2)/2 with one MUFU operation for
// both (tanh.approx.f16x2, relative error about 2^-11 -- the precision the
// fp16 result keeps anyway; the logits are rounded to fp16 first, |x| stays
// far inside its range).
__device__ __forceinline__ uint32_t sigmoid2_h(float x0, float x1) {
    const __half2 hx = __floats2half2_rn(0.5f * x0, 0.5f * x1);
    uint32_t t;
    asm("tanh.approx.f16x2 %0, %1;" : "=r"(t) : "r"(*reinterpret_cast<const uint32_t*>(&hx)));
    const __half2 half2v = __floats2half2_rn(0.5f, 0.5f);
    const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&t), half2v, half2v);
    return *reinterpret_cast<const uint32_t*>(&r);
}

// The gate's value of two logits as fp16 for gate function FN (0..4).
template <int FN>
__device__ __forceinline__ uint32_t gate_value2_h(float x0, float x1) {
    if (FN == 0 || FN == 2) return sigmoid2_h(x0, x1);
    const __half2 r = __floats2half2_rn(gate_value(x0, FN), gate_value(x1, FN));
    return *reinterpret_cast<const uint32_t*>(&r);
}

template <int FN, bool STATS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
gate_sigmoid_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmG, const SigArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* full = bars;              // [NS] even CTA: both CTAs' halves of the chunk landed
    uint64_t* empty = bars + kNS;       // [NS] both: the MMAs reading the stage completed
    uint64_t* acc_full = bars + 2 * kNS;     // both: the accumulator is complete
    uint64_t* drain = bars + 2 * kNS + 1;    // even
    uint64_t* grp_ready = bars + 2 * kNS + 2;   // [4] the 4 warps staging 128-column group g are done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    int* abort_word = reinterpret_cast<int*>(smem + kOffMisc + 4);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = pair::cta_rank();
    const pair::PairAbort ab{abort_word, pair::map_to(abort_word, rank ^ 1u)};
    const int tile = (int)pair::cluster_id();
    const int r0 = (tile % args.row_tiles) * 256;   // the pair's first row
    const int c0 = (tile / args.row_tiles) * 512;   // the pair's first column

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
        tma_prefetch_desc(&tmG);
    }
    if (warp == 1) {
        pair::tmem_alloc(tmem_slot, 512);
        tc_fence_before();
    }
    __syncthreads();
    pair::cluster_sync();
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
    pdl_trigger();   // the attention kernel may start; it reads the gate only in its epilogues

    if (warp == 0) {
        // ---- TMA producer: this CTA's rows of X and its 256 columns of W_g
        if (lane == 0) {
            for (int kc = 0; kc < args.nkc; ++kc) {
                const int s = kc % kNS;
                const uint32_t ph = (kc / kNS) & 1;
                if (!pair::wait(&empty[s], ph ^ 1u, ab, args.ctl)) break;
                if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * kStage);   // both CTAs' bytes
                const uint32_t fb = pair::map_to(&full[s], 0);
                uint8_t* st = smem + s * kStage;
                pair::tma_load_2d(st, &tmX, kc * 64, r0 + (int)rank * 128, fb);
                // W_g viewed as (64 columns, d_model rows, cols/64 blocks): four 64-column blocks
                pair::tma_load_3d(st + kXBytes, &tmW, 0, kc * 64, (c0 + (int)rank * 256) / 64, fb);
            }
            // ---- then the stores: each 128-column group of the staged fp16 tile
            // as soon as its 4 warps are done (group g = tile columns [128 g, 128 g + 128))
            // (rows / columns past the end of the output are clipped by the copy)
            bool ok = true;
            for (int g = 0; g < 4 && ok; ++g) {   // (groups 0 and 1 are staged first, in parallel)
                if (!(ok = pair::wait(&grp_ready[g], 0, ab, args.ctl))) break;
                tma_store_3d(&tmG, smem + g * 32768, 0, r0 + (int)rank * 128, (c0 + g * 128) / 64);
                tma_store_commit();
            }
            tma_store_wait_read0();   // the staging area stays valid until the copies have read it
        }
    } else if (warp == 1) {
        // ---- MMA issue (even CTA): D[256 x 512] += X[256 x 64] W_g[64 x 512] per chunk, as two N = 256 MMAs
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
                // X: K-major, one 64-column box; W_g: MN-major, 64-column blocks 8 KB apart;
                // MMA h reads blocks 2h, 2h + 1 of each CTA
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
        // ---- epilogue: sigma, fp16, 512 bytes of one row per thread
        const int qd = warp & 3;
        const int half = (warp - 2) >> 2;      // which 256 accumulator columns
        const int row = qd * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const bool ok = __all_sync(0xffffffffu, pair::wait(acc_full, 0, ab, args.ctl));
        tc_fence_after();
        // gate statistics of the fp16 values this thread stores: per-thread totals,
        // and per-thread bin counters in the idle ring past the staged tile,
        // bin-major [64 bins][256 threads] (64 KB): each thread owns its counters,
        // a warp's 32 counters of one bin lie in 32 different banks, and the
        // increments are shared-memory reductions whose result nobody waits for
        const int et = (int)threadIdx.x - 64;   // epilogue thread 0..255
        unsigned long long st_fx = 0;
        unsigned st_n = 0, st_below = 0;
        unsigned* st_h = reinterpret_cast<unsigned*>(smem + 8 * 16384);
        if (STATS)
            for (int k = 0; k < args.st.n_bins; ++k) st_h[k * 256 + et] = 0;
        const bool row_ok = r0 + (int)rank * 128 + row < args.rows;
        if (ok) {
            // (every MMA has completed, so the ring is idle: stage the tile there as
            // [8 blocks of 64 columns][128 rows], 128-byte rows, 128B swizzle)
            uint32_t buf[2][32];
            tmem_ld32(tmem + lane_base + half * 256, buf[0]);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                tmem_wait_ld_regs(buf[k & 1]);
                if (k + 1 < 8) tmem_ld32(tmem + lane_base + half * 256 + (k + 1) * 32, buf[(k + 1) & 1]);
                const uint32_t* v = buf[k & 1];
                const int c = half * 256 + k * 32;   // accumulator column -> tile column (see the column order above)
                const int tc = 256 * ((c & 255) >> 7) + 128 * (c >> 8) + (c & 127);
                uint32_t hv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    hv[e] = gate_value2_h<FN>(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                }
                uint8_t* blk = smem + (tc >> 6) * 16384;
                const uint32_t chunk0 = (uint32_t)(tc & 63) >> 3;   // 16-byte chunk of the 128-byte row
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4*>(blk + sw128_offset((uint32_t)row, chunk0 + q)) =
                        make_uint4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]);
                if ((k & 3) == 3) {
                    // this warp's rows of 128-column group (half, then 2 + half) are staged:
                    // make them visible to the bulk copy and tell the storing thread
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&grp_ready[(k >> 2) * 2 + half]);
                }
            }
        }
        if (STATS && ok) {
            // this thread's 256 staged values, read back from the staging blocks (its
            // own writes) as fp16 pairs, with few instructions per score (the pass
            // runs on two warps per scheduler while the tensor pipe waits for it):
            // - sum: float32 pairs, four partial sums of up to 64 scores each (at
            //   most 64, so each partial is within 64 * 2^-24 of the exact sum),
            //   rounded to fixed point once per thread;
            // - below the threshold: a fp16 score s is below t exactly when it is
            //   below t rounded up to fp16 (no fp16 value lies in between); the
            //   packed comparison gives 1.0 or 0.0 per score and the packed fp16
            //   counters stay exact (at most 128 per half);
            // - bin: s n_bins + 2^23 rounded down (one fused multiply-add) holds
            //   floor(s n_bins) in its low bits; the unsigned difference from 2^23's
            //   bit pattern clamped to n_bins - 1 keeps any input on a counter.
            const float nbf = (float)args.st.n_bins;
            const uint32_t last_bin = (uint32_t)args.st.n_bins - 1u;
            const __half2 thr2 = __half2half2(__float2half_ru(args.st.threshold));
            const uint32_t h_addr = smem_u32(st_h + et);   // this thread's counter of bin 0
            float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
            __half2 below2 = __float2half2_rn(0.f);
            auto count_bin = [&](float sv) {
                uint32_t bin = __float_as_uint(__fmaf_rd(sv, nbf, 8388608.0f)) - 0x4B000000u;
                bin = bin < last_bin ? bin : last_bin;
                asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(h_addr + (bin << 10)));
            };
#pragma unroll 1
            for (int k = 0; k < 8; ++k) {
                const int c = half * 256 + k * 32;
                const int tc = 256 * ((c & 255) >> 7) + 128 * (c >> 8) + (c & 127);
                const int col0 = c0 + tc;   // the gate column of the chunk's first value
                if (!row_ok || col0 >= args.cols) continue;
                const bool whole = col0 + 32 <= args.cols;
                const uint8_t* blk = smem + (tc >> 6) * 16384;
                const uint32_t chunk0 = (uint32_t)(tc & 63) >> 3;
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    const uint4 w4 = *reinterpret_cast<const uint4*>(blk + sw128_offset((uint32_t)row, chunk0 + q));
                    const uint32_t ws4[4] = {w4.x, w4.y, w4.z, w4.w};
                    if (whole) {
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const __half2 h2 = *reinterpret_cast<const __half2*>(&ws4[x]);
                            const float2 f2 = __half22float2(h2);
                            if (x & 1) acc1 = __fadd2_rn(acc1, f2);
                            else acc0 = __fadd2_rn(acc0, f2);
                            below2 = __hadd2(below2, __hlt2(h2, thr2));
                            count_bin(f2.x);
                            count_bin(f2.y);
                        }
                    } else {
                        // the last columns of the gate: scores past them are not counted
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            if (col0 + 8 * q + j >= args.cols) break;
                            const __half hs = __ushort_as_half((unsigned short)(ws4[j >> 1] >> (16 * (j & 1))));
                            const float sv = __half2float(hs);
                            acc0.x += sv;
                            st_below += __hlt(hs, __low2half(thr2)) ? 1u : 0u;
                            count_bin(sv);
                        }
                    }
                }
                st_n += whole ? 32u : (uint32_t)(args.cols - col0);
            }
            const float sum = (acc0.x + acc0.y) + (acc1.x + acc1.y);
            st_fx = __float2ull_rn(sum * 4294967296.0f);   // score * 2^32
            st_below += (uint32_t)(__low2float(below2) + __high2float(below2));
        }
        if (STATS) {
            // this warp's totals and histogram into the call's counters
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) {
                st_fx += __shfl_xor_sync(0xffffffffu, st_fx, sh);
                st_n += __shfl_xor_sync(0xffffffffu, st_n, sh);
                st_below += __shfl_xor_sync(0xffffffffu, st_below, sh);
            }
            if (lane == 0 && st_n) {
                atomicAdd(args.st.out, (unsigned long long)st_n);
                atomicAdd(args.st.out + 1, st_fx);
                if (st_below) atomicAdd(args.st.out + 2, (unsigned long long)st_below);
            }
            // the CTA's histogram: 4 threads per bin each add 64 threads' counters
            named_bar_sync(1, 256);
            const int kb = et >> 2, q = et & 3;
            unsigned hsum = 0;
            if (kb < args.st.n_bins)
                for (int u = 0; u < 64; ++u) hsum += st_h[kb * 256 + q * 64 + u];
            hsum += __shfl_xor_sync(0xffffffffu, hsum, 1);
            hsum += __shfl_xor_sync(0xffffffffu, hsum, 2);
            if (kb < args.st.n_bins && q == 0 && hsum) atomicAdd(args.st.out + 3 + kb, (unsigned long long)hsum);
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

// The input-independent gate: out[k] = fp16(value(theta[k])) for the H_q * d_k
// parameters ("GatedAttention [2025]", sec. 1.4.2 (iii): a free q x d_k
// parameter, then the gate function, multiplied with the SDPA output). Runs
// first in the call, like the gate GEMM: it zeroes the attention kernel's
// per-call state and lets it start.
__global__ void __launch_bounds__(256) gate_static_kernel(const __nv_bfloat16* __restrict__ theta,
                                                          __half* __restrict__ out, int n, int fn, ZeroJob zero) {
    pdl_wait();
    if (blockIdx.x == 0 && zero.n > 0) {
        for (int k = threadIdx.x; k < zero.n; k += blockDim.x) zero.p[k] = 0;
        __threadfence();
        __syncthreads();
    }
    pdl_trigger();
    for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < n; k += gridDim.x * blockDim.x)
        out[k] = __float2half_rn(gate_value(__bfloat162float(theta[k]), fn));
}

bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* d, const cuuint64_t* st,
              const cuuint32_t* box) {
    cuuint32_t es[3] = {1, 1, 1};
    return encode_tiled_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, st, box, es,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {
template <int FN, bool STATS = false>
cudaError_t launch_gate_value_t(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                cudaStream_t s, ZeroJob zero) {
    alignas(64) CUtensorMap tmX, tmW, tmG;
    const int rows = p.B * p.Lq, cols = gate_cols(p);
    if (rows == 0) return cudaSuccess;
    {
        const cuuint64_t d[2] = {(cuuint64_t)p.d_model, (cuuint64_t)rows};
        const cuuint64_t st[1] = {(cuuint64_t)p.d_model * 2};
        const cuuint32_t box[2] = {64, 128};
        if (!make_map(&tmX, p.X, 2, d, st, box)) return cudaErrorInvalidValue;
    }
    {
        // (64 columns, d_model rows, cols/64 column blocks; the blocks 128 bytes apart)
        const cuuint64_t d[3] = {64, (cuuint64_t)p.d_model, (cuuint64_t)cols / 64};
        const cuuint64_t st[2] = {(cuuint64_t)cols * 2, 128};
        const cuuint32_t box[3] = {64, 64, 4};
        if (!make_map(&tmW, p.Wg, 3, d, st, box)) return cudaErrorInvalidValue;
    }
    {
        // output (fp16, [rows, cols]) as (64 columns, rows, cols/64 blocks): 128 rows x 128 columns per copy
        const cuuint64_t d[3] = {64, (cuuint64_t)rows, (cuuint64_t)cols / 64};
        const cuuint64_t st[2] = {(cuuint64_t)cols * 2, 128};
        const cuuint32_t box[3] = {64, 128, 2};
        const cuuint32_t es[3] = {1, 1, 1};
        if (encode_tiled_fn()(&tmG, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, ws + w.gate_sig, d, st, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    SigArgs a;
    a.out = reinterpret_cast<__half*>(ws + w.gate_sig);
    a.rows = rows;
    a.cols = cols;
    a.d_model = p.d_model;
    a.row_tiles = (rows + 255) / 256;
    a.nkc = (p.d_model + 63) / 64;
    a.zero = zero;
    a.st = p.stats;
    a.ctl.err = rt.err;
    a.ctl.limit_ns = rt.limit_ns;
    static PerDeviceSetup setup;   // per template instance
    cudaError_t r = setup_once_per_device(setup, [](int&) {
        return cudaFuncSetAttribute(gate_sigmoid_kernel<FN, STATS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemBytes);
    });
    if (r != cudaSuccess) return r;
    const long tiles = (long)a.row_tiles * ((cols + 511) / 512);
    return launch_dependent(gate_sigmoid_kernel<FN, STATS>, dim3((unsigned)(2 * tiles)), dim3(kThreads), kSmemBytes, s, tmX,
                            tmW, tmG, a);
}
}  // namespace

namespace {
// The head-shared gate read as an average over the heads ("GatedAttention
// [2025]", sec. 1.3.2 (ii): the n x q x d_k scores averaged over the q query
// heads into an n x d_k score that every head uses). Both kernels run between
// the gate kernel and the attention kernel as programmatic dependents: they
// let the attention kernel start at once (it reads the gate only in its
// epilogues, after waiting for this kernel) and wait for the gate kernel
// before they read its output.
//
// Elementwise: g [rows, H_q d_k] fp16 values; each thread averages one row's 8
// consecutive columns c..c+7 over the heads (16-byte loads, fp32 sums) and
// writes the average over head 0's values (only this thread touches them).
__global__ void gate_average_values_kernel(__half* __restrict__ g, int rows, int Hq, int dk) {
    pdl_trigger();
    pdl_wait();
    const int chunks = dk / 8;
    const long t = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (long)rows * chunks) return;
    const long r = t / chunks;
    const int c = (int)(t % chunks) * 8;
    __half* row = g + r * (long)Hq * dk;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int h = 0; h < Hq; ++h) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + (long)h * dk + c);
        const __half2* hv = reinterpret_cast<const __half2*>(&v);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(hv[e]);
            acc[2 * e] += f.x;
            acc[2 * e + 1] += f.y;
        }
    }
    const float inv = 1.0f / (float)Hq;
    uint4 out;
    __half2* ho = reinterpret_cast<__half2*>(&out);
#pragma unroll
    for (int e = 0; e < 4; ++e) ho[e] = __floats2half2_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv);
    *reinterpret_cast<uint4*>(row + c) = out;
}

// Headwise: gl [rows, H_q] fp32 logits (one split); each thread turns one
// row's H_q logits into values f(gl_h), averages them and writes the average,
// a value, over column 0 (the attention epilogue then applies the identity).
__global__ void gate_average_logits_kernel(float* __restrict__ gl, int rows, int Hq, int fn) {
    pdl_trigger();
    pdl_wait();
    const long r = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    float* row = gl + r * Hq;
    float acc = 0.f;
    for (int h = 0; h < Hq; ++h) acc += gate_value(row[h], fn);
    row[0] = acc / (float)Hq;
}
}  // namespace

cudaError_t launch_gate_average_bf16(const Problem& p, const WorkspacePlan& w, char* ws, cudaStream_t s) {
    const int rows = p.B * p.Lq;
    if (rows == 0) return cudaSuccess;
    if (p.gate_mode == 7) {
        if (p.dk % 8 != 0) return cudaErrorInvalidValue;
        const long n = (long)rows * (p.dk / 8);
        return launch_dependent(gate_average_values_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s,
                                reinterpret_cast<__half*>(ws + w.gate_sig), rows, p.Hq, p.dk);
    }
    if (p.gate_mode == 6) {
        if (w.gate_splits != 1) return cudaErrorInvalidValue;   // (prefill plans one split)
        return launch_dependent(gate_average_logits_kernel, dim3((unsigned)((rows + 255) / 256)), dim3(256), 0, s,
                                reinterpret_cast<float*>(ws + w.gate_part), rows, p.Hq, p.gate_fn);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_gate_sigmoid_bf16(const Problem& p, const WorkspacePlan& w, char* ws, const Runtime& rt,
                                     cudaStream_t s, ZeroJob zero) {
    if (p.gate_mode == 5) {
        const int n = p.Hq * p.dk;
        return launch_dependent(gate_static_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s,
                                static_cast<const __nv_bfloat16*>(p.Wg), reinterpret_cast<__half*>(ws + w.gate_sig),
                                n, p.gate_fn, zero);
    }
    if (p.stats.out) return launch_gate_value_t<0, true>(p, w, ws, rt, s, zero);   // (sigmoid gate only)
    switch (p.gate_fn) {
    case 1: return launch_gate_value_t<1>(p, w, ws, rt, s, zero);
    case 3: return launch_gate_value_t<3>(p, w, ws, rt, s, zero);
    case 4: return launch_gate_value_t<4>(p, w, ws, rt, s, zero);
    default: return launch_gate_value_t<0>(p, w, ws, rt, s, zero);   // sigmoid (multiplied or added)
    }
}

}  // namespace gsdpa
