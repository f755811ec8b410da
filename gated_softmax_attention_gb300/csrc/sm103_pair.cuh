// sm103_pair.cuh -- inline-PTX building blocks for kernels that run on a pair
// of CTAs (a cluster of two, one per SM) sharing tcgen05 MMAs with
// .cta_group::2: the even CTA issues every MMA; each MMA reads the A rows and
// one half of the B columns from each CTA's shared memory (or A from each
// CTA's tensor memory) at the same offsets, and writes each CTA's 128 rows of
// D into that CTA's tensor memory.
//
// Barriers that the issuing CTA waits on live in its shared memory and the
// other CTA reaches them through `mapa`; MMA completions are multicast to the
// same barrier offset in both CTAs. Written from the PTX ISA's descriptions
// of these instructions; no library headers are used.
#pragma once
#include "sm103_ptx.cuh"

namespace gsdpa {
namespace pair {

__device__ __forceinline__ uint32_t cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t n_clusters() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Every thread of both CTAs; orders earlier shared-memory writes (barrier
// initialisation) before anything the other CTA does after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address, in the cluster shared window, of the object at `p` (a local
// shared-memory pointer) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to(const void* p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    return a;
}

// Arrive on a barrier given by its cluster address (either CTA). Default
// (CTA-scope release) semantics: what the arrival publishes here is tensor
// memory, ordered by tcgen05.wait::st and tcgen05.fence::before_thread_sync
// in the arriving thread and tcgen05.fence::after_thread_sync in the waiter;
// a cluster-scope release would cost about a thousand cycles per arrival.
__device__ __forceinline__ void arrive_remote(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
// Cluster-scope release arrive: orders this thread's earlier stores to the
// other CTA's shared memory before the arrival (rare: about a thousand cycles).
__device__ __forceinline__ void arrive_remote_release(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
// Wait with cluster-scope acquire (pairs with arrive_remote_release).
__device__ __forceinline__ bool try_wait_acquire_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void store_remote_u32(uint32_t addr_cluster, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr_cluster), "r"(v) : "memory");
}

// Bounded wait (see mbar_wait): on giving up it records ERR_WAIT_TIMEOUT and
// raises the abort flag of both CTAs, so that the other CTA's waits end too.
// The limit is checked after the first unsuccessful retry and then every 32
// tries (each try may suspend the thread for a while), so that a wait that is
// not over at once gives up promptly under a tiny limit.
struct PairAbort {
    volatile int* local;   // this CTA's flag
    uint32_t peer;         // the other CTA's flag, cluster address
};
static __device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity, const PairAbort& ab, const WaitCtl& ctl) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 1) {
            if (*ab.local) return false;
            if (globaltimer_ns() - t0 > ctl.limit_ns) {
                atomicOr(ctl.err, ERR_WAIT_TIMEOUT);
                *ab.local = 1;
                store_remote_u32(ab.peer, 1u);
                __threadfence_block();
                return false;
            }
        }
    }
}

// wait() with cluster-scope acquire, for barriers armed by arrive_remote_release.
static __device__ __forceinline__ bool wait_acquire_cluster(uint64_t* bar, uint32_t parity, const PairAbort& ab,
                                                            const WaitCtl& ctl) {
    if (try_wait_acquire_cluster(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (try_wait_acquire_cluster(bar, parity)) return true;
        if ((it & 31u) == 1) {
            if (*ab.local) return false;
            if (globaltimer_ns() - t0 > ctl.limit_ns) {
                atomicOr(ctl.err, ERR_WAIT_TIMEOUT);
                *ab.local = 1;
                store_remote_u32(ab.peer, 1u);
                __threadfence_block();
                return false;
            }
        }
    }
}

// TMA tile loads into this CTA's shared memory whose completion (bytes) is
// signalled on a barrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, int c0, int c1, int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* m, int c0, int c1, int c2, int c3, int c4,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
        : "memory");
}

// Tensor memory for the pair: one warp of EACH CTA executes these together.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Pair MMAs, issued by one elected lane of a converged warp of the even CTA.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, uint32_t b_hi,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b64 da, db;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "mov.b64 da, {%1, %2};\n\t"
        "mov.b64 db, {%3, %4};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b64 db;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "mov.b64 db, {%2, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive (once) on the barrier at `bar`'s offset in both CTAs when every MMA
// issued so far by this thread has completed.
__device__ __forceinline__ void commit_both(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
            smem_u32(bar)),
        "h"((unsigned short)3)
        : "memory");
}

}  // namespace pair
}  // namespace gsdpa

namespace gsdpa {
namespace pair {
// Pair forms of mma_ss_k128 / mma_ts_k128 (cta_group::2, issued by the even CTA).
template <uint32_t A_BLK, uint32_t B_BLK>
__device__ __forceinline__ void mma_ss_k128(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b32 al, bl;\n\t.reg .b64 da, db;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "mov.b64 da, {%1, %3};\n\t"
        "mov.b64 db, {%2, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %4, p;\n\t"
        "add.u32 al, %1, 2;\n\t"
        "add.u32 bl, %2, 2;\n\t"
        "mov.b64 da, {al, %3};\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %4, 1;\n\t"
        "add.u32 al, %1, 4;\n\t"
        "add.u32 bl, %2, 4;\n\t"
        "mov.b64 da, {al, %3};\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %4, 1;\n\t"
        "add.u32 al, %1, 6;\n\t"
        "add.u32 bl, %2, 6;\n\t"
        "mov.b64 da, {al, %3};\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %4, 1;\n\t"
        "add.u32 al, %1, %6;\n\t"
        "add.u32 bl, %2, %10;\n\t"
        "mov.b64 da, {al, %3};\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %4, 1;\n\t"
        "add.u32 al, %1, %7;\n\t"
        "add.u32 bl, %2, %11;\n\t"
        "mov.b64 da, {al, %3};\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %4, 1;\n\t"
        "add.u32 al, %1, %8;\n\t"
        "add.u32 bl, %2, %12;\n\t"
        "mov.b64 da, {al, %3};\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %4, 1;\n\t"
        "add.u32 al, %1, %9;\n\t"
        "add.u32 bl, %2, %13;\n\t"
        "mov.b64 da, {al, %3};\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %4, 1;\n\t"
        "}"
        ::"r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate),
        "n"((A_BLK >> 4) + 0), "n"((A_BLK >> 4) + 2), "n"((A_BLK >> 4) + 4), "n"((A_BLK >> 4) + 6),
        "n"((B_BLK >> 4) + 0), "n"((B_BLK >> 4) + 2), "n"((B_BLK >> 4) + 4), "n"((B_BLK >> 4) + 6)
        : "memory");
}
__device__ __forceinline__ void mma_ts_k128(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t hi,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b32 ta, bl;\n\t.reg .b64 db;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "mov.b64 db, {%2, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], db, %4, p;\n\t"
        "add.u32 ta, %1, 8;\n\t"
        "add.u32 bl, %2, 128;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], db, %4, 1;\n\t"
        "add.u32 ta, %1, 16;\n\t"
        "add.u32 bl, %2, 256;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], db, %4, 1;\n\t"
        "add.u32 ta, %1, 24;\n\t"
        "add.u32 bl, %2, 384;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], db, %4, 1;\n\t"
        "add.u32 ta, %1, 32;\n\t"
        "add.u32 bl, %2, 512;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], db, %4, 1;\n\t"
        "add.u32 ta, %1, 40;\n\t"
        "add.u32 bl, %2, 640;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], db, %4, 1;\n\t"
        "add.u32 ta, %1, 48;\n\t"
        "add.u32 bl, %2, 768;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], db, %4, 1;\n\t"
        "add.u32 ta, %1, 56;\n\t"
        "add.u32 bl, %2, 896;\n\t"
        "mov.b64 db, {bl, %3};\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], db, %4, 1;\n\t"
        "}"
        ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate)
        : "memory");
}
}  // namespace pair
}  // namespace gsdpa
