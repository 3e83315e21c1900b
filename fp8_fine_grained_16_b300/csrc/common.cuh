// common.cuh -- shared device helpers for libfp8bs: argument checks, E4M3
// conversion, and thin inline-PTX wrappers for the Blackwell async machinery
// (mbarrier, TMA bulk tensor copies, tcgen05 MMA / tensor memory).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp8bs.h"

#define FP8_DEV __device__ __forceinline__

namespace fp8bs {

constexpr float kE4M3Max = 448.0f;
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;   // 2 s for any single pipeline wait

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- bf16 / E4M3
FP8_DEV float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
FP8_DEV float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> two E4M3 codes, round to nearest even, saturating to +-448.
// Returns the pair packed little-endian: byte 0 = lo, byte 1 = hi.
FP8_DEV uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two fp32 -> bf16x2 (round to nearest even), lo in the low half.
FP8_DEV uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Scale of one tile from its max-abs value.  Returns s, writes inv.
// Default: s = amax/448, inv = 448/amax (IEEE divisions).  pow2: s = 2^e with
// e the least integer such that 448*2^e >= amax, taken from the fp32 bits.
FP8_DEV float tile_scale(float amax, bool pow2, float& inv) {
    float a = fmaxf(amax, 0x1p-64f);
    if (!pow2) {
        inv = __fdiv_rn(kE4M3Max, a);
        return __fdiv_rn(a, kE4M3Max);
    }
    uint32_t bits = __float_as_uint(a);              // a is normal (>= 2^-64)
    int E = int((bits >> 23) & 0xFFu) - 127;
    uint32_t frac = bits & 0x7FFFFFu;                // mantissa - 1 in units of 2^-23
    int e = (frac <= 0x600000u) ? E - 8 : E - 7;      // 0x600000 = 0.75 * 2^23 (448 = 1.75 * 2^8)
    inv = __uint_as_float(uint32_t(127 - e) << 23);
    return __uint_as_float(uint32_t(127 + e) << 23);
}

// ---------------------------------------------------------------- dependent launches
// A kernel launched with programmatic stream serialisation (launch_pdl, or
// the GEMMs' own launches) may start while the kernel before it on the stream
// is still running; it must call pdl_wait() before it reads anything that
// kernel writes (the wait returns once that kernel has completed and its
// writes are visible; in a kernel launched without the attribute it returns
// at once).  pdl_launch_dependents() lets the next such kernel start early.
FP8_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
FP8_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- misc PTX
FP8_DEV uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

FP8_DEV uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
FP8_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
FP8_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

FP8_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
FP8_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
FP8_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of the phase (much cheaper than try_wait when the
// phase has already completed).
FP8_DEV bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with the given parity, giving up after
// timeout_ns or as soon as *abort becomes non-zero.  On a timeout the waiter
// raises *abort itself.  Returns true when the phase completed.  A phase that
// is already complete is caught by the non-blocking probe first.
FP8_DEV bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                               uint64_t timeout_ns = kWaitTimeoutNs) {
    if (mbar_test_wait(bar, parity)) return true;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                *abort = 1;
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------- TMA
FP8_DEV void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
FP8_DEV void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}
FP8_DEV void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
FP8_DEV void tma_load_1d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t c0) {
    asm volatile(
        "cp.async.bulk.tensor.1d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0)
        : "memory");
}

// Tensor store from this CTA's shared memory (the box of `map` at (c0, c1)),
// tracked by the issuing thread's bulk-async groups.
FP8_DEV void tma_store_2d(const CUtensorMap* map, const void* src, int32_t c0, int32_t c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(c0), "r"(c1)
                 : "memory");
}
FP8_DEV void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every committed store of this thread has finished reading shared memory
FP8_DEV void bulk_wait_group_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// all but the most recent committed store of this thread have finished reading shared memory
FP8_DEV void bulk_wait_group_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// every committed store of this thread is complete
FP8_DEV void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// shared-memory writes of this thread made visible to the async proxy (TMA)
FP8_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---------------------------------------------------------------- tcgen05
// Ordering of tcgen05 operations around thread synchronisation (barriers,
// mbarrier waits) between the threads that issue and observe them.
FP8_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
FP8_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// One CTA: TMEM allocation (one warp), MMA and commit.
FP8_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
FP8_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
FP8_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D(tmem) (+)= A(smem) * B(smem)^T, E4M3 x E4M3 -> F32, one CTA (M = 128).
FP8_DEV void umma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every tcgen05 op this thread issued is done.
FP8_DEV void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// ---------------------------------------------------------------- CTA pairs
// A cluster of two CTAs on neighbouring SMs drives one tcgen05 MMA of M=256
// (each CTA holds 128 rows of A and half of the B tile in its own shared
// memory at the same offsets; each CTA's TMEM receives its 128 rows of D).
FP8_DEV uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Shared-memory address of the same variable in CTA `rank` of the cluster.
FP8_DEV uint32_t mapa_shared(const void* p, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
    return out;
}
// Arrive on an mbarrier given by its shared::cluster address (possibly the peer's).
FP8_DEV void mbar_arrive_cluster(uint32_t bar_cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster_addr) : "memory");
}
// All threads of both CTAs: arrive and wait (release / acquire at cluster scope).
FP8_DEV void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// TMA tile loads into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (given as a shared::cluster address).
FP8_DEV void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster_addr, int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(c0), "r"(c1)
        : "memory");
}
FP8_DEV void tma_load_3d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster_addr, int32_t c0, int32_t c1,
                              int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// TMEM allocation shared by the pair: one warp of each CTA executes it.
FP8_DEV void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
FP8_DEV void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
FP8_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D(tmem of both CTAs) (+)= A(smem of both) * B(smem of both)^T, E4M3 -> F32,
// issued by one thread of the leader CTA.
FP8_DEV void umma_e4m3_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// When every tcgen05 op this thread issued is done, arrive once on the
// mbarrier at this shared offset in each CTA of `cta_mask`.
FP8_DEV void umma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Block-scaled form (kind::mxf8f6f4, one UE8M0 scale per 32 K elements per
// row of A and per row of B): D (+)= (sA .* A) * (sB .* B)^T over K = 32, the
// scales read from tensor memory at sfa / sfb.  Where each scale sits (each
// CTA's own TMEM, measured on B300):
//   A row m (of the CTA's 128)    lane m,                    column sfa + m/32
//   B row n, for D rows in lanes  lanes 32q .. 32q+31 (every column sfb + n/32,
//     32q .. 32q+31                q), at lane 32q + n%32
// and in each 32-bit word the byte chosen by the scale-ID fields of idesc.
// Called by a whole converged warp: one lane, picked by elect.sync, issues
// the MMA (the operands are warp-uniform, so they stay in uniform registers).
// PAIR: cta_group::2 (M = 256 across a CTA pair); otherwise cta_group::1.
template <bool PAIR>
FP8_DEV void umma_mx_e4m3_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                uint32_t sfb, uint32_t accumulate) {
    if constexpr (PAIR)
        asm volatile(
            "{\n\t.reg .pred pe, pa;\n\t"
            "elect.sync _|pe, 0xffffffff;\n\t"
            "setp.ne.b32 pa, %6, 0;\n\t"
            "@pe tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], pa;\n\t}" ::"r"(
                d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred pe, pa;\n\t"
            "elect.sync _|pe, 0xffffffff;\n\t"
            "setp.ne.b32 pa, %6, 0;\n\t"
            "@pe tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], pa;\n\t}" ::"r"(
                d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
}

// The same MMA (accumulating), issued between a non-blocking probe of one or
// two mbarrier phases and the use of the probe's result, so that the probe's
// latency overlaps the issue of the MMA (which waits for the tensor core to
// accept it).  Returns true when every probed phase has completed; with
// bar1 == 0 only bar0 is probed.  Whole converged warp, as above.
template <bool PAIR>
FP8_DEV bool umma_mx_e4m3_probe_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                      uint32_t sfb, uint32_t bar0, uint32_t par0, uint32_t bar1, uint32_t par1) {
    uint32_t ok;
    if constexpr (PAIR)
        asm volatile(
            "{\n\t.reg .pred p0, p1, pe;\n\t"
            "mbarrier.test_wait.parity.shared::cta.b64 p0, [%7], %8;\n\t"
            "setp.eq.u32 p1, %9, 0;\n\t"
            "@!p1 mbarrier.test_wait.parity.shared::cta.b64 p1, [%9], %10;\n\t"
            "elect.sync _|pe, 0xffffffff;\n\t"
            "@pe tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], %2, %3, %4, [%5], [%6], 1;\n\t"
            "and.pred p0, p0, p1;\n\t"
            "selp.u32 %0, 1, 0, p0;\n\t}"
            : "=r"(ok)
            : "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(bar0), "r"(par0), "r"(bar1),
              "r"(par1)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p0, p1, pe;\n\t"
            "mbarrier.test_wait.parity.shared::cta.b64 p0, [%7], %8;\n\t"
            "setp.eq.u32 p1, %9, 0;\n\t"
            "@!p1 mbarrier.test_wait.parity.shared::cta.b64 p1, [%9], %10;\n\t"
            "elect.sync _|pe, 0xffffffff;\n\t"
            "@pe tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], %2, %3, %4, [%5], [%6], 1;\n\t"
            "and.pred p0, p0, p1;\n\t"
            "selp.u32 %0, 1, 0, p0;\n\t}"
            : "=r"(ok)
            : "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(bar0), "r"(par0), "r"(bar1),
              "r"(par1)
            : "memory");
    return ok != 0;
}

// umma_commit issued by one elected lane of a converged warp (one CTA).
FP8_DEV void umma_commit_elect(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred pe;\n\t"
        "elect.sync _|pe, 0xffffffff;\n\t"
        "@pe tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

// umma_commit_pair issued by one elected lane of a converged warp.
FP8_DEV void umma_commit_pair_elect(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "{\n\t.reg .pred pe;\n\t"
        "elect.sync _|pe, 0xffffffff;\n\t"
        "@pe tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Stores into tensor memory: thread i of the warp writes lane (base lane + i),
// 4 or 8 consecutive 32-bit columns from `col` (taddr = lane << 16 | col).
FP8_DEV void tmem_st_32x32b_x4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v0), "r"(v1),
                 "r"(v2), "r"(v3)
                 : "memory");
}
FP8_DEV void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}
FP8_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns; thread i of the warp gets lane
// (base lane + i), columns [col, col+32).
FP8_DEV void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}
// 32 lanes x 64 consecutive 32-bit columns into one register array.
FP8_DEV void tmem_ld_32x32b_x64(uint32_t taddr, uint32_t (&v)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]),
          "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]),
          "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]),
          "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]),
          "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
        : "r"(taddr)
        : "memory");
}
// 16 lanes x 128 consecutive 32-bit columns (shape 16x256b, 16 repetitions)
// into 64 registers.  Thread t of the warp gets, for repetition k (columns
// 8k .. 8k+7): v[4k], v[4k+1] = lane base + t/4, columns 8k + 2(t%4) and
// 8k + 2(t%4) + 1; v[4k+2], v[4k+3] = the same columns of lane base + 8 + t/4
// (measured on B300 against a 32x32b store).
FP8_DEV void tmem_ld_16x256b_x16(uint32_t taddr, uint32_t (&v)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]),
          "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]),
          "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]),
          "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]),
          "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
        : "r"(taddr)
        : "memory");
}
// tcgen05.wait::ld naming the 64 registers a preceding x64 load wrote.
FP8_DEV void tmem_wait_ld_regs64(uint32_t (&v)[64]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
          "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]),
          "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]),
          "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31]),
          "+r"(v[32]), "+r"(v[33]), "+r"(v[34]), "+r"(v[35]), "+r"(v[36]), "+r"(v[37]), "+r"(v[38]), "+r"(v[39]),
          "+r"(v[40]), "+r"(v[41]), "+r"(v[42]), "+r"(v[43]), "+r"(v[44]), "+r"(v[45]), "+r"(v[46]), "+r"(v[47]),
          "+r"(v[48]), "+r"(v[49]), "+r"(v[50]), "+r"(v[51]), "+r"(v[52]), "+r"(v[53]), "+r"(v[54]), "+r"(v[55]),
          "+r"(v[56]), "+r"(v[57]), "+r"(v[58]), "+r"(v[59]), "+r"(v[60]), "+r"(v[61]), "+r"(v[62]), "+r"(v[63])
        :
        : "memory");
}

// tcgen05.wait::ld that also names the registers a preceding tcgen05.ld
// wrote, so that the compiler cannot move their uses above the wait.
FP8_DEV void tmem_wait_ld_regs(uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
          "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]),
          "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]),
          "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
        :
        : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored as rows
// of 128 bytes with the 128-byte swizzle (the layout a TMA load with
// CU_TENSOR_MAP_SWIZZLE_128B writes).  Groups of 8 rows are 1024 bytes apart.
// The tile base must be 1024-byte aligned; stepping along K inside the
// 128-byte row is done by adding the byte offset to the start address.
FP8_DEV uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFFu);     // start address >> 4
    d |= uint64_t(1) << 16;                     // leading byte offset (unused for swizzled K-major)
    d |= uint64_t(1024 >> 4) << 32;             // stride byte offset: 8 rows x 128 B
    d |= uint64_t(1) << 46;                     // descriptor version for tcgen05
    d |= uint64_t(2) << 61;                     // swizzle mode: 128B
    return d;
}

// Instruction descriptor, kind::f8f6f4: D = F32, A = B = E4M3, both K-major,
// tile M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4)                     // D format: F32
           | (0u << 7) | (0u << 10)      // A, B format: E4M3
           | (0u << 15) | (0u << 16)     // A, B K-major
           | (uint32_t(N >> 3) << 17)    // N / 8
           | (uint32_t(M >> 4) << 24);   // M / 16
}

// Instruction descriptor, kind::mxf8f6f4 with block scaling: D = F32,
// A = B = E4M3, both K-major, tile M x N, UE8M0 scales, scale byte 0 of each
// 32-bit TMEM word for both A and B.
__host__ __device__ constexpr uint32_t idesc_mx_e4m3(int M, int N) {
    return (0u << 4)                     // B scale byte (scale ID)
           | (0u << 7) | (0u << 10)      // A, B format: E4M3
           | (0u << 15) | (0u << 16)     // A, B K-major
           | (uint32_t(N >> 3) << 17)    // N / 8
           | (1u << 23)                  // scale format: UE8M0
           | (uint32_t(M >> 4) << 24)    // M / 16
           | (0u << 29);                 // A scale byte (scale ID)
}

}  // namespace fp8bs
