// Bulk copies (TMA, 1-D cp.async.bulk) and mbarriers for sm_103a, in inline
// PTX. Only plain global -> own-CTA shared memory copies: no multicast.
//
// Every wait is bounded by the GPU's global nanosecond timer; a wait that runs
// out returns false and the caller records BEAM_ERR_TIMEOUT in the device
// status word instead of spinning forever.
#pragma once

#include <cstdint>

namespace beam {

// bulk prefetch of [p, p + bytes) into L2 (p and bytes multiples of 16)
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// L2 cache policies: evict_last keeps lines ahead of normal and evict_first
// ones; evict_first lines are the first to go. A later access with another
// policy sets the line's priority anew.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// The same prefetch, with the lines marked evict_last so that the write
// stream of the rows being finished does not push them out before they are
// read. Every caller reads the prefetched lines with an evict_first load (or
// overwrites them with evict_first stores), which drops the priority again:
// no evict_last line outlives the kernel.
__device__ __forceinline__ void prefetch_l2_keep(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;"
                 :: "l"(p), "r"(bytes), "l"(l2_evict_last()) : "memory");
}

// Programmatic dependent launch. A kernel launched with programmatic stream
// serialisation may start while the previous kernel on the stream still runs;
// pdl_wait() returns once that kernel has completed and its writes are
// visible (at once when the launch had no such dependency). pdl_trigger()
// lets the next kernel on the stream start its own prologue early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ unsigned int g_status_word;  // bit 0: a bounded wait gave up

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

// make the initialised barriers visible to the bulk-copy (async) proxy
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// one arrival that also announces `bytes` of transactions to come
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// wait for the phase with the given parity to complete, at most limit_ns
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// global -> shared bulk copy completing `bytes` transactions on `bar`
// (both addresses 16-byte aligned, bytes a multiple of 16)
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_u32(dst_smem)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void report_timeout() { atomicOr(&g_status_word, 1u); }

}  // namespace beam
