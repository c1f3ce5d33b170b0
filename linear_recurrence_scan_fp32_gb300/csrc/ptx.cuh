// ptx.cuh -- thin inline-PTX wrappers used by the sm_103a kernels:
// mbarrier phases, TMA tensor loads into shared memory, and the gpu-scope
// relaxed 64-bit words that carry look-back state between CTAs.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace linrec {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier -------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make the initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.
// Returns false if it did not complete within max_polls polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t max_polls) {
    for (uint32_t i = 0; i < max_polls; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i > 64) __nanosleep(256);
    }
    return false;
}

// ---- programmatic dependent launch ------------------------------------------
// A kernel launched with launch_dependent() may be scheduled while the work before
// it on the stream is finishing.  pdl_wait() blocks until that work has completed
// and its writes are visible: every thread calls it before its first access to
// global memory.  pdl_release() lets the launch after this one be scheduled (a
// CTA calls it when its own work is done; exiting counts as well).

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// A barrier for `threads` threads (a multiple of 32) of the CTA on hardware barrier `id`
// (1 .. 15; 0 is __syncthreads): lets groups of warps synchronise among themselves.
__device__ __forceinline__ void bar_sync_group(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---- TMA ------------------------------------------------------------------

__device__ __forceinline__ void tmap_prefetch(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled tensor load of one box into shared memory, completing on `bar`.
// Coordinates are element indices {x = innermost, y, z}; x*4 bytes must be a
// multiple of 16 for fp32 (the callers pass x as a multiple of the tile width,
// itself a multiple of 4).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
          "r"(smem_u32(bar))
        : "memory");
}

// ---- gpu-scope relaxed 64-bit words ---------------------------------------
// A look-back word packs {tag (high 32 bits), fp32 value bits (low 32)} so a
// reader sees the tag and the value from one single-copy-atomic access.

__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Two adjacent words in one access; each 64-bit element is itself single-copy atomic.
__device__ __forceinline__ void st_relaxed_v2_u64(unsigned long long *p, unsigned long long x, unsigned long long y) {
    asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(x), "l"(y) : "memory");
}

__device__ __forceinline__ void ld_relaxed_v2_u64(const unsigned long long *p, unsigned long long &x,
                                                  unsigned long long &y) {
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(x), "=l"(y) : "l"(p) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long pack_word(uint32_t tag, float v) {
    return (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(v);
}
__device__ __forceinline__ uint32_t word_tag(unsigned long long w) { return static_cast<uint32_t>(w >> 32); }
__device__ __forceinline__ float word_val(unsigned long long w) {
    return __uint_as_float(static_cast<uint32_t>(w & 0xffffffffull));
}

// A launch tags its words with tag_of(epoch); the last CTA to finish stores
// next_epoch(epoch).  Tags run through 1 .. 2^32 - 1 (0 is never a tag, so zeroed
// memory never reads as published) and two consecutive launches never share one,
// whatever value the epoch word holds, 0xffffffff included.
__device__ __forceinline__ uint32_t tag_of(uint32_t epoch) { return epoch % 0xffffffffu + 1u; }
__device__ __forceinline__ uint32_t next_epoch(uint32_t epoch) { return tag_of(epoch) % 0xffffffffu; }

}  // namespace linrec
