// Thin wrappers over the sm_100-family asynchronous-copy and barrier PTX used by
// the TMA-fed kernels: mbarriers (with bounded waits), 2-D tiled TMA loads,
// L2 cache policies.  Written from the PTX ISA's descriptions of
// mbarrier.*, cp.async.bulk.tensor.* and createpolicy.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace tfl {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

// Makes initialised mbarriers visible to the async proxy (TMA) and other threads.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `bar` with the given parity to complete.  Each
// try_wait suspends the thread in hardware until the phase completes or a
// short time limit passes, so the loop needs no sleep of its own and wakes as
// soon as the phase completes.  Gives up after `limit` polls or about a second
// (global timer), whichever comes first: sets kStatusDevice in *status and
// returns false, so a broken pipeline ends the kernel instead of hanging the GPU.
constexpr uint32_t kMbarSpinLimit = 1u << 24;
constexpr uint64_t kMbarWaitNs = 1000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                                          uint32_t limit = kMbarSpinLimit) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0u && global_ns() - t0 > kMbarWaitNs) break;
    }
    atomicOr(status, kStatusDevice);
    return false;
}

// The same wait that also gives up at once when *abort is raised (a wait
// between warps of one CTA whose partner may have stopped).
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                   int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1; i < kMbarSpinLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0u) {
            if (*abort) return false;
            if (global_ns() - t0 > kMbarWaitNs) break;
        }
    }
    atomicOr(status, kStatusDevice);
    *abort = 1;
    return false;
}

// After an abort: waits, bounded, for the copies of the last `issued` (at
// most depth) stages a producer armed on a ring of `depth` stages whose next
// stage is (stage, phase), so that no copy lands in shared memory after the
// CTA has exited.  Older stages were refilled only after their consumers
// released them, so their copies have landed.  A wait that runs out leaves
// kStatusDevice set.
__device__ __forceinline__ void drain_ring(uint64_t* full, int depth, int stage, uint32_t phase, long long issued,
                                           int* status) {
    const int n = issued < depth ? (int)issued : depth;
    for (int i = 0; i < n; ++i) {
        if (stage == 0) {
            stage = depth - 1;
            phase ^= 1u;
        } else {
            --stage;
        }
        mbar_wait(&full[stage], phase, status);
    }
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2-D tiled TMA load of the box at (x = inner element index, y = row) into
// shared memory; completion is counted in bytes on `bar`.  x * element size
// must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 3-D tiled TMA load of the box at (x, y, z) (x = innermost element index).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ bool elect_lane0() { return (threadIdx.x & 31) == 0; }

// Named barrier over `count` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// The same barrier returning whether `pred` held for any (or) / every (and)
// participating thread: a decision all of them share, so that no thread leaves
// a loop that others stay in (an abort flag read at different moments could
// otherwise differ between threads).
__device__ __forceinline__ bool named_barrier_or(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool named_barrier_and(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Address of 16-byte chunk c of row r in a tile written by TMA with 128-byte
// swizzling (rows of 128 bytes, 1024-byte aligned tile): chunks are permuted
// within each row by XOR with (row mod 8).
__device__ __forceinline__ const void* sw128_chunk(const void* tile, int r, int c) {
    return static_cast<const char*>(tile) + r * 128 + ((c ^ (r & 7)) << 4);
}

}  // namespace tfl
