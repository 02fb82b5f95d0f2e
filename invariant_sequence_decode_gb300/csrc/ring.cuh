// ring.cuh - pieces shared by the kernels that stream weights through a ring
// of shared-memory stages filled by the tensor memory accelerator (TMA):
// mbarrier operations, bounded waits, tiled tensor copies, and the host-side
// tensor-map cache and per-device launch state.
//
// Every wait here is bounded (about one second on the global timer and 2^26
// polls); a wait that runs out adds one to the calling file's device counter
// and returns false, so a stalled copy surfaces as a counted error instead of
// a hung stream.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"

namespace luce {

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // about one second

// Wait for the phase of parity `parity` to complete, for limit_ns at most
// (and at most 2^26 polls, should the timer not advance); false, with one
// more expiry counted in *counter, if it did not.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, unsigned int* counter,
                                          uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try(b, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t polls = 0; !mbar_try(b, parity); ++polls)
        if (global_ns() - t0 > limit_ns || polls >= (1u << 26)) {
            atomicAdd(counter, 1u);
            return false;
        }
    return true;
}

// Before a ring's producer thread returns: wait for the copies of the last
// stages it issued (stage it went to slot it % S, phase parity (it / S) & 1;
// no later phase of those slots follows), for kWaitLimitNs in all, so that
// no tensor copy is still landing in this CTA's shared memory once the CTA
// may exit - also after a consumer's or the producer's own wait expired.  On
// a healthy run the consumers wait for the same phases, so this waits for
// nothing they do not; it polls with a short sleep in between, leaving the
// issue slots to the consumer warps.  An expiry here is counted like any
// other.
template <int S>
__device__ __forceinline__ void ring_drain(uint64_t* full, int issued, unsigned int* counter)
{
    const uint64_t t0 = global_ns();
    for (int it = issued > S ? issued - S : 0; it < issued; ++it)
        for (uint32_t polls = 0; !mbar_try(&full[it % S], (it / S) & 1); ++polls) {
            if (global_ns() - t0 > kWaitLimitNs || polls >= (1u << 22)) {
                atomicAdd(counter, 1u);
                return;
            }
            __nanosleep(128);
        }
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, int x, int y, int z, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_addr(dst)),
        "l"(m), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, int x, int y, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_addr(dst)),
        "l"(m), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_addr(p)));
    return v;
}

// ---------------------------------------------------------------- host side

constexpr int kMaxDevices = 64;

// The calling thread's current device, or -1 (also when it is >= kMaxDevices).
int current_device();

// Multiprocessor count of the current device (cached per device); 0 on error.
int sm_count();

// A tiled tensor map of `rank` (2 or 3) dims (dims[0] innermost, strides in
// bytes for dims 1..rank-1), zero fill outside the tensor, with the given
// swizzle.  Maps are pure functions of their inputs and are kept in a small
// table keyed by them.  false when the driver refuses the map.
bool encode_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
                const cuuint64_t* strides, const cuuint32_t* box,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE);

// Raises `kernel`'s dynamic shared-memory limit to `bytes` once per device;
// `done` is the kernel's own per-device flag table.
template <typename Kern>
cudaError_t set_smem_once(Kern kernel, int bytes, std::atomic<bool> (&done)[kMaxDevices])
{
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
    return e;
}

}  // namespace luce
