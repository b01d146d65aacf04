// Device helpers shared by the CUDA translation units of liboscar.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace oscar {

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
    return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}

// Loads element i of a K/V/q row stored as bf16 (dtype 0) or fp32 (dtype 1)
// and returns its bf16-rounded value when `to_bf16` is set.
__device__ __forceinline__ float load_elem(const void* base, int64_t i, int dtype) {
    if (dtype == 0) return bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(base)[i]);
    return reinterpret_cast<const float*>(base)[i];
}

// 2^x with the hardware approximation (ex2.approx.ftz.f32: relative error
// about 2^-22, subnormal results flushed to zero); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Block-wide exclusive scan of one int per thread (warp shuffles, then the
// warp totals); *total receives the sum.  scratch: one int per warp.  All
// threads of the block participate.
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? scratch[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        if (lane < nw) scratch[lane] = w;
    }
    __syncthreads();
    *total = scratch[nw - 1];
    return (warp ? scratch[warp - 1] : 0) + x - v;
}

// Programmatic dependent launch: wait for the previous grid of the stream (its
// completion and memory), then let the next grid be scheduled.  Both are no-ops
// for a grid launched without the programmatic attribute.
__device__ __forceinline__ void grid_dep_sync() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2 prefetch hint for the 128-byte line at p (no data returns; nothing waits).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

__device__ __forceinline__ void set_status(int* word, int bits) {
    if (word) atomicOr(word, bits);
}

// ---- mbarrier / bulk-copy primitives (inline PTX, sm_90+) -------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}

#ifndef OSCAR_MBAR_SUSPEND_NS
#define OSCAR_MBAR_SUSPEND_NS 0   // 0: the hardware's default time slice per try_wait
#endif

// Tests the phase with the given parity (a waiting thread may be suspended
// for a while before the test returns false).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
#if OSCAR_MBAR_SUSPEND_NS > 0
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity), "r"((unsigned)OSCAR_MBAR_SUSPEND_NS) : "memory");
#else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
#endif
    return ok != 0;
}

// Waits for the phase with the given parity to complete, for at most
// `budget` SM clock cycles.  On giving up it sets OSCAR_DEV_TIMEOUT in the
// status word, drops the caller's budget to zero (every later wait makes a
// single attempt) and returns false.  Callers carry on regardless (every
// address they use derives from indices, not from the awaited data), so warps
// that share named barriers stay matched and the kernel ends quickly.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* status,
                                                  long long& budget) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15u) == 0 && clock64() - t0 > budget) break;
    }
    set_status(status, 8 /* OSCAR_DEV_TIMEOUT */);
    budget = 0;
    return false;
}

// 4-byte asynchronous copy global -> shared (cp.async, completion by groups).
__device__ __forceinline__ void cp_async4(void* dst_smem, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(smem_addr(dst_smem)), "l"(src) : "memory");
}
// 8-byte asynchronous copy global -> shared (both addresses 8-byte aligned).
__device__ __forceinline__ void cp_async8(void* dst_smem, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" :: "r"(smem_addr(dst_smem)), "l"(src) : "memory");
}
// 16-byte asynchronous copy global -> shared (both addresses 16-byte aligned).
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_addr(dst_smem)), "l"(src) : "memory");
}
// Arrives on `bar` once every cp.async this thread issued before has landed
// (the arrival does not raise the barrier's pending count: the expected count
// at init must include it).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_addr(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// (s, z) of group gi from the pair array at `p`: fp16 pairs (4 bytes) or E4M3
// pairs (2 bytes); both convert exactly.
__device__ __forceinline__ float2 load_sz(const uint8_t* p, int gi, bool fp8) {
    if (fp8) {
        const unsigned short v = *reinterpret_cast<const unsigned short*>(p + 2 * gi);
        uint32_t h;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(v));     // exact: every E4M3 value is an fp16
        return __half22float2(*reinterpret_cast<const __half2*>(&h));
    }
    return __half22float2(*reinterpret_cast<const __half2*>(p + 4 * gi));
}

}  // namespace oscar
