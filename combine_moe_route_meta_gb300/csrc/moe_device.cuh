// moe_device.cuh -- device helpers shared by the route-meta, dispatch and combine kernels.
//
// Everything here is written for sm_103a. The number-format conversions use the
// hardware cvt instructions (round-to-nearest-even, satfinite); the library's GPU
// tests compare them exhaustively on their decision points against an independent
// CPU implementation of the formats.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe_dispatch.h"

namespace moe {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------
// status word: first error wins
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
    if (status != nullptr) atomicCAS(reinterpret_cast<int*>(status), MOE_OK, code);
}

// ---------------------------------------------------------------------------
// memory access with cache hints
// ---------------------------------------------------------------------------
// 16-byte read-only load that does not allocate in L1 (each byte is read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_v2(void* p, uint2 v) {
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// ---------------------------------------------------------------------------
// bf16 <-> fp32
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// two fp32 -> packed bf16x2, round-to-nearest-even; `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// unpack 8 bf16 (one uint4) into fp32
__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// ---------------------------------------------------------------------------
// FP8 E4M3 / FP4 E2M1 conversions (hardware cvt, RNE, satfinite)
// ---------------------------------------------------------------------------
// two fp32 -> two e4m3 codes in one 16-bit word; `lo` lands in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// two fp32 -> two e2m1 codes in one byte; `lo` lands in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// exact value of an e4m3 code (through f16, which holds every e4m3 value exactly)
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    uint32_t h2;
    uint16_t c = static_cast<uint16_t>(code & 0xffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
}

// ---------------------------------------------------------------------------
// block-wide staging of small metadata arrays into shared memory
// ---------------------------------------------------------------------------
// Each thread issues all of its loads (up to 8) before any of its stores, so the copy costs
// one memory round trip; a plain strided loop would wait for every load in turn.
template <typename Src>
__device__ __forceinline__ void stage_to_shared(const Src* __restrict__ src, int* dst, int n) {
    for (int j0 = threadIdx.x; j0 < n; j0 += 8 * int(blockDim.x)) {
        Src v[8];
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const int j = j0 + u * int(blockDim.x);
            v[u] = j < n ? __ldg(src + j) : Src(0);
        }
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const int j = j0 + u * int(blockDim.x);
            if (j < n) dst[j] = int(v[u]);
        }
    }
}

// ---------------------------------------------------------------------------
// bulk (TMA) copies and mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// make mbarrier initialisation visible to the async (bulk copy) proxy
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// global -> shared bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned);
// completion is signalled on `bar` as transaction bytes
__device__ __forceinline__ void bulk_load(uint32_t dst_smem, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst_smem),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// shared -> global bulk copy, tracked in the issuing thread's bulk group
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src_smem), "r"(bytes)
                 : "memory");
}
// the same with an L2 cache policy (createpolicy) for the written lines
__device__ __forceinline__ void bulk_store_hint(void* dst, uint32_t src_smem, uint32_t bytes, uint64_t policy) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
                 "r"(src_smem), "r"(bytes), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// L2 policy that keeps the lines it covers in L2 ahead of normally cached ones: for data that a
// later kernel of the same call reads back (the row-major scale rows of the swizzled layout).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void st_v4_hint(void* ptr, uint4 v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w), "l"(policy)
                 : "memory");
}
// wait until at most N of this thread's committed bulk groups still read shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// generic-proxy shared-memory writes become visible to later bulk copies
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Global nanosecond clock (%globaltimer).
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// One test of phase `parity` of an mbarrier (the thread may be suspended for a short,
// hardware-defined time while the phase is pending).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Limits of the bounded waits: a bulk row load normally lands within microseconds.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // ring waits: 1 s
constexpr uint64_t kDrainLimitNs = 100000000ull;  // draining loads after a timeout: 0.1 s
constexpr int kWaitMinPolls = 64;

// Bounded wait for phase `parity` of an mbarrier: true once the phase completes, false
// when it is still pending after limit_ns of wall-clock time and at least kWaitMinPolls
// tests (the poll floor keeps a long preemption of the context from counting as a
// timeout). The caller reports MOE_ERR_TIMEOUT instead of hanging.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    int polls = 1;
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (polls < kWaitMinPolls)
            polls++;
        else if (global_ns() - t0 > limit_ns)
            return false;
    }
}

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
// Wait until the kernels this launch depends on have completed and flushed memory.
// A no-op when the kernel was not launched as a programmatic dependent.
// No kernel here issues griddepcontrol.launch_dependents: a dependent is released as the
// blocks of the kernel before it exit. Releasing it at the start of a kernel let its blocks
// take SM resources while they waited, which slowed the large dispatch/combine steps by up to
// 30 % on GB300 (measured), and gained nothing at decode sizes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace moe
