// Device-side building blocks shared by the kernels: bulk-copy (TMA) and
// mbarrier PTX with bounded waits, programmatic dependent launch, warp
// reductions, fp16 decode, activations, and the device error word.
#pragma once
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace qg {

constexpr unsigned FULL = 0xffffffffu;

// Bits of the device error word (a kernel that gives up on a bounded wait sets
// one and returns; the host maps a non-zero word to QG_ERR_TIMEOUT).
enum : unsigned {
    DEVERR_FULL_WAIT = 1u,    // consumer waited too long for a bulk copy
    DEVERR_EMPTY_WAIT = 2u,   // producer waited too long for a free ring slot
    DEVERR_DRAIN_WAIT = 4u,   // copies still in flight at an error exit
};

// ~1-2 s at GB300 clocks: far above any legitimate wait, short enough that a
// broken pipeline returns an error instead of holding the GPU.
constexpr long long kWaitCycles = 2000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// A thread whose phase is not complete is suspended in hardware until it
// completes or kSuspendNs pass (the time-limit operand of try_wait), so a
// waiting warp takes no issue slots from the warps doing the work.
constexpr unsigned kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    unsigned done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return done != 0;
}
// Bounded wait for the phase with `parity` to complete; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
    if (mbar_try_wait(bar, parity)) return true;
    long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitCycles) return false;
    }
    return true;
}

// ------------------------------------------------------ bulk copy (TMA 1-D)
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// Global -> shared bulk copy completing on `bar`.  dst, src 16-byte aligned;
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Tiled 2-D tensor copy (TMA) of the box at element coordinates (x, y) of the
// tensor map at `tmap` (a __grid_constant__ kernel parameter) into shared
// memory at dst (128-byte aligned), completing on `bar`.  x times the element
// size must be a multiple of 16 bytes; rows past the tensor read as zeros and
// still count toward the box's bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Hint the TMA engine to pull [src, src + bytes) into L2 (no shared memory
// involved); src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Prefetch ranges for the kernel that runs next: each CTA of the current
// kernel pulls its 1/gridDim share of every range into L2, so that the next
// kernel's bulk copies hit L2 even when its CTAs become resident late.
struct L2Prefetch {
    const uint8_t* p[2];
    unsigned long long bytes[2];
    __device__ void issue() const {
        const unsigned long long nb = gridDim.x * gridDim.y;
        const unsigned long long id = blockIdx.x + static_cast<unsigned long long>(blockIdx.y) * gridDim.x;
        for (int i = 0; i < 2; ++i) {
            if (!p[i] || bytes[i] == 0) continue;
            const unsigned long long units = (bytes[i] + 15) / 16;  // 16-byte units
            const unsigned long long u0 = units * id / nb, u1 = units * (id + 1) / nb;
            for (unsigned long long u = u0; u < u1; u += 4096) {  // at most 64 KB per instruction
                const unsigned long long n = (u1 - u < 4096 ? u1 - u : 4096);
                bulk_prefetch_l2(p[i] + 16 * u, static_cast<unsigned>(16 * n));
            }
        }
    }
};

// ------------------------------------------- programmatic dependent launch
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Named barrier over the first `nthreads` threads (the consumer warps).
__device__ __forceinline__ void bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
    return v;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long w = __shfl_xor_sync(FULL, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// --------------------------------------------------------------- numerics
__device__ __forceinline__ float f16_to_f32(uint16_t bits) {
    return __half2float(__ushort_as_half(bits));
}
// x / (1 + exp(-x)) and 1 / (1 + exp(-x)) with the quotient taken as a
// reciprocal-multiply (2 ulp): activations of magnitude ~100 make exp(-x)
// overflow to inf, where an IEEE division would take its slow path; here the
// reciprocal of inf is 0 and the result the same signed zero.
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.0f + expf(-x)); }
__device__ __forceinline__ float sigmoid(float x) { return __fdividef(1.0f, 1.0f + expf(-x)); }
__device__ __forceinline__ float softplus(float x) { return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x))); }

// Loads of activations written by an earlier kernel: cached in L2 only.
__device__ __forceinline__ float ldcg(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float4 ldcg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

// Order-preserving key of a logit for a max-reduction that keeps the lowest
// index on ties: the float's total-order bits above (0xffffffff - index).
// -0 is folded into +0 (equal values tie); NaN maps to key 0 (never wins).
__device__ __forceinline__ unsigned long long argmax_key(float v, unsigned idx) {
    if (v != v) return 0ull;
    v = v + 0.0f;
    unsigned b = __float_as_uint(v);
    unsigned ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return (static_cast<unsigned long long>(ord) << 32) | (0xffffffffu - idx);
}
__device__ __forceinline__ unsigned argmax_key_index(unsigned long long key) {
    return 0xffffffffu - static_cast<unsigned>(key & 0xffffffffull);
}

}  // namespace qg
