// pa_device.cuh -- device-side building blocks for the sm_103a kernels:
// mbarrier waits with iteration limits, TMA tensor copies, bf16 unpacking,
// and the exp2 instruction.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedattn.h"

namespace pa {

// Every mbarrier wait gives up after this many polls (each poll may suspend
// the thread for a hardware-chosen time).  A healthy pipeline completes each
// wait within microseconds; giving up sets PA_DEV_TIMEOUT and ends the CTA.
constexpr uint32_t kWaitPollLimit = 1u << 20;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Non-blocking probe of a phase's completion (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}


// Waits for the phase with the given parity to complete.  Returns false if
// the poll limit ran out or *abort became non-zero (another thread gave up).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const volatile int *abort) {
    for (uint32_t i = 0; i < kWaitPollLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
    }
    return false;
}

// 4-D tiled TMA load global -> shared, completion signalled on `bar` as bytes.
// Coordinates are innermost first.  Out-of-range boxes are zero-filled.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1,
                                            int c2, int c3, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar)),
        "l"(policy)
        : "memory");
}

// 5-D tiled TMA load global -> shared (coordinates innermost first).
__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1,
                                            int c2, int c3, int c4, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_addr(bar)),
        "l"(policy)
        : "memory");
}

// Prefetch of a 5-D tiled box into L2 (no shared-memory destination, no
// completion to wait for); coordinates innermost first.
__device__ __forceinline__ void tma_prefetch_l2_5d(const CUtensorMap *map, int c0, int c1, int c2, int c3, int c4) {
    asm volatile("cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %2, %3, %4, %5}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
                 : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// bf16 pair in one 32-bit word -> two floats (exact: bf16 is the top half of fp32).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 2^x with the hardware approximation instruction (ex2.approx, relative error
// about 2^-22); exp2(-inf) = +0.
// max(a, b, c) in one instruction (three-input max.f32, sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Per-warpgroup register budget (all 128 threads of the warpgroup execute it):
// dec returns registers to the CTA's pool, inc waits until the pool holds
// enough.  The sum over warpgroups must stay within what the CTA was launched
// with (threads x registers per thread at launch); the host checks the
// kernel's launch register count before it launches a kernel that uses these.
template <int R>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}

// Named barrier over the first `threads` threads of the CTA (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// x = head + residual with both parts in bf16 (packed pairs for elements a, b).
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t &head, uint32_t &resid) {
    head = pack_bf16(a, b);
    const float2 h = make_float2(__uint_as_float(head << 16), __uint_as_float(head & 0xffff0000u));
    const float2 r = __ffma2_rn(h, make_float2(-1.f, -1.f), make_float2(a, b));  // (a, b) - head, exact
    resid = pack_bf16(r.x, r.y);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// The same split with both parts in f16.
__device__ __forceinline__ void split_f16(float a, float b, uint32_t &head, uint32_t &resid) {
    head = pack_f16(a, b);
    const float2 h = __half22float2(*reinterpret_cast<const __half2 *>(&head));
    const float2 r = __ffma2_rn(h, make_float2(-1.f, -1.f), make_float2(a, b));
    resid = pack_f16(r.x, r.y);
}

// The fp8-cache kernels multiply in f16, so q (bf16, 8 exponent bits) is
// brought into f16's range first: the row (or head) is scaled by the power of
// two 2^e that puts its largest |element| in [2^14, 2^15), and 2^-e joins the
// softmax scale.  `amax` is the largest bf16 bit pattern of the row with the
// sign cleared (for non-NaN values the integer order is the order of the
// magnitudes), E its exponent field, e = 141 - E, kept in [-100, 64] so that
// both 2^e and scale * 2^-e are normal binary32 numbers.  Every element
// within 2^38 of the largest keeps all its bits (f16 subnormals reach 2^-24).
__device__ __forceinline__ float f16_prescale(uint32_t amax) {
    const int e = min(64, max(-100, 141 - (int)(amax >> 7)));
    return __uint_as_float((uint32_t)(127 + e) << 23);
}

// The larger magnitude of a bf16 pair, as a bit pattern with the sign cleared.
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t w) {
    return max(w & 0x7fffu, (w >> 16) & 0x7fffu);
}

// Two bf16 (packed) times a power of two -> two f16 (packed), exact when the
// scaled values lie in f16's normal range.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float s) {
    return pack_f16(__uint_as_float(w << 16) * s, __uint_as_float(w & 0xffff0000u) * s);
}

// Eight bf16 (one 16-byte vector) -> eight e4m3 codes of x / s: the division
// in binary32, rounding to nearest even and saturating to +-448
// (cvt ... satfinite); the quantiser of the fp8 cache.
__device__ __forceinline__ uint32_t e4m3x2_div(uint32_t two_bf16, float s) {
    const float lo = __fdiv_rn(bf16lo(two_bf16), s), hi = __fdiv_rn(bf16hi(two_bf16), s);
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint2 e4m3x8_div(uint4 w, float s) {
    return make_uint2(e4m3x2_div(w.x, s) | (e4m3x2_div(w.y, s) << 16), e4m3x2_div(w.z, s) | (e4m3x2_div(w.w, s) << 16));
}

// Bulk copy shared -> global of `bytes` (a multiple of 16; both addresses
// 16-byte aligned) in the calling thread's bulk group.
__device__ __forceinline__ void bulk_store_s2g(void *gdst, const void *ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_addr(ssrc)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk copy of this thread has read its source
// (the shared memory may then be reused; the writes complete before the grid
// does).
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

__device__ __forceinline__ void set_status(int32_t *status, int bits) {
    if (status) atomicOr(status, bits);
}

}  // namespace pa
