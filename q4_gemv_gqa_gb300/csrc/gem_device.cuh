// gem_device.cuh — device-side building blocks shared by the sm_103a kernels:
// mbarrier + TMA (cp.async.bulk.tensor) staging, programmatic dependent launch,
// bounded waits that report instead of hanging, and small numeric helpers.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "gem_internal.h"

namespace gem {

// ---- programmatic dependent launch --------------------------------------------------
// The rule every kernel of the library keeps:
//   (1) a thread executes pdl_trigger() only after it has itself returned from pdl_wait()
//       (pdl_wait_trigger() does both), and no other thread of the CTA triggers earlier;
//   (2) every CTA executes pdl_wait() (in at least one thread) before it exits.
// griddepcontrol.wait returns once the preceding kernel of the stream has completed and its
// writes are visible.  So by (1) the next kernel is launched only when every CTA of this one
// has passed its wait, i.e. when the kernel BEFORE this one has completed; and by (2) the
// completion of a kernel implies the completion of every earlier one.  Consequently a kernel
// may read before its own pdl_wait() any data that the immediately preceding kernel does not
// write: weights, positions, and K/V rows written by any kernel two or more launches back
// (the previous decode step's appended rows included).  Data written by the immediately
// preceding kernel is read only after the wait.  Nothing is written before the wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_trigger() {
    pdl_wait();
    pdl_trigger();
}

// ---- shared-memory addresses and mbarriers --------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// ---- run-time controls of the bounded waits ----------------------------------------------
// Each translation unit with kernels holds its own copy of these two words (module-scope
// device variables exist per module); gem_set_wait_limit() and gem_set_test_injection()
// write every registered copy on the current device.
//   g_wait_limit_ns  wall-time limit of every device-side wait (default GEM_WAIT_LIMIT_NS);
//   g_test_inject    GEM_INJECT_* bits: make one bounded wait run out on purpose (tests of
//                    the timeout path; 0 in normal use).
static __device__ unsigned long long g_wait_limit_ns = GEM_WAIT_LIMIT_NS;
static __device__ int g_test_inject = 0;
namespace {
struct DeviceControlsRegistration {
    DeviceControlsRegistration() { register_device_controls(&g_wait_limit_ns, &g_test_inject); }
};
const DeviceControlsRegistration g_device_controls_registration;
}  // namespace

__device__ __forceinline__ uint64_t wait_limit_ns() {
    return *reinterpret_cast<const volatile unsigned long long*>(&g_wait_limit_ns);
}
__device__ __forceinline__ int test_inject() { return *reinterpret_cast<const volatile int*>(&g_test_inject); }

// Wait for phase `parity` of `bar`.  Gives up after wait_limit_ns() of wall time, records
// GEM_DEVFLAG_TIMEOUT in *status and returns false.  A healthy wait takes microseconds;
// the limit only guards against a copy that never lands.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const uint64_t limit = wait_limit_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit) {
            if (status) atomicOr(status, GEM_DEVFLAG_TIMEOUT);
            return false;
        }
    }
}

// After a wait gave up: give the copies of ring stages [first, last] a bounded chance to
// land before the CTA exits, so none of them writes into shared memory it no longer owns.
// Called by the thread that issued the copies.
__device__ __forceinline__ void drain_stages(uint64_t* bars, int ns, int first, int last) {
    for (int s = first; s <= last; ++s) (void)mbar_wait(&bars[s % ns], static_cast<uint32_t>((s / ns) & 1), nullptr);
}

// Words that a kernel sets to zero for a later launch (CTA 0's threads, after the wait).
__device__ __forceinline__ void clear_words(unsigned* w, int n, int tid, int nthreads) {
    if (w && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        for (int i = tid; i < n; i += nthreads) w[i] = 0u;
}

// ---- TMA -------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int32_t c0, int32_t c1,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// ---- warp helpers ----------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Packed fp32 pair FMA (one instruction for two lanes of arithmetic).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t ra, rb, rc, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

// Packed fp32 pair add.
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    uint64_t ra, rb, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

// ---- tensor-core fragments (mma.sync m16n8k16, f16 inputs, f32 accumulate) ---------------
__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                            uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t& r0, uint32_t& r1, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x2_trans(uint32_t& r0, uint32_t& r1, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                                  uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// fp32 -> (hi, lo) binary16 pair with hi + lo == x to about 2^-22 relative.
__device__ __forceinline__ void split_hi_lo(float x, __half& hi, __half& lo) {
    hi = __float2half_rn(x);
    lo = __float2half_rn(x - __half2float(hi));
}

// ---- shared by the RoPE and attention paths ----------------------------------------------
// cos and sin of an fp64 angle in fp32: the angle is reduced to [-pi, pi] with a two-part
// 2*pi (Cody and Waite's additive argument reduction), which keeps the reduced angle exact
// to ~1e-13 for the positions of a decode cache; fp32 sincosf is then accurate.
__device__ __forceinline__ void rope_cos_sin(double ang, float& c, float& s) {
    const double two_pi_hi = 6.283185307179586;        // 2*pi rounded to double
    const double two_pi_lo = 2.4492935982947064e-16;   // 2*pi - two_pi_hi
    const double k = rint(ang * 0.15915494309189535);  // ang / (2*pi)
    double r = fma(-k, two_pi_hi, ang);
    r = fma(-k, two_pi_lo, r);
    sincosf(static_cast<float>(r), &s, &c);
}

// Byte offset of (row r, element c) of a binary16 tile stored by TMA as D/64 boxes of
// [tp rows][64 elements] with the 128-byte swizzle (16-byte chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t swz(int r, int c, int tp) {
    const int box = c >> 6, cc = c & 63;
    return static_cast<uint32_t>(box * tp * 128 + r * 128 + ((((cc >> 3) ^ r) & 7) << 4) + ((cc & 7) << 1));
}

}  // namespace gem
