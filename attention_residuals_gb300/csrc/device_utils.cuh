// device_utils.cuh -- sm_103a building blocks for the AttnRes kernels:
// shared-memory mbarriers with bounded waits, 1-D TMA bulk copies, small
// async copies, bf16 packing and warp/CTA reductions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace attnres {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but lets the thread sleep for up to `hint_ns` while the
// phase is incomplete (it wakes as soon as the phase completes).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// How long a wait on a shared-memory barrier lasts before the kernel gives
// up on it (nanoseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Wait for the phase with the given parity to complete.  Gives up after
// about two seconds: records `where` in *err (first failure wins), sets
// *abort so the calling CTA stops waiting from then on, and returns false.
// Once *abort is set every later wait returns immediately.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned* err, unsigned where) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
        if (((++spins) & 15u) == 0u) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                atomicCAS(err, 0u, where);
                *abort = 1;
                return false;
            }
        }
    }
    return true;
}

// ------------------------------------------------------------ async copies
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void tma_load_1d(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Atomic adds to global memory without a returned value (reductions
// performed at L2): four consecutive floats (16-byte aligned) or one.
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}
__device__ __forceinline__ void red_add_f32(float* p, float a) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(a) : "memory");
}

// 4-byte asynchronous copy global -> shared (Ampere-style cp.async).
__device__ __forceinline__ void cp_async_4(void* dst_smem, const void* src_gmem) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst_smem)),
                 "l"(src_gmem)
                 : "memory");
}

// 8-byte asynchronous copy global -> shared (both addresses 8-byte aligned).
__device__ __forceinline__ void cp_async_8(void* dst_smem, const void* src_gmem) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst_smem)), "l"(src_gmem) : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed.
// The arrival counts against the barrier's expected count (.noinc).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// --------------------------------------------------------- named barriers
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ bf16
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        f[2 * k] = __uint_as_float(w[k] << 16);
        f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 r;
    r.x = pack_bf16x2(f[0], f[1]);
    r.y = pack_bf16x2(f[2], f[3]);
    r.z = pack_bf16x2(f[4], f[5]);
    r.w = pack_bf16x2(f[6], f[7]);
    return r;
}

// bf16 pair (low half = lower address) -> packed FP32 pair.
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Packed FP32 fused multiply-add and multiply (one FFMA2 / FMUL2 on sm_100
// and later).  Run-time compiled builds (NVRTC) issue the PTX instructions
// directly: with NVRTC's intrinsics for them the run-time compiled forward
// used more registers and spilled, where the nvcc build did not.
#ifdef __CUDACC_RTC__
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\tmov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
        "mov.b64 pc, {%6, %7};\n\tfma.rn.f32x2 pd, pa, pb, pc;\n\tmov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pd;\n\tmov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
        "mul.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
#else
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
#endif

__device__ __forceinline__ uint32_t pack_f2(float2 v) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(v.y), "f"(v.x));
    return r;
}

__device__ __forceinline__ uint32_t u4_get(const uint4& v, int k) {
    return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__device__ __forceinline__ uint4 ld_shared_v4(const void* p) {
    return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Streaming 16-byte global store (evict-first in L2).
// Tensor-core fragments (warp-wide): ldmatrix of four / two 8x8 bf16 tiles
// (each lane gives one 16-byte row address; .trans transposes each tile) and
// the m16n8k16 bf16 MMA with FP32 accumulators, d += A (16 x 16, row-major) *
// B (16 x 8, column-major).  The products of bf16 values are exact in FP32.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2_trans(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the kernel before it on the stream is still
// running; pdl_wait() then blocks until that kernel has finished and its
// memory is visible (a no-op for an ordinary launch), so it must come before
// the kernel's first global memory access.  pdl_launch_dependents() lets the
// next kernel start launching (its CTAs take SMs as this kernel's CTAs leave).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Bring `bytes` (a multiple of 16) at a 16-byte aligned global address into
// L2 ahead of its use (no shared memory, no completion to wait for).
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// 16-byte store with an L2 cache-eviction policy (createpolicy).
__device__ __forceinline__ void st_global_v4_policy(void* p, const uint4& v, uint64_t pol) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void st_global_cs_v4(void* p, const uint4& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// ------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// Reduce-scatter of K (power of two, <= 32) per-lane values over a warp:
// K/2 + K/4 + ... + 1 shuffles halve the vector, then plain butterflies
// finish.  Afterwards lane l holds, in v[0], the warp total of element
// (l >> (5 - log2 K)).
template <int K, int OFF, int N>
__device__ __forceinline__ void reduce_scatter_step(float (&v)[N], int lane) {
    if constexpr (OFF > 0) {
        if constexpr (K > 1) {
            const bool upper = (lane & OFF) != 0;
#pragma unroll
            for (int i = 0; i < K / 2; ++i) {
                const float send = upper ? v[i] : v[i + K / 2];
                const float keep = upper ? v[i + K / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
            }
            reduce_scatter_step<K / 2, OFF / 2>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], OFF);
            reduce_scatter_step<1, OFF / 2>(v, lane);
        }
    }
}

template <int K>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[K], int lane) {
    static_assert(K >= 1 && K <= 32 && (K & (K - 1)) == 0, "K must be a power of two <= 32");
    reduce_scatter_step<K, 16>(v, lane);
}

template <int K>
__device__ __forceinline__ constexpr int log2_const() {
    return K <= 1 ? 0 : 1 + log2_const<K / 2>();
}


// ------------------------------------------------ 32-bit shared addressing
__device__ __forceinline__ void mbar_arrive_s(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_test_s(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_test_sleep_s(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait on a barrier given by its 32-bit shared address (see mbar_wait).
// `abort` points at the CTA's control words in shared memory: abort[0] is the
// abort flag; a kernel that sets abort[2] to a nonzero number of microseconds
// (a test of the recovery path) shortens the limit, read only here, after the
// first test of the barrier has failed.
static __device__ __noinline__ bool mbar_wait_slow_s(uint32_t bar, uint32_t parity, volatile int* abort,
                                              unsigned* err, unsigned where, bool ctl_limit) {
    if (*abort) return false;
    const uint64_t limit_ns = (ctl_limit && abort[2] > 0) ? static_cast<uint64_t>(abort[2]) * 1000ull : kWaitLimitNs;
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (!mbar_test_sleep_s(bar, parity, 20000u)) {
        if (((++spins) & 15u) == 0u) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                atomicCAS(err, 0u, where);
                *abort = 1;
                return false;
            }
        }
    }
    return true;
}

__device__ __forceinline__ bool mbar_wait_s(uint32_t bar, uint32_t parity, volatile int* abort,
                                            unsigned* err, unsigned where) {
    if (mbar_test_s(bar, parity)) return true;
    return mbar_wait_slow_s(bar, parity, abort, err, where, false);
}

// As mbar_wait_s, with the limit abort[2] (microseconds) when that word is nonzero.
__device__ __forceinline__ bool mbar_wait_ctl_s(uint32_t bar, uint32_t parity, volatile int* abort,
                                                unsigned* err, unsigned where) {
    if (mbar_test_s(bar, parity)) return true;
    return mbar_wait_slow_s(bar, parity, abort, err, where, true);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ float4 lds128f(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}


// Arrive on a slot's "empty" barrier once the shared-memory loads that read
// the slot have returned their data: `dep` must be computed from every one
// of those loads, so the arrive cannot issue while a load is in flight (a
// later bulk copy into the slot would otherwise race with it).
__device__ __forceinline__ void mbar_arrive_after(uint32_t bar, uint32_t dep) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar), "r"(dep)
                 : "memory");
}


// Key statistics of one 16-byte vector of bf16 pairs, on bf16 operands
// directly (fma.rn.f32.bf16: one FFMA each, exact products, FP32 sums):
//   s0 += x_lo^2, s1 += x_hi^2, t0 += q_lo*x_lo, t1 += q_hi*x_hi
// for each of the four 32-bit words of x and q.
__device__ __forceinline__ void bf16_sq_dot(const uint4& x, const uint4& q, float& s0, float& s1,
                                            float& t0, float& t1) {
    asm("{\n\t.reg .b16 xl, xh, ql, qh;\n\t"
        "mov.b32 {xl, xh}, %4;\n\tmov.b32 {ql, qh}, %8;\n\t"
        "fma.rn.f32.bf16 %0, xl, xl, %0;\n\tfma.rn.f32.bf16 %1, xh, xh, %1;\n\t"
        "fma.rn.f32.bf16 %2, ql, xl, %2;\n\tfma.rn.f32.bf16 %3, qh, xh, %3;\n\t"
        "mov.b32 {xl, xh}, %5;\n\tmov.b32 {ql, qh}, %9;\n\t"
        "fma.rn.f32.bf16 %0, xl, xl, %0;\n\tfma.rn.f32.bf16 %1, xh, xh, %1;\n\t"
        "fma.rn.f32.bf16 %2, ql, xl, %2;\n\tfma.rn.f32.bf16 %3, qh, xh, %3;\n\t"
        "mov.b32 {xl, xh}, %6;\n\tmov.b32 {ql, qh}, %10;\n\t"
        "fma.rn.f32.bf16 %0, xl, xl, %0;\n\tfma.rn.f32.bf16 %1, xh, xh, %1;\n\t"
        "fma.rn.f32.bf16 %2, ql, xl, %2;\n\tfma.rn.f32.bf16 %3, qh, xh, %3;\n\t"
        "mov.b32 {xl, xh}, %7;\n\tmov.b32 {ql, qh}, %11;\n\t"
        "fma.rn.f32.bf16 %0, xl, xl, %0;\n\tfma.rn.f32.bf16 %1, xh, xh, %1;\n\t"
        "fma.rn.f32.bf16 %2, ql, xl, %2;\n\tfma.rn.f32.bf16 %3, qh, xh, %3;\n\t}"
        : "+f"(s0), "+f"(s1), "+f"(t0), "+f"(t1)
        : "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w), "r"(q.x), "r"(q.y), "r"(q.z), "r"(q.w));
}

// t0 += x_lo * y_lo, t1 += x_hi * y_hi over the four 32-bit words of two
// bf16x8 vectors (fma.rn.f32.bf16: exact products, FP32 sums).
__device__ __forceinline__ void bf16_dot8(const uint4& x, const uint4& y, float& t0, float& t1) {
    asm("{\n\t.reg .b16 xl, xh, yl, yh;\n\t"
        "mov.b32 {xl, xh}, %2;\n\tmov.b32 {yl, yh}, %6;\n\t"
        "fma.rn.f32.bf16 %0, yl, xl, %0;\n\tfma.rn.f32.bf16 %1, yh, xh, %1;\n\t"
        "mov.b32 {xl, xh}, %3;\n\tmov.b32 {yl, yh}, %7;\n\t"
        "fma.rn.f32.bf16 %0, yl, xl, %0;\n\tfma.rn.f32.bf16 %1, yh, xh, %1;\n\t"
        "mov.b32 {xl, xh}, %4;\n\tmov.b32 {yl, yh}, %8;\n\t"
        "fma.rn.f32.bf16 %0, yl, xl, %0;\n\tfma.rn.f32.bf16 %1, yh, xh, %1;\n\t"
        "mov.b32 {xl, xh}, %5;\n\tmov.b32 {yl, yh}, %9;\n\t"
        "fma.rn.f32.bf16 %0, yl, xl, %0;\n\tfma.rn.f32.bf16 %1, yh, xh, %1;\n\t}"
        : "+f"(t0), "+f"(t1)
        : "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w), "r"(y.x), "r"(y.y), "r"(y.z), "r"(y.w));
}

// s0 += x_lo^2, s1 += x_hi^2 over the four words of a bf16x8 vector.
__device__ __forceinline__ void bf16_sq8(const uint4& x, float& s0, float& s1) { bf16_dot8(x, x, s0, s1); }

// Zero the bf16 halves of x (channels j0 .. j0+7) outside [lo, hi).
__device__ __forceinline__ uint4 mask_bf16x8(const uint4& x, int j0, int lo, int hi) {
    uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int j = j0 + 2 * kk;
        if (j < lo || j >= hi) w[kk] &= 0xffff0000u;
        if (j + 1 < lo || j + 1 >= hi) w[kk] &= 0x0000ffffu;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void sts128(uint32_t addr, const uint4& v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// a + b for two bf16x8 vectors: each pair widened exactly to FP32, added
// once, rounded to bf16 (nearest, ties to even) -- a bf16 tensor add.
__device__ __forceinline__ uint4 add_bf16x8(const uint4& a, const uint4& b) {
    const float2 one = make_float2(1.0f, 1.0f);
    uint32_t w[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) w[kk] = pack_f2(ffma2(one, bf2_to_f2(u4_get(a, kk)), bf2_to_f2(u4_get(b, kk))));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// ------------------------------------------------------ thread-block clusters
// This CTA's rank inside its cluster, the cluster's index and the number of
// clusters in the grid (x dimension).
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_index_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Shared::cluster address of the same shared-memory location in CTA `rank`
// of this cluster (distributed shared memory).
__device__ __forceinline__ uint32_t cluster_map(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}

// Store one float into another CTA's shared memory (address from cluster_map).
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster; release at cluster
// scope orders this thread's earlier stores (local or remote) before it.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}

// Wait on a local mbarrier whose arrivals come from other CTAs of the
// cluster: acquire at cluster scope, so their stores before arriving are
// visible afterwards.  Bounded like mbar_wait_s (about two seconds).
__device__ __forceinline__ bool mbar_test_cluster_s(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_poll_cluster_s(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

static __device__ __noinline__ bool mbar_wait_cluster_s(uint32_t bar, uint32_t parity, volatile int* abort,
                                                        unsigned* err, unsigned where) {
    if (mbar_poll_cluster_s(bar, parity)) return true;
    if (*abort) return false;
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (!mbar_test_cluster_s(bar, parity, 20000u)) {
        if (((++spins) & 15u) == 0u) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                atomicCAS(err, 0u, where);
                *abort = 1;
                return false;
            }
        }
    }
    return true;
}

// Every thread of every CTA of the cluster meets here (release / acquire at
// cluster scope).  Only at kernel start (after barrier initialisation) and
// end (so no CTA exits while a peer may still address its shared memory),
// where every thread arrives after finitely many bounded waits.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Position in the shared-memory row ring: row address, slot index, phase.
struct RingCursor {
    uint32_t row;
    int slot;
    uint32_t phase;
    __device__ __forceinline__ void next(uint32_t slot_bytes, int slots, uint32_t ring_lo) {
        row += slot_bytes;
        if (++slot == slots) {
            slot = 0;
            row = ring_lo;
            phase ^= 1u;
        }
    }
};

}  // namespace attnres
