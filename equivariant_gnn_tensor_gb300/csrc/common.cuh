// Device-side helpers: mbarrier / bulk-copy (TMA) / cp.async PTX wrappers,
// the bounded pipeline wait, and bf16 unpacking. sm_100+ only.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tpconv.h"
#include "tables.h"

namespace tpc {

// An mbarrier wait gives up after about this long, so a lost copy turns into a
// status bit instead of a hung GPU. Kernels take their main-loop limit as a
// parameter (this value unless a test shortens it); the waits that let copies
// in flight land before a failed warp exits always use this one.
constexpr uint64_t kWaitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__host__ __device__ constexpr int round_up_dev(int v, int a) { return (v + a - 1) / a * a; }

// Arrive on `bar` once all cp.async copies this thread issued so far have
// landed (does not count as an extra expected arrival: .noinc).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
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

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Probe that may suspend the thread in hardware for up to about `hint_ns`
// while the phase is incomplete (no issue slots spent spinning).
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
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

// Non-blocking probe: true when the phase with this parity has completed.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: true when the phase completed, false once about `limit_ns`
// have passed since the first probe found it incomplete. The clock is read
// only on that slow path, after every suspended probe. (A try_wait probe may
// itself suspend for a system-dependent time, so limits under 2 us use
// non-blocking probes instead.)
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns = kWaitNs) {
    if (limit_ns < 2000u) {
        const uint64_t t0 = global_ns();
        for (;;) {
            if (mbar_test_wait(bar, parity)) return true;
            if (global_ns() - t0 > limit_ns) return false;
        }
    }
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_hint(bar, parity, 2000u)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared (TMA engine), completion counted in bytes on
// `bar`. dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 16-byte asynchronous global -> shared copy through the load/store unit
// (bypasses L1). dst and src must be 16-byte aligned.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// Close this thread's open group of cp.async copies.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most n of this thread's cp.async groups are still pending
// (n in 0..7; larger n waits for n = 7).
__device__ __forceinline__ void cp_async_wait_pending(int n) {
    switch (n) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
        case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
        case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}

__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void set_status(int *status, int bits) {
    if (status) atomicOr(status, bits);
}

// float value of element q of a row of T (float or bf16)
template <typename T>
struct Elem;
template <>
struct Elem<float> {
    static constexpr int kBytes = 4;
};
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kBytes = 2;
};

// Load CPT consecutive elements starting at p (aligned to CPT elements) as floats.
template <int CPT>
__device__ __forceinline__ void load_vec(const float *p, float (&v)[CPT]) {
    if constexpr (CPT == 4) {
        float4 t = *reinterpret_cast<const float4 *>(p);
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else if constexpr (CPT == 2) {
        float2 t = *reinterpret_cast<const float2 *>(p);
        v[0] = t.x; v[1] = t.y;
    } else {
#pragma unroll
        for (int c = 0; c < CPT; ++c) v[c] = p[c];
    }
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int CPT>
__device__ __forceinline__ void load_vec(const __nv_bfloat16 *p, float (&v)[CPT]) {
    if constexpr (CPT == 4) {
        uint2 t = *reinterpret_cast<const uint2 *>(p);
        v[0] = bf16lo(t.x); v[1] = bf16hi(t.x); v[2] = bf16lo(t.y); v[3] = bf16hi(t.y);
    } else if constexpr (CPT == 2) {
        uint32_t t = *reinterpret_cast<const uint32_t *>(p);
        v[0] = bf16lo(t); v[1] = bf16hi(t);
    } else {
#pragma unroll
        for (int c = 0; c < CPT; ++c) v[c] = __bfloat162float(p[c]);
    }
}

template <int CPT>
__device__ __forceinline__ void store_vec(float *p, const float (&v)[CPT]) {
    if constexpr (CPT == 4) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    } else if constexpr (CPT == 2) {
        *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
    } else {
#pragma unroll
        for (int c = 0; c < CPT; ++c) p[c] = v[c];
    }
}

// Real spherical harmonics of degrees 0..L (L <= 3) of (x, y, z) into
// Y[l*l + m + l], "component" normalisation, real basis m = -l..l with z as
// pole and no Condon-Shortley sign ("cuEquivariance in PyTorch", Spherical
// harmonics and a NumPy reference). With `unit` the vector is first scaled
// to unit length (a zero vector gives Y_0 = 1 and zeros); otherwise these are
// the raw homogeneous polynomials. The polynomials are the Cartesian forms of
// the real harmonics times sqrt(4 pi):
//   l=1: sqrt(3) (y, z, x)
//   l=2: sqrt(15) xy, sqrt(15) yz, sqrt(5)/2 (2z^2-x^2-y^2), sqrt(15) xz, sqrt(15)/2 (x^2-y^2)
//   l=3: sqrt(70)/4 y(3x^2-y^2), sqrt(105) xyz, sqrt(42)/4 y(4z^2-x^2-y^2),
//        sqrt(7)/2 z(2z^2-3x^2-3y^2), sqrt(42)/4 x(4z^2-x^2-y^2),
//        sqrt(105)/2 z(x^2-y^2), sqrt(70)/4 x(x^2-3y^2)
template <int L>
__device__ __forceinline__ void real_sh_upto(float x, float y, float z, bool unit, float (&Y)[16]) {
    if (unit) {
        const float r2 = x * x + y * y + z * z;
        const float inv = r2 > 0.f ? rsqrtf(r2) : 0.f;
        x *= inv;
        y *= inv;
        z *= inv;
    }
    Y[0] = 1.f;
    if constexpr (L >= 1) {
        const float s3 = 1.7320508075688772f;
        Y[1] = s3 * y;
        Y[2] = s3 * z;
        Y[3] = s3 * x;
    }
    const float x2 = x * x, y2 = y * y, z2 = z * z;
    if constexpr (L >= 2) {
        const float s15 = 3.872983346207417f, s5h = 1.118033988749895f;
        Y[4] = s15 * x * y;
        Y[5] = s15 * y * z;
        Y[6] = s5h * (2.f * z2 - x2 - y2);
        Y[7] = s15 * x * z;
        Y[8] = 0.5f * s15 * (x2 - y2);
    }
    if constexpr (L >= 3) {
        const float c70 = 2.0916500663351889f;   // sqrt(70)/4
        const float c105 = 10.246950765959598f;  // sqrt(105)
        const float c42 = 1.6201851746019651f;   // sqrt(42)/4
        const float c7 = 1.3228756555322954f;    // sqrt(7)/2
        Y[9] = c70 * y * (3.f * x2 - y2);
        Y[10] = c105 * x * y * z;
        Y[11] = c42 * y * (4.f * z2 - x2 - y2);
        Y[12] = c7 * z * (2.f * z2 - 3.f * x2 - 3.f * y2);
        Y[13] = c42 * x * (4.f * z2 - x2 - y2);
        Y[14] = 0.5f * c105 * z * (x2 - y2);
        Y[15] = c70 * x * (x2 - 3.f * y2);
    }
}

// Copy the parts of the tables the kernels read into shared memory.
struct SmemTables {
    uint16_t rec_ptr[kMaxM + 1];
    uint16_t rec_j[kMaxTerms];
    float rec_c[kMaxTerms];
};

}  // namespace tpc
