// qpack_dev.cuh — device-side building blocks shared by the qpack kernels (sm_103a).
//
// Format traits follow the byte table of the 2/3/5/6-bit quantization article (lpnh.cn/news/2857666, §2.3)
// and the INT4 layout of the DBHOO-CIM article (pwwt.cn/news/4452170, §3.2, §4.1); where the pages leave a bit
// order open, fields are little-endian with weight i at the lowest free bit. The PTX wrappers cover the mbarrier / bulk-copy pipeline used by the streaming kernels.
#pragma once

#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace qpack {

enum : int { FMT_Q4G32 = 0, FMT_Q2S = 1, FMT_Q3S = 2, FMT_Q5S = 3, FMT_Q6S = 4, FMT_Q4G32H = 5, FMT_Q4G16 = 6,
             FMT_Q4G32A = 7 };
enum : int { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2 };

// Bits OR-ed into a per-translation-unit device fault word when a bounded wait gives up, or when a decode product met
// an inf or nan activation (its outputs are then nan; the public value is QPACK_FAULT_NONFINITE_X).
enum : int { FAULT_WAIT_FULL = 1, FAULT_WAIT_EMPTY = 2, FAULT_WAIT_MMA = 4, FAULT_WAIT_TMEM = 8, FAULT_NONFINITE_X = 16 };

template <int F> struct Fmt;
// INT4 symmetric group 32: 16 code bytes per group, fp32 scale in a separate array.
template <> struct Fmt<FMT_Q4G32> {
    static constexpr int bits = 4, nsub = 8, sublen = 32, lmax = 0, bytes = 128;  // per 256 weights of codes
    static constexpr bool asym = false, sb = false;
    static constexpr int offset = 8;        // stored u = q + 8
};
// INT4 symmetric group 32 with fp16 group scales: the same codes, 2-byte scales in the separate array.
template <> struct Fmt<FMT_Q4G32H> {
    static constexpr int bits = 4, nsub = 8, sublen = 32, lmax = 0, bytes = 128;
    static constexpr bool asym = false, sb = false;
    static constexpr int offset = 8;
};
// INT4 symmetric group 16 (fp32 scales): the same codes, one scale per 16 weights.
template <> struct Fmt<FMT_Q4G16> {
    static constexpr int bits = 4, nsub = 16, sublen = 16, lmax = 0, bytes = 128;
    static constexpr bool asym = false, sb = false;
    static constexpr int offset = 8;
};
// INT4 asymmetric group 32: unsigned codes u = q (no offset), an fp32 (scale, zero point) pair per group.
template <> struct Fmt<FMT_Q4G32A> {
    static constexpr int bits = 4, nsub = 8, sublen = 32, lmax = 0, bytes = 128;
    static constexpr bool asym = true, sb = false;
    static constexpr int offset = 0;
};
// The INT4 formats share their code layout; only the group size, the offset and the scale words differ.
template <int F> constexpr bool kInt4 = (F == FMT_Q4G32 || F == FMT_Q4G32H || F == FMT_Q4G16 || F == FMT_Q4G32A);
template <> struct Fmt<FMT_Q2S> {
    static constexpr int bits = 2, nsub = 16, sublen = 16, lmax = 15, bytes = 84;
    static constexpr bool asym = true, sb = true;
    static constexpr int offset = 0;
};
template <> struct Fmt<FMT_Q3S> {
    static constexpr int bits = 3, nsub = 16, sublen = 16, lmax = 63, bytes = 110;
    static constexpr bool asym = false, sb = true;
    static constexpr int offset = 4;
};
template <> struct Fmt<FMT_Q5S> {
    static constexpr int bits = 5, nsub = 8, sublen = 32, lmax = 63, bytes = 176;
    static constexpr bool asym = true, sb = true;
    static constexpr int offset = 0;
};
template <> struct Fmt<FMT_Q6S> {
    static constexpr int bits = 6, nsub = 16, sublen = 16, lmax = 127, bytes = 210;
    static constexpr bool asym = false, sb = true;
    static constexpr int offset = 32;
};

__host__ __device__ constexpr int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// ------------------------------------------------------------------------------------------------------------
// Small device helpers
// ------------------------------------------------------------------------------------------------------------
__device__ __forceinline__ float clampf_ord(float v, float lo, float hi) {
    // Same comparison order as the written definition: v < lo ? lo : (v > hi ? hi : v).
    return v < lo ? lo : (v > hi ? hi : v);
}

__device__ __forceinline__ float h2f_bits(uint16_t h) { return __half2float(__ushort_as_half(h)); }
__device__ __forceinline__ uint16_t f2h_bits(float f) { return __half_as_ushort(__float2half_rn(f)); }

template <int WDT> __device__ __forceinline__ void load8(const void *W, int64_t idx, float *w);
template <> __device__ __forceinline__ void load8<DT_F32>(const void *W, int64_t idx, float *w) {
    const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(W) + idx);
    float4 a = __ldg(p), b = __ldg(p + 1);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}
template <> __device__ __forceinline__ void load8<DT_F16>(const void *W, int64_t idx, float *w) {
    uint4 v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(W) + idx));
    uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        w[2 * i] = h2f_bits(uint16_t(u[i] & 0xFFFFu));
        w[2 * i + 1] = h2f_bits(uint16_t(u[i] >> 16));
    }
}
template <> __device__ __forceinline__ void load8<DT_BF16>(const void *W, int64_t idx, float *w) {
    uint4 v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(W) + idx));
    uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        w[2 * i] = __uint_as_float(u[i] << 16);
        w[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
}

// ------------------------------------------------------------------------------------------------------------
// mbarrier + bulk-copy wrappers (PTX ISA: mbarrier, cp.async.bulk). Every wait is bounded.
// ------------------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
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

// Bounded wait: returns false (and the caller records a fault) after `limit` failed polls. try_wait itself
// suspends for a hardware-defined interval, so the limit corresponds to seconds, not microseconds.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit = (1u << 22)) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Same, with a suspend-time hint (ns) per poll: a waiting thread yields its issue slots to the other warps of its
// SM sub-partition instead of polling (used by producer threads that wait on consumers).
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_bounded_hint(uint64_t *bar, uint32_t parity, uint32_t ns = 200,
                                                       uint32_t limit = (1u << 22)) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait_hint(bar, parity, ns)) return true;
    return false;
}

// Shared-memory atomic add with acquire-release semantics at CTA scope; returns the old value.
__device__ __forceinline__ uint32_t atom_add_acq_rel_cta(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_u32(p)), "r"(v) : "memory");
    return old;
}

// 1-D bulk copy global -> shared, completion signalled on `bar` as transaction bytes.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Programmatic dependent launch: allow the next grid in the stream to start launching / wait until the previous
// grid has completed and its memory is visible (both are no-ops for a normally launched grid).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// fp32 += fp16 * fp16 with an exact product (PTX mixed-precision fma, sm_100+).
__device__ __forceinline__ float fma_h(uint16_t a, uint16_t b, float c) {
    float d;
    asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
    return d;
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
    // (a & mask) | orv in one LOP3 (immediate truth table 0xEA = (A & B) | C).
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(orv));
    return d;
}

__device__ __forceinline__ uint32_t lop3_sel(uint32_t a, uint32_t b, uint32_t c) {
    // c ? a : b, bitwise (truth table 0xE4 = (A & C) | (B & ~C)).
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

}  // namespace qpack
