// qpack_quot.cuh — rounded quotients for the quantizers (codes = rint(v / scale) with IEEE division) without a
// division per value.
#pragma once
#include <cuda_runtime.h>

namespace qpack {

// q_i = rint(fl(v_i / s)) for a lane's n values, given rs = fl(1 / s) correctly rounded. The product
// t = fl(v * rs) is within (2^-24 + 2^-24 + 2^-48) |v / s| of v / s, and fl(v / s) within 2^-24 |v / s|, so
// |t - fl(v / s)| <= 2^-22 |t| (tiny results lie far from every half-integer). Where t is farther than 2^-21 |t|
// from the nearest half-integer, rint(t) is rint(fl(v / s)); a lane with any value nearer than that (or a NaN) takes
// all n true quotients instead, behind one branch.
template <int n>
__device__ __forceinline__ void rint_quot(const float *v, float s, float rs, float *q) {
    bool near = false;
#pragma unroll
    for (int i = 0; i < n; ++i) {
        const float t = __fmul_rn(v[i], rs);
        q[i] = rintf(t);
        near |= !(fabsf(__fsub_rn(t, q[i])) <= __fmaf_rn(fabsf(t), -0x1p-21f, 0.5f));
    }
    if (near) {
#pragma unroll
        for (int i = 0; i < n; ++i) q[i] = rintf(__fdiv_rn(v[i], s));
    }
}

// Codes c_i = int(clamp(rint(fl(v_i / s)) + add, lo, hi)) + off for a lane's n values (add a small integer, so the
// sum is exact; the clamp in the order v < lo ? lo : (v > hi ? hi : v)), with rint_quot's test of the product
// t = fl(v * rs). A value that passes the test has |t| <= 2^20, so fl(t + 1.5 * 2^23) is 1.5 * 2^23 + rint(t)
// exactly (round to nearest, ties to even, with a spacing of 1 there) and rint(t) is that sum's bit pattern less the
// bit pattern of 1.5 * 2^23: the code needs no rounding or float-to-integer instruction (both on the SM's
// quarter-rate conversion pipe), and the clamp is taken on integers. A lane with any value that fails the test takes
// the written definition with the true quotients, behind one branch.
template <int n>
__device__ __forceinline__ void rint_codes(const float *v, float s, float rs, int add, int lo, int hi, int off,
                                           uint8_t *c) {
    constexpr float kMagic = 12582912.0f;        // 1.5 * 2^23
    constexpr int kMagicBits = 0x4B400000;       // its bit pattern
    bool near = false;
#pragma unroll
    for (int i = 0; i < n; ++i) {
        const float t = __fmul_rn(v[i], rs);
        const float y = __fadd_rn(t, kMagic);
        const float q = __fsub_rn(y, kMagic);
        near |= !(fabsf(__fsub_rn(t, q)) <= __fmaf_rn(fabsf(t), -0x1p-21f, 0.5f));
        const int k = __float_as_int(y) - kMagicBits + add;
        c[i] = uint8_t((k < lo ? lo : (k > hi ? hi : k)) + off);
    }
    if (near) {
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float q = __fadd_rn(rintf(__fdiv_rn(v[i], s)), float(add));
            const float u = q < float(lo) ? float(lo) : (q > float(hi) ? float(hi) : q);
            c[i] = uint8_t(int(u) + off);
        }
    }
}

}  // namespace qpack
