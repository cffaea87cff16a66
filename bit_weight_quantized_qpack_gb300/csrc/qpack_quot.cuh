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
__device__ __forceinline__ void rint_quot8(const float v[8], float s, float rs, float q[8]) { rint_quot<8>(v, s, rs, q); }

}  // namespace qpack
