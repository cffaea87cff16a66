// qpack_kv.cu — 8-bit KV cache: quantize fp16 keys/values to int8 codes with one fp16 scale per 32 consecutive
// elements (2/3/5/6-bit article, lpnh.cn/news/2857666, §4.1: half the cache size at about 1.06 bytes per element),
// and dequantize them back to fp16 (Mix-Quant article, lnrk.cn/news/34246, §2.3: the cache is dequantized in bulk
// when decoding switches to fp16).
//
// Per group: d = fp16(max|v| / 127) (the rounded scale is the one used), q = clamp(rint(v / d), -127, 127), 0 when
// d is 0; dequant v' = fp16(d * q). Both kernels are HBM streams (2 + 34/32 bytes per element either way). A warp
// takes 32 groups (1024 elements) at a time: lane l holds elements 8 (32 j + l) .. +7 for j = 0..3, so each of its
// 16-byte loads (and the 8-byte code stores) is one fully coalesced warp access. The four lanes of a group reduce
// its max with two shuffles.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qpack_dev.cuh"
#include "qpack_launch.h"
#include "qpack_quot.cuh"

namespace qpack {
namespace {

constexpr int KV_THREADS = 256;

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }
__device__ __forceinline__ uint16_t f2h(float f) { return __half_as_ushort(__float2half_rn(f)); }

__global__ void __launch_bounds__(KV_THREADS) kv_quantize_kernel(const uint4 *__restrict__ v, int64_t ngroups,
                                                                  uint2 *__restrict__ q, uint16_t *__restrict__ sc) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = int64_t(gridDim.x) * (KV_THREADS / 32);
    for (int64_t c = int64_t(blockIdx.x) * (KV_THREADS / 32) + (threadIdx.x >> 5); c * 32 < ngroups; c += warps) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t piece = c * 128 + 32 * j + lane;            // 8-element piece; group = piece / 4
            const bool live = piece / 4 < ngroups;                    // uniform across the group's four lanes
            uint4 w = make_uint4(0u, 0u, 0u, 0u);
            if (live) w = __ldcs(v + piece);                          // read once: streaming
            const uint32_t hw[4] = {w.x, w.y, w.z, w.w};
            float x[8];
            float a = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[2 * e] = h2f(uint16_t(hw[e] & 0xFFFFu));
                x[2 * e + 1] = h2f(uint16_t(hw[e] >> 16));
                a = fmaxf(a, fmaxf(fabsf(x[2 * e]), fabsf(x[2 * e + 1])));
            }
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            const uint16_t d16 = f2h(__fdiv_rn(a, 127.0f));
            const float d = h2f(d16);
            // clamp(rint(v / d), -127, 127) as two's-complement bytes, rounded as the true quotient is
            uint8_t cb[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (d > 0.0f) rint_codes<8>(x, d, __frcp_rn(d), 0, -127, 127, 0, cb);
            uint32_t packed[2] = {0u, 0u};
#pragma unroll
            for (int e = 0; e < 8; ++e) packed[e >> 2] |= uint32_t(cb[e]) << (8 * (e & 3));
            if (live) {
                q[piece] = make_uint2(packed[0], packed[1]);
                if ((lane & 3) == 0) sc[piece / 4] = d16;
            }
        }
    }
}

__global__ void __launch_bounds__(KV_THREADS) kv_dequant_kernel(const uint2 *__restrict__ q,
                                                                 const uint16_t *__restrict__ sc, int64_t ngroups,
                                                                 uint4 *__restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = int64_t(gridDim.x) * (KV_THREADS / 32);
    for (int64_t c = int64_t(blockIdx.x) * (KV_THREADS / 32) + (threadIdx.x >> 5); c * 32 < ngroups; c += warps) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t piece = c * 128 + 32 * j + lane;
            if (piece / 4 >= ngroups) continue;
            const uint2 cw = __ldcs(q + piece);
            const float d = h2f(__ldg(sc + piece / 4));
            const uint32_t cc[2] = {cw.x, cw.y};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float lo = d * float(int8_t(uint8_t(cc[e >> 1] >> (16 * (e & 1)))));
                const float hi = d * float(int8_t(uint8_t(cc[e >> 1] >> (16 * (e & 1) + 8))));
                o[e] = uint32_t(f2h(lo)) | (uint32_t(f2h(hi)) << 16);
            }
            __stcs(out + piece, make_uint4(o[0], o[1], o[2], o[3]));
        }
    }
}

int kv_grid(int64_t ngroups) {
    const int64_t chunks = (ngroups + 31) / 32;                       // one warp per 32 groups
    const int64_t blocks = (chunks + KV_THREADS / 32 - 1) / (KV_THREADS / 32);
    const int64_t cap = int64_t(num_sms()) * 8;                       // 8 blocks of 256 threads per SM
    return int(blocks < cap ? blocks : cap);
}

}  // namespace

cudaError_t launch_kv_quantize(const uint16_t *v, int64_t n, int8_t *q, uint16_t *scales, cudaStream_t s) {
    const int64_t ng = n / 32;
    kv_quantize_kernel<<<kv_grid(ng), KV_THREADS, 0, s>>>(reinterpret_cast<const uint4 *>(v), ng,
                                                          reinterpret_cast<uint2 *>(q), scales);
    return cudaGetLastError();
}

cudaError_t launch_kv_dequant(const int8_t *q, const uint16_t *scales, int64_t n, uint16_t *out, cudaStream_t s) {
    const int64_t ng = n / 32;
    kv_dequant_kernel<<<kv_grid(ng), KV_THREADS, 0, s>>>(reinterpret_cast<const uint2 *>(q), scales, ng,
                                                         reinterpret_cast<uint4 *>(out));
    return cudaGetLastError();
}

}  // namespace qpack
