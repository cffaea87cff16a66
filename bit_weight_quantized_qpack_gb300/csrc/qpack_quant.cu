// qpack_quant.cu — quantize, pack, fused quantize+pack, unpack and dequantize kernels (sm_103a).
//
// The quantizers (quant16_kernel) give each half-warp one 256-weight block of a row (a super-block, or eight INT4
// groups), lane ll owning weights 16 ll .. 16 ll + 15; pack, unpack and dequantize (block_kernel) give each warp one
// block, lane l owning weights 8 l .. 8 l + 7. Loads are 16-byte vectors, the per-group / per-sub-block reductions
// are shuffles, and every floating-point step uses an explicitly rounded intrinsic (no FMA contraction) so that
// codes, scales and dequantized values are bit-identical to the formats' IEEE fp32 definition (round to nearest
// even, true division, no FMA). The per-weight quotients are taken from one correctly rounded reciprocal per group
// (rint_quot), which provably rounds to the same integer as the true quotient except within a stated distance of
// a half-integer, where the true quotient is computed instead; the quantizers (but Q6S's) read the rounded code from
// the bits of the quotient plus 1.5 * 2^23 and clamp it as an integer (rint_codes), keeping the quarter-rate rounding
// and conversion instructions off the path (Q5S 80 -> 72 us, Q2S 66 -> 61 us on a 14336x4096 matrix).
//
// Quantizers: INT4 group-32 per the DBHOO-CIM article (pwwt.cn/news/4452170) §3.1; two-level round-to-nearest
// super-blocks per the 2/3/5/6-bit article (lpnh.cn/news/2857666) §2.1 and §2.3 (sub-block scales from each
// sub-block's own range, an fp16 super-block scale used rounded, integer sub-block scales against it, codes against
// the rounded sub-block scale). Packing: §3.2 of the INT4 article (low nibble first), §2.2 (8 three-bit codes in 3
// bytes, four 6-bit fields in 3 bytes) and §2.3 (4-bit plane + high-bit plane) of the 2/3/5/6-bit article.
#include <cuda_runtime.h>

#include "qpack_dev.cuh"
#include "qpack_launch.h"
#include "qpack_quot.cuh"

namespace qpack {

enum : int { MODE_QUANT_PARTS = 0, MODE_QUANT_PACKED = 1, MODE_PACK = 2, MODE_UNPACK = 3, MODE_DEQUANT = 4 };


// Per-lane state of one 256-weight block.
struct LaneBlock {
    uint8_t u[8];     // stored codes (q + offset)
    int L, M;         // this lane's sub-block scale / minimum integers
    uint16_t d16, dm16;
    float gscale;     // INT4: this lane's group scale
    float gzero;      // Q4G32A: the group's zero point as stored (an integer value); M holds it as an int
};

// ------------------------------------------------------------------------------------------------------------
// Packing of one block (byte offsets as written in each branch). `blk` points at the block's first packed byte;
// `valid` is false for lanes beyond a partial INT4 row tail.
// ------------------------------------------------------------------------------------------------------------
__device__ __forceinline__ void st_u16(uint8_t *p, uint32_t v) { *reinterpret_cast<uint16_t *>(p) = uint16_t(v); }
__device__ __forceinline__ void st_u32(uint8_t *p, uint32_t v) { *reinterpret_cast<uint32_t *>(p) = v; }

template <int F>
__device__ __forceinline__ void pack_lane(const LaneBlock &B, int lane, bool valid, uint8_t *blk) {
    if constexpr (kInt4<F>) {
        uint32_t v = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) v |= uint32_t(B.u[i] & 15u) << (4 * i);
        if (valid) st_u32(blk + 4 * lane, v);
    } else if constexpr (F == FMT_Q2S) {
        uint32_t v = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) v |= uint32_t(B.u[i] & 3u) << (2 * i);
        st_u16(blk + 2 * lane, v);
        if ((lane & 1) == 0) blk[64 + (lane >> 1)] = uint8_t((B.L & 15) | ((B.M & 15) << 4));
        if (lane == 0) { st_u16(blk + 80, B.d16); st_u16(blk + 82, B.dm16); }
    } else if constexpr (F == FMT_Q3S) {
        uint32_t v = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) v |= uint32_t(B.u[i] & 7u) << (3 * i);
        uint8_t *p = blk + 3 * lane;
        p[0] = uint8_t(v); p[1] = uint8_t(v >> 8); p[2] = uint8_t(v >> 16);
        // 16 six-bit sub-scales, 4 per 3 bytes: lane r < 4 packs L_{4r..4r+3}; L_j lives in lane 2j.
        uint32_t f = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            int Lk = __shfl_sync(0xffffffffu, B.L, 8 * (lane & 3) + 2 * k);
            f |= uint32_t(Lk & 63) << (6 * k);
        }
        if (lane < 4) {
            uint8_t *q = blk + 96 + 3 * lane;
            q[0] = uint8_t(f); q[1] = uint8_t(f >> 8); q[2] = uint8_t(f >> 16);
        }
        if (lane == 0) st_u16(blk + 108, B.d16);
    } else if constexpr (F == FMT_Q5S) {
        // high-bit word of the lane's 32-weight unit (lanes 4c .. 4c + 3; this lane = code word j = lane & 3):
        // weight 8j + 2b at bit 8b + 4 + j, weight 8j + 2b + 1 at bit 8((b + 1) & 3) + j
        const uint32_t j = uint32_t(lane) & 3u;
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t b = uint32_t(i) >> 1, pos = (i & 1) ? 8u * ((b + 1u) & 3u) + j : 8u * b + 4u + j;
            lo |= uint32_t(B.u[i] & 15u) << (4 * i);
            hi |= uint32_t((B.u[i] >> 4) & 1u) << pos;
        }
        hi |= __shfl_xor_sync(0xffffffffu, hi, 1);
        hi |= __shfl_xor_sync(0xffffffffu, hi, 2);
        st_u32(blk + 4 * lane, lo);
        if (j == 0) st_u32(blk + 128 + lane, hi);
        // fields 0..7 = L_0..L_7 (sub-block j in lanes 4j..4j+3), fields 8..15 = M_0..M_7; lane r < 4 packs
        // fields 4r..4r+3.
        const int r = lane & 3;
        uint32_t f = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int src = 16 * (r & 1) + 4 * k;
            int Lk = __shfl_sync(0xffffffffu, B.L, src);
            int Mk = __shfl_sync(0xffffffffu, B.M, src);
            f |= uint32_t((r >= 2 ? Mk : Lk) & 63) << (6 * k);
        }
        if (lane < 4) {
            uint8_t *q = blk + 160 + 3 * lane;
            q[0] = uint8_t(f); q[1] = uint8_t(f >> 8); q[2] = uint8_t(f >> 16);
        }
        if (lane == 0) st_u32(blk + 172, uint32_t(B.d16) | (uint32_t(B.dm16) << 16));
    } else {  // Q6S
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            lo |= uint32_t(B.u[i] & 15u) << (4 * i);
            hi |= uint32_t((B.u[i] >> 4) & 3u) << (2 * i);
        }
        st_u16(blk + 4 * lane, lo & 0xFFFFu);          // block start is only 2-byte aligned
        st_u16(blk + 4 * lane + 2, lo >> 16);
        st_u16(blk + 128 + 2 * lane, hi);
        if ((lane & 1) == 0) blk[192 + (lane >> 1)] = uint8_t(B.L);
        if (lane == 0) st_u16(blk + 208, B.d16);
    }
}

// ------------------------------------------------------------------------------------------------------------
// Unpacking of one block from global memory into per-lane state.
// ------------------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_u16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }
__device__ __forceinline__ uint32_t ld_u32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ uint32_t ld_u24(const uint8_t *p) {
    return uint32_t(p[0]) | (uint32_t(p[1]) << 8) | (uint32_t(p[2]) << 16);
}

template <int F>
__device__ __forceinline__ void unpack_lane(const uint8_t *blk, int lane, bool valid, LaneBlock &B) {
    if constexpr (kInt4<F>) {
        uint32_t v = valid ? ld_u32(blk + 4 * lane) : 0x88888888u;
#pragma unroll
        for (int i = 0; i < 8; ++i) B.u[i] = uint8_t((v >> (4 * i)) & 15u);
        B.L = B.M = 0; B.d16 = B.dm16 = 0;
    } else if constexpr (F == FMT_Q2S) {
        uint32_t v = ld_u16(blk + 2 * lane);
#pragma unroll
        for (int i = 0; i < 8; ++i) B.u[i] = uint8_t((v >> (2 * i)) & 3u);
        uint32_t lm = blk[64 + (lane >> 1)];
        B.L = int(lm & 15u); B.M = int(lm >> 4);
        B.d16 = uint16_t(ld_u16(blk + 80)); B.dm16 = uint16_t(ld_u16(blk + 82));
    } else if constexpr (F == FMT_Q3S) {
        uint32_t v = ld_u24(blk + 3 * lane);
#pragma unroll
        for (int i = 0; i < 8; ++i) B.u[i] = uint8_t((v >> (3 * i)) & 7u);
        const int j = lane >> 1;
        uint32_t f = ld_u24(blk + 96 + 3 * (j >> 2));
        B.L = int((f >> (6 * (j & 3))) & 63u); B.M = 0;
        B.d16 = uint16_t(ld_u16(blk + 108)); B.dm16 = 0;
    } else if constexpr (F == FMT_Q5S) {
        const uint32_t cw = uint32_t(lane) & 3u;   // the lane's code word within its unit
        uint32_t lo = ld_u32(blk + 4 * lane), hi = ld_u32(blk + 128 + 4 * (lane >> 2));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t b = uint32_t(i) >> 1, pos = (i & 1) ? 8u * ((b + 1u) & 3u) + cw : 8u * b + 4u + cw;
            B.u[i] = uint8_t(((lo >> (4 * i)) & 15u) | (((hi >> pos) & 1u) << 4));
        }
        const int j = lane >> 2;
        uint32_t fl = ld_u24(blk + 160 + 3 * (j >> 2)), fm = ld_u24(blk + 166 + 3 * (j >> 2));
        B.L = int((fl >> (6 * (j & 3))) & 63u);
        B.M = int((fm >> (6 * (j & 3))) & 63u);
        B.d16 = uint16_t(ld_u16(blk + 172)); B.dm16 = uint16_t(ld_u16(blk + 174));
    } else {  // Q6S
        uint32_t lo = ld_u16(blk + 4 * lane) | (ld_u16(blk + 4 * lane + 2) << 16), hi = ld_u16(blk + 128 + 2 * lane);
#pragma unroll
        for (int i = 0; i < 8; ++i) B.u[i] = uint8_t(((lo >> (4 * i)) & 15u) | (((hi >> (2 * i)) & 3u) << 4));
        B.L = int(int8_t(blk[192 + (lane >> 1)])); B.M = 0;
        B.d16 = uint16_t(ld_u16(blk + 208)); B.dm16 = 0;
    }
}

// Dequantize a lane's 8 weights (Q4G32 w' = s * q; super-blocks (d * L) * q, minus dmin * M when asymmetric).
template <int F>
__device__ __forceinline__ void dequant_lane(const LaneBlock &B, float out[8]) {
    using T = Fmt<F>;
    if constexpr (kInt4<F>) {      // gscale: the fp32 scale, or the fp16 scale widened; q - z for Q4G32A
        const int z = F == FMT_Q4G32A ? B.M : 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = __fmul_rn(B.gscale, float(int(B.u[i]) - z));
    } else {
        const float D = h2f_bits(B.d16);
        const float es = __fmul_rn(D, float(B.L));
        const float em = T::asym ? __fmul_rn(h2f_bits(B.dm16), float(B.M)) : 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float v = __fmul_rn(es, float(int(B.u[i]) - T::offset));
            if (T::asym) v = __fsub_rn(v, em);
            out[i] = v;
        }
    }
}

// A lane's 8 input weights as loaded (two 16-byte vectors for fp32, one for fp16 / bf16): the quantizers load the
// next block's while they work on the current one.
struct Raw8 {
    uint4 v0, v1;
};
template <int WDT>
__device__ __forceinline__ Raw8 ld_raw8(const void *W, int64_t idx) {
    Raw8 r;
    if constexpr (WDT == DT_F32) {
        const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const float *>(W) + idx);
        r.v0 = __ldg(p);
        r.v1 = __ldg(p + 1);
    } else {
        r.v0 = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(W) + idx));
        r.v1 = make_uint4(0u, 0u, 0u, 0u);
    }
    return r;
}
template <int WDT>
__device__ __forceinline__ void cvt_raw8(const Raw8 &r, float *w) {
    if constexpr (WDT == DT_F32) {
        const uint32_t u[8] = {r.v0.x, r.v0.y, r.v0.z, r.v0.w, r.v1.x, r.v1.y, r.v1.z, r.v1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = __uint_as_float(u[i]);
    } else {
        const uint32_t u[4] = {r.v0.x, r.v0.y, r.v0.z, r.v0.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (WDT == DT_F16) {
                w[2 * i] = h2f_bits(uint16_t(u[i] & 0xFFFFu));
                w[2 * i + 1] = h2f_bits(uint16_t(u[i] >> 16));
            } else {
                w[2 * i] = __uint_as_float(u[i] << 16);
                w[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
            }
        }
    }
}

// ------------------------------------------------------------------------------------------------------------
// The block kernel (pack, unpack, dequantize): one warp per 256-weight block, 8 weights a lane.
// ------------------------------------------------------------------------------------------------------------
template <int F, int MODE, int WDT>
__global__ void __launch_bounds__(256) block_kernel(BlockArgs a) {
    using T = Fmt<F>;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int64_t total = a.N * a.nbk;
    static_assert(MODE == MODE_PACK || MODE == MODE_UNPACK || MODE == MODE_DEQUANT, "quantizers: quant16_kernel");
    // (row, block) of this warp's first block and of the grid stride: one division each, then additions
    int64_t r = warp0 / a.nbk, b = warp0 - r * a.nbk;
    const int64_t sr = nwarps / a.nbk, sb = nwarps - sr * a.nbk;
    for (int64_t wb = warp0; wb < total; wb += nwarps, r += sr, b += sb) {
        if (b >= a.nbk) { b -= a.nbk; ++r; }
        const int64_t k0 = 256 * b + 8 * lane;           // first weight of this lane within the row
        const bool valid = k0 < a.K;                      // only INT4 rows can end inside a block
        LaneBlock B;
        B.gscale = B.gzero = 0.0f;
        const int j = lane / (T::sublen / 8);             // this lane's group / sub-block within the block
        if constexpr (MODE == MODE_PACK) {
            if (valid) {
                uint2 c = *reinterpret_cast<const uint2 *>(a.codes + r * a.K + k0);
                uint32_t cw[2] = {c.x, c.y};
#pragma unroll
                for (int i = 0; i < 8; ++i) B.u[i] = uint8_t(int(int8_t(cw[i >> 2] >> (8 * (i & 3)))) + T::offset);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) B.u[i] = uint8_t(T::offset);
            }
            if constexpr (F == FMT_Q4G32 || F == FMT_Q4G16) {
                B.gscale = valid ? a.gscale[r * (a.K / T::sublen) + T::nsub * b + j] : 0.0f;
                B.L = B.M = 0; B.d16 = B.dm16 = 0;
            } else if constexpr (F == FMT_Q4G32H) {
                B.d16 = valid ? a.d[r * (a.K / 32) + 8 * b + j] : uint16_t(0);
                B.gscale = h2f_bits(B.d16);
                B.L = B.M = 0; B.dm16 = 0;
            } else if constexpr (F == FMT_Q4G32A) {
                const int64_t e = r * (a.K / 16) + 2 * (8 * b + j);
                B.gscale = valid ? a.gscale[e] : 0.0f;
                B.gzero = valid ? a.gscale[e + 1] : 0.0f;
                B.L = B.M = 0; B.d16 = B.dm16 = 0;
            } else {
                const int64_t sb = r * a.nbk + b;
                B.L = a.sub_scale[sb * T::nsub + j];
                B.M = T::asym ? a.sub_min[sb * T::nsub + j] : 0;
                B.d16 = a.d[sb];
                B.dm16 = T::asym ? a.dmin[sb] : uint16_t(0);
            }
        } else {  // UNPACK / DEQUANT read packed bytes
            const uint8_t *blk = a.packed_in + r * a.row_stride + b * T::bytes;
            unpack_lane<F>(blk, lane, valid, B);
            if constexpr (F == FMT_Q4G32 || F == FMT_Q4G16) B.gscale = valid ? a.gs_in[r * a.scale_stride + T::nsub * b + j] : 0.0f;
            if constexpr (F == FMT_Q4G32H) {
                const uint16_t *g16 = reinterpret_cast<const uint16_t *>(a.gs_in);
                B.d16 = valid ? g16[r * a.scale_stride + 8 * b + j] : uint16_t(0);
                B.gscale = h2f_bits(B.d16);
            }
            if constexpr (F == FMT_Q4G32A) {
                const int64_t e = r * a.scale_stride + 2 * (8 * b + j);
                B.gscale = valid ? a.gs_in[e] : 0.0f;
                B.gzero = valid ? a.gs_in[e + 1] : 0.0f;
                B.M = int(B.gzero);
            }
        }

        if constexpr (MODE == MODE_UNPACK) {
            if (valid) {
                uint32_t cw[2] = {0u, 0u};
#pragma unroll
                for (int i = 0; i < 8; ++i) cw[i >> 2] |= uint32_t(uint8_t(int(B.u[i]) - T::offset)) << (8 * (i & 3));
                *reinterpret_cast<uint2 *>(a.codes + r * a.K + k0) = make_uint2(cw[0], cw[1]);
            }
            const bool first_of_sub = (lane % (T::sublen / 8)) == 0;
            if constexpr (F == FMT_Q4G32 || F == FMT_Q4G16) {
                if (valid && first_of_sub) a.gscale[r * (a.K / T::sublen) + T::nsub * b + j] = B.gscale;
            } else if constexpr (F == FMT_Q4G32H) {
                if (valid && first_of_sub) a.d[r * (a.K / 32) + 8 * b + j] = B.d16;
            } else if constexpr (F == FMT_Q4G32A) {
                if (valid && first_of_sub) {
                    const int64_t e = r * (a.K / 16) + 2 * (8 * b + j);
                    a.gscale[e] = B.gscale;
                    a.gscale[e + 1] = B.gzero;
                }
            } else {
                const int64_t sb = r * a.nbk + b;
                if (first_of_sub) {
                    a.sub_scale[sb * T::nsub + j] = uint8_t(B.L);
                    if (T::asym) a.sub_min[sb * T::nsub + j] = uint8_t(B.M);
                }
                if (lane == 0) {
                    a.d[sb] = B.d16;
                    if (T::asym) a.dmin[sb] = B.dm16;
                }
            }
        } else if constexpr (MODE == MODE_PACK) {
            uint8_t *row = a.packed + r * a.row_stride;
            pack_lane<F>(B, lane, valid, row + b * T::bytes);
            if constexpr (F == FMT_Q4G32 || F == FMT_Q4G16) {
                const bool first_of_group = (lane % (T::sublen / 8)) == 0;
                if (valid && first_of_group) a.gs_out[r * a.scale_stride + T::nsub * b + j] = B.gscale;
                if (b == a.nbk - 1) {                      // zero the scale-row padding
                    const int64_t g0 = a.K / T::sublen;
                    if (g0 + lane < a.scale_stride) a.gs_out[r * a.scale_stride + g0 + lane] = 0.0f;
                }
            } else if constexpr (F == FMT_Q4G32A) {
                if (valid && (lane & 3) == 0) {
                    const int64_t e = r * a.scale_stride + 2 * (8 * b + j);
                    a.gs_out[e] = B.gscale;
                    a.gs_out[e + 1] = B.gzero;
                }
                if (b == a.nbk - 1) {                      // zero the scale-row padding
                    const int64_t g0 = a.K / 16;
                    if (g0 + lane < a.scale_stride) a.gs_out[r * a.scale_stride + g0 + lane] = 0.0f;
                }
            } else if constexpr (F == FMT_Q4G32H) {
                uint16_t *g16 = reinterpret_cast<uint16_t *>(a.gs_out);
                const bool first_of_group = (lane & 3) == 0;
                if (valid && first_of_group) g16[r * a.scale_stride + 8 * b + j] = B.d16;
                if (b == a.nbk - 1) {                      // zero the scale-row padding
                    const int64_t g0 = a.K / 32;
                    if (g0 + lane < a.scale_stride) g16[r * a.scale_stride + g0 + lane] = 0;
                }
            } else {
                if (b == a.nbk - 1) {                      // zero the row padding (< 16 bytes)
                    const int64_t used = a.nbk * T::bytes;
                    if (used + lane < a.row_stride) row[used + lane] = 0;
                }
            }
        } else {  // DEQUANT
            if (valid) {
                float o[8];
                dequant_lane<F>(B, o);
                float4 *dst = reinterpret_cast<float4 *>(a.out + r * a.K + k0);
                dst[0] = make_float4(o[0], o[1], o[2], o[3]);
                dst[1] = make_float4(o[4], o[5], o[6], o[7]);
            }
        }
    }
}

// ------------------------------------------------------------------------------------------------------------
// Quantizers with 16 weights a lane. Each half-warp owns one 256-weight block: lane ll = lane & 15 holds weights
// 16 ll .. 16 ll + 15, so a warp quantizes two blocks per pass and every per-block step (the reductions, the
// super-block scale, the sub-block integers, the index and address arithmetic) serves twice the weights it does
// with 8 weights a lane. Every shuffle stays inside the half-warp (xor offsets below 16); groups and sub-blocks of
// 16 weights are one lane, those of 32 two neighbouring lanes.
// ------------------------------------------------------------------------------------------------------------
struct LaneQ {
    uint8_t u[16];    // stored codes (q + offset)
    int L, M;         // the lane's sub-block scale / minimum integers (INT4 asymmetric: M = z)
    uint16_t d16, dm16;
    float gscale;     // INT4: the lane's group scale
    float gzero;      // Q4G32A: the group's zero point as stored
};

template <int F>
__device__ __forceinline__ float grp_max16(float v) {           // over the lanes of a group / sub-block
    if constexpr (Fmt<F>::sublen == 32) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
    return v;
}
template <int F>
__device__ __forceinline__ float grp_min16(float v) {
    if constexpr (Fmt<F>::sublen == 32) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, 1));
    return v;
}
__device__ __forceinline__ float block_max16(float v) {          // over the 16 lanes of a block
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Quantization of the lane's 16 weights: INT4 s = max|w| / 8 (floor 1e-12), q = clamp(rint(w / s), -8, 7) (fp16
// scale: the fp16-rounded s; asymmetric: s = (hi - lo) / 15, z = rint(-lo / s)); super-blocks: the sub-block scale
// (and minimum) from its own range, d (and dmin) = fp16(max over the block / Lmax), integer L_j (M_j) against the
// rounded d, codes against d * L_j. Returns the RANGE flag (an fp16 scale that overflowed).
template <int F>
__device__ __forceinline__ int quantize16(const float w[16], LaneQ &B) {
    using T = Fmt<F>;
    B.gscale = B.gzero = 0.0f;
    B.L = B.M = 0;
    B.d16 = B.dm16 = 0;
    if constexpr (F == FMT_Q4G32 || F == FMT_Q4G16) {
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(w[i]));
        a = grp_max16<F>(a);
        float s = __fmul_rn(a, 0.125f);                   // a / 8: the same real number, rounded the same way
        if (s < 1e-12f) s = 1e-12f;
        rint_codes<16>(w, s, __frcp_rn(s), 0, -8, 7, 8, B.u);
        B.gscale = s;
        return 0;
    } else if constexpr (F == FMT_Q4G32A) {
        float lo = 0.0f, hi = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) { lo = fminf(lo, w[i]); hi = fmaxf(hi, w[i]); }
        lo = grp_min16<F>(lo);
        hi = grp_max16<F>(hi);
        float s = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
        if (s < 1e-12f) s = 1e-12f;
        const int z = int(clampf_ord(rintf(__fdiv_rn(-lo, s)), 0.0f, 15.0f));
        rint_codes<16>(w, s, __frcp_rn(s), z, 0, 15, 0, B.u);
        B.gscale = s;
        B.gzero = float(z);
        B.M = z;
        return 0;
    } else if constexpr (F == FMT_Q4G32H) {
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(w[i]));
        a = grp_max16<F>(a);
        const uint16_t s16 = f2h_bits(__fmul_rn(a, 0.125f));
        const float D = h2f_bits(s16);
        if (D > 0.0f) {
            rint_codes<16>(w, D, __frcp_rn(D), 0, -8, 7, 8, B.u);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) B.u[i] = 8;
        }
        B.gscale = D;
        B.d16 = s16;
        return ((s16 & 0x7FFFu) == 0x7C00u) ? 1 : 0;
    } else if constexpr (!T::asym) {
        const float half_range = float(1 << (T::bits - 1));
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(w[i]));
        a = grp_max16<F>(a);
        const float s = __fmul_rn(a, 1.0f / half_range);
        const float smax = block_max16(s);
        const uint16_t d16 = f2h_bits(__fdiv_rn(smax, float(T::lmax)));
        const float D = h2f_bits(d16);
        float L = 0.0f;
        if (D > 0.0f) L = clampf_ord(rintf(__fdiv_rn(s, D)), 0.0f, float(T::lmax));
        const float e = __fmul_rn(D, L);
        if constexpr (F == FMT_Q6S) {
            // the rounding and conversion instructions measured 2% faster here than rint_codes (Q3S: 3% slower)
            float q[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) q[i] = 0.0f;
            if (e > 0.0f) {
                rint_quot<16>(w, e, __frcp_rn(e), q);
#pragma unroll
                for (int i = 0; i < 16; ++i) q[i] = clampf_ord(q[i], -half_range, half_range - 1.0f);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) B.u[i] = uint8_t(int(q[i]) + T::offset);
        } else if (e > 0.0f) {
            rint_codes<16>(w, e, __frcp_rn(e), 0, -(1 << (T::bits - 1)), (1 << (T::bits - 1)) - 1, T::offset, B.u);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) B.u[i] = uint8_t(T::offset);
        }
        B.L = int(L);
        B.d16 = d16;
        return ((d16 & 0x7FFFu) == 0x7C00u) ? 1 : 0;
    } else {
        const float levels = float((1 << T::bits) - 1);
        float lo = 0.0f, hi = -INFINITY;
#pragma unroll
        for (int i = 0; i < 16; ++i) { lo = fminf(lo, w[i]); hi = fmaxf(hi, w[i]); }
        lo = grp_min16<F>(lo);
        hi = grp_max16<F>(hi);
        const float s = __fdiv_rn(__fsub_rn(hi, lo), levels);
        const float m = __fsub_rn(0.0f, lo);
        const float smax = fmaxf(0.0f, block_max16(s));
        const float mmax = fmaxf(0.0f, block_max16(m));
        const uint16_t d16 = f2h_bits(__fdiv_rn(smax, float(T::lmax)));
        const uint16_t dm16 = f2h_bits(__fdiv_rn(mmax, float(T::lmax)));
        const float D = h2f_bits(d16), Dm = h2f_bits(dm16);
        float L = 0.0f, M = 0.0f;
        if (D > 0.0f) L = clampf_ord(rintf(__fdiv_rn(s, D)), 0.0f, float(T::lmax));
        if (Dm > 0.0f) M = clampf_ord(rintf(__fdiv_rn(m, Dm)), 0.0f, float(T::lmax));
        const float es = __fmul_rn(D, L), em = __fmul_rn(Dm, M);
        if (es > 0.0f) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __fadd_rn(w[i], em);
            rint_codes<16>(v, es, __frcp_rn(es), 0, 0, (1 << T::bits) - 1, 0, B.u);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) B.u[i] = 0;
        }
        B.L = int(L);
        B.M = int(M);
        B.d16 = d16;
        B.dm16 = dm16;
        return (((d16 & 0x7FFFu) == 0x7C00u) || ((dm16 & 0x7FFFu) == 0x7C00u)) ? 1 : 0;
    }
}

// Packed bytes of one block from its 16 lanes (the byte layouts of pack_lane; `blk` = the block's first byte, `on`
// false for a half-warp without a block or an INT4 lane past the row's end). Every lane runs the shuffles.
template <int F>
__device__ __forceinline__ void pack16(const LaneQ &B, int lane, bool on, uint8_t *blk) {
    const int ll = lane & 15, hb = lane & 16;
    if constexpr (kInt4<F>) {
        uint32_t v0 = 0, v1 = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v0 |= uint32_t(B.u[i] & 15u) << (4 * i);
            v1 |= uint32_t(B.u[8 + i] & 15u) << (4 * i);
        }
        if (on) *reinterpret_cast<uint2 *>(blk + 8 * ll) = make_uint2(v0, v1);
    } else if constexpr (F == FMT_Q2S) {
        uint32_t v = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) v |= uint32_t(B.u[i] & 3u) << (2 * i);
        if (on) {
            st_u32(blk + 4 * ll, v);
            blk[64 + ll] = uint8_t((B.L & 15) | ((B.M & 15) << 4));
            if (ll == 0) { st_u16(blk + 80, B.d16); st_u16(blk + 82, B.dm16); }
        }
    } else if constexpr (F == FMT_Q3S) {
        uint64_t v = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) v |= uint64_t(B.u[i] & 7u) << (3 * i);
        // 16 six-bit sub-scales, 4 per 3 bytes: lane r < 4 packs L_{4r..4r+3}; L_j lives in lane j
        uint32_t f = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int Lk = __shfl_sync(0xffffffffu, B.L, hb | (4 * (ll & 3) + k));
            f |= uint32_t(Lk & 63) << (6 * k);
        }
        if (on) {
            uint8_t *p = blk + 6 * ll;                     // 2-byte aligned
            st_u16(p, uint32_t(v));
            st_u16(p + 2, uint32_t(v >> 16));
            st_u16(p + 4, uint32_t(v >> 32));
            if (ll < 4) {
                uint8_t *q = blk + 96 + 3 * ll;
                q[0] = uint8_t(f); q[1] = uint8_t(f >> 8); q[2] = uint8_t(f >> 16);
            }
            if (ll == 0) st_u16(blk + 108, B.d16);
        }
    } else if constexpr (F == FMT_Q5S) {
        // high-bit word of the lane's 32-weight unit c = ll >> 1 (this lane: code words j = 2 (ll & 1), + 1):
        // weight 8j + 2b at bit 8b + 4 + j, weight 8j + 2b + 1 at bit 8((b + 1) & 3) + j
        // (positions for code words 0, 1, then shifted by 2 for the odd lane's words 2, 3)
        uint32_t lo0 = 0, lo1 = 0, hi = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t j = uint32_t(i) >> 3, b = (uint32_t(i) >> 1) & 3u;
            const uint32_t pos = (i & 1) ? 8u * ((b + 1u) & 3u) + j : 8u * b + 4u + j;
            if (i < 8) lo0 |= uint32_t(B.u[i] & 15u) << (4 * i);
            else lo1 |= uint32_t(B.u[i] & 15u) << (4 * (i - 8));
            hi |= uint32_t((B.u[i] >> 4) & 1u) << pos;
        }
        hi <<= 2 * (ll & 1);
        hi |= __shfl_xor_sync(0xffffffffu, hi, 1);
        // fields 0..7 = L_0..L_7 (sub-block j in lanes 2j, 2j + 1), 8..15 = M_0..M_7; lane r < 4 packs 4r..4r+3
        const int r = ll & 3;
        uint32_t f = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int src = hb | (8 * (r & 1) + 2 * k);
            const int Lk = __shfl_sync(0xffffffffu, B.L, src);
            const int Mk = __shfl_sync(0xffffffffu, B.M, src);
            f |= uint32_t((r >= 2 ? Mk : Lk) & 63) << (6 * k);
        }
        if (on) {
            *reinterpret_cast<uint2 *>(blk + 8 * ll) = make_uint2(lo0, lo1);
            if ((ll & 1) == 0) st_u32(blk + 128 + 2 * ll, hi);
            if (ll < 4) {
                uint8_t *q = blk + 160 + 3 * ll;
                q[0] = uint8_t(f); q[1] = uint8_t(f >> 8); q[2] = uint8_t(f >> 16);
            }
            if (ll == 0) st_u32(blk + 172, uint32_t(B.d16) | (uint32_t(B.dm16) << 16));
        }
    } else {  // Q6S
        uint32_t lo0 = 0, lo1 = 0, hi = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            lo0 |= uint32_t(B.u[i] & 15u) << (4 * i);
            lo1 |= uint32_t(B.u[8 + i] & 15u) << (4 * i);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) hi |= uint32_t((B.u[i] >> 4) & 3u) << (2 * i);
        if (on) {
            uint8_t *p = blk + 8 * ll;                     // the block start is only 2-byte aligned
            st_u16(p, lo0 & 0xFFFFu); st_u16(p + 2, lo0 >> 16);
            st_u16(p + 4, lo1 & 0xFFFFu); st_u16(p + 6, lo1 >> 16);
            st_u16(blk + 128 + 4 * ll, hi & 0xFFFFu);
            st_u16(blk + 128 + 4 * ll + 2, hi >> 16);
            blk[192 + ll] = uint8_t(B.L);
            if (ll == 0) st_u16(blk + 208, B.d16);
        }
    }
}

// A lane's 16 input weights as loaded (four 16-byte vectors for fp32, two for fp16 / bf16).
struct Raw16 {
    Raw8 p0, p1;
};
template <int WDT>
__device__ __forceinline__ Raw16 ld_raw16(const void *W, int64_t idx) {
    return Raw16{ld_raw8<WDT>(W, idx), ld_raw8<WDT>(W, idx + 8)};
}

template <int F, int MODE, int WDT>
__global__ void __launch_bounds__(256) quant16_kernel(BlockArgs a) {
    using T = Fmt<F>;
    const int lane = threadIdx.x & 31, hw = lane >> 4, ll = lane & 15;
    const int64_t warp0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int64_t total = a.N * a.nbk;                    // 256-weight blocks
    const int64_t npairs = (total + 1) / 2;               // a warp takes blocks 2 p and 2 p + 1 of pair p
    const int64_t step = 2 * nwarps;                      // blocks between a half-warp's passes
    int64_t blk = 2 * warp0 + hw;
    int64_t r = blk / a.nbk, b = blk - r * a.nbk;
    const int64_t sr = step / a.nbk, sb = step - sr * a.nbk;
    int flags = 0;
    Raw16 nxt = {};
    if (blk < total && 256 * b + 16 * ll < a.K) nxt = ld_raw16<WDT>(a.W, r * a.K + 256 * b + 16 * ll);
    for (int64_t pv = warp0; pv < npairs; pv += nwarps, blk += step, r += sr, b += sb) {
        if (b >= a.nbk) { b -= a.nbk; ++r; }
        const bool live = blk < total;                    // the grid's last pair may hold a single block
        const int64_t k0 = 256 * b + 16 * ll;             // first weight of this lane within the row
        const bool valid = live && k0 < a.K;              // only INT4 rows can end inside a block
        const Raw16 cur = nxt;
        {
            int64_t r2 = r + sr, b2 = b + sb;
            if (b2 >= a.nbk) { b2 -= a.nbk; ++r2; }
            if (blk + step < total && 256 * b2 + 16 * ll < a.K)
                nxt = ld_raw16<WDT>(a.W, r2 * a.K + 256 * b2 + 16 * ll);
        }
        float w[16];
        if (valid) {
            cvt_raw8<WDT>(cur.p0, w);
            cvt_raw8<WDT>(cur.p1, w + 8);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = 0.0f;
        }
        LaneQ B;
        flags |= quantize16<F>(w, B);
        const int j = ll / (T::sublen / 16);              // this lane's group / sub-block within the block
        const bool first_of_sub = (ll % (T::sublen / 16)) == 0;
        if constexpr (MODE == MODE_QUANT_PARTS) {
            if (valid) {
                uint32_t cw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int i = 0; i < 16; ++i) cw[i >> 2] |= uint32_t(uint8_t(int(B.u[i]) - T::offset)) << (8 * (i & 3));
                uint2 *dst = reinterpret_cast<uint2 *>(a.codes + r * a.K + k0);
                dst[0] = make_uint2(cw[0], cw[1]);
                dst[1] = make_uint2(cw[2], cw[3]);
            }
            if constexpr (F == FMT_Q4G32 || F == FMT_Q4G16) {
                if (valid && first_of_sub) a.gscale[r * (a.K / T::sublen) + T::nsub * b + j] = B.gscale;
            } else if constexpr (F == FMT_Q4G32H) {
                if (valid && first_of_sub) a.d[r * (a.K / 32) + 8 * b + j] = B.d16;
            } else if constexpr (F == FMT_Q4G32A) {
                if (valid && first_of_sub) {
                    const int64_t e = r * (a.K / 16) + 2 * (8 * b + j);
                    a.gscale[e] = B.gscale;
                    a.gscale[e + 1] = B.gzero;
                }
            } else if (live) {
                const int64_t sbk = r * a.nbk + b;
                if (first_of_sub) {
                    a.sub_scale[sbk * T::nsub + j] = uint8_t(B.L);
                    if (T::asym) a.sub_min[sbk * T::nsub + j] = uint8_t(B.M);
                }
                if (ll == 0) {
                    a.d[sbk] = B.d16;
                    if (T::asym) a.dmin[sbk] = B.dm16;
                }
            }
        } else {
            uint8_t *row = a.packed + (live ? r : 0) * a.row_stride;
            pack16<F>(B, lane, kInt4<F> ? valid : live, row + b * T::bytes);
            if (live) {
                if constexpr (F == FMT_Q4G32 || F == FMT_Q4G16) {
                    if (valid && first_of_sub) a.gs_out[r * a.scale_stride + T::nsub * b + j] = B.gscale;
                    if (b == a.nbk - 1) {                  // zero the scale-row padding
                        const int64_t g0 = a.K / T::sublen;
                        if (g0 + ll < a.scale_stride) a.gs_out[r * a.scale_stride + g0 + ll] = 0.0f;
                    }
                } else if constexpr (F == FMT_Q4G32A) {
                    if (valid && first_of_sub) {
                        const int64_t e = r * a.scale_stride + 2 * (8 * b + j);
                        a.gs_out[e] = B.gscale;
                        a.gs_out[e + 1] = B.gzero;
                    }
                    if (b == a.nbk - 1) {
                        const int64_t g0 = a.K / 16;
                        if (g0 + ll < a.scale_stride) a.gs_out[r * a.scale_stride + g0 + ll] = 0.0f;
                    }
                } else if constexpr (F == FMT_Q4G32H) {
                    uint16_t *g16 = reinterpret_cast<uint16_t *>(a.gs_out);
                    if (valid && first_of_sub) g16[r * a.scale_stride + 8 * b + j] = B.d16;
                    if (b == a.nbk - 1) {
                        const int64_t g0 = a.K / 32;
                        if (g0 + ll < a.scale_stride) g16[r * a.scale_stride + g0 + ll] = 0;
                    }
                } else {
                    if (b == a.nbk - 1) {                  // zero the row padding (< 16 bytes)
                        const int64_t used = a.nbk * T::bytes;
                        if (used + ll < a.row_stride) row[used + ll] = 0;
                    }
                }
            }
        }
    }
    flags = __any_sync(0xffffffffu, flags != 0) ? 1 : 0;
    if (flags && lane == 0 && a.status) atomicOr(a.status, 1);
}

template <int F, int MODE, int WDT>
static cudaError_t launch_quant16(const BlockArgs &a, cudaStream_t s) {
    const int64_t pairs = (a.N * a.nbk + 1) / 2;
    int64_t blocks = (pairs + 7) / 8;
    const int64_t cap = int64_t(num_sms()) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return cudaSuccess;
    quant16_kernel<F, MODE, WDT><<<unsigned(blocks), 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <int F, int MODE, int WDT>
static cudaError_t launch_block(const BlockArgs &a, cudaStream_t s) {
    const int64_t warps = a.N * a.nbk;
    int64_t blocks = (warps + 7) / 8;
    const int64_t cap = int64_t(num_sms()) * 16;          // ~4 waves of resident CTAs (measured: faster than 1)
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return cudaSuccess;
    block_kernel<F, MODE, WDT><<<unsigned(blocks), 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <int F, int MODE>
static cudaError_t launch_wdt(const BlockArgs &a, int wdt, cudaStream_t s) {
    switch (wdt) {
        case DT_F32: return launch_quant16<F, MODE, DT_F32>(a, s);
        case DT_F16: return launch_quant16<F, MODE, DT_F16>(a, s);
        default: return launch_quant16<F, MODE, DT_BF16>(a, s);
    }
}

template <int F>
static cudaError_t launch_mode(const BlockArgs &a, int mode, int wdt, cudaStream_t s) {
    switch (mode) {
        case MODE_QUANT_PARTS: return launch_wdt<F, MODE_QUANT_PARTS>(a, wdt, s);
        case MODE_QUANT_PACKED: return launch_wdt<F, MODE_QUANT_PACKED>(a, wdt, s);
        case MODE_PACK: return launch_block<F, MODE_PACK, DT_F32>(a, s);
        case MODE_UNPACK: return launch_block<F, MODE_UNPACK, DT_F32>(a, s);
        default: return launch_block<F, MODE_DEQUANT, DT_F32>(a, s);
    }
}

cudaError_t launch_block_op(int fmt, int mode, int wdt, const BlockArgs &a, cudaStream_t s) {
    switch (fmt) {
        case FMT_Q4G32: return launch_mode<FMT_Q4G32>(a, mode, wdt, s);
        case FMT_Q2S: return launch_mode<FMT_Q2S>(a, mode, wdt, s);
        case FMT_Q3S: return launch_mode<FMT_Q3S>(a, mode, wdt, s);
        case FMT_Q5S: return launch_mode<FMT_Q5S>(a, mode, wdt, s);
        case FMT_Q6S: return launch_mode<FMT_Q6S>(a, mode, wdt, s);
        case FMT_Q4G32H: return launch_mode<FMT_Q4G32H>(a, mode, wdt, s);
        case FMT_Q4G16: return launch_mode<FMT_Q4G16>(a, mode, wdt, s);
        default: return launch_mode<FMT_Q4G32A>(a, mode, wdt, s);
    }
}

}  // namespace qpack
