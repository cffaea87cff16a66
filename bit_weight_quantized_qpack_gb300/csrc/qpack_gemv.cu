// qpack_gemv.cu — fused dequant-GEMV (batch 1) and small-batch GEMM (M <= 16) over packed low-bit weights.
//
// The decode-phase product is a pure stream over the packed weights: every weight byte is read from HBM once
// (2/3/5/6-bit article, lpnh.cn/news/2857666, §1.2: time per token = weight bytes / bandwidth; DBHOO-CIM
// article, pwwt.cn/news/4452170, §3.3: dequantization must stay fused, never materialised).
//
// Structure (one CTA per SM, persistent):
//   warp 8      producer: streams (4-row tile x 4096-weight chunk) segments of the packed rows into a ring of
//               shared-memory stages with 1-D bulk copies (cp.async.bulk, completion on an mbarrier), evict-first
//               in L2 because each byte is used once.
//   warps 0..7  consumers: warp pair p owns row p of the tile; each lane unpacks two 32-weight units per stage.
// Unpacking (2/3/5/6-bit article §3.3: separate unpack from multiply-add, factor s*(q.x) + m*sum(x)): codes are
// OR-ed into the mantissa of an fp16 1024.0 with one LOP3 per pair of weights, so a half holds 1024 + u*2^p
// exactly; an fp32 FMA with fp16 inputs (exact product) accumulates (1024 + u*2^p)*x per bit-position class p,
// and the constant 1024*sum(x) terms, the symmetric code offsets and the asymmetric minima are removed per
// sub-block with activation sums that each CTA precomputes once from x into shared memory.
#include <cuda_runtime.h>

#include "qpack_dev.cuh"
#include "qpack_launch.h"

namespace qpack {

__device__ int g_fault_gemv = 0;

namespace {

constexpr int NCW = 8;                   // consumer warps
constexpr int NTHREADS = (NCW + 1) * 32; // + producer warp
constexpr int TILE_R = 4;                // rows per tile (one warp pair per row)
constexpr int CHW = 4096;                // weights per chunk
constexpr int UPC = CHW / 32;            // 32-weight units per chunk
constexpr uint32_t MAGIC2 = 0x64006400u; // fp16 1024.0 in both halves
constexpr int SMEM_BUDGET = 220 * 1024;

template <int F> struct Geo {
    // bytes of one row's chunk in shared memory (codes; Q4G32 scales are a separate region)
    static constexpr int chunk_bytes = Fmt<F>::sb ? (CHW / 256) * Fmt<F>::bytes : CHW / 2;
    static constexpr int scale_bytes = Fmt<F>::sb ? 0 : (CHW / 32) * 4;
    static constexpr int stage_bytes = TILE_R * (chunk_bytes + scale_bytes);
    // activation-derived constants per 32-weight unit
    static constexpr int consts_per_unit = (F == FMT_Q4G32) ? 1 : (F == FMT_Q2S) ? 4 : (F == FMT_Q3S) ? 2 : (F == FMT_Q5S) ? 2 : 2;
};

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ uint16_t lo16(uint32_t v) { return uint16_t(v & 0xFFFFu); }
__device__ __forceinline__ uint16_t hi16(uint32_t v) { return uint16_t(v >> 16); }

// Accumulate a half2 of magic-coded weights against two activation halves.
__device__ __forceinline__ float fma2h(uint32_t codes, uint16_t xa, uint16_t xb, float acc) {
    acc = fma_h(lo16(codes), xa, acc);
    return fma_h(hi16(codes), xb, acc);
}

// x halves of a unit: xv[t] holds x[2t], x[2t+1].
__device__ __forceinline__ uint16_t xh(const uint32_t *xv, int i) {
    return (i & 1) ? hi16(xv[i >> 1]) : lo16(xv[i >> 1]);
}

__device__ __forceinline__ void load_x_unit(const uint16_t *xs, int64_t k0, uint32_t xv[16]) {
    const uint4 *p = reinterpret_cast<const uint4 *>(xs + k0);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        uint4 v = p[t];
        xv[4 * t] = v.x; xv[4 * t + 1] = v.y; xv[4 * t + 2] = v.z; xv[4 * t + 3] = v.w;
    }
}

__device__ __forceinline__ uint32_t lds32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }

// Read `n` consecutive 32-bit words starting at a 2-byte aligned shared-memory address.
template <int n>
__device__ __forceinline__ void lds_words_a2(const uint8_t *p, uint32_t *w) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t *base = reinterpret_cast<const uint32_t *>(a & ~uintptr_t(3));
    const uint32_t sh = uint32_t(a & 3u) * 8u;   // 0 or 16
    uint32_t r[n + 1];
#pragma unroll
    for (int i = 0; i <= n; ++i) r[i] = base[i];
#pragma unroll
    for (int i = 0; i < n; ++i) w[i] = __funnelshift_r(r[i], r[i + 1], sh);
}

// INT4-style nibble word: 8 weights, nibble k at bits 4k. Accumulates class p=0 (even k) and p=4 (odd k).
// `hb` (optional) holds high bits already positioned for the four pairs (see callers).
__device__ __forceinline__ void nib_word(uint32_t c, const uint32_t *xv, int i0, float &a0, float &a4) {
    const uint32_t c2 = c >> 8;
    a0 = fma2h(lop3_and_or(c, 0x000F000Fu, MAGIC2), xh(xv, i0 + 0), xh(xv, i0 + 4), a0);
    a4 = fma2h(lop3_and_or(c, 0x00F000F0u, MAGIC2), xh(xv, i0 + 1), xh(xv, i0 + 5), a4);
    a0 = fma2h(lop3_and_or(c2, 0x000F000Fu, MAGIC2), xh(xv, i0 + 2), xh(xv, i0 + 6), a0);
    a4 = fma2h(lop3_and_or(c2, 0x00F000F0u, MAGIC2), xh(xv, i0 + 3), xh(xv, i0 + 7), a4);
}

// Nibble word with extra high bits merged above each nibble. X holds, for the pairs (0,4),(1,5),(2,6),(3,7),
// the high bits already shifted so that (X << s_k) & mask_k lands them just above the pair's nibbles.
template <int HB>   // 1 (5-bit) or 2 (6-bit) high bits
__device__ __forceinline__ void nib_word_hi(uint32_t c, uint32_t X, const uint32_t *xv, int i0, float &a0, float &a4) {
    constexpr uint32_t mlo = (HB == 1) ? 0x00100010u : 0x00300030u;   // bits 4(+5) of each half
    constexpr uint32_t mhi = (HB == 1) ? 0x01000100u : 0x03000300u;   // bits 8(+9) of each half
    // shifts that bring pair k's high bits of X to the target positions
    constexpr int s0 = (HB == 1) ? 4 : 4, s1 = (HB == 1) ? 7 : 6, s2 = (HB == 1) ? 2 : 0, s3 = (HB == 1) ? 5 : 2;
    const uint32_t c2 = c >> 8;
    uint32_t h;
    h = lop3_and_or(c, 0x000F000Fu, MAGIC2);
    h = lop3_and_or(X << s0, mlo, h);
    a0 = fma2h(h, xh(xv, i0 + 0), xh(xv, i0 + 4), a0);
    h = lop3_and_or(c, 0x00F000F0u, MAGIC2);
    h = lop3_and_or(X << s1, mhi, h);
    a4 = fma2h(h, xh(xv, i0 + 1), xh(xv, i0 + 5), a4);
    h = lop3_and_or(c2, 0x000F000Fu, MAGIC2);
    h = lop3_and_or(X << s2, mlo, h);
    a0 = fma2h(h, xh(xv, i0 + 2), xh(xv, i0 + 6), a0);
    h = lop3_and_or(c2, 0x00F000F0u, MAGIC2);
    h = lop3_and_or(X << s3, mhi, h);
    a4 = fma2h(h, xh(xv, i0 + 3), xh(xv, i0 + 7), a4);
}

// 2-bit word: 16 weights, weight 4b+k at bits 8b+2k. Classes p = 2k (k = 0..3).
__device__ __forceinline__ void crumb_word(uint32_t c, const uint32_t *xv, int i0, float a[4]) {
    const uint32_t c2 = c >> 8;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t m = (3u << (2 * k)) * 0x00010001u;
        a[k] = fma2h(lop3_and_or(c, m, MAGIC2), xh(xv, i0 + k), xh(xv, i0 + 8 + k), a[k]);
        a[k] = fma2h(lop3_and_or(c2, m, MAGIC2), xh(xv, i0 + 4 + k), xh(xv, i0 + 12 + k), a[k]);
    }
}

// 3-bit group: 24-bit value v (bits above 23 ignored), code t at bits 3t, weights i0..i0+7.
// Classes: p=0 {0,3,4,7}, p=3 {1,5}, p=6 {2,6}.
__device__ __forceinline__ void tri_group(uint32_t v, const uint32_t *xv, int i0, float &a0, float &a3, float &a6) {
    const uint32_t Y = lop3_sel(v, v << 4, 0x00000FFFu);   // codes 0..3 in the low half, 4..7 in the high half
    const uint32_t Y9 = Y >> 9;
    a0 = fma2h(lop3_and_or(Y, 0x00070007u, MAGIC2), xh(xv, i0 + 0), xh(xv, i0 + 4), a0);
    a3 = fma2h(lop3_and_or(Y, 0x00380038u, MAGIC2), xh(xv, i0 + 1), xh(xv, i0 + 5), a3);
    a6 = fma2h(lop3_and_or(Y, 0x01C001C0u, MAGIC2), xh(xv, i0 + 2), xh(xv, i0 + 6), a6);
    a0 = fma2h(lop3_and_or(Y9, 0x00070007u, MAGIC2), xh(xv, i0 + 3), xh(xv, i0 + 7), a0);
}

__device__ __forceinline__ float hbits(const uint8_t *p) { return h2f_bits(*reinterpret_cast<const uint16_t *>(p)); }

// ------------------------------------------------------------------------------------------------------------
// Batch-1 unit dot products. `row` = the row's chunk in shared memory (codes), `uc` = unit within the chunk,
// `cst` = activation constants of this unit, `xv` = the unit's 32 activations. Returns sum_i w'_i * x_i.
// ------------------------------------------------------------------------------------------------------------
template <int F> struct Unit1;

template <> struct Unit1<FMT_Q4G32> {
    // constants: C = 1032*S_even + 72*S_odd
    static __device__ __forceinline__ float dot(const uint8_t *row, const float *scl, int uc, const float *cst,
                                                const uint32_t *xv) {
        const uint4 c = *reinterpret_cast<const uint4 *>(row + 16 * uc);
        float a0 = 0.f, a4 = 0.f;
        nib_word(c.x, xv, 0, a0, a4);
        nib_word(c.y, xv, 8, a0, a4);
        nib_word(c.z, xv, 16, a0, a4);
        nib_word(c.w, xv, 24, a0, a4);
        return scl[uc] * (fmaf(a4, 0.0625f, a0) - cst[0]);
    }
    static __device__ __forceinline__ void consts(const uint16_t *xs, int64_t u, float *out) {
        float se = 0.f, so = 0.f;
        for (int i = 0; i < 32; i += 2) { se += h2f_bits(xs[32 * u + i]); so += h2f_bits(xs[32 * u + i + 1]); }
        out[0] = 1032.0f * se + 72.0f * so;
    }
};

template <> struct Unit1<FMT_Q2S> {
    // constants per sub-block j (16 weights): C_j = 1024 * sum_k 4^-k S_{j,k}, S_j
    static __device__ __forceinline__ float dot(const uint8_t *row, const float *, int uc, const float *cst,
                                                const uint32_t *xv) {
        const int sbk = uc >> 3, su = uc & 7;
        const uint8_t *blk = row + sbk * 84;
        const uint32_t w0 = lds32(blk + 8 * su), w1 = lds32(blk + 8 * su + 4);
        const float D = hbits(blk + 80), Dm = hbits(blk + 82);
        const uint32_t lm = *reinterpret_cast<const uint16_t *>(blk + 64 + 2 * su);
        float r = 0.f;
        {
            float a[4] = {0.f, 0.f, 0.f, 0.f};
            crumb_word(w0, xv, 0, a);
            const float t = fmaf(a[3], 0.015625f, fmaf(a[2], 0.0625f, fmaf(a[1], 0.25f, a[0]))) - cst[0];
            r = fmaf(D * float(lm & 15u), t, r);
            r = fmaf(-Dm * float((lm >> 4) & 15u), cst[1], r);
        }
        {
            float a[4] = {0.f, 0.f, 0.f, 0.f};
            crumb_word(w1, xv, 16, a);
            const float t = fmaf(a[3], 0.015625f, fmaf(a[2], 0.0625f, fmaf(a[1], 0.25f, a[0]))) - cst[2];
            r = fmaf(D * float((lm >> 8) & 15u), t, r);
            r = fmaf(-Dm * float((lm >> 12) & 15u), cst[3], r);
        }
        return r;
    }
    static __device__ __forceinline__ void consts(const uint16_t *xs, int64_t u, float *out) {
        for (int h = 0; h < 2; ++h) {
            float S[4] = {0.f, 0.f, 0.f, 0.f};
            for (int i = 0; i < 16; ++i) S[i & 3] += h2f_bits(xs[32 * u + 16 * h + i]);
            out[2 * h] = 1024.0f * (S[0] + 0.25f * S[1] + 0.0625f * S[2] + 0.015625f * S[3]);
            out[2 * h + 1] = S[0] + S[1] + S[2] + S[3];
        }
    }
};

template <> struct Unit1<FMT_Q3S> {
    // constants per sub-block j: C_j = 1024*(S0 + S3/8 + S6/64) + 4*(S0 + S3 + S6)
    static __device__ __forceinline__ float dot(const uint8_t *row, const float *, int uc, const float *cst,
                                                const uint32_t *xv) {
        const int sbk = uc >> 3, su = uc & 7;
        const uint8_t *blk = row + sbk * 110;
        uint32_t s[3];
        lds_words_a2<3>(blk + 12 * su, s);
        const uint32_t v1 = __funnelshift_r(s[0], s[1], 24);
        const uint32_t v2 = __funnelshift_r(s[1], s[2], 16);
        const uint32_t v3 = s[2] >> 8;
        const float D = hbits(blk + 108);
        const uint8_t *fb = blk + 96 + 3 * (su >> 1);
        const uint32_t f = uint32_t(fb[0]) | (uint32_t(fb[1]) << 8) | (uint32_t(fb[2]) << 16);
        const int j0 = (2 * su) & 3;
        const float L0 = float((f >> (6 * j0)) & 63u), L1 = float((f >> (6 * (j0 + 1))) & 63u);
        float a0 = 0.f, a3 = 0.f, a6 = 0.f;
        tri_group(s[0], xv, 0, a0, a3, a6);
        tri_group(v1, xv, 8, a0, a3, a6);
        float r = D * L0 * (fmaf(a6, 0.015625f, fmaf(a3, 0.125f, a0)) - cst[0]);
        a0 = a3 = a6 = 0.f;
        tri_group(v2, xv, 16, a0, a3, a6);
        tri_group(v3, xv, 24, a0, a3, a6);
        r = fmaf(D * L1, fmaf(a6, 0.015625f, fmaf(a3, 0.125f, a0)) - cst[1], r);
        return r;
    }
    static __device__ __forceinline__ void consts(const uint16_t *xs, int64_t u, float *out) {
        for (int h = 0; h < 2; ++h) {
            float S0 = 0.f, S3 = 0.f, S6 = 0.f;
            for (int i = 0; i < 16; ++i) {
                const float v = h2f_bits(xs[32 * u + 16 * h + i]);
                const int t = i & 7;
                if (t == 1 || t == 5) S3 += v; else if (t == 2 || t == 6) S6 += v; else S0 += v;
            }
            out[h] = 1024.0f * (S0 + 0.125f * S3 + 0.015625f * S6) + 4.0f * (S0 + S3 + S6);
        }
    }
};

template <> struct Unit1<FMT_Q5S> {
    // constants per unit (one sub-block of 32): C = 1024*S_even + 64*S_odd, S
    static __device__ __forceinline__ float dot(const uint8_t *row, const float *, int uc, const float *cst,
                                                const uint32_t *xv) {
        const int sbk = uc >> 3, su = uc & 7;
        const uint8_t *blk = row + sbk * 176;
        const uint4 c = *reinterpret_cast<const uint4 *>(blk + 16 * su);
        const uint32_t H = lds32(blk + 128 + 4 * su);
        const float D = hbits(blk + 172), Dm = hbits(blk + 174);
        // 6-bit fields: L_su = field su, M_su = field 8 + su
        const uint8_t *fl = blk + 160 + 3 * (su >> 2);
        const uint8_t *fm = blk + 166 + 3 * (su >> 2);
        const uint32_t vl = uint32_t(fl[0]) | (uint32_t(fl[1]) << 8) | (uint32_t(fl[2]) << 16);
        const uint32_t vm = uint32_t(fm[0]) | (uint32_t(fm[1]) << 8) | (uint32_t(fm[2]) << 16);
        const float L = float((vl >> (6 * (su & 3))) & 63u), M = float((vm >> (6 * (su & 3))) & 63u);
        float a0 = 0.f, a4 = 0.f;
        // X_t: high bits of weights 8t..8t+3 at bits 0..3, of 8t+4..8t+7 at bits 16..19 (garbage elsewhere).
        nib_word_hi<1>(c.x, lop3_sel(H, H << 12, 0x0000FFFFu), xv, 0, a0, a4);
        nib_word_hi<1>(c.y, lop3_sel(H >> 8, H << 4, 0x0000FFFFu), xv, 8, a0, a4);
        nib_word_hi<1>(c.z, lop3_sel(H >> 16, H >> 4, 0x0000FFFFu), xv, 16, a0, a4);
        nib_word_hi<1>(c.w, lop3_sel(H >> 24, H >> 12, 0x0000FFFFu), xv, 24, a0, a4);
        const float t = fmaf(a4, 0.0625f, a0) - cst[0];
        return fmaf(D * L, t, -(Dm * M) * cst[1]);
    }
    static __device__ __forceinline__ void consts(const uint16_t *xs, int64_t u, float *out) {
        float se = 0.f, so = 0.f;
        for (int i = 0; i < 32; i += 2) { se += h2f_bits(xs[32 * u + i]); so += h2f_bits(xs[32 * u + i + 1]); }
        out[0] = 1024.0f * se + 64.0f * so;
        out[1] = se + so;
    }
};

template <> struct Unit1<FMT_Q6S> {
    // constants per sub-block j (16): C_j = 1056*S_even + 96*S_odd
    static __device__ __forceinline__ float dot(const uint8_t *row, const float *, int uc, const float *cst,
                                                const uint32_t *xv) {
        const int sbk = uc >> 3, su = uc & 7;
        const uint8_t *blk = row + sbk * 210;
        uint32_t c[4], h[2];
        lds_words_a2<4>(blk + 16 * su, c);
        lds_words_a2<2>(blk + 128 + 8 * su, h);
        const float D = hbits(blk + 208);
        const float L0 = float(int8_t(blk[192 + 2 * su])), L1 = float(int8_t(blk[193 + 2 * su]));
        // X_t: high-2 byte pair (2t, 2t+1) of the sub-block's high word spread to bytes 0 and 2.
        float a0 = 0.f, a4 = 0.f;
        nib_word_hi<2>(c[0], __byte_perm(h[0], 0u, 0x4140u), xv, 0, a0, a4);
        nib_word_hi<2>(c[1], __byte_perm(h[0], 0u, 0x4342u), xv, 8, a0, a4);
        float r = D * L0 * (fmaf(a4, 0.0625f, a0) - cst[0]);
        a0 = a4 = 0.f;
        nib_word_hi<2>(c[2], __byte_perm(h[1], 0u, 0x4140u), xv, 16, a0, a4);
        nib_word_hi<2>(c[3], __byte_perm(h[1], 0u, 0x4342u), xv, 24, a0, a4);
        return fmaf(D * L1, fmaf(a4, 0.0625f, a0) - cst[1], r);
    }
    static __device__ __forceinline__ void consts(const uint16_t *xs, int64_t u, float *out) {
        for (int h = 0; h < 2; ++h) {
            float se = 0.f, so = 0.f;
            for (int i = 0; i < 16; i += 2) { se += h2f_bits(xs[32 * u + 16 * h + i]); so += h2f_bits(xs[32 * u + 16 * h + i + 1]); }
            out[h] = 1056.0f * se + 96.0f * so;
        }
    }
};

// ------------------------------------------------------------------------------------------------------------
// Exact unit decode for the small-batch path: 32 dequantized fp32 weights (same roundings as FORMATS.md).
// ------------------------------------------------------------------------------------------------------------
template <int F>
__device__ __forceinline__ void decode_unit(const uint8_t *row, const float *scl, int uc, float w[32]) {
    if constexpr (F == FMT_Q4G32) {
        const uint4 c = *reinterpret_cast<const uint4 *>(row + 16 * uc);
        const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
        const float s = scl[uc];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = __fmul_rn(s, float(int((cw[i >> 3] >> (4 * (i & 7))) & 15u) - 8));
    } else if constexpr (F == FMT_Q2S) {
        const int sbk = uc >> 3, su = uc & 7;
        const uint8_t *blk = row + sbk * 84;
        const uint32_t cw[2] = {lds32(blk + 8 * su), lds32(blk + 8 * su + 4)};
        const float D = hbits(blk + 80), Dm = hbits(blk + 82);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t lm = blk[64 + 2 * su + h];
            const float es = __fmul_rn(D, float(lm & 15u)), em = __fmul_rn(Dm, float(lm >> 4));
#pragma unroll
            for (int i = 0; i < 16; ++i)
                w[16 * h + i] = __fsub_rn(__fmul_rn(es, float((cw[h] >> (2 * i)) & 3u)), em);
        }
    } else if constexpr (F == FMT_Q3S) {
        const int sbk = uc >> 3, su = uc & 7;
        const uint8_t *blk = row + sbk * 110;
        uint32_t s[3];
        lds_words_a2<3>(blk + 12 * su, s);
        const uint32_t v[4] = {s[0], __funnelshift_r(s[0], s[1], 24), __funnelshift_r(s[1], s[2], 16), s[2] >> 8};
        const float D = hbits(blk + 108);
        const uint8_t *fb = blk + 96 + 3 * (su >> 1);
        const uint32_t f = uint32_t(fb[0]) | (uint32_t(fb[1]) << 8) | (uint32_t(fb[2]) << 16);
        const int j0 = (2 * su) & 3;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float es = __fmul_rn(D, float((f >> (6 * (j0 + h))) & 63u));
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int g = 2 * h + (i >> 3), t = i & 7;
                w[16 * h + i] = __fmul_rn(es, float(int((v[g] >> (3 * t)) & 7u) - 4));
            }
        }
    } else if constexpr (F == FMT_Q5S) {
        const int sbk = uc >> 3, su = uc & 7;
        const uint8_t *blk = row + sbk * 176;
        const uint4 c = *reinterpret_cast<const uint4 *>(blk + 16 * su);
        const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
        const uint32_t H = lds32(blk + 128 + 4 * su);
        const float D = hbits(blk + 172), Dm = hbits(blk + 174);
        const uint8_t *fl = blk + 160 + 3 * (su >> 2), *fm = blk + 166 + 3 * (su >> 2);
        const uint32_t vl = uint32_t(fl[0]) | (uint32_t(fl[1]) << 8) | (uint32_t(fl[2]) << 16);
        const uint32_t vm = uint32_t(fm[0]) | (uint32_t(fm[1]) << 8) | (uint32_t(fm[2]) << 16);
        const float es = __fmul_rn(D, float((vl >> (6 * (su & 3))) & 63u));
        const float em = __fmul_rn(Dm, float((vm >> (6 * (su & 3))) & 63u));
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t u = ((cw[i >> 3] >> (4 * (i & 7))) & 15u) | (((H >> i) & 1u) << 4);
            w[i] = __fsub_rn(__fmul_rn(es, float(u)), em);
        }
    } else {
        const int sbk = uc >> 3, su = uc & 7;
        const uint8_t *blk = row + sbk * 210;
        uint32_t c[4], h[2];
        lds_words_a2<4>(blk + 16 * su, c);
        lds_words_a2<2>(blk + 128 + 8 * su, h);
        const float D = hbits(blk + 208);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const float es = __fmul_rn(D, float(int8_t(blk[192 + 2 * su + hh])));
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int ii = 16 * hh + i;
                const uint32_t u = ((c[ii >> 3] >> (4 * (ii & 7))) & 15u) | (((h[hh] >> (2 * i)) & 3u) << 4);
                w[ii] = __fmul_rn(es, float(int(u) - 32));
            }
        }
    }
}

struct Smem {
    uint64_t *full, *empty;
    float *red;        // [2][NCW][MT]
    uint16_t *xs;      // batch-1: x [K] (fp16)
    float *cst;        // batch-1: per-unit activation constants
    uint8_t *stages;   // NS x stage_bytes
};

}  // namespace

// ------------------------------------------------------------------------------------------------------------
// The streaming kernel. MT = 1: batch-1 GEMV with the magic-offset unpack; MT > 1: small-batch GEMM with exact
// per-unit dequantization and M FMAs per weight (activations read through L1).
// ------------------------------------------------------------------------------------------------------------
template <int F, int MT>
__global__ void __launch_bounds__(NTHREADS, 1) stream_kernel(GemvArgs a, int NS) {
    using G = Geo<F>;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t N = a.N, K = a.K;
    const int64_t ntiles = (N + TILE_R - 1) / TILE_R;
    const int nchunks = int((K + CHW - 1) / CHW);
    const int64_t units_row = K / 32;

    // ---- carve shared memory ----
    uint8_t *p = smem_raw;
    uint64_t *full = reinterpret_cast<uint64_t *>(p);
    uint64_t *empty = full + NS;
    p += round_up(16 * NS, 128);
    float *red = reinterpret_cast<float *>(p);
    p += round_up(2 * NCW * MT * 4, 128);
    uint16_t *xs = nullptr;
    float *cst = nullptr;
    if constexpr (MT == 1) {
        xs = reinterpret_cast<uint16_t *>(p);
        p += round_up(2 * K, 128);
        cst = reinterpret_cast<float *>(p);
        p += round_up(4 * units_row * G::consts_per_unit, 128);
    }
    uint8_t *stages = p;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], NCW); }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NCW) {
        // ================================= producer =================================
        const uint64_t pol = l2_evict_first_policy();
        int it = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            const int64_t r0 = tile * TILE_R;
            const int rows = int(imin64(TILE_R, N - r0));
            for (int c = 0; c < nchunks; ++c) {
                const int s = it % NS;
                const uint32_t ph = uint32_t(it / NS) & 1u;
                if (it >= NS) {
                    bool ok = true;
                    if (lane == 0) ok = mbar_wait_bounded(&empty[s], ph ^ 1u);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    // A consumer stopped releasing stages: record it and stop producing. Consumers then give up
                    // on their next bounded wait, so nothing is left waiting.
                    if (!ok) { if (lane == 0) atomicOr(&g_fault_gemv, FAULT_WAIT_EMPTY); return; }
                }
                int64_t cbytes, sbytes = 0;
                const int64_t koff = int64_t(c) * CHW;
                if constexpr (Fmt<F>::sb) {
                    const int64_t off = (koff / 256) * Fmt<F>::bytes;
                    cbytes = imin64(G::chunk_bytes, a.row_stride - off);
                } else {
                    cbytes = imin64(G::chunk_bytes, (K - koff) / 2);
                    sbytes = imin64(G::scale_bytes, (a.scale_stride - koff / 32) * 4);
                }
                uint8_t *st = stages + int64_t(s) * G::stage_bytes;
                if (lane == 0) mbar_arrive_expect_tx(&full[s], uint32_t(rows * (cbytes + sbytes)));
                __syncwarp();
                if (lane < rows) {
                    const int64_t r = r0 + lane;
                    const uint8_t *src;
                    if constexpr (Fmt<F>::sb) src = a.packed + r * a.row_stride + (koff / 256) * Fmt<F>::bytes;
                    else src = a.packed + r * a.row_stride + koff / 2;
                    bulk_g2s(st + lane * G::chunk_bytes, src, uint32_t(cbytes), &full[s], pol);
                } else if (!Fmt<F>::sb && lane >= 8 && lane < 8 + rows) {
                    const int64_t r = r0 + (lane - 8);
                    const uint8_t *src = reinterpret_cast<const uint8_t *>(a.gscale + r * a.scale_stride + koff / 32);
                    bulk_g2s(st + TILE_R * G::chunk_bytes + (lane - 8) * G::scale_bytes, src, uint32_t(sbytes),
                             &full[s], pol);
                }
                ++it;
            }
        }
        return;
    }

    // =================================== consumers ===================================
    if constexpr (MT == 1) {
        // x -> shared memory, then per-unit activation constants (once per CTA)
        const uint4 *xg = reinterpret_cast<const uint4 *>(a.X);
        uint4 *xd = reinterpret_cast<uint4 *>(xs);
        for (int64_t i = tid; i < K / 8; i += NCW * 32) xd[i] = xg[i];
        named_bar_sync(1, NCW * 32);
        for (int64_t u = tid; u < units_row; u += NCW * 32) Unit1<F>::consts(xs, u, cst + u * G::consts_per_unit);
        named_bar_sync(1, NCW * 32);
    }

    const int pair = warp >> 1, half = warp & 1;    // warp pair `pair` owns row `pair` of the tile
    int it = 0, tcount = 0;
    bool dead = false;   // set after a bounded wait gave up: skip all further waits and work, keep the barriers
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tcount) {
        const int64_t r0 = tile * TILE_R;
        const bool row_ok = (r0 + pair) < N;
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
        for (int c = 0; c < nchunks; ++c) {
            const int s = it % NS;
            const uint32_t ph = uint32_t(it / NS) & 1u;
            if (!dead) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait_bounded(&full[s], ph);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) { if (lane == 0) atomicOr(&g_fault_gemv, FAULT_WAIT_FULL); dead = true; }
            }
            const int64_t koff = int64_t(c) * CHW;
            const int units = int(imin64(UPC, (K - koff) / 32));
            const uint8_t *st = stages + int64_t(s) * G::stage_bytes;
            const uint8_t *row = st + pair * G::chunk_bytes;
            const float *scl = reinterpret_cast<const float *>(st + TILE_R * G::chunk_bytes + pair * G::scale_bytes);
            if (row_ok && !dead) {
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    const int uc = 64 * half + 32 * v + lane;
                    if (uc < units) {
                        if constexpr (MT == 1) {
                            uint32_t xv[16];
                            load_x_unit(xs, koff + 32 * uc, xv);
                            acc[0] += Unit1<F>::dot(row, scl, uc, cst + (koff / 32 + uc) * G::consts_per_unit, xv);
                        } else {
                            float w[32];
                            decode_unit<F>(row, scl, uc, w);
#pragma unroll
                            for (int m = 0; m < MT; ++m) {
                                if (m < a.M) {
                                    const uint4 *xp = reinterpret_cast<const uint4 *>(a.X + m * a.ldx + koff + 32 * uc);
                                    float t = 0.f;
#pragma unroll
                                    for (int q = 0; q < 4; ++q) {
                                        const uint4 xq = __ldg(xp + q);
                                        const uint32_t xw[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
                                        for (int e = 0; e < 4; ++e) {
                                            t = fmaf(w[8 * q + 2 * e], h2f_bits(lo16(xw[e])), t);
                                            t = fmaf(w[8 * q + 2 * e + 1], h2f_bits(hi16(xw[e])), t);
                                        }
                                    }
                                    acc[m] += t;
                                }
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            ++it;
        }
        // ---- reduce the row over the warp pair ----
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float v = acc[m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[m] = v;
        }
        float *rb = red + (tcount & 1) * NCW * MT;
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < MT; ++m) rb[warp * MT + m] = acc[m];
        }
        named_bar_sync(2 + pair, 64);
        if (half == 0 && row_ok && lane < MT && lane < a.M) {
            const float v = rb[(2 * pair) * MT + lane] + rb[(2 * pair + 1) * MT + lane];
            a.Y[int64_t(lane) * a.ldy + r0 + pair] = v;
        }
    }
}

template <int F, int MT>
static cudaError_t launch_stream(const GemvArgs &a, cudaStream_t s) {
    using G = Geo<F>;
    const int64_t units_row = a.K / 32;
    int64_t fixed = 128 /*barrier area upper bound for NS <= 8 is recomputed below*/;
    int64_t extra = round_up(2 * NCW * MT * 4, 128);
    if (MT == 1) extra += round_up(2 * a.K, 128) + round_up(4 * units_row * G::consts_per_unit, 128);
    // choose the stage count so that barriers + extras + stages fit
    int NS = 0;
    for (int ns = 16; ns >= 2; --ns) {
        const int64_t tot = round_up(16 * ns, 128) + extra + int64_t(ns) * G::stage_bytes + 16;
        if (tot <= SMEM_BUDGET) { NS = ns; fixed = tot; break; }
    }
    if (NS == 0) return cudaErrorInvalidValue;
    const size_t smem = size_t(fixed);
    auto kern = stream_kernel<F, MT>;
    // Raise the dynamic shared-memory limit once per device (not per launch, so launches can be graph-captured).
    static int opted[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (opted[dev] == 0) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BUDGET);
        if (e != cudaSuccess) return e;
        opted[dev] = 1;
    }
    const int64_t ntiles = (a.N + TILE_R - 1) / TILE_R;
    int grid = num_sms();
    if (ntiles < grid) grid = int(ntiles);
    if (grid < 1) return cudaSuccess;
    kern<<<grid, NTHREADS, smem, s>>>(a, NS);
    return cudaGetLastError();
}

template <int F>
static cudaError_t launch_fmt(const GemvArgs &a, cudaStream_t s) {
    if (a.M <= 1) return launch_stream<F, 1>(a, s);
    if (a.M <= 2) return launch_stream<F, 2>(a, s);
    if (a.M <= 4) return launch_stream<F, 4>(a, s);
    if (a.M <= 8) return launch_stream<F, 8>(a, s);
    return launch_stream<F, 16>(a, s);
}

cudaError_t launch_gemv(int fmt, const GemvArgs &a, cudaStream_t s) {
    switch (fmt) {
        case FMT_Q4G32: return launch_fmt<FMT_Q4G32>(a, s);
        case FMT_Q2S: return launch_fmt<FMT_Q2S>(a, s);
        case FMT_Q3S: return launch_fmt<FMT_Q3S>(a, s);
        case FMT_Q5S: return launch_fmt<FMT_Q5S>(a, s);
        default: return launch_fmt<FMT_Q6S>(a, s);
    }
}

cudaError_t fetch_fault_gemv(int32_t *flags) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_fault_gemv, sizeof(int));
    if (e != cudaSuccess) return e;
    *flags |= v;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_fault_gemv, &zero, sizeof(int));
}

}  // namespace qpack
