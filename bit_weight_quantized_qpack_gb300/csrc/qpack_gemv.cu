// qpack_gemv.cu — fused dequant-GEMV (batch 1) and small-batch GEMM (M <= 16) over packed low-bit weights.
//
// The decode-phase product is a pure stream over the packed weights: every weight byte is read from HBM once
// (2/3/5/6-bit article, lpnh.cn/news/2857666, §1.2: time per token = weight bytes / bandwidth; DBHOO-CIM
// article, pwwt.cn/news/4452170, §3.3: dequantization must stay fused, never materialised).
//
// Batch-1 kernel (gemv1_kernel), one persistent CTA per SM:
//   warp 16      producer: streams (4-row tile x 4096-weight chunk) segments of the packed rows into a ring of
//                shared-memory stages with 1-D bulk copies (cp.async.bulk, completion on an mbarrier), L2
//                evict-first because each byte is used once.
//   warps 0..15  two consumer groups of 8 warps; group g consumes the stages whose item index has parity g. In
//                a group, lane l of warp w owns the 32-weight unit uc = (32w + l) mod 128 of the rows
//                (32w + l) div 128 and that + 2, so its activations are loaded once for two rows.
// Unpacking (2/3/5/6-bit article §3.3: separate unpack from multiply-add, factor s*(q.x) + m*sum(x)): codes are
// OR-ed into the mantissa of an fp16 1024.0 with one LOP3 per pair of weights, so a half holds 1024 + u*2^p
// exactly, p being the code's bit position inside its 16-bit half. The activations are staged in shared memory
// pre-scaled by 2^-p of the code they meet (x' = fp16(x * 2^-p), exact unless subnormal), so one fp32 FMA with
// fp16 inputs (exact product) per weight accumulates 1024*x' + u*x for every class into one accumulator. The
// 1024*sum(x') terms, the symmetric code offsets and the asymmetric minima are removed per sub-block with
// activation sums that each CTA precomputes once. Per-row results are combined without a block barrier: each
// warp reduces its two rows, publishes the partials and bumps a per-tile counter; the warp completing the count
// sums the partials in a fixed order (deterministic) and writes y.
//
// Small-batch kernel (stream_kernel, M = 2..16): same producer; each unit is dequantized exactly to fp32
// registers and multiplied against the M activation rows.
#include <cuda_runtime.h>

#include "qpack_dev.cuh"
#include "qpack_launch.h"

namespace qpack {

__device__ int g_fault_gemv = 0;

namespace {

constexpr int TILE_R = 4;                // rows per tile
constexpr int CHW = 4096;                // weights per chunk (stage width)
constexpr int UPC = CHW / 32;            // 32-weight units per chunk
constexpr uint32_t MAGIC2 = 0x64006400u; // fp16 1024.0 in both halves
constexpr uint32_t MAGICF = 0x4B000000u; // fp32 2^23

template <int F> struct Geo {
    // bytes of one row's chunk in shared memory (codes; Q4G32 scales are a separate region)
    static constexpr int chunk_bytes = Fmt<F>::sb ? (CHW / 256) * Fmt<F>::bytes : CHW / 2;
    static constexpr int scale_bytes = Fmt<F>::sb ? 0 : (CHW / 32) * 4;
    static constexpr int stage_bytes = TILE_R * (chunk_bytes + scale_bytes);
};

__device__ __forceinline__ uint16_t lo16(uint32_t v) { return uint16_t(v & 0xFFFFu); }
__device__ __forceinline__ uint16_t hi16(uint32_t v) { return uint16_t(v >> 16); }
__device__ __forceinline__ uint32_t lds32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ float hbits(const uint8_t *p) { return h2f_bits(*reinterpret_cast<const uint16_t *>(p)); }
__device__ __forceinline__ float small_int_f(uint32_t bits_or_magic) { return __uint_as_float(bits_or_magic) - 8388608.0f; }

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

// acc += lo(codes) * xa + hi(codes) * xb with exact products (fp16 x fp16 -> fp32 FMA).
__device__ __forceinline__ float fma2h(uint32_t codes, uint16_t xa, uint16_t xb, float acc) {
    acc = fma_h(lo16(codes), xa, acc);
    return fma_h(hi16(codes), xb, acc);
}
// x halves of a unit: xv[t] holds x'[2t], x'[2t+1].
__device__ __forceinline__ uint16_t xh(const uint32_t *xv, int i) { return (i & 1) ? hi16(xv[i >> 1]) : lo16(xv[i >> 1]); }

// ------------------------------------------------------------------------------------------------------------
// Unpack + multiply helpers. Two accumulators (a, b) only for instruction-level parallelism.
// ------------------------------------------------------------------------------------------------------------
// 8 nibbles, nibble k at bits 4k (weights i0 + k). Bit classes: even k at p = 0, odd k at p = 4.
__device__ __forceinline__ void nib_word(uint32_t c, const uint32_t *xv, int i0, float &a, float &b) {
    const uint32_t c2 = c >> 8;
    a = fma2h(lop3_and_or(c, 0x000F000Fu, MAGIC2), xh(xv, i0 + 0), xh(xv, i0 + 4), a);
    b = fma2h(lop3_and_or(c, 0x00F000F0u, MAGIC2), xh(xv, i0 + 1), xh(xv, i0 + 5), b);
    a = fma2h(lop3_and_or(c2, 0x000F000Fu, MAGIC2), xh(xv, i0 + 2), xh(xv, i0 + 6), a);
    b = fma2h(lop3_and_or(c2, 0x00F000F0u, MAGIC2), xh(xv, i0 + 3), xh(xv, i0 + 7), b);
}
// Nibble word with HB extra high bits merged just above each nibble. X holds the high bits of weights
// i0..i0+3 at bits HB*k (k = 0..3) and of weights i0+4..i0+7 at bits 16 + HB*k; (X << s_k) & mask lands pair
// k's high bits right above its nibbles.
template <int HB>
__device__ __forceinline__ void nib_word_hi(uint32_t c, uint32_t X, const uint32_t *xv, int i0, float &a, float &b) {
    constexpr uint32_t mlo = (HB == 1) ? 0x00100010u : 0x00300030u;
    constexpr uint32_t mhi = (HB == 1) ? 0x01000100u : 0x03000300u;
    constexpr int s0 = 4, s1 = (HB == 1) ? 7 : 6, s2 = (HB == 1) ? 2 : 0, s3 = (HB == 1) ? 5 : 2;
    const uint32_t c2 = c >> 8;
    a = fma2h(lop3_and_or(X << s0, mlo, lop3_and_or(c, 0x000F000Fu, MAGIC2)), xh(xv, i0 + 0), xh(xv, i0 + 4), a);
    b = fma2h(lop3_and_or(X << s1, mhi, lop3_and_or(c, 0x00F000F0u, MAGIC2)), xh(xv, i0 + 1), xh(xv, i0 + 5), b);
    a = fma2h(lop3_and_or(X << s2, mlo, lop3_and_or(c2, 0x000F000Fu, MAGIC2)), xh(xv, i0 + 2), xh(xv, i0 + 6), a);
    b = fma2h(lop3_and_or(X << s3, mhi, lop3_and_or(c2, 0x00F000F0u, MAGIC2)), xh(xv, i0 + 3), xh(xv, i0 + 7), b);
}
// 16 two-bit codes, weight 4b + k at bits 8b + 2k (weights i0 + ...). Bit class p = 2k.
__device__ __forceinline__ void crumb_word(uint32_t c, const uint32_t *xv, int i0, float &a, float &b) {
    const uint32_t c2 = c >> 8;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t m = (3u << (2 * k)) * 0x00010001u;
        a = fma2h(lop3_and_or(c, m, MAGIC2), xh(xv, i0 + k), xh(xv, i0 + 8 + k), a);
        b = fma2h(lop3_and_or(c2, m, MAGIC2), xh(xv, i0 + 4 + k), xh(xv, i0 + 12 + k), b);
    }
}
// Two 3-byte code groups (weights 8g..8g+7 and 8g+8..8g+15 of a unit, bytes b0 b1 b2 | b3 b4 b5) spread by three
// byte permutes: W0 = (b0 b1 | b3 b4), W1 = (b1 b2 | b4 b5), W2 = (b2 b2 | b5 b5). Code t of the first group then
// sits in the low half and code t of the second group in the high half, both at bit p = 3t mod 8 (t = 0..7 ->
// p = 0, 3, 6, 1, 4, 7, 2, 5), so one LOP3 per pair yields 1024 + u*2^p in both halves. xv word w0 + t holds the
// two matching staged activations.
__device__ __forceinline__ void tri_pair(uint32_t W0, uint32_t W1, uint32_t W2, const uint32_t *xv, int w0, float &acc) {
    acc = fma2h(lop3_and_or(W0, 0x00070007u, MAGIC2), lo16(xv[w0 + 0]), hi16(xv[w0 + 0]), acc);
    acc = fma2h(lop3_and_or(W0, 0x00380038u, MAGIC2), lo16(xv[w0 + 1]), hi16(xv[w0 + 1]), acc);
    acc = fma2h(lop3_and_or(W0, 0x01C001C0u, MAGIC2), lo16(xv[w0 + 2]), hi16(xv[w0 + 2]), acc);
    acc = fma2h(lop3_and_or(W1, 0x000E000Eu, MAGIC2), lo16(xv[w0 + 3]), hi16(xv[w0 + 3]), acc);
    acc = fma2h(lop3_and_or(W1, 0x00700070u, MAGIC2), lo16(xv[w0 + 4]), hi16(xv[w0 + 4]), acc);
    acc = fma2h(lop3_and_or(W1, 0x03800380u, MAGIC2), lo16(xv[w0 + 5]), hi16(xv[w0 + 5]), acc);
    acc = fma2h(lop3_and_or(W2, 0x001C001Cu, MAGIC2), lo16(xv[w0 + 6]), hi16(xv[w0 + 6]), acc);
    acc = fma2h(lop3_and_or(W2, 0x00E000E0u, MAGIC2), lo16(xv[w0 + 7]), hi16(xv[w0 + 7]), acc);
}

// 2^e for a small integer e, exactly (e is a compile-time constant where it is used).
__host__ __device__ constexpr float pow2f(int e) { return e >= 0 ? float(1u << e) : 1.0f / float(1u << (-e)); }

// Bit-class shift p of staging slot i (0..31) of a unit: the activation in that slot is staged as x * 2^(E - p),
// E being the vector's scale exponent. Slot i is half (i & 1) of staged word i >> 1. For every format but Q3S slot i
// holds element i; for Q3S word 8*pi + t holds elements 16*pi + t and 16*pi + 8 + t (see tri_pair).
template <int F>
__host__ __device__ constexpr int xshift(int i) {
    if constexpr (F == FMT_Q2S) return 2 * (i & 3);
    else if constexpr (F == FMT_Q3S) return (3 * ((i >> 1) & 7)) & 7;
    else return (i & 1) ? 4 : 0;
}
// Element (0..15, within a half-unit) staged in half h of word k (0..7) of that half-unit.
template <int F>
__host__ __device__ constexpr int slot_elem(int k, int h) {
    if constexpr (F == FMT_Q3S) return 8 * h + k;
    else return 2 * k + h;
}

// Activation constants per unit (XC<F>::n floats), from the staged x' (see the file comment).
template <int F> struct XC;
template <> struct XC<FMT_Q4G32> { static constexpr int n = 1; };   // C
template <> struct XC<FMT_Q2S> { static constexpr int n = 4; };     // C0, S0, C1, S1 (two sub-blocks)
template <> struct XC<FMT_Q3S> { static constexpr int n = 2; };     // C0, C1
template <> struct XC<FMT_Q5S> { static constexpr int n = 2; };     // C, S
template <> struct XC<FMT_Q6S> { static constexpr int n = 2; };     // C0, C1

template <int F>
__device__ __forceinline__ void unit_consts(const float xp[32], const float xt[32], float *out) {
    // xp = staged x' (as fp32), xt = 2^p * x' (the activation the integer code effectively multiplies)
    float sp[2] = {0.f, 0.f}, st[2] = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 32; ++i) { sp[i >> 4] += xp[i]; st[i >> 4] += xt[i]; }
    if constexpr (F == FMT_Q4G32) {
        out[0] = 1024.0f * (sp[0] + sp[1]) + 8.0f * (st[0] + st[1]);
    } else if constexpr (F == FMT_Q2S) {
        out[0] = 1024.0f * sp[0]; out[1] = st[0];
        out[2] = 1024.0f * sp[1]; out[3] = st[1];
    } else if constexpr (F == FMT_Q3S) {
        out[0] = 1024.0f * sp[0] + 4.0f * st[0];
        out[1] = 1024.0f * sp[1] + 4.0f * st[1];
    } else if constexpr (F == FMT_Q5S) {
        out[0] = 1024.0f * (sp[0] + sp[1]);
        out[1] = st[0] + st[1];
    } else {
        out[0] = 1024.0f * sp[0] + 32.0f * st[0];
        out[1] = 1024.0f * sp[1] + 32.0f * st[1];
    }
}

// ------------------------------------------------------------------------------------------------------------
// Per-lane geometry of one unit position (uc) within a 4096-weight chunk: byte offsets relative to the unit's
// aligned code base, so that both rows of a lane use immediate offsets.
// ------------------------------------------------------------------------------------------------------------
struct LaneGeo {
    uint32_t ubase;      // aligned byte offset of the unit's codes within a row chunk
    int32_t o1, o2, o3;  // format-specific byte offsets relative to ubase
    uint32_t sh0, sh1;   // format-specific shifts
    uint32_t p0, p1, p2, q0, q1, q2;   // Q3S byte-permute selectors of the two group pairs
};

template <int F>
__device__ __forceinline__ LaneGeo lane_geo(int uc) {
    LaneGeo g = {0u, 0, 0, 0, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    const uint32_t sbk = uint32_t(uc) >> 3, su = uint32_t(uc) & 7u;
    if constexpr (F == FMT_Q4G32) {
        g.ubase = 16u * uc;
    } else if constexpr (F == FMT_Q2S) {
        g.ubase = 84u * sbk + 8u * su;
        g.o1 = int32_t(64u + 2u * su) - int32_t(8u * su);     // L|M bytes of the two sub-blocks
        g.o2 = int32_t(80u) - int32_t(8u * su);               // d, dmin
    } else if constexpr (F == FMT_Q3S) {
        const uint32_t a = 110u * sbk + 12u * su;             // code start, 2-byte aligned
        const uint32_t o = a & 3u;                            // 0 or 2
        g.ubase = a - o;
        g.o1 = int32_t(4u + 2u * o);                          // word pair holding the second group pair's 6 bytes
        const uint32_t fa = 110u * sbk + 96u + 3u * (su >> 1);
        uint32_t fw = fa & ~3u, fs = 8u * (fa & 3u) + 6u * ((2u * su) & 3u);
        if (fs >= 32u) { fw += 4u; fs -= 32u; }
        g.o2 = int32_t(fw) - int32_t(g.ubase);                // word pair holding L_j0, L_j0+1 at bits fs..
        g.sh1 = fs;
        g.o3 = int32_t(110u * sbk + 108u) - int32_t(g.ubase); // d
        // the first group pair starts at byte o of (w0, w1), the second at byte 2 - o of its word pair
        const uint32_t s0 = o * 0x1111u, s1 = (2u - o) * 0x1111u;
        g.p0 = 0x4310u + s0; g.p1 = 0x5421u + s0; g.p2 = 0x5522u + s0;
        g.q0 = 0x4310u + s1; g.q1 = 0x5421u + s1; g.q2 = 0x5522u + s1;
    } else if constexpr (F == FMT_Q5S) {
        g.ubase = 176u * sbk + 16u * su;
        g.o1 = int32_t(128u + 4u * su) - int32_t(16u * su);   // high-bit plane word
        g.o2 = int32_t(160u) - int32_t(16u * su);             // 16 six-bit fields + d + dmin (16-byte aligned)
        g.sh0 = 6u * su;                                      // bit of L_su in the field run
        g.sh1 = 48u + 6u * su;                                // bit of M_su
    } else {
        const uint32_t a = 210u * sbk + 16u * su;
        g.ubase = a & ~3u;
        g.sh0 = (a & 3u) * 8u;
        g.o1 = int32_t(((210u * sbk + 128u + 8u * su) & ~3u)) - int32_t(g.ubase);   // high-2 plane (same alignment)
        g.o2 = int32_t(210u * sbk + 192u + 2u * su) - int32_t(g.ubase);            // two int8 sub-scales
        g.o3 = int32_t(210u * sbk + 208u) - int32_t(g.ubase);                      // d
    }
    return g;
}

// sum_i w'_i x_i over one 32-weight unit of one row; `u` = aligned unit base in shared memory, `sp` = this
// row's group-scale pointer (Q4G32), `c` = the unit's activation constants, `xv` = its staged activations.
// Each sub-block accumulator starts at -C (the activation constant), so no separate subtraction is needed.
template <int F>
__device__ __forceinline__ float row_dot(const uint8_t *u, const float *sp, const LaneGeo &g, const float *c,
                                         const uint32_t *xv) {
    if constexpr (F == FMT_Q4G32) {
        const uint4 w = *reinterpret_cast<const uint4 *>(u);
        float a = -c[0], b = 0.f;
        nib_word(w.x, xv, 0, a, b);
        nib_word(w.y, xv, 8, a, b);
        nib_word(w.z, xv, 16, a, b);
        nib_word(w.w, xv, 24, a, b);
        return sp[0] * (a + b);
    } else if constexpr (F == FMT_Q2S) {
        const uint32_t w0 = lds32(u), w1 = lds32(u + 4);
        const uint32_t dd = lds32(u + g.o2);
        const float2 Dd = __half22float2(*reinterpret_cast<const __half2 *>(&dd));
        const uint32_t lm = *reinterpret_cast<const uint16_t *>(u + g.o1);
        const float L0 = small_int_f(lop3_and_or(lm, 0xFu, MAGICF));
        const float M0 = small_int_f(lop3_and_or(lm >> 4, 0xFu, MAGICF));
        const float L1 = small_int_f(lop3_and_or(lm >> 8, 0xFu, MAGICF));
        const float M1 = small_int_f(lop3_and_or(lm >> 12, 0xFu, MAGICF));
        float a0 = -c[0], b0 = 0.f, a1 = -c[2], b1 = 0.f;
        crumb_word(w0, xv, 0, a0, b0);
        crumb_word(w1, xv, 16, a1, b1);
        float r = (Dd.x * L0) * (a0 + b0);
        r = fmaf(Dd.x * L1, a1 + b1, r);
        r = fmaf(-(Dd.y * M0), c[1], r);
        return fmaf(-(Dd.y * M1), c[3], r);
    } else if constexpr (F == FMT_Q3S) {
        const uint32_t *wp = reinterpret_cast<const uint32_t *>(u);
        const uint32_t w0 = wp[0], w1 = wp[1];
        const uint32_t *qp = reinterpret_cast<const uint32_t *>(u + g.o1);
        const uint32_t w2 = qp[0], w3 = qp[1];
        const uint32_t *fp = reinterpret_cast<const uint32_t *>(u + g.o2);
        const uint32_t f = __funnelshift_r(fp[0], fp[1], g.sh1);
        const float L0 = small_int_f(lop3_and_or(f, 63u, MAGICF));
        const float L1 = small_int_f(lop3_and_or(f >> 6, 63u, MAGICF));
        const float D = hbits(u + g.o3);
        float a0 = -c[0], a1 = -c[1];
        tri_pair(__byte_perm(w0, w1, g.p0), __byte_perm(w0, w1, g.p1), __byte_perm(w0, w1, g.p2), xv, 0, a0);
        tri_pair(__byte_perm(w2, w3, g.q0), __byte_perm(w2, w3, g.q1), __byte_perm(w2, w3, g.q2), xv, 8, a1);
        return fmaf(D * L1, a1, (D * L0) * a0);
    } else if constexpr (F == FMT_Q5S) {
        const uint4 w = *reinterpret_cast<const uint4 *>(u);
        const uint32_t H = lds32(u + g.o1);
        const uint4 fld = *reinterpret_cast<const uint4 *>(u + g.o2);
        const float2 Dd = __half22float2(*reinterpret_cast<const __half2 *>(&fld.w));
        const uint64_t lo64 = (uint64_t(fld.y) << 32) | fld.x, hi64 = (uint64_t(fld.z) << 32) | fld.y;
        const float L = small_int_f(lop3_and_or(uint32_t(lo64 >> g.sh0), 63u, MAGICF));
        const float M = small_int_f(lop3_and_or(uint32_t(hi64 >> (g.sh1 - 32u)), 63u, MAGICF));
        float a = -c[0], b = 0.f;
        nib_word_hi<1>(w.x, lop3_sel(H, H << 12, 0x0000FFFFu), xv, 0, a, b);
        nib_word_hi<1>(w.y, lop3_sel(H >> 8, H << 4, 0x0000FFFFu), xv, 8, a, b);
        nib_word_hi<1>(w.z, lop3_sel(H >> 16, H >> 4, 0x0000FFFFu), xv, 16, a, b);
        nib_word_hi<1>(w.w, lop3_sel(H >> 24, H >> 12, 0x0000FFFFu), xv, 24, a, b);
        return fmaf(Dd.x * L, a + b, -(Dd.y * M) * c[1]);
    } else {
        const uint32_t sh = g.sh0;
        const uint32_t *wp = reinterpret_cast<const uint32_t *>(u);
        const uint32_t r0 = wp[0], r1 = wp[1], r2 = wp[2], r3 = wp[3], r4 = wp[4];
        const uint32_t *hp = reinterpret_cast<const uint32_t *>(u + g.o1);
        const uint32_t q0 = hp[0], q1 = hp[1], q2 = hp[2];
        const uint32_t h0 = __funnelshift_r(q0, q1, sh), h1 = __funnelshift_r(q1, q2, sh);
        const uint32_t lv = *reinterpret_cast<const uint16_t *>(u + g.o2);
        // int8 -> float exactly: (b ^ 0x80) | 2^23 as fp32, minus 2^23 + 128
        const float L0 = __uint_as_float((lv & 0xFFu) ^ (MAGICF | 0x80u)) - 8388736.0f;
        const float L1 = __uint_as_float(((lv >> 8) & 0xFFu) ^ (MAGICF | 0x80u)) - 8388736.0f;
        const float D = hbits(u + g.o3);
        float a0 = -c[0], b0 = 0.f, a1 = -c[1], b1 = 0.f;
        nib_word_hi<2>(__funnelshift_r(r0, r1, sh), __byte_perm(h0, 0u, 0x4140u), xv, 0, a0, b0);
        nib_word_hi<2>(__funnelshift_r(r1, r2, sh), __byte_perm(h0, 0u, 0x4342u), xv, 8, a0, b0);
        nib_word_hi<2>(__funnelshift_r(r2, r3, sh), __byte_perm(h1, 0u, 0x4140u), xv, 16, a1, b1);
        nib_word_hi<2>(__funnelshift_r(r3, r4, sh), __byte_perm(h1, 0u, 0x4342u), xv, 24, a1, b1);
        return fmaf(D * L1, a1 + b1, (D * L0) * (a0 + b0));
    }
}

// Staged activations: within each 4096-weight chunk c, the 16 words of unit uc are four 16-byte vectors at vector
// index (c * 4 + t) * 128 + uc (t = 0..3), so consecutive lanes (consecutive units) read consecutive 16-byte vectors
// and the four loads of a unit sit at constant 2 KB offsets. Half-unit hh (elements 16 hh .. 16 hh + 15) is words
// 8 hh .. 8 hh + 7, i.e. vectors t = 2 hh and 2 hh + 1.
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }   // -126 <= e <= 127

// Stage one half-unit: xr = its 16 raw fp16 activations in element order, E = the vector's scale exponent.
template <int F>
__device__ __forceinline__ void stage_half_unit(const uint16_t *xr, int E, uint32_t w[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float f0 = h2f_bits(xr[slot_elem<F>(k, 0)]) * exp2i(E - xshift<F>(2 * k));
        const float f1 = h2f_bits(xr[slot_elem<F>(k, 1)]) * exp2i(E - xshift<F>(2 * k + 1));
        w[k] = uint32_t(f2h_bits(f0)) | (uint32_t(f2h_bits(f1)) << 16);
    }
}
__device__ __forceinline__ void load_xp(const uint16_t *xs, uint32_t c, uint32_t uc, uint32_t xv[16]) {
    const uint4 *p = reinterpret_cast<const uint4 *>(xs) + c * 512u + uc;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint4 v = p[t * 128];
        xv[4 * t] = v.x; xv[4 * t + 1] = v.y; xv[4 * t + 2] = v.z; xv[4 * t + 3] = v.w;
    }
}

}  // namespace

// ------------------------------------------------------------------------------------------------------------
// Batch-1 fused dequant-GEMV kernel: NG consumer groups of 8 warps + 1 producer warp (TR lanes per group).
// ------------------------------------------------------------------------------------------------------------
constexpr int G1_NG = 3;     // consumer groups
template <int F, int NS, int NG, int TR>
struct G1Layout {
    static constexpr int CW = 8 * NG;                  // consumer warps
    static constexpr int THREADS = (CW + 1) * 32;
    static constexpr int NSLOT = NS + 2;               // per-tile reduction slots (tiles in flight <= NS + 1)
    static constexpr int RPL = TR / 2;                 // rows per lane (rows rlo, rlo + 2, ...)
    static constexpr int RED_PER_SLOT = NG * 8 * RPL;  // one partial per (group, warp, lane row)
    static constexpr int STAGE = TR * (Geo<F>::chunk_bytes + Geo<F>::scale_bytes);
    static __host__ __device__ uint32_t bar_bytes() { return uint32_t(round_up(16 * NS, 128)); }
    static __host__ __device__ uint32_t red_bytes() {
        return uint32_t(round_up(16 + NSLOT * 4 + NSLOT * RED_PER_SLOT * 4, 128));
    }
    static __host__ __device__ uint32_t x_bytes(uint32_t K) { return uint32_t(round_up(int64_t((K + CHW - 1) / CHW) * CHW * 2, 128)); }
    static __host__ __device__ uint32_t c_bytes(uint32_t K) { return uint32_t(round_up(4 * int64_t(K / 32) * XC<F>::n, 128)); }
    // + 32: the Q3S unpack reads the word pair holding a unit's scale fields, up to 4 bytes past its row chunk
    static __host__ __device__ uint32_t total(uint32_t K) {
        return bar_bytes() + red_bytes() + x_bytes(K) + c_bytes(K) + uint32_t(NS) * STAGE + 32;
    }
};

// Sum R per-lane values over the warp, one value per row: after the call, lanes j * (32 / R) (j < R) hold the warp
// sum of v[j]. log2(R) transposing exchanges, then a butterfly inside each group of 32 / R lanes.
template <int R>
__device__ __forceinline__ float warp_rows_sum(float (&v)[R], int lane) {
    int off = 16;
#pragma unroll
    for (int n = R; n > 1; n >>= 1, off >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int k = 0; k < n / 2; ++k) {
            const float keep = up ? v[k + n / 2] : v[k];
            const float send = up ? v[k] : v[k + n / 2];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float r = v[0];
#pragma unroll
    for (int o = off; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

template <int F, int NS, int NG, int TR, bool FULLK>
__global__ void __launch_bounds__(G1Layout<F, NS, NG, TR>::THREADS, 1) gemv1_kernel(GemvArgs a) {
    using G = Geo<F>;
    using LY = G1Layout<F, NS, NG, TR>;
    constexpr int NSLOT = LY::NSLOT;
    constexpr int CW = LY::CW;
    constexpr int RPL = LY::RPL;
    constexpr uint32_t STAGE = uint32_t(LY::STAGE);
    constexpr uint32_t NSG = uint32_t(NS / NG);       // stages per consumer group
    static_assert(NS % NG == 0, "each consumer group owns NS / NG stages");
    static_assert(NG * TR <= 32, "producer lanes: TR per group");
    static_assert(RPL >= 1 && (RPL & (RPL - 1)) == 0 && RPL <= 8, "rows per lane: a power of two");
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t N = uint32_t(a.N), K = uint32_t(a.K);
    // this CTA's rows: a contiguous range, the row counts of any two CTAs differ by at most one
    const uint32_t rq = N / gridDim.x, rm = N % gridDim.x, b = blockIdx.x;
    const uint32_t rbeg = b * rq + min(b, rm), rend = rbeg + rq + (b < rm ? 1u : 0u);
    const uint32_t ntl = (rend - rbeg + TR - 1) / TR;  // row tiles of this CTA (the last one may be ragged)
    const uint32_t nch = (K + CHW - 1) / CHW;
    const uint32_t U = K / 32;                        // units per row

    uint8_t *p = smem_raw;
    uint64_t *full = reinterpret_cast<uint64_t *>(p);
    uint64_t *empty = full + NS;
    p += LY::bar_bytes();
    int *misc = reinterpret_cast<int *>(p);           // [0]: max |x| as float bits
    int *cnt = misc + 4;
    float *red = reinterpret_cast<float *>(p + 16 + NSLOT * 4);
    p += LY::red_bytes();
    uint16_t *xs = reinterpret_cast<uint16_t *>(p);
    p += LY::x_bytes(K);
    float *cst = reinterpret_cast<float *>(p);
    p += LY::c_bytes(K);
    uint8_t *stages = p;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 8); }
        for (int s = 0; s < NSLOT; ++s) cnt[s] = 0;
        misc[0] = 0;
        fence_mbar_init();
    }
    pdl_launch_dependents();     // the next product may begin launching; it still waits for us before reading
    __syncthreads();

    if (warp == CW) {
        // ------------------------------------ producer ------------------------------------
        // Item i of this CTA is (local tile i / nch, chunk i mod nch); group g consumes items g, g + NG, ... from
        // its private sub-ring of stages [g*NSG, (g+1)*NSG), so every mbarrier is waited on only by the one group
        // that consumed its previous phase (a parity wait is only meaningful one phase ahead). Producer lanes
        // g*TR .. g*TR+TR-1 serve group g: lane r copies row r of the tile (bulk copies issued by one thread are
        // processed one after another, so rows go out from different lanes), or lane 0 copies the whole tile when
        // its rows are contiguous. The lanes advance in rounds (round k = every group's k-th item), and a round
        // starts only once every group has released the stage it reuses, so no group runs more than NSG rounds
        // ahead of another: the per-tile reduction slots, reused every NSLOT = NS + 2 tiles, depend on that bound.
        constexpr uint32_t PMASK = (NG * TR >= 32) ? 0xffffffffu : ((1u << (NG * TR)) - 1u);
        const int pg = lane / TR, pr = lane % TR;
        if (pg < NG) {
            // Packed weights are read before the previous grid has finished only when the caller opted in
            // (QPACK_OPT_WEIGHT_PREFETCH: weights are not written by the kernel just before this one).
            if (!a.weight_prefetch) pdl_wait();
            const uint64_t pol = l2_evict_first_policy();
            const bool whole_rows = (K == uint32_t(CHW));        // a tile of whole rows is one contiguous range
            uint32_t k = 0, issued = 0, c = uint32_t(pg), lt = 0;
            while (c >= nch) { c -= nch; ++lt; }
            while (true) {
                const bool have = lt < ntl;
                if (!__any_sync(PMASK, have)) break;
                const uint32_t s = uint32_t(pg) * NSG + k % NSG, ph = (k / NSG) & 1u;
                bool bad = false;
                if (have && pr == 0 && k >= NSG && !mbar_wait_bounded(&empty[s], ph ^ 1u)) {
                    // A consumer stopped releasing stages: record it and stop producing; consumers then give up
                    // on their next bounded wait, so nothing is left waiting.
                    atomicOr(&g_fault_gemv, FAULT_WAIT_EMPTY);
                    bad = true;
                }
                if (__any_sync(PMASK, bad)) break;
                const uint32_t r0 = rbeg + lt * TR;
                const uint32_t rows = have ? min(uint32_t(TR), rend - r0) : 0u;
                const uint32_t koff = c * CHW;
                uint32_t cbytes, sbytes = 0;
                if constexpr (Fmt<F>::sb) {
                    const uint32_t off = (koff / 256) * Fmt<F>::bytes;
                    cbytes = min(uint32_t(G::chunk_bytes), uint32_t(a.row_stride) - off);
                } else {
                    cbytes = min(uint32_t(G::chunk_bytes), (K - koff) / 2);
                    sbytes = min(uint32_t(G::scale_bytes), (uint32_t(a.scale_stride) - koff / 32) * 4);
                }
                uint8_t *st = stages + s * STAGE;
                if (have && pr == 0) mbar_arrive_expect_tx(&full[s], rows * (cbytes + sbytes));
                __syncwarp(PMASK);                               // expect_tx before any of this item's copies
                if (have) {
                    const uint8_t *src0 =
                        a.packed + int64_t(r0) * a.row_stride + (Fmt<F>::sb ? (koff / 256) * Fmt<F>::bytes : koff / 2);
                    const uint8_t *ssrc0 =
                        Fmt<F>::sb ? nullptr : reinterpret_cast<const uint8_t *>(a.gscale + int64_t(r0) * a.scale_stride + koff / 32);
                    if (whole_rows) {
                        if (pr == 0) bulk_g2s(st, src0, rows * cbytes, &full[s], pol);
                        if constexpr (!Fmt<F>::sb) {
                            if (pr == 1 % TR) bulk_g2s(st + TR * G::chunk_bytes, ssrc0, rows * sbytes, &full[s], pol);
                        }
                    } else if (uint32_t(pr) < rows) {
                        bulk_g2s(st + pr * G::chunk_bytes, src0 + int64_t(pr) * a.row_stride, cbytes, &full[s], pol);
                        if constexpr (!Fmt<F>::sb)
                            bulk_g2s(st + TR * G::chunk_bytes + pr * G::scale_bytes,
                                     ssrc0 + int64_t(pr) * a.scale_stride * 4, sbytes, &full[s], pol);
                    }
                    ++issued;
                }
                ++k;
                c += NG;
                while (c >= nch) { c -= nch; ++lt; }
            }
            // Drain: wait (bounded) until the last fill of each of the group's stages has landed, so the CTA never
            // exits with bulk copies still writing its shared memory (consumers that gave up may exit early).
            if (pr == 0) {
                for (uint32_t j = (issued > NSG ? issued - NSG : 0u); j < issued; ++j) {
                    if (!mbar_wait_bounded(&full[uint32_t(pg) * NSG + j % NSG], (j / NSG) & 1u)) {
                        atomicOr(&g_fault_gemv, FAULT_WAIT_FULL);
                        break;
                    }
                }
            }
        }
        return;
    }

    // -------------------------------------- consumers --------------------------------------
    pdl_wait();                  // x (and y) may belong to the previous grid
    int E;                       // scale exponent: activations are staged as x * 2^E, with max |x| * 2^E in [2^14, 2^15)
    {
        const uint4 *xg = reinterpret_cast<const uint4 *>(a.X);
        // pass 1: max |x| over the whole vector (fp16 magnitudes order like their bit patterns)
        uint32_t m = 0;
        for (uint32_t v = tid; v < K / 8; v += CW * 32) {
            const uint4 raw = __ldg(xg + v);
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) m = max(m, max(w[e] & 0x7FFFu, (w[e] >> 16) & 0x7FFFu));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) atomicMax(misc, int(m));
        named_bar_sync(1, CW * 32);
        const float xm = h2f_bits(uint16_t(min(uint32_t(misc[0]), 0x7BFFu)));   // inf / nan inputs: clamp the exponent
        E = (xm > 0.f) ? 14 - (int((__float_as_uint(xm) >> 23) & 255u) - 127) : 0;
        // pass 2: stage x' = fp16(x * 2^(E - p)) half-unit by half-unit (16 activations, 8 words, 2 vectors)
        uint4 *xd = reinterpret_cast<uint4 *>(xs);
        for (uint32_t h = tid; h < K / 16; h += CW * 32) {
            const uint4 r0 = __ldg(xg + 2 * h), r1 = __ldg(xg + 2 * h + 1);
            const uint32_t rw[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
            uint16_t xr[16];
#pragma unroll
            for (int e = 0; e < 8; ++e) { xr[2 * e] = lo16(rw[e]); xr[2 * e + 1] = hi16(rw[e]); }
            uint32_t w[8];
            stage_half_unit<F>(xr, E, w);
            const uint32_t u = h >> 1, hh = h & 1u, cc = u >> 7, uu = u & 127u;
            xd[(cc * 4 + 2 * hh) * 128 + uu] = make_uint4(w[0], w[1], w[2], w[3]);
            xd[(cc * 4 + 2 * hh + 1) * 128 + uu] = make_uint4(w[4], w[5], w[6], w[7]);
        }
        named_bar_sync(1, CW * 32);
        for (uint32_t u = tid; u < U; u += CW * 32) {
            uint32_t xv[16];
            load_xp(xs, u >> 7, u & 127u, xv);
            float xp[32], xt[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                xp[i] = h2f_bits(xh(xv, i));
                xt[i] = xp[i] * pow2f(xshift<F>(i));
            }
            unit_consts<F>(xp, xt, cst + u * XC<F>::n);
        }
        named_bar_sync(1, CW * 32);
    }
    const float unscale = exp2i(-E);
    const uint32_t group = uint32_t(warp) >> 3, wg = uint32_t(warp) & 7u;
    const uint32_t gl = wg * 32u + uint32_t(lane);
    const int uc = int(gl & 127u);
    const uint32_t rlo = gl >> 7;                      // rows rlo, rlo + 2, ..., rlo + TR - 2 of the tile
    const LaneGeo geo = lane_geo<F>(uc);
    const uint32_t uoff0 = rlo * uint32_t(G::chunk_bytes) + geo.ubase;
    const uint32_t soff0 = TR * uint32_t(G::chunk_bytes) + rlo * uint32_t(G::scale_bytes) + 4u * uint32_t(uc);

    // own items: the group's k-th item is item group + NG*k, in stage group*NSG + k mod NSG
    uint32_t sl = 0, ph = 0;
    uint32_t lt = 0, c = group, ib = 0, slot = 0;      // ib = item index of the tile's first chunk
    while (c >= nch && lt < ntl) { c -= nch; ++lt; ib += nch; if (++slot == uint32_t(NSLOT)) slot = 0; }
    bool dead = false;
    float acc[RPL];
#pragma unroll
    for (int j = 0; j < RPL; ++j) acc[j] = 0.f;
    while (lt < ntl) {
        const uint32_t r0 = rbeg + lt * TR;
        const uint32_t s = group * NSG + sl;
        if (!dead && !mbar_wait_bounded(&full[s], ph)) {
            if (lane == 0) atomicOr(&g_fault_gemv, FAULT_WAIT_FULL);
            dead = true;
        }
        {
            const uint8_t *st = stages + s * STAGE;
            uint32_t ucv = uint32_t(uc);
            bool use = !dead;
            if constexpr (!FULLK) {
                const uint32_t units = min(uint32_t(UPC), (K - c * CHW) / 32);
                use = use && (uint32_t(uc) < units);
                ucv = min(ucv, units - 1);                 // stay on this item's data
            }
            uint32_t xv[16];
            load_xp(xs, c, ucv, xv);
            float cv[XC<F>::n];
            const float *cp = cst + (c * UPC + ucv) * XC<F>::n;
#pragma unroll
            for (int q = 0; q < XC<F>::n; ++q) cv[q] = cp[q];
            const uint8_t *u0 = st + uoff0;
            const float *sp0 = reinterpret_cast<const float *>(st + soff0);
#pragma unroll
            for (int j = 0; j < RPL; ++j) {
                const float d = row_dot<F>(u0 + 2 * j * G::chunk_bytes, sp0 + 2 * j * (G::scale_bytes / 4), geo, cv, xv);
                acc[j] += use ? d : 0.f;
            }
        }
        if (c + NG >= nch) {
            // this group's last item of the tile: one value per (warp, row) into the tile's slot, then a counter;
            // the warp completing the count sums the tile's partials in a fixed order and writes y.
            const float v = warp_rows_sum<RPL>(acc, lane);
            float *rs = red + slot * LY::RED_PER_SLOT + (group * 8 + wg) * RPL;
            if ((lane & (32 / RPL - 1)) == 0) rs[lane / (32 / RPL)] = v;
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                __threadfence_block();
                const int expected = 8 * int(min(uint32_t(NG), nch));
                last = (atomicAdd(&cnt[slot], 1) == expected - 1);
                if (last) __threadfence_block();
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                // lane r < TR: tile row r = 2 j + rl, summed over the four warps holding rows of parity rl in every
                // contributing group
                if (lane < TR) {
                    const int rl = lane & 1, j = lane >> 1;
                    const float *sb = red + slot * LY::RED_PER_SLOT;
                    float yv = 0.f;
#pragma unroll
                    for (int gr = 0; gr < NG; ++gr) {
                        bool contributed = nch >= uint32_t(NG);
                        if (!contributed) {
                            for (uint32_t cc = 0; cc < nch; ++cc) contributed |= ((ib + cc) % NG) == uint32_t(gr);
                        }
                        if (contributed) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) yv += sb[(gr * 8 + 4 * rl + q) * RPL + j];
                        }
                    }
                    if (r0 + uint32_t(lane) < rend) a.Y[r0 + lane] = yv * unscale;
                }
                __syncwarp();
                if (lane == 0) cnt[slot] = 0;
            }
#pragma unroll
            for (int j = 0; j < RPL; ++j) acc[j] = 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++sl == NSG) { sl = 0; ph ^= 1u; }
        c += NG;
        while (c >= nch) {
            c -= nch;
            ++lt;
            ib += nch;
            if (++slot == uint32_t(NSLOT)) slot = 0;
        }
    }
}

template <int F, int NS, int NG, int TR, bool FULLK>
static cudaError_t try_launch_gemv1(const GemvArgs &a, cudaStream_t st, bool *launched) {
    using LY = G1Layout<F, NS, NG, TR>;
    *launched = false;
    const uint32_t smem = LY::total(uint32_t(a.K));
    if (smem > 227u * 1024u) return cudaSuccess;
    static int opted[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!opted[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemv1_kernel<F, NS, NG, TR, FULLK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             227 * 1024);
        if (e != cudaSuccess) return e;
        opted[dev] = 1;
    }
    int grid = num_sms();
    if (a.N < grid) grid = int(a.N);                   // every CTA gets at least one row
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(unsigned(LY::THREADS));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = a.weight_prefetch ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    *launched = true;
    return cudaLaunchKernelEx(&cfg, gemv1_kernel<F, NS, NG, TR, FULLK>, a);
}

// Largest ring (a multiple of G1_NG stages, so every group owns the same number) that fits beside the staged
// activations; about 200 KB of stages keeps far more bytes in flight per SM than the memory latency needs.
template <int F, int TR, bool FULLK>
static cudaError_t launch_gemv1_k(const GemvArgs &a, cudaStream_t st) {
    bool done = false;
    cudaError_t e;
    constexpr int SB = G1Layout<F, 3, G1_NG, TR>::STAGE;
    if constexpr (SB * 15 <= 200 * 1024) {
        e = try_launch_gemv1<F, 15, G1_NG, TR, FULLK>(a, st, &done);
        if (e != cudaSuccess || done) return e;
    }
    if constexpr (SB * 12 <= 200 * 1024) {
        e = try_launch_gemv1<F, 12, G1_NG, TR, FULLK>(a, st, &done);
        if (e != cudaSuccess || done) return e;
    }
    e = try_launch_gemv1<F, 9, G1_NG, TR, FULLK>(a, st, &done);
    if (e != cudaSuccess || done) return e;
    e = try_launch_gemv1<F, 6, G1_NG, TR, FULLK>(a, st, &done);
    if (e != cudaSuccess || done) return e;
    e = try_launch_gemv1<F, 3, G1_NG, TR, FULLK>(a, st, &done);
    if (e != cudaSuccess || done) return e;
    return cudaErrorInvalidValue;
}

#ifndef QPACK_G1_TR
#define QPACK_G1_TR 8
#endif
template <int F>
static cudaError_t launch_gemv1(const GemvArgs &a, cudaStream_t st) {
    if (a.K % CHW == 0) return launch_gemv1_k<F, QPACK_G1_TR, true>(a, st);
    return launch_gemv1_k<F, QPACK_G1_TR, false>(a, st);
}

namespace {
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


}  // namespace

// ------------------------------------------------------------------------------------------------------------
// Small-batch kernel (M = 2..16): 8 consumer warps, warp pair p owns row p of the 4-row tile; each lane
// dequantizes two 32-weight units exactly and multiplies them against the M activation rows (read through L1).
// ------------------------------------------------------------------------------------------------------------
constexpr int NCW = 8;
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr int SMEM_BUDGET = 220 * 1024;

template <int F, int MT>
__global__ void __launch_bounds__(NTHREADS, 1) stream_kernel(GemvArgs a, int NS) {
    using G = Geo<F>;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t N = a.N, K = a.K;
    const int64_t ntiles = (N + TILE_R - 1) / TILE_R;
    const int nchunks = int((K + CHW - 1) / CHW);

    uint8_t *p = smem_raw;
    uint64_t *full = reinterpret_cast<uint64_t *>(p);
    uint64_t *empty = full + NS;
    p += round_up(16 * NS, 128);
    float *red = reinterpret_cast<float *>(p);
    p += round_up(2 * NCW * MT * 4, 128);
    uint8_t *stages = p;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], NCW); }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NCW) {
        const uint64_t pol = l2_evict_first_policy();
        int it = 0;
        bool bad = false;
        for (int64_t tile = blockIdx.x; tile < ntiles && !bad; tile += gridDim.x) {
            const int64_t r0 = tile * TILE_R;
            const int rows = int(N - r0 < TILE_R ? N - r0 : TILE_R);
            for (int c = 0; c < nchunks; ++c) {
                const int s = it % NS;
                const uint32_t ph = uint32_t(it / NS) & 1u;
                if (it >= NS) {
                    bool ok = true;
                    if (lane == 0) ok = mbar_wait_bounded(&empty[s], ph ^ 1u);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) { if (lane == 0) atomicOr(&g_fault_gemv, FAULT_WAIT_EMPTY); bad = true; break; }
                }
                int64_t cbytes, sbytes = 0;
                const int64_t koff = int64_t(c) * CHW;
                if constexpr (Fmt<F>::sb) {
                    const int64_t off = (koff / 256) * Fmt<F>::bytes;
                    cbytes = a.row_stride - off < G::chunk_bytes ? a.row_stride - off : G::chunk_bytes;
                } else {
                    cbytes = (K - koff) / 2 < G::chunk_bytes ? (K - koff) / 2 : G::chunk_bytes;
                    const int64_t sb = (a.scale_stride - koff / 32) * 4;
                    sbytes = sb < G::scale_bytes ? sb : G::scale_bytes;
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
        // Drain: wait (bounded) for the last fill of each stage, so the CTA never exits with bulk copies in flight.
        if (lane == 0) {
            for (int j = (it > NS ? it - NS : 0); j < it; ++j) {
                if (!mbar_wait_bounded(&full[j % NS], uint32_t(j / NS) & 1u)) {
                    atomicOr(&g_fault_gemv, FAULT_WAIT_FULL);
                    break;
                }
            }
        }
        return;
    }

    const int pair = warp >> 1, half = warp & 1;    // warp pair `pair` owns row `pair` of the tile
    int it = 0, tcount = 0;
    bool dead = false;
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
            const int units = int((K - koff) / 32 < UPC ? (K - koff) / 32 : UPC);
            const uint8_t *st = stages + int64_t(s) * G::stage_bytes;
            const uint8_t *row = st + pair * G::chunk_bytes;
            const float *scl = reinterpret_cast<const float *>(st + TILE_R * G::chunk_bytes + pair * G::scale_bytes);
            if (row_ok && !dead) {
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    const int uc = 64 * half + 32 * v + lane;
                    if (uc < units) {
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
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            ++it;
        }
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
    const int64_t extra = round_up(2 * NCW * MT * 4, 128);
    int NS = 0;
    int64_t tot = 0;
    for (int ns = 16; ns >= 2; --ns) {
        tot = round_up(16 * ns, 128) + extra + int64_t(ns) * G::stage_bytes + 32;
        if (tot <= SMEM_BUDGET) { NS = ns; break; }
    }
    if (NS == 0) return cudaErrorInvalidValue;
    static int opted[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!opted[dev]) {
        cudaError_t e = cudaFuncSetAttribute(stream_kernel<F, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BUDGET);
        if (e != cudaSuccess) return e;
        opted[dev] = 1;
    }
    const int64_t ntiles = (a.N + TILE_R - 1) / TILE_R;
    int grid = num_sms();
    if (ntiles < grid) grid = int(ntiles);
    if (grid < 1) return cudaSuccess;
    stream_kernel<F, MT><<<grid, NTHREADS, size_t(tot), s>>>(a, NS);
    return cudaGetLastError();
}

template <int F>
static cudaError_t launch_fmt(const GemvArgs &a, cudaStream_t s) {
    if (a.M <= 1) return launch_gemv1<F>(a, s);
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
