// qpack_gemv.cu — fused dequant-GEMV (batch 1) and small-batch GEMM (M <= 16) over packed low-bit weights.
//
// The decode-phase product is a pure stream over the packed weights: every weight byte is read from HBM once
// (2/3/5/6-bit article, lpnh.cn/news/2857666, §1.2: time per token = weight bytes / bandwidth; DBHOO-CIM
// article, pwwt.cn/news/4452170, §3.3: dequantization must stay fused, never materialised).
//
// Batch-1 kernel (gemv1_kernel<F, 1>), one persistent CTA per SM:
//   warp 16      producer: 2-D TMA tensor copies of (row tile x K chunk) boxes of the packed rows into a ring of
//                shared-memory stages (completion on mbarriers, L2 evict-first because each byte is used once).
//   warps 0..15  consumers: row class x K part of every stage; lane l owns one 32-weight unit of each chunk.
// Unpacking (2/3/5/6-bit article §3.3: separate unpack from multiply-add, factor s*(q.x) + m*sum(x)): codes are
// OR-ed into the mantissa of an fp16 1024.0 with one LOP3 per pair of weights, so a half holds 1024 + u*2^p
// exactly, p being the code's bit position inside its 16-bit half. The activations are staged in shared memory
// pre-scaled by 2^-p of the code they meet (x' = fp16(x * 2^-p), exact unless subnormal), so one fp32 FMA with
// fp16 inputs (exact product) per weight accumulates 1024*x' + u*x for every class into one accumulator. The
// 1024*sum(x') terms, the symmetric code offsets and the asymmetric minima are removed per sub-block with
// activation sums that each CTA precomputes once. Per row, each warp reduces its lanes' sums with shuffles and
// stores one partial per K part in shared memory; the partials are scaled back by each part's power of two and
// summed in a fixed order (deterministic) before y is written.
//
// Small batches (M = 2..16) use the same kernel with MT activation rows: each unit-row is unpacked once and
// multiplied against every staged activation row; rows beyond what shared memory holds go in further launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "qpack_dev.cuh"
#include "qpack_launch.h"

namespace qpack {

__device__ int g_fault_gemv = 0;

namespace {

constexpr uint32_t MAGIC2 = 0x64006400u; // fp16 1024.0 in both halves
constexpr uint32_t MAGICF = 0x4B000000u; // fp32 2^23

__device__ __forceinline__ uint16_t lo16(uint32_t v) { return uint16_t(v & 0xFFFFu); }
__device__ __forceinline__ uint16_t hi16(uint32_t v) { return uint16_t(v >> 16); }
__device__ __forceinline__ uint32_t lds32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ float small_int_f(uint32_t bits_or_magic) { return __uint_as_float(bits_or_magic) - 8388608.0f; }

// acc += lo(codes) * xa + hi(codes) * xb with exact products (fp16 x fp16 -> fp32 FMA).
__device__ __forceinline__ float fma2h(uint32_t codes, uint16_t xa, uint16_t xb, float acc) {
    acc = fma_h(lo16(codes), xa, acc);
    return fma_h(hi16(codes), xb, acc);
}
// x halves of a unit: xv[t] holds x'[2t], x'[2t+1].
__device__ __forceinline__ uint16_t xh(const uint32_t *xv, int i) { return (i & 1) ? hi16(xv[i >> 1]) : lo16(xv[i >> 1]); }

// Two-way integer dot products: c + a.h0 * b.byte(k) + a.h1 * b.byte(k + 1), a = two signed 16-bit values, b = four
// unsigned bytes, k = 0 (lo) or 2 (hi). Exact in int32.
__device__ __forceinline__ int32_t dp2a_lo(uint32_t a, uint32_t b, int32_t c) {
    int32_t d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int32_t dp2a_hi(uint32_t a, uint32_t b, int32_t c) {
    int32_t d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// One Q4G32 code word (weights 8j..8j+7, weight 8j+2b in the low nibble of byte b, 8j+2b+1 in the high nibble) against
// the unit's 16-bit activations A[0..3] = (x0, x2), (x4, x6), (x1, x3), (x5, x7) of those weights: the low nibbles
// add u * x to lo, the high nibbles, masked in place, add 16 u * x to hi.
__device__ __forceinline__ void nib_dp(uint32_t c, const uint32_t *A, int32_t &lo, int32_t &hi) {
    const uint32_t l = c & 0x0F0F0F0Fu, h = c & 0xF0F0F0F0u;
    lo = dp2a_lo(A[0], l, lo);
    lo = dp2a_hi(A[1], l, lo);
    hi = dp2a_lo(A[2], h, hi);
    hi = dp2a_hi(A[3], h, hi);
}

// ------------------------------------------------------------------------------------------------------------
// Unpack + multiply helpers. Two accumulators (a, b) only for instruction-level parallelism.
// ------------------------------------------------------------------------------------------------------------
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
template <> struct XC<FMT_Q4G32> { static constexpr int n = 2; };   // C (int bits), 2^-(E+4)
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
    static_assert(F != FMT_Q4G32, "Q4G32 activations are staged as 16-bit integers (stage_unit_i16)");
    if constexpr (F == FMT_Q2S) {
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

// fp16 pair arithmetic on raw bits: the two halves of a + b (each rounded; exact for the small integers used here).
__device__ __forceinline__ uint32_t hadd2_bits(uint32_t a, uint32_t b) {
    const __half2 r = __hadd2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
    return *reinterpret_cast<const uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t lop3_xor_or(uint32_t a, uint32_t b, uint32_t c) {
    // (a ^ b) | c in one LOP3 (truth table 0xBE)
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xBE;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
constexpr uint32_t HNEG1024 = 0xE400E400u;   // fp16 -1024 in both halves
constexpr uint32_t HNEG1152 = 0xE480E480u;   // fp16 -1152 = -(1024 + 128) in both halves

// acc += sum_i w'_i x_i over one 32-weight unit of one row when `on`, else acc is left unchanged; `u` = aligned unit
// base in shared memory, `sp` = this row's group-scale pointer (Q4G32), `c` = the unit's activation constants,
// `xv` = its staged activations. Each sub-block accumulator starts at -C (the activation constant), so no separate
// subtraction is needed. Sub-block scale integers are turned into exact fp16 values with the 1024 mantissa trick and
// multiplied by the raw fp16 super-block scale with exact fp16 x fp16 -> fp32 products; masking zeroes that scale.
template <int F>
__device__ __forceinline__ void row_acc(const uint8_t *u, const float *sp, const LaneGeo &g, const float *c,
                                        const uint32_t *xv, bool on, float &acc) {
    if constexpr (F == FMT_Q4G32) {
        // 16 * sum (u - 8) x_i in int32 (exact), then one conversion and the group scale times 2^-(E+4)
        const uint4 w = *reinterpret_cast<const uint4 *>(u);
        const float s = on ? sp[0] : 0.f;
        int32_t lo = 0, hi = __float_as_int(c[0]);
        nib_dp(w.x, xv + 0, lo, hi);
        nib_dp(w.y, xv + 4, lo, hi);
        nib_dp(w.z, xv + 8, lo, hi);
        nib_dp(w.w, xv + 12, lo, hi);
        acc = fmaf(float(16 * lo + hi), s * c[1], acc);
    } else if constexpr (F == FMT_Q2S) {
        const uint32_t w0 = lds32(u), w1 = lds32(u + 4);
        const uint32_t dd = on ? lds32(u + g.o2) : 0u;                   // d (low half), dmin (high half)
        const uint32_t lm = *reinterpret_cast<const uint16_t *>(u + g.o1);
        const uint32_t t = __byte_perm(lm, 0u, 0x4140u);                 // L0 | M0 << 4 at byte 0, L1 | M1 << 4 at byte 2
        const uint32_t hl = hadd2_bits(lop3_and_or(t, 0x000F000Fu, MAGIC2), HNEG1024);        // (L0, L1)
        const uint32_t hm = hadd2_bits(lop3_and_or(t >> 4, 0x000F000Fu, MAGIC2), HNEG1024);   // (M0, M1)
        float a0 = -c[0], b0 = 0.f, a1 = -c[2], b1 = 0.f;
        crumb_word(w0, xv, 0, a0, b0);
        crumb_word(w1, xv, 16, a1, b1);
        acc = fmaf(fma_h(lo16(hl), lo16(dd), 0.f), a0 + b0, acc);
        acc = fmaf(fma_h(hi16(hl), lo16(dd), 0.f), a1 + b1, acc);
        acc = fmaf(-fma_h(lo16(hm), hi16(dd), 0.f), c[1], acc);
        acc = fmaf(-fma_h(hi16(hm), hi16(dd), 0.f), c[3], acc);
    } else if constexpr (F == FMT_Q3S) {
        const uint32_t *wp = reinterpret_cast<const uint32_t *>(u);
        const uint32_t w0 = wp[0], w1 = wp[1];
        const uint32_t *qp = reinterpret_cast<const uint32_t *>(u + g.o1);
        const uint32_t w2 = qp[0], w3 = qp[1];
        const uint32_t *fp = reinterpret_cast<const uint32_t *>(u + g.o2);
        const uint32_t f = __funnelshift_r(fp[0], fp[1], g.sh1);          // L_j0 at bits 0..5, L_j0+1 at bits 6..11
        const uint32_t lh = hadd2_bits(lop3_and_or(lop3_sel(f << 10, f, 0xFFFF0000u), 0x003F003Fu, MAGIC2), HNEG1024);
        const uint16_t D = on ? *reinterpret_cast<const uint16_t *>(u + g.o3) : uint16_t(0);
        float a0 = -c[0], a1 = -c[1];
        tri_pair(__byte_perm(w0, w1, g.p0), __byte_perm(w0, w1, g.p1), __byte_perm(w0, w1, g.p2), xv, 0, a0);
        tri_pair(__byte_perm(w2, w3, g.q0), __byte_perm(w2, w3, g.q1), __byte_perm(w2, w3, g.q2), xv, 8, a1);
        acc = fmaf(fma_h(lo16(lh), D, 0.f), a0, acc);
        acc = fmaf(fma_h(hi16(lh), D, 0.f), a1, acc);
    } else if constexpr (F == FMT_Q5S) {
        const uint4 w = *reinterpret_cast<const uint4 *>(u);
        const uint32_t H = lds32(u + g.o1);
        const uint4 fld = *reinterpret_cast<const uint4 *>(u + g.o2);
        const uint32_t ddw = on ? fld.w : 0u;
        const float2 Dd = __half22float2(*reinterpret_cast<const __half2 *>(&ddw));
        const uint64_t lo64 = (uint64_t(fld.y) << 32) | fld.x, hi64 = (uint64_t(fld.z) << 32) | fld.y;
        const float L = small_int_f(lop3_and_or(uint32_t(lo64 >> g.sh0), 63u, MAGICF));
        const float M = small_int_f(lop3_and_or(uint32_t(hi64 >> (g.sh1 - 32u)), 63u, MAGICF));
        float a = -c[0], b = 0.f;
        nib_word_hi<1>(w.x, lop3_sel(H, H << 12, 0x0000FFFFu), xv, 0, a, b);
        nib_word_hi<1>(w.y, lop3_sel(H >> 8, H << 4, 0x0000FFFFu), xv, 8, a, b);
        nib_word_hi<1>(w.z, lop3_sel(H >> 16, H >> 4, 0x0000FFFFu), xv, 16, a, b);
        nib_word_hi<1>(w.w, lop3_sel(H >> 24, H >> 12, 0x0000FFFFu), xv, 24, a, b);
        acc = fmaf(Dd.x * L, a + b, acc);
        acc = fmaf(-(Dd.y * M), c[1], acc);
    } else {
        const uint32_t sh = g.sh0;
        const uint32_t *wp = reinterpret_cast<const uint32_t *>(u);
        const uint32_t r0 = wp[0], r1 = wp[1], r2 = wp[2], r3 = wp[3], r4 = wp[4];
        const uint32_t *hp = reinterpret_cast<const uint32_t *>(u + g.o1);
        const uint32_t q0 = hp[0], q1 = hp[1], q2 = hp[2];
        const uint32_t h0 = __funnelshift_r(q0, q1, sh), h1 = __funnelshift_r(q1, q2, sh);
        const uint32_t lv = *reinterpret_cast<const uint16_t *>(u + g.o2);
        // int8 pair -> exact fp16 pair: (b ^ 0x80) in the mantissa of 1024, minus 1024 + 128
        const uint32_t lh = hadd2_bits(lop3_xor_or(__byte_perm(lv, 0u, 0x4140u), 0x00800080u, MAGIC2), HNEG1152);
        const uint16_t D = on ? *reinterpret_cast<const uint16_t *>(u + g.o3) : uint16_t(0);
        float a0 = -c[0], b0 = 0.f, a1 = -c[1], b1 = 0.f;
        nib_word_hi<2>(__funnelshift_r(r0, r1, sh), __byte_perm(h0, 0u, 0x4140u), xv, 0, a0, b0);
        nib_word_hi<2>(__funnelshift_r(r1, r2, sh), __byte_perm(h0, 0u, 0x4342u), xv, 8, a0, b0);
        nib_word_hi<2>(__funnelshift_r(r2, r3, sh), __byte_perm(h1, 0u, 0x4140u), xv, 16, a1, b1);
        nib_word_hi<2>(__funnelshift_r(r3, r4, sh), __byte_perm(h1, 0u, 0x4342u), xv, 24, a1, b1);
        acc = fmaf(fma_h(lo16(lh), D, 0.f), a0 + b0, acc);
        acc = fmaf(fma_h(hi16(lh), D, 0.f), a1 + b1, acc);
    }
}

// ------------------------------------------------------------------------------------------------------------
// Multi-row form of the same math (small-batch products): a unit-row is unpacked once into 16 words of fp16 code
// pairs (the LOP3 outputs of row_acc, in the same order) plus its sub-block scale factors, then multiplied against
// several staged activation rows. hw[j] holds the codes of staging slots hslot<F>(j, 0) (low half) and
// hslot<F>(j, 1) (high half); words 0..7 belong to sub-block 0 and 8..15 to sub-block 1 (formats with one 32-weight
// sub-block use the same split for two independent accumulators).
// ------------------------------------------------------------------------------------------------------------
template <int F>
__host__ __device__ constexpr int hslot(int j, int h) {
    if constexpr (F == FMT_Q3S) return 2 * j + h;
    else if constexpr (F == FMT_Q2S) return 16 * (j / 8) + 4 * (j % 2) + (j % 8) / 2 + 8 * h;
    else return 8 * (j / 4) + j % 4 + 4 * h;
}
struct URow {
    uint32_t hw[16];
    float f0, f1;   // sub-block scale factors (w' = f * code for the symmetric part)
    float g0, g1;   // minima factors of the asymmetric formats (dmin * M_j), else 0
};
template <int HB>
__device__ __forceinline__ void unpack_nib_hi(uint32_t c, uint32_t X, uint32_t *hw) {
    constexpr uint32_t mlo = (HB == 1) ? 0x00100010u : 0x00300030u;
    constexpr uint32_t mhi = (HB == 1) ? 0x01000100u : 0x03000300u;
    constexpr int s0 = 4, s1 = (HB == 1) ? 7 : 6, s2 = (HB == 1) ? 2 : 0, s3 = (HB == 1) ? 5 : 2;
    const uint32_t c2 = c >> 8;
    hw[0] = lop3_and_or(X << s0, mlo, lop3_and_or(c, 0x000F000Fu, MAGIC2));
    hw[1] = lop3_and_or(X << s1, mhi, lop3_and_or(c, 0x00F000F0u, MAGIC2));
    hw[2] = lop3_and_or(X << s2, mlo, lop3_and_or(c2, 0x000F000Fu, MAGIC2));
    hw[3] = lop3_and_or(X << s3, mhi, lop3_and_or(c2, 0x00F000F0u, MAGIC2));
}
__device__ __forceinline__ void unpack_crumb(uint32_t c, uint32_t *hw) {
    const uint32_t c2 = c >> 8;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t m = (3u << (2 * k)) * 0x00010001u;
        hw[2 * k] = lop3_and_or(c, m, MAGIC2);
        hw[2 * k + 1] = lop3_and_or(c2, m, MAGIC2);
    }
}
__device__ __forceinline__ void unpack_tri(uint32_t W0, uint32_t W1, uint32_t W2, uint32_t *hw) {
    hw[0] = lop3_and_or(W0, 0x00070007u, MAGIC2);
    hw[1] = lop3_and_or(W0, 0x00380038u, MAGIC2);
    hw[2] = lop3_and_or(W0, 0x01C001C0u, MAGIC2);
    hw[3] = lop3_and_or(W1, 0x000E000Eu, MAGIC2);
    hw[4] = lop3_and_or(W1, 0x00700070u, MAGIC2);
    hw[5] = lop3_and_or(W1, 0x03800380u, MAGIC2);
    hw[6] = lop3_and_or(W2, 0x001C001Cu, MAGIC2);
    hw[7] = lop3_and_or(W2, 0x00E000E0u, MAGIC2);
}

// Unpack one unit-row (same operands as row_acc); `on` false zeroes its scale factors.
template <int F>
__device__ __forceinline__ void unpack_row(const uint8_t *u, const float *sp, const LaneGeo &g, bool on, URow &r) {
    r.g0 = r.g1 = 0.f;
    if constexpr (F == FMT_Q4G32) {
        const uint4 w = *reinterpret_cast<const uint4 *>(u);
        r.f0 = r.f1 = on ? sp[0] : 0.f;
        // the dp2a operands: hw[2j] = low nibbles of word j in place, hw[2j + 1] = its high nibbles in place
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) { r.hw[2 * j] = wv[j] & 0x0F0F0F0Fu; r.hw[2 * j + 1] = wv[j] & 0xF0F0F0F0u; }
    } else if constexpr (F == FMT_Q2S) {
        const uint32_t w0 = lds32(u), w1 = lds32(u + 4);
        const uint32_t dd = on ? lds32(u + g.o2) : 0u;
        const uint32_t lm = *reinterpret_cast<const uint16_t *>(u + g.o1);
        const uint32_t t = __byte_perm(lm, 0u, 0x4140u);
        const uint32_t hl = hadd2_bits(lop3_and_or(t, 0x000F000Fu, MAGIC2), HNEG1024);
        const uint32_t hm = hadd2_bits(lop3_and_or(t >> 4, 0x000F000Fu, MAGIC2), HNEG1024);
        r.f0 = fma_h(lo16(hl), lo16(dd), 0.f);
        r.f1 = fma_h(hi16(hl), lo16(dd), 0.f);
        r.g0 = fma_h(lo16(hm), hi16(dd), 0.f);
        r.g1 = fma_h(hi16(hm), hi16(dd), 0.f);
        unpack_crumb(w0, r.hw); unpack_crumb(w1, r.hw + 8);
    } else if constexpr (F == FMT_Q3S) {
        const uint32_t *wp = reinterpret_cast<const uint32_t *>(u);
        const uint32_t w0 = wp[0], w1 = wp[1];
        const uint32_t *qp = reinterpret_cast<const uint32_t *>(u + g.o1);
        const uint32_t w2 = qp[0], w3 = qp[1];
        const uint32_t *fp = reinterpret_cast<const uint32_t *>(u + g.o2);
        const uint32_t f = __funnelshift_r(fp[0], fp[1], g.sh1);
        const uint32_t lh = hadd2_bits(lop3_and_or(lop3_sel(f << 10, f, 0xFFFF0000u), 0x003F003Fu, MAGIC2), HNEG1024);
        const uint16_t D = on ? *reinterpret_cast<const uint16_t *>(u + g.o3) : uint16_t(0);
        r.f0 = fma_h(lo16(lh), D, 0.f);
        r.f1 = fma_h(hi16(lh), D, 0.f);
        unpack_tri(__byte_perm(w0, w1, g.p0), __byte_perm(w0, w1, g.p1), __byte_perm(w0, w1, g.p2), r.hw);
        unpack_tri(__byte_perm(w2, w3, g.q0), __byte_perm(w2, w3, g.q1), __byte_perm(w2, w3, g.q2), r.hw + 8);
    } else if constexpr (F == FMT_Q5S) {
        const uint4 w = *reinterpret_cast<const uint4 *>(u);
        const uint32_t H = lds32(u + g.o1);
        const uint4 fld = *reinterpret_cast<const uint4 *>(u + g.o2);
        const uint32_t ddw = on ? fld.w : 0u;
        const float2 Dd = __half22float2(*reinterpret_cast<const __half2 *>(&ddw));
        const uint64_t lo64 = (uint64_t(fld.y) << 32) | fld.x, hi64 = (uint64_t(fld.z) << 32) | fld.y;
        const float L = small_int_f(lop3_and_or(uint32_t(lo64 >> g.sh0), 63u, MAGICF));
        const float Mv = small_int_f(lop3_and_or(uint32_t(hi64 >> (g.sh1 - 32u)), 63u, MAGICF));
        r.f0 = r.f1 = Dd.x * L;
        r.g0 = Dd.y * Mv;
        unpack_nib_hi<1>(w.x, lop3_sel(H, H << 12, 0x0000FFFFu), r.hw);
        unpack_nib_hi<1>(w.y, lop3_sel(H >> 8, H << 4, 0x0000FFFFu), r.hw + 4);
        unpack_nib_hi<1>(w.z, lop3_sel(H >> 16, H >> 4, 0x0000FFFFu), r.hw + 8);
        unpack_nib_hi<1>(w.w, lop3_sel(H >> 24, H >> 12, 0x0000FFFFu), r.hw + 12);
    } else {
        const uint32_t sh = g.sh0;
        const uint32_t *wp = reinterpret_cast<const uint32_t *>(u);
        const uint32_t r0 = wp[0], r1 = wp[1], r2 = wp[2], r3 = wp[3], r4 = wp[4];
        const uint32_t *hp = reinterpret_cast<const uint32_t *>(u + g.o1);
        const uint32_t q0 = hp[0], q1 = hp[1], q2 = hp[2];
        const uint32_t h0 = __funnelshift_r(q0, q1, sh), h1 = __funnelshift_r(q1, q2, sh);
        const uint32_t lv = *reinterpret_cast<const uint16_t *>(u + g.o2);
        const uint32_t lh = hadd2_bits(lop3_xor_or(__byte_perm(lv, 0u, 0x4140u), 0x00800080u, MAGIC2), HNEG1152);
        const uint16_t D = on ? *reinterpret_cast<const uint16_t *>(u + g.o3) : uint16_t(0);
        r.f0 = fma_h(lo16(lh), D, 0.f);
        r.f1 = fma_h(hi16(lh), D, 0.f);
        unpack_nib_hi<2>(__funnelshift_r(r0, r1, sh), __byte_perm(h0, 0u, 0x4140u), r.hw);
        unpack_nib_hi<2>(__funnelshift_r(r1, r2, sh), __byte_perm(h0, 0u, 0x4342u), r.hw + 4);
        unpack_nib_hi<2>(__funnelshift_r(r2, r3, sh), __byte_perm(h1, 0u, 0x4140u), r.hw + 8);
        unpack_nib_hi<2>(__funnelshift_r(r3, r4, sh), __byte_perm(h1, 0u, 0x4342u), r.hw + 12);
    }
}

// acc += sum_i w'_i x_i of an unpacked unit-row against one staged activation row (xv, c: that row's unit constants).
template <int F>
__device__ __forceinline__ void dot_row(const URow &r, const uint32_t *xv, const float *c, float &acc) {
    if constexpr (F == FMT_Q4G32) {
        int32_t lo = 0, hi = __float_as_int(c[0]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            lo = dp2a_lo(xv[4 * j], r.hw[2 * j], lo);
            lo = dp2a_hi(xv[4 * j + 1], r.hw[2 * j], lo);
            hi = dp2a_lo(xv[4 * j + 2], r.hw[2 * j + 1], hi);
            hi = dp2a_hi(xv[4 * j + 3], r.hw[2 * j + 1], hi);
        }
        acc = fmaf(float(16 * lo + hi), r.f0 * c[1], acc);
        return;
    }
    float a0, a1;
    if constexpr (F == FMT_Q5S) { a0 = -c[0]; a1 = 0.f; }
    else if constexpr (F == FMT_Q2S) { a0 = -c[0]; a1 = -c[2]; }
    else { a0 = -c[0]; a1 = -c[1]; }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        a0 = fma_h(lo16(r.hw[j]), xh(xv, hslot<F>(j, 0)), a0);
        a0 = fma_h(hi16(r.hw[j]), xh(xv, hslot<F>(j, 1)), a0);
        a1 = fma_h(lo16(r.hw[8 + j]), xh(xv, hslot<F>(8 + j, 0)), a1);
        a1 = fma_h(hi16(r.hw[8 + j]), xh(xv, hslot<F>(8 + j, 1)), a1);
    }
    if constexpr (F == FMT_Q5S) {
        acc = fmaf(r.f0, a0 + a1, acc);
        acc = fmaf(-r.g0, c[1], acc);
    } else {
        acc = fmaf(r.f0, a0, acc);
        acc = fmaf(r.f1, a1, acc);
        if constexpr (F == FMT_Q2S) {
            acc = fmaf(-r.g0, c[1], acc);
            acc = fmaf(-r.g1, c[3], acc);
        }
    }
}

// Staged activations: the 16 words of unit u are four 16-byte vectors at vector index t * U + u (t = 0..3, U = K / 32
// units per row), so consecutive lanes (consecutive units) read consecutive vectors. Half-unit hh (elements
// 16 hh .. 16 hh + 15) is words 8 hh .. 8 hh + 7, i.e. vectors t = 2 hh and 2 hh + 1.
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
__device__ __forceinline__ void load_xp(const uint4 *xs, uint32_t U, uint32_t u, uint32_t xv[16]) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint4 v = xs[t * U + u];
        xv[4 * t] = v.x; xv[4 * t + 1] = v.y; xv[4 * t + 2] = v.z; xv[4 * t + 3] = v.w;
    }
}
// Scale exponent of a K part from its max |x| (fp16 magnitude bits): x * 2^E has max in [2^14, 2^15); 0 for an all-zero
// part; inf / nan inputs clamp to the largest finite magnitude.
__device__ __forceinline__ int part_exponent(uint32_t mbits) {
    const float xm = h2f_bits(uint16_t(min(mbits, 0x7BFFu)));
    return (xm > 0.f) ? 14 - (int((__float_as_uint(xm) >> 23) & 255u) - 127) : 0;
}

// Stage one unit: raw = its 32 fp16 activations (four 16-byte vectors), E = the part's scale exponent. Writes the
// unit's four staged vectors (x' = fp16(x * 2^(E - p)), see stage_half_unit) and its activation constants.
// Q4G32 staging: the unit's 32 activations as 16-bit integers xi = rint(x * 2^E), E = the unit's own exponent (max
// |x| * 2^E in [2^14, 2^15), so |xi| <= 32752; an inf clamps to 32767, a nan gives 0), vector j holding the dp2a
// operands of code word j (see nib_dp). Constants: -128 * sum(xi) as int bits (the code offset 8, times the 16 of
// the high-nibble accumulator) and 2^-(E+4).
__device__ __forceinline__ void stage_unit_i16(const uint4 (&raw)[4], uint4 *xs, float *cst, uint32_t U, uint32_t u) {
    const uint32_t hx[16] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w, raw[1].x, raw[1].y, raw[1].z, raw[1].w,
                             raw[2].x, raw[2].y, raw[2].z, raw[2].w, raw[3].x, raw[3].y, raw[3].z, raw[3].w};
    uint32_t mx = 0;
#pragma unroll
    for (int e = 0; e < 16; ++e) mx = max(mx, max(hx[e] & 0x7FFFu, (hx[e] >> 16) & 0x7FFFu));
    const int E = part_exponent(mx);
    const float sc = exp2i(E);
    int32_t xi[32], sum = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int32_t v = __float2int_rn(h2f_bits((i & 1) ? hi16(hx[i >> 1]) : lo16(hx[i >> 1])) * sc);
        xi[i] = min(max(v, -32767), 32767);
        sum += xi[i];
    }
    auto pk = [&](int i0, int i1) { return (uint32_t(xi[i0]) & 0xFFFFu) | (uint32_t(xi[i1]) << 16); };
#pragma unroll
    for (int j = 0; j < 4; ++j)
        xs[j * U + u] = make_uint4(pk(8 * j, 8 * j + 2), pk(8 * j + 4, 8 * j + 6), pk(8 * j + 1, 8 * j + 3),
                                   pk(8 * j + 5, 8 * j + 7));
    cst[2 * u] = __int_as_float(-128 * sum);
    cst[2 * u + 1] = exp2i(-(E + 4));
}

template <int F>
__device__ __forceinline__ void stage_unit(const uint4 (&raw)[4], int E, uint4 *xs, float *cst, uint32_t U, uint32_t u) {
    if constexpr (F == FMT_Q4G32) {
        stage_unit_i16(raw, xs, cst, U, u);   // per-unit exponent; E (the part's) is not used
    } else {
        uint32_t w[16];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const uint32_t rw[8] = {raw[2 * hh].x, raw[2 * hh].y, raw[2 * hh].z, raw[2 * hh].w,
                                    raw[2 * hh + 1].x, raw[2 * hh + 1].y, raw[2 * hh + 1].z, raw[2 * hh + 1].w};
            uint16_t xr[16];
#pragma unroll
            for (int e = 0; e < 8; ++e) { xr[2 * e] = lo16(rw[e]); xr[2 * e + 1] = hi16(rw[e]); }
            stage_half_unit<F>(xr, E, w + 8 * hh);
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) xs[t * U + u] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
        float xp[32], xt[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            xp[i] = h2f_bits(xh(w, i));
            xt[i] = xp[i] * pow2f(xshift<F>(i));
        }
        unit_consts<F>(xp, xt, cst + u * XC<F>::n);
    }
}

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

// 2-D tensor copy global -> shared (box of the tensor map at coordinates {x, y}), completion on `bar` as bytes.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

}  // namespace

// ------------------------------------------------------------------------------------------------------------
// Fused dequant-GEMV kernel for MT activation rows (MT = 1: the batch-1 decode product; MT = 2..16: small batches).
//
// The packed matrix is read through a 2-D TMA tensor map over (rows x 8-byte words): one tensor copy moves a tile of
// TR rows x one K chunk (CHW weights) into a shared-memory stage, so every stage has the same compile-time layout
// (row r of the chunk at r * CB bytes) whatever K is; words past the row end and rows past N arrive as zeros and are
// masked by the consumers. One CTA per SM; the next product in the stream, launched as a programmatic dependent,
// starts streaming its weights as soon as this CTA leaves its SM.
// Warp 16 is the producer (one lane issues the first copies; every later copy is issued by the consumer warp that
// releases a stage last). Warps 0..15 consume every stage together: warp w handles row class rc = w / P (rows rc,
// rc + RC, ...: RW rows) over K part q = w % P of the chunk (32 units; lane l owns unit 32 q + l of every chunk).
// With MT = 1 a lane unpacks and multiplies in one pass (row_acc); with MT > 1 it unpacks each unit-row once
// (unpack_row) and multiplies it against the MT staged activation rows (dot_row), so every weight is read and
// unpacked once for the whole batch. Row sums accumulate over the chunks of a tile; then each warp reduces its lanes
// with shuffles and stores one partial per (row, activation row, part), and the P partials are summed in a fixed
// order (deterministic). Activations are staged per (row, part) with a power-of-two scale (max |x| * 2^E in
// [2^14, 2^15)).
// ------------------------------------------------------------------------------------------------------------
constexpr int G1_CW = 16;                      // consumer warps
template <int F, int MT = 1> struct T1 {
    static constexpr int CHW = (F == FMT_Q5S || F == FMT_Q6S) ? 2048 : 4096;      // weights per K chunk
    static constexpr int UPC = CHW / 32;                                          // units per chunk
    static constexpr int P = UPC / 32;                                            // K parts of 32 units
    static constexpr int RC = G1_CW / P;                                          // row classes
    static constexpr int RW = MT > 2 ? 2 : (F == FMT_Q4G32 ? 4 : (P == 4 ? 8 : 4)); // rows per warp and stage
    static constexpr int TR = RC * RW;                                            // rows per tile
    static constexpr int PR = MT > 1 ? (256 / MT > TR ? 256 / MT : TR) : 256;     // rows per partial-sum round
    static constexpr int CB = Fmt<F>::sb ? (CHW / 256) * Fmt<F>::bytes : CHW / 2; // code bytes per row chunk
    static constexpr int SB = Fmt<F>::sb ? 0 : (CHW / 32) * 4;                    // Q4G32 scale bytes per row chunk
    static constexpr int TX = TR * (CB + SB);                                     // bytes a stage receives
    static constexpr int STAGE = (TX + 127) / 128 * 128;
    static_assert(CB % 16 == 0 && CB / 8 <= 256 && SB / 8 <= 256, "tensor-map box limits");
    static_assert(PR % TR == 0 && RW * MT <= 32, "tile and reduction shapes");
};
constexpr int G1_THREADS = (G1_CW + 1) * 32;
constexpr int G1_MAXNS = 16;                   // stages in the ring at most
constexpr int G1_PRE = 1;                      // stage fills issued before the activations are staged
constexpr uint32_t G1_HDR = 1024;              // mbarriers, release counters, per-(row, part) scales

struct G1Plan {
    uint32_t off_part, off_xs, off_cst, off_stages, smem;
    int ns;
};

template <int F, int MT>
__global__ void __launch_bounds__(G1_THREADS, 1)
    gemv1_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_scales,
                 GemvArgs a, G1Plan pl) {
    using T = T1<F, MT>;
    constexpr int P = T::P, RC = T::RC, RW = T::RW, TR = T::TR, CB = T::CB, SB = T::SB, UPC = T::UPC, PR = T::PR;
    constexpr int NX = XC<F>::n;
    constexpr uint32_t NT = G1_CW * 32;
    extern __shared__ __align__(1024) uint8_t smem_g1[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t N = uint32_t(a.N), K = uint32_t(a.K), U = K / 32;
    const uint32_t Mg = uint32_t(a.M);                     // activation rows of this launch (<= MT)
    // this CTA's rows: a contiguous range; the row counts of any two CTAs differ by at most one
    const uint32_t rq = N / gridDim.x, rm = N % gridDim.x, b = blockIdx.x;
    const uint32_t rbeg = b * rq + min(b, rm), nrows = rq + (b < rm ? 1u : 0u);
    const uint32_t nch = (U + UPC - 1) / UPC;              // K chunks per row
    const uint32_t nit = (nrows + TR - 1) / TR * nch;      // stages of this CTA: tiles x chunks
    const uint32_t NS = uint32_t(pl.ns);

    uint64_t *full = reinterpret_cast<uint64_t *>(smem_g1);                  // [NS] stage filled
    uint32_t *rel = reinterpret_cast<uint32_t *>(smem_g1 + G1_MAXNS * 8);    // [NS] warps done with the stage
    uint64_t *xready = reinterpret_cast<uint64_t *>(smem_g1 + G1_MAXNS * 12);  // activations staged
    float *uscale = reinterpret_cast<float *>(smem_g1 + 256);                // [MT][P]: 2^-E per (row, part)
    uint32_t *pmax = reinterpret_cast<uint32_t *>(smem_g1 + 512);            // [MT][P]: max |x| bits
    float *part = reinterpret_cast<float *>(smem_g1 + pl.off_part);
    uint4 *xs = reinterpret_cast<uint4 *>(smem_g1 + pl.off_xs);              // [MT][4][U]
    float *cst = reinterpret_cast<float *>(smem_g1 + pl.off_cst);            // [MT][U][NX]
    uint8_t *stages = smem_g1 + pl.off_stages;

    if (tid == 0) {
        for (uint32_t s = 0; s < NS; ++s) { mbar_init(&full[s], 1); rel[s] = 0; }
        for (int i = 0; i < MT * P; ++i) pmax[i] = 0;
        mbar_init(xready, 1);
        fence_mbar_init();
    }
    pdl_launch_dependents();     // the next product may begin launching; it still waits for us before reading x
    __syncthreads();
    const uint64_t pol = l2_evict_first_policy();
    // Fill of item j (tile j / nch, chunk j % nch) into stage j % NS.
    auto fill = [&](uint32_t j) {
        const uint32_t s = j % NS, tj = j / nch, cj = j - tj * nch;
        uint8_t *st = stages + s * uint32_t(T::STAGE);
        mbar_arrive_expect_tx(&full[s], uint32_t(T::TX));
        tma_load_2d(st, &tm_codes, int(cj * (CB / 8)), int(rbeg + tj * TR), &full[s], pol);
        if constexpr (SB > 0) tma_load_2d(st + TR * CB, &tm_scales, int(cj * (SB / 8)), int(rbeg + tj * TR), &full[s], pol);
    };

    if (warp == G1_CW) {
        // ------------------------------------ producer ------------------------------------
        if (lane == 0) {
            // Packed weights are read before the previous grid has finished only when the caller opted in
            // (QPACK_OPT_WEIGHT_PREFETCH: weights are not written by the kernel just before this one). Only the first
            // G1_PRE fills go out before the activations are staged: a deeper early prefetch fills the memory queues
            // and delays the activation loads on the critical path.
            if (!a.weight_prefetch) pdl_wait();
            uint32_t j = 0;
            for (; j < nit && j < NS && j < uint32_t(G1_PRE); ++j) fill(j);
            if (j < nit && j < NS) {
                if (!mbar_wait_bounded_hint(xready, 0u)) atomicOr(&g_fault_gemv, FAULT_WAIT_FULL);
                for (; j < nit && j < NS; ++j) fill(j);
            }
        }
        return;
    }

    // -------------------------------------- consumers --------------------------------------
    const uint32_t rc = uint32_t(warp) / P, q = uint32_t(warp) % P;
    const uint32_t uc = q * 32u + uint32_t(lane);           // this lane's unit within every chunk
    pdl_wait();                  // x (and y) may belong to the previous grid
    {
        const uint4 *xg = reinterpret_cast<const uint4 *>(a.X);
        if constexpr (MT == 1) {
            // Thread t handles units t, t + NT, ... (K <= 32768). A warp's 32 consecutive units are one 32-unit run of
            // one chunk, i.e. of one K part, so a part's max |x| is a warp max plus one shared atomic per warp; after
            // a barrier every thread stages its units from registers.
            constexpr int HU = int((1024 + NT - 1) / NT);   // units per thread at the largest K
            uint4 raw[HU][4];
#pragma unroll
            for (int h = 0; h < HU; ++h) {
                const uint32_t u = uint32_t(tid) + h * NT;
                uint32_t mx = 0;
                if (u < U) {
#pragma unroll
                    for (int t = 0; t < 4; ++t) raw[h][t] = __ldg(xg + 4 * u + t);
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const uint32_t w[4] = {raw[h][t].x, raw[h][t].y, raw[h][t].z, raw[h][t].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) mx = max(mx, max(w[e] & 0x7FFFu, (w[e] >> 16) & 0x7FFFu));
                    }
                }
                if (F != FMT_Q4G32 && uint32_t(tid - lane) + h * NT < U) {   // the warp's first unit exists
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    if (lane == 0) atomicMax(&pmax[((uint32_t(tid) + h * NT) % UPC) / 32], mx);
                }
            }
            if constexpr (F != FMT_Q4G32) named_bar_sync(1, G1_CW * 32);   // Q4G32: per-unit exponents
#pragma unroll
            for (int h = 0; h < HU; ++h) {
                const uint32_t u = uint32_t(tid) + h * NT;
                if (u < U) stage_unit<F>(raw[h], part_exponent(pmax[(u % UPC) / 32]), xs, cst, U, u);
            }
        } else {
            // MT x U units (activation row m, unit u): item i = m * Upad + u, Upad = U rounded up to 32, so a warp's 32
            // consecutive items are one 32-unit run of one chunk of one row, i.e. of one (row, K part). Two passes:
            // the max, then (after a barrier) a reload and the staging. Rows m >= Mg of a short group stage zeros.
            const uint32_t Upad = (U + 31) / 32 * 32, items = uint32_t(MT) * Upad;
            for (uint32_t it = uint32_t(tid); F != FMT_Q4G32 && it < items; it += NT) {   // Q4G32: per-unit exponents
                const uint32_t m = it / Upad, u = it - m * Upad;
                uint32_t mx = 0;
                if (u < U && m < Mg) {
                    const uint4 *xr = xg + (int64_t(m) * a.ldx) / 8 + 4 * u;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const uint4 v = __ldg(xr + t);
                        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) mx = max(mx, max(w[e] & 0x7FFFu, (w[e] >> 16) & 0x7FFFu));
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                if (lane == 0) atomicMax(&pmax[m * P + (u % UPC) / 32], mx);
            }
            if constexpr (F != FMT_Q4G32) named_bar_sync(1, G1_CW * 32);
            for (uint32_t it = uint32_t(tid); it < items; it += NT) {
                const uint32_t m = it / Upad, u = it - m * Upad;
                if (u < U) {
                    uint4 raw[4] = {};
                    if (m < Mg) {
                        const uint4 *xr = xg + (int64_t(m) * a.ldx) / 8 + 4 * u;
#pragma unroll
                        for (int t = 0; t < 4; ++t) raw[t] = __ldg(xr + t);
                    }
                    stage_unit<F>(raw, part_exponent(pmax[m * P + (u % UPC) / 32]), xs + m * 4 * U, cst + m * U * NX, U, u);
                }
            }
        }
        if (tid < MT * P) uscale[tid] = exp2i(-part_exponent(pmax[tid]));
        // every consumer meets here: masked lanes read the last unit's staged activations, whichever part staged it
        named_bar_sync(1, G1_CW * 32);
        if (tid == 0) mbar_arrive(xready);
    }

    const LaneGeo geo = lane_geo<F>(int(uc));
    const bool last_full = (U % UPC) == 0;                 // every lane has a unit in the last chunk too
    uint32_t ph = 0, s = 0, c = 0, t = 0;
    bool dead = false;
    float acc[RW * MT];
#pragma unroll
    for (int i = 0; i < RW * MT; ++i) acc[i] = 0.f;
    for (uint32_t k = 0; k < nit; ++k) {
        if (!dead && !mbar_wait_bounded(&full[s], ph)) {
            if (lane == 0) atomicOr(&g_fault_gemv, FAULT_WAIT_FULL);
            dead = true;
        }
        const uint32_t rows = min(uint32_t(TR), nrows - t * TR);
        if (!dead) {
            const uint8_t *st = stages + s * uint32_t(T::STAGE);
            const uint8_t *ub = st + rc * CB + geo.ubase;
            const float *sp = reinterpret_cast<const float *>(st + TR * CB + rc * SB) + uc;
            const uint32_t u = c * UPC + uc;
            const bool uv = u < U;
            const uint32_t uu = uv ? u : U - 1;
            const bool full_tile = rows == uint32_t(TR) && (last_full || c + 1 < nch);
            if constexpr (MT == 1) {
                uint32_t xv[16];
                load_xp(xs, U, uu, xv);
                float cv[NX];
#pragma unroll
                for (int cc = 0; cc < NX; ++cc) cv[cc] = cst[uu * NX + cc];
                if (full_tile) {
#pragma unroll
                    for (int i = 0; i < RW; ++i)
                        row_acc<F>(ub + i * RC * CB, sp + i * RC * (SB / 4), geo, cv, xv, true, acc[i]);
                } else {
                    // ragged tile or chunk: rows past the tile's end are skipped (uniform branches), lanes past K masked
#pragma unroll
                    for (int i = 0; i < RW; ++i)
                        if (rc + uint32_t(RC * i) < rows)
                            row_acc<F>(ub + i * RC * CB, sp + i * RC * (SB / 4), geo, cv, xv, uv, acc[i]);
                }
            } else if constexpr (MT == 2) {
                // both activation rows stay in registers; each unit-row is unpacked once and used twice
                uint32_t xv0[16], xv1[16];
                load_xp(xs, U, uu, xv0);
                load_xp(xs + 4 * U, U, uu, xv1);
                float cv0[NX], cv1[NX];
#pragma unroll
                for (int cc = 0; cc < NX; ++cc) { cv0[cc] = cst[uu * NX + cc]; cv1[cc] = cst[(U + uu) * NX + cc]; }
#pragma unroll
                for (int i = 0; i < RW; ++i) {
                    if (full_tile || rc + uint32_t(RC * i) < rows) {
                        URow ur;
                        unpack_row<F>(ub + i * RC * CB, sp + i * RC * (SB / 4), geo, full_tile || uv, ur);
                        dot_row<F>(ur, xv0, cv0, acc[2 * i]);
                        dot_row<F>(ur, xv1, cv1, acc[2 * i + 1]);
                    }
                }
            } else {
                // each unit-row unpacked once, then multiplied against every activation row
                URow ur[RW];
#pragma unroll
                for (int i = 0; i < RW; ++i)
                    unpack_row<F>(ub + i * RC * CB, sp + i * RC * (SB / 4), geo,
                                  full_tile || (uv && rc + uint32_t(RC * i) < rows), ur[i]);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    uint32_t xv[16];
                    load_xp(xs + m * 4 * U, U, uu, xv);
                    float cv[NX];
#pragma unroll
                    for (int cc = 0; cc < NX; ++cc) cv[cc] = cst[(m * U + uu) * NX + cc];
#pragma unroll
                    for (int i = 0; i < RW; ++i) dot_row<F>(ur[i], xv, cv, acc[i * MT + m]);
                }
            }
            // Release the stage; the warp that releases it last refills it with item k + NS (acq_rel: the other
            // warps' reads of the stage happen before the copy is issued).
            __syncwarp();
            if (lane == 0) {
                const uint32_t n = atom_add_acq_rel_cta(&rel[s], 1u);
                if (n % G1_CW == G1_CW - 1 && k + NS < nit) fill(k + NS);
            }
        }
        if (++s == NS) { s = 0; ph ^= 1u; }
        if (++c < nch) continue;

        // tile done: one partial per (row, activation row, part); after the reduction lanes j * (32 / (RW MT)) hold
        // value j = i * MT + m, i.e. row rc + RC * i and activation row m
        c = 0;
        constexpr int R = RW * MT;
        const float v = warp_rows_sum<R>(acc, lane);
#pragma unroll
        for (int i = 0; i < R; ++i) acc[i] = 0.f;
        const uint32_t lr = (t * TR) % PR;                   // tile's first row within the round
        if ((lane & (32 / R - 1)) == 0) {
            const uint32_t j = uint32_t(lane) / (32 / R), i = j / MT, m = j % MT;
            const uint32_t r = rc + uint32_t(RC) * i;
            if (r < rows) part[((lr + r) * MT + m) * P + q] = v;
        }
        const uint32_t done = t * TR + rows;                // rows of this CTA finished after this tile
        ++t;
        if (done == nrows || done % PR == 0) {
            named_bar_sync(1, G1_CW * 32);
            const uint32_t base = (done - 1) / PR * PR, cnt = done - base;
            for (uint32_t e = uint32_t(tid); e < cnt * MT; e += G1_CW * 32) {
                const uint32_t r = e / MT, m = e - r * MT;
                float yv = 0.f;
#pragma unroll
                for (int pp = 0; pp < P; ++pp) yv = fmaf(part[(r * MT + m) * P + pp], uscale[m * P + pp], yv);
                if (m < Mg) a.Y[int64_t(m) * a.ldy + rbeg + base + r] = yv;
            }
            if (done != nrows) named_bar_sync(1, G1_CW * 32);   // partials of the next round overwrite these
        }
    }
    // Never leave with a copy still writing shared memory: the last fill of every stage has landed (bounded; only a
    // warp that gave up on a wait can get here before that).
    if (dead && lane == 0) {
        for (uint32_t j = (nit > NS ? nit - NS : 0u); j < nit; ++j)
            if (!mbar_wait_bounded(&full[j % NS], (j / NS) & 1u)) break;
    }
}

// Shared-memory plan of one launch: returns false when two stages plus the staged activations do not fit `budget`.
template <int F, int MT>
static bool plan_gemv1(const GemvArgs &a, uint32_t budget, G1Plan *pl) {
    using T = T1<F, MT>;
    const uint32_t U = uint32_t(a.K / 32);
    pl->off_part = G1_HDR;
    pl->off_xs = pl->off_part + uint32_t(T::PR * MT * T::P * 4);
    pl->off_cst = pl->off_xs + uint32_t(round_up(int64_t(MT) * U * 64, 128));
    pl->off_stages = uint32_t(round_up(pl->off_cst + int64_t(MT) * U * XC<F>::n * 4, 1024));
    // + 32: the Q3S / Q6S unpack reads up to 4 bytes past a row chunk
    const int64_t room = int64_t(budget) - pl->off_stages - 32;
    if (room < int64_t(T::STAGE) * 2) return false;
    pl->ns = int(room / T::STAGE < G1_MAXNS ? room / T::STAGE : G1_MAXNS);
    pl->smem = pl->off_stages + uint32_t(pl->ns) * uint32_t(T::STAGE) + 32;
    return true;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Tensor map over a row-major byte matrix [rows][stride] viewed as 8-byte words: boxes of box_words x box_rows.
static cudaError_t encode_rows(CUtensorMap *m, const void *base, int64_t rows, int64_t stride_bytes,
                               uint32_t box_words, uint32_t box_rows) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {cuuint64_t(stride_bytes / 8), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(stride_bytes)};
    const cuuint32_t box[2] = {box_words, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// One launch for activation rows [0, a.M) of `a` (a.M <= MT). The plan must already be known to fit.
template <int F, int MT>
static cudaError_t launch_gemv_mt(const GemvArgs &a, const G1Plan &pl, cudaStream_t st) {
    using T = T1<F, MT>;
    CUtensorMap tmc, tms;
    cudaError_t e = encode_rows(&tmc, a.packed, a.N, a.row_stride, uint32_t(T::CB / 8), uint32_t(T::TR));
    if (e != cudaSuccess) return e;
    if constexpr (T::SB > 0) {
        e = encode_rows(&tms, a.gscale, a.N, a.scale_stride * 4, uint32_t(T::SB / 8), uint32_t(T::TR));
        if (e != cudaSuccess) return e;
    } else {
        tms = tmc;
    }
    static int opted[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!opted[dev]) {
        e = cudaFuncSetAttribute(gemv1_kernel<F, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        opted[dev] = 1;
    }
    int grid = num_sms();
    if (a.N < grid) grid = int(a.N);                   // every CTA gets at least one row
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(unsigned(G1_THREADS));
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = a.weight_prefetch ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv1_kernel<F, MT>, tmc, tms, a, pl);
}

// Activation rows in groups of MT (their staged activations share one SM's shared memory with the weight ring):
// every group is one launch over the whole packed matrix.
template <int F, int MT>
static cudaError_t launch_groups(const GemvArgs &a, const G1Plan &pl, cudaStream_t st) {
    for (int m0 = 0; m0 < a.M; m0 += MT) {
        GemvArgs g = a;
        g.X = a.X + int64_t(m0) * a.ldx;
        g.Y = a.Y + int64_t(m0) * a.ldy;
        g.M = a.M - m0 < MT ? a.M - m0 : MT;
        const cudaError_t e = launch_gemv_mt<F, MT>(g, pl, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int F>
static cudaError_t launch_fmt(const GemvArgs &a, cudaStream_t s) {
    G1Plan pl;
    constexpr uint32_t BUDGET = 227u * 1024u;
    if (a.M <= 1) {
        if (!plan_gemv1<F, 1>(a, BUDGET, &pl)) return cudaErrorInvalidValue;
        return launch_gemv_mt<F, 1>(a, pl, s);
    }
    // the widest group that still leaves a ring of at least three stages
    if (a.M > 8 && plan_gemv1<F, 16>(a, BUDGET, &pl) && pl.ns >= 3) return launch_groups<F, 16>(a, pl, s);
    if (a.M > 4 && plan_gemv1<F, 8>(a, BUDGET, &pl) && pl.ns >= 3) return launch_groups<F, 8>(a, pl, s);
    if (a.M > 2 && plan_gemv1<F, 4>(a, BUDGET, &pl) && pl.ns >= 3) return launch_groups<F, 4>(a, pl, s);
    if (plan_gemv1<F, 2>(a, BUDGET, &pl)) return launch_groups<F, 2>(a, pl, s);
    // long rows of the widest formats: one row of activations per launch
    if (!plan_gemv1<F, 1>(a, BUDGET, &pl)) return cudaErrorInvalidValue;
    return launch_groups<F, 1>(a, pl, s);
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
