// qpack_gemv.cu — fused dequant-GEMV (batch 1) and small-batch GEMM (M <= 16) over packed low-bit weights.
//
// The decode-phase product is a pure stream over the packed weights: every weight byte is read from HBM once
// (2/3/5/6-bit article, lpnh.cn/news/2857666, §1.2: time per token = weight bytes / bandwidth; DBHOO-CIM
// article, pwwt.cn/news/4452170, §3.3: dequantization must stay fused, never materialised).
//
// Batch-1 kernel (gemv1_kernel<F, 1>), one persistent CTA of 16 warps per SM: 2-D TMA tensor copies of (row tile x
// K chunk) boxes of the packed rows stream into a ring of shared-memory stages (completion on mbarriers, L2
// evict-first because each byte is used once); warp w takes row class x K part of every stage, lane l one 32-weight
// unit of each chunk. Thread 0 issues the first copies; every later copy is issued by the warp that frees a stage.
// Unpacking (2/3/5/6-bit article §3.3: separate unpack from multiply-add, factor s*(q.x) + m*sum(x)) works on integers:
// each unit-row is unpacked with masks, byte permutes and shifts into eight words whose bytes each hold one code,
// possibly shifted left inside its byte by a known "bit class"; the activations are staged once per launch as 16-bit
// fixed point with a per-unit power-of-two scale, in the order the code bytes meet them. dp2a (two 16 x 8-bit
// products per instruction) accumulates exact int32 sums per class, the classes are folded with integer
// multiply-adds, and each sub-block-row needs one conversion and one fp32 FMA with its scale; the symmetric code
// offsets ride in the accumulators' start values and the asymmetric minima use per-unit activation sums. Per row,
// each warp reduces its lanes' sums with shuffles and stores one partial per K part in shared memory; the partials
// are summed in a fixed order (deterministic) before y is written.
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

constexpr uint32_t MAGIC2 = 0x64006400u;   // fp16 1024.0 in both halves
constexpr uint32_t MAGICF = 0x4B000000u;   // fp32 2^23
constexpr uint32_t HNEG1024 = 0xE400E400u; // fp16 -1024 in both halves
constexpr uint32_t HNEG1152 = 0xE480E480u; // fp16 -1152 = -(1024 + 128) in both halves

__device__ __forceinline__ uint16_t lo16(uint32_t v) { return uint16_t(v & 0xFFFFu); }
__device__ __forceinline__ uint16_t hi16(uint32_t v) { return uint16_t(v >> 16); }
__device__ __forceinline__ uint32_t lds32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ float small_int_f(uint32_t bits_or_magic) { return __uint_as_float(bits_or_magic) - 8388608.0f; }

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

// ------------------------------------------------------------------------------------------------------------
// Integer decode. A unit-row (32 weights of one row) is unpacked into eight 32-bit code words (DRow::v) whose bytes
// each hold one code, possibly shifted left inside its byte by a "bit class" p (the byte is u * 2^p). Staged word
// a = 2w + h holds the two 16-bit activations that meet byte pair h (bytes 0-1 or 2-3) of code word w; dp_elem<F>
// says which of the unit's 32 weights each one belongs to. Both bytes of a pair always share one class, so one dp2a
// adds 2^p (u0 x0 + u1 x1) to the accumulator of class p; the classes are folded with exact integer multiply-adds
// (sum_p 2^(P - p) acc_p = 2^P sum u x), converted once per sub-block-row and scaled.
// ------------------------------------------------------------------------------------------------------------
template <int F>
__host__ __device__ constexpr int dp_elem(int a, int e) {
    const int w = a >> 1, h = a & 1;
    if constexpr (kInt4<F> || F == FMT_Q5S) {
        // word 2j + p: byte b holds weight 8j + 2b + p (p = 0: the low nibbles of code word j, p = 1: the high ones)
        return 8 * (w >> 1) + (w & 1) + 4 * h + 2 * e;
    } else if constexpr (F == FMT_Q3S) {
        // sub-block s = w / 4 (3-byte groups g = 2s, 2s + 1, codes c_t, c'_t = weights 16s + t, 16s + 8 + t):
        // word 0 = (c0 c'0 | c6 c'6), 1 = (c1 c'1 | c7 c'7), 2 = (c3 c'3 | c4 c'4), 3 = (c2 c5 | c'2 c'5)
        const int k = w & 3, t = 4 * k + 2 * h + e;
        const int tab = (t == 0) ? 0 : (t == 1) ? 8 : (t == 2) ? 6 : (t == 3) ? 14 : (t == 4) ? 1 : (t == 5) ? 9
                      : (t == 6) ? 7 : (t == 7) ? 15 : (t == 8) ? 3 : (t == 9) ? 11 : (t == 10) ? 4 : (t == 11) ? 12
                      : (t == 12) ? 2 : (t == 13) ? 5 : (t == 14) ? 10 : 13;
        return 16 * (w >> 2) + tab;
    } else {
        // Q2S, Q6S: word 4s + k: byte b holds weight 16s + 4b + k
        return 16 * (w >> 2) + (w & 3) + 8 * h + 4 * e;
    }
}

// Activation constants of one 32-element unit (four floats; "int" = int32 bits). The unit is staged as two halves of
// 16 activations (weights 0-15 and 16-31 of the unit), each with its own step sigma_h (see the activation staging
// below); Sx_h = the sum of the staged integers of half h.
//   INT4 symmetric (Q4G32, Q4G32H, Q4G16), Q3S, Q6S: int -128 Sx_0, int -128 Sx_1, sigma_0 2^-P, sigma_1 2^-P
//     (P = 4, 5, 2: the bit class the folded integer sum ends at, so float(sum) * scale * c needs no other factor)
//   Q4G32A:                                          int -16 Sx_0, int -16 Sx_1, sigma_0 / 16, sigma_1 / 16
//   Q2S:                                             Sx_0 sigma_0, Sx_1 sigma_1, sigma_0, sigma_1
//   Q5S:                                             Sx_0 sigma_0 + Sx_1 sigma_1, sigma_0, sigma_1, 0
constexpr int NXC = 4;

struct DRow {
    uint32_t v[8];   // code words (see dp_elem)
    float f0, f1;    // sub-block scale factors D * L_j (Q4G32: the group scale; Q5S: f0 only)
    float g0, g1;    // minima factors Dm * M_j of the asymmetric formats (Q4G32A g0: the bits of the int32 z)
};

// ------------------------------------------------------------------------------------------------------------
// Per-lane geometry of one unit position (uc) within a K chunk: byte offsets relative to the unit's aligned code
// base, so that every row of a lane uses immediate offsets.
// ------------------------------------------------------------------------------------------------------------
struct LaneGeo {
    uint32_t ubase;      // aligned byte offset of the unit's codes within a row chunk
    int32_t o1, o2, o3;  // format-specific byte offsets relative to ubase
    uint32_t sh0, sh1;   // format-specific shifts
    uint32_t p[4], q[4]; // Q3S byte-permute selectors of the two sub-blocks (words P, Q, R, S)
};

template <int F>
__device__ __forceinline__ LaneGeo lane_geo(int uc) {
    LaneGeo g = {};
    const uint32_t sbk = uint32_t(uc) >> 3, su = uint32_t(uc) & 7u;
    if constexpr (kInt4<F>) {
        g.ubase = 16u * uc;
    } else if constexpr (F == FMT_Q2S) {
        g.ubase = 84u * sbk + 8u * su;
        g.o1 = int32_t(64u + 2u * su) - int32_t(8u * su);     // L|M bytes of the two sub-blocks
        g.o2 = int32_t(80u) - int32_t(8u * su);               // d, dmin
    } else if constexpr (F == FMT_Q3S) {
        const uint32_t a = 110u * sbk + 12u * su;             // code start, 2-byte aligned
        const uint32_t o = a & 3u;                            // 0 or 2
        g.ubase = a - o;
        g.o1 = int32_t(4u + 2u * o);                          // word pair holding the second sub-block's 6 bytes
        const uint32_t fa = 110u * sbk + 96u + 3u * (su >> 1);
        uint32_t fw = fa & ~3u, fs = 8u * (fa & 3u) + 6u * ((2u * su) & 3u);
        if (fs >= 32u) { fw += 4u; fs -= 32u; }
        g.o2 = int32_t(fw) - int32_t(g.ubase);                // word pair holding L_j0, L_j0+1 at bits fs..
        g.sh1 = fs;
        g.o3 = int32_t(110u * sbk + 108u) - int32_t(g.ubase); // d
        // bytes b0..b5 of a sub-block start at byte o (first) or 2 - o (second) of their word pair:
        // P = (b0 b3 b2 b5), Q = (b1 b4 b1 b4), R = (b0 b1 b3 b4), S = (b1 b2 b4 b5)
        const uint32_t base[4] = {0x5230u, 0x4141u, 0x4310u, 0x5421u};
#pragma unroll
        for (int i = 0; i < 4; ++i) { g.p[i] = base[i] + o * 0x1111u; g.q[i] = base[i] + (2u - o) * 0x1111u; }
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

// Q3S sub-block of two 3-byte groups (b0 b1 b2 | b3 b4 b5, code t of a group at bits 3t of its 24-bit value) from its
// word pair and the four selectors: P & 0x1C1C0707 = (c0 c'0 at bit 0 | c6 c'6 at bit 2), P & 0xE0E03838 = (c1 c'1 at
// bit 3 | c7 c'7 at bit 5), Q & 0x70700E0E = (c3 c'3 at bit 1 | c4 c'4 at bit 4); the codes c2 (bits 6..8) and c5
// (bits 15..17) straddle bytes and are shifted down from the 16-bit windows R = (b1b0 | b4b3), S = (b2b1 | b5b4).
__device__ __forceinline__ void unpack_tri_dp(uint32_t wa, uint32_t wb, const uint32_t *sel, uint32_t *v) {
    const uint32_t P = __byte_perm(wa, wb, sel[0]), Q = __byte_perm(wa, wb, sel[1]);
    const uint32_t R = __byte_perm(wa, wb, sel[2]), S = __byte_perm(wa, wb, sel[3]);
    v[0] = P & 0x1C1C0707u;
    v[1] = P & 0xE0E03838u;
    v[2] = Q & 0x70700E0Eu;
    v[3] = ((R >> 6) & 0x00070007u) | ((S << 1) & 0x07000700u);
}
// Q6S sub-block: low-4 plane words A (weights 0..7) and B (8..15), high-2 plane word H (weight 4b + k at bits 2k of
// byte b). Words k = 0..3 hold weight 4b + k in byte b: k even at bit 0 (nibble | high bits << 4), k odd at bit 2.
__device__ __forceinline__ void unpack_six_dp(uint32_t A, uint32_t B, uint32_t H, uint32_t *v) {
    const uint32_t P0 = __byte_perm(A, B, 0x6420u), P1 = __byte_perm(A, B, 0x7531u), Hs = H << 4;
    v[0] = (P0 & 0x0F0F0F0Fu) | (Hs & 0x30303030u);
    v[1] = ((P0 >> 2) & 0x3C3C3C3Cu) | (Hs & 0xC0C0C0C0u);
    v[2] = (P1 & 0x0F0F0F0Fu) | (H & 0x30303030u);
    v[3] = ((P1 >> 2) & 0x3C3C3C3Cu) | (H & 0xC0C0C0C0u);
}

// Unpack one unit-row: `u` = aligned unit base in shared memory, `sp` = this row's group-scale pointer (Q4G32);
// `on` false zeroes its scale factors (a masked lane or row). Sub-block scale integers become exact fp16 values with
// the 1024 mantissa trick and are multiplied by the raw fp16 super-block scale with exact fp16 x fp16 -> fp32 products.
template <int F>
__device__ __forceinline__ void unpack_dp(const uint8_t *u, const uint8_t *sp, const LaneGeo &g, bool on, DRow &r) {
    r.f1 = r.g0 = r.g1 = 0.f;
    if constexpr (kInt4<F>) {
        const uint4 w = *reinterpret_cast<const uint4 *>(u);
        // the unit's group scale(s) at sp: fp32 (Q4G32), fp16 (Q4G32H), two fp32 (Q4G16: weights 0-15, 16-31), or
        // the fp32 pair (s, z) (Q4G32A; z + 2^23 puts the integer z in the low mantissa bits, exactly, and z is kept
        // as an int32)
        if constexpr (F == FMT_Q4G32) {
            r.f0 = on ? *reinterpret_cast<const float *>(sp) : 0.f;
        } else if constexpr (F == FMT_Q4G32H) {
            r.f0 = on ? h2f_bits(*reinterpret_cast<const uint16_t *>(sp)) : 0.f;
        } else if constexpr (F == FMT_Q4G32A) {
            const float2 s2 = *reinterpret_cast<const float2 *>(sp);
            r.f0 = on ? s2.x : 0.f;
            r.g0 = __int_as_float(__float_as_int(__fadd_rn(s2.y, 8388608.0f)) - 0x4B000000);
        } else {
            const float2 s2 = *reinterpret_cast<const float2 *>(sp);
            r.f0 = on ? s2.x : 0.f;
            r.f1 = on ? s2.y : 0.f;
        }
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) { r.v[2 * j] = wv[j] & 0x0F0F0F0Fu; r.v[2 * j + 1] = wv[j] & 0xF0F0F0F0u; }
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
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            r.v[k] = (w0 >> (2 * k)) & 0x03030303u;
            r.v[4 + k] = (w1 >> (2 * k)) & 0x03030303u;
        }
    } else if constexpr (F == FMT_Q3S) {
        const uint32_t *wp = reinterpret_cast<const uint32_t *>(u);
        const uint32_t *qp = reinterpret_cast<const uint32_t *>(u + g.o1);
        const uint32_t *fp = reinterpret_cast<const uint32_t *>(u + g.o2);
        const uint32_t f = __funnelshift_r(fp[0], fp[1], g.sh1);          // L_j0 at bits 0..5, L_j0+1 at bits 6..11
        const uint32_t lh = hadd2_bits(lop3_and_or(lop3_sel(f << 10, f, 0xFFFF0000u), 0x003F003Fu, MAGIC2), HNEG1024);
        const uint16_t D = on ? *reinterpret_cast<const uint16_t *>(u + g.o3) : uint16_t(0);
        r.f0 = fma_h(lo16(lh), D, 0.f);
        r.f1 = fma_h(hi16(lh), D, 0.f);
        unpack_tri_dp(wp[0], wp[1], g.p, r.v);
        unpack_tri_dp(qp[0], qp[1], g.q, r.v + 4);
    } else if constexpr (F == FMT_Q5S) {
        const uint4 w = *reinterpret_cast<const uint4 *>(u);
        const uint32_t H = lds32(u + g.o1);                               // the unit's high-bit word
        const uint4 fld = *reinterpret_cast<const uint4 *>(u + g.o2);
        const uint32_t ddw = on ? fld.w : 0u;
        const float2 Dd = __half22float2(*reinterpret_cast<const __half2 *>(&ddw));
        const uint64_t lo64 = (uint64_t(fld.y) << 32) | fld.x, hi64 = (uint64_t(fld.z) << 32) | fld.y;
        const float L = small_int_f(lop3_and_or(uint32_t(lo64 >> g.sh0), 63u, MAGICF));
        const float Mv = small_int_f(lop3_and_or(uint32_t(hi64 >> (g.sh1 - 32u)), 63u, MAGICF));
        r.f0 = Dd.x * L;
        r.g0 = Dd.y * Mv;
        // word 2j (2j + 1): the even (odd) weights' nibbles of code word j with their fifth bits. hj = bit lane j of the
        // high-bit word: bit 8b + 4 = weight 8j + 2b, bit 8((b + 1) & 3) = weight 8j + 2b + 1. The even codes take
        // hj's bits 4 beside the low nibbles (one select); the odd codes take hj's bits 0 beside the high nibbles, and
        // one funnel shift by 4 (hj supplying the top bits) moves them down into whole bytes.
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t hj = (H >> j) & 0x11111111u;
            r.v[2 * j] = lop3_sel(wv[j], hj, 0x0F0F0F0Fu);
            r.v[2 * j + 1] = __funnelshift_r(lop3_sel(wv[j], hj, 0xF0F0F0F0u), hj, 4);
        }
    } else {
        const uint32_t sh = g.sh0;
        const uint32_t *wp = reinterpret_cast<const uint32_t *>(u);
        const uint32_t r0 = wp[0], r1 = wp[1], r2 = wp[2], r3 = wp[3], r4 = wp[4];
        const uint32_t *hp = reinterpret_cast<const uint32_t *>(u + g.o1);
        const uint32_t q0 = hp[0], q1 = hp[1], q2 = hp[2];
        const uint32_t lv = *reinterpret_cast<const uint16_t *>(u + g.o2);
        // int8 pair -> exact fp16 pair: (b ^ 0x80) in the mantissa of 1024, minus 1024 + 128
        const uint32_t lh = hadd2_bits(lop3_xor_or(__byte_perm(lv, 0u, 0x4140u), 0x00800080u, MAGIC2), HNEG1152);
        const uint16_t D = on ? *reinterpret_cast<const uint16_t *>(u + g.o3) : uint16_t(0);
        r.f0 = fma_h(lo16(lh), D, 0.f);
        r.f1 = fma_h(hi16(lh), D, 0.f);
        unpack_six_dp(__funnelshift_r(r0, r1, sh), __funnelshift_r(r1, r2, sh), __funnelshift_r(q0, q1, sh), r.v);
        unpack_six_dp(__funnelshift_r(r2, r3, sh), __funnelshift_r(r3, r4, sh), __funnelshift_r(q1, q2, sh), r.v + 4);
    }
}

// acc += sum_i w'_i x_i of an unpacked unit-row against one staged activation row (xv: its 16 staged words, words
// 0-7 = half 0 = weights 0-15 and words 8-15 = half 1; c: its unit constants). Every half's integer sum is converted
// once and scaled with its own sigma_h.
template <int F>
__device__ __forceinline__ void dot_dp(const DRow &r, const uint32_t *xv, const float *c, float &acc) {
    if constexpr (kInt4<F>) {
        // per half g (code words 2g, 2g + 1): lo = even weights at class 0, hi = odd weights at class 4, hi starting
        // at -128 Sx_g (the code offset 8) -> 16 lo + hi = 16 sum q x; Q4G32A starts hi at z (-16 Sx_g) -> 16 sum (u - z) x.
        // Q4G16 has one scale per half, the other INT4 formats one per unit.
        float tg[2];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            int32_t lo = 0, hi = __float_as_int(c[g]);
            if constexpr (F == FMT_Q4G32A) hi *= __float_as_int(r.g0);
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * g + jj;
                lo = dp2a_lo(xv[4 * j], r.v[2 * j], lo);
                lo = dp2a_hi(xv[4 * j + 1], r.v[2 * j], lo);
                hi = dp2a_lo(xv[4 * j + 2], r.v[2 * j + 1], hi);
                hi = dp2a_hi(xv[4 * j + 3], r.v[2 * j + 1], hi);
            }
            tg[g] = float(16 * lo + hi);
        }
        if constexpr (F == FMT_Q4G16) {
            acc = fmaf(tg[0], r.f0 * c[2], acc);
            acc = fmaf(tg[1], r.f1 * c[3], acc);
        } else {
            // one scale for the unit: sigma-weighted halves first, then the scale
            acc = fmaf(fmaf(tg[1], c[3], tg[0] * c[2]), r.f0, acc);
        }
    } else if constexpr (F == FMT_Q5S) {
        // one chain per half, every byte at class 0; the sigma-weighted halves first, then the sub-block scale
        int32_t a[2] = {0, 0};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            a[j >> 1] = dp2a_lo(xv[4 * j], r.v[2 * j], a[j >> 1]);
            a[j >> 1] = dp2a_hi(xv[4 * j + 1], r.v[2 * j], a[j >> 1]);
            a[j >> 1] = dp2a_lo(xv[4 * j + 2], r.v[2 * j + 1], a[j >> 1]);
            a[j >> 1] = dp2a_hi(xv[4 * j + 3], r.v[2 * j + 1], a[j >> 1]);
        }
        acc = fmaf(fmaf(float(a[1]), c[2], float(a[0]) * c[1]), r.f0, acc);
        acc = fmaf(-r.g0, c[0], acc);
    } else if constexpr (F == FMT_Q2S) {
        const float fs[2] = {r.f0, r.f1}, gs[2] = {r.g0, r.g1};
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            int32_t t = 0;                                      // every byte at class 0
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                t = dp2a_lo(xv[8 * s + 2 * k], r.v[4 * s + k], t);
                t = dp2a_hi(xv[8 * s + 2 * k + 1], r.v[4 * s + k], t);
            }
            acc = fmaf(float(t), fs[s] * c[2 + s], acc);
            acc = fmaf(-gs[s], c[s], acc);
        }
    } else if constexpr (F == FMT_Q3S) {
        const float fs[2] = {r.f0, r.f1};
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const uint32_t *v = r.v + 4 * s;
            const uint32_t *x = xv + 8 * s;
            // class accumulators a_p (p = bit class); a5 starts at -128 Sx_s (the code offset 4, times 32)
            int32_t a0 = dp2a_lo(x[0], v[0], 0);
            const int32_t a2 = dp2a_hi(x[1], v[0], 0);
            const int32_t a3 = dp2a_lo(x[2], v[1], 0);
            const int32_t a5 = dp2a_hi(x[3], v[1], __float_as_int(c[s]));
            const int32_t a1 = dp2a_lo(x[4], v[2], 0);
            const int32_t a4 = dp2a_hi(x[5], v[2], 0);
            a0 = dp2a_lo(x[6], v[3], a0);
            a0 = dp2a_hi(x[7], v[3], a0);
            const int32_t t = ((((a0 * 2 + a1) * 2 + a2) * 2 + a3) * 2 + a4) * 2 + a5;   // 32 sum (u - 4) x
            acc = fmaf(float(t), fs[s] * c[2 + s], acc);
        }
    } else {
        const float fs[2] = {r.f0, r.f1};
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const uint32_t *v = r.v + 4 * s;
            const uint32_t *x = xv + 8 * s;
            int32_t a0 = 0, a2 = __float_as_int(c[s]);           // classes 0 and 2; a2 starts at -128 Sx_s
            a0 = dp2a_lo(x[0], v[0], a0);
            a0 = dp2a_hi(x[1], v[0], a0);
            a2 = dp2a_lo(x[2], v[1], a2);
            a2 = dp2a_hi(x[3], v[1], a2);
            a0 = dp2a_lo(x[4], v[2], a0);
            a0 = dp2a_hi(x[5], v[2], a0);
            a2 = dp2a_lo(x[6], v[3], a2);
            a2 = dp2a_hi(x[7], v[3], a2);
            acc = fmaf(float(4 * a0 + a2), fs[s] * c[2 + s], acc);  // 4 sum (u - 32) x
        }
    }
}

// ------------------------------------------------------------------------------------------------------------
// Activation staging. A unit's 32 fp16 activations are taken as two halves of 16 (elements 0-15 and 16-31). Half h
// gets the step sigma_h = fl(m_h * fl(1/32767)), m_h = its largest |x|, and its activations become 16-bit integers
// xi = rint(x * inv_h) with inv_h = fl(1 / sigma_h), the product rounded once: fma(x, inv_h, 1.5 * 2^23) lands in
// [2^23, 2^24), where the fp32 spacing is 1, so its bits are 0x4B400000 + xi and their low 16 bits are xi as a 16-bit
// two's-complement integer (no float-to-int conversion). |xi| <= 32767 and the largest element maps to +-32767.
// Every staged value xi * sigma_h is within m_h / 65000 of x (half a step plus the fp32 roundings of sigma and of
// its reciprocal), which bounds the product error at sqrt(15) / 65000 * ||w'|| * ||x|| (the largest element of each
// half is staged exactly to 2.4e-7 relative). An all-zero half has sigma 0; a half holding an inf or a nan has
// sigma = nan, so every product it enters is nan, and the kernel reports it in the fault word. The 16 staged words are
// in dp_elem order: words 0-7 carry half 0, words 8-15 half 1.
// ------------------------------------------------------------------------------------------------------------
__device__ __forceinline__ void load_xp(const uint4 *xs, uint32_t U, uint32_t u, uint32_t xv[16]) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint4 v = xs[t * U + u];
        xv[4 * t] = v.x; xv[4 * t + 1] = v.y; xv[4 * t + 2] = v.z; xv[4 * t + 3] = v.w;
    }
}

// Largest fp16 magnitude pattern among the 16 values of two 16-byte vectors (0x7C00 or more: an inf or a nan).
__device__ __forceinline__ uint32_t half_max_bits(const uint4 &p, const uint4 &q) {
    constexpr uint32_t M = 0x7FFF7FFFu;
    const uint32_t a = __vmaxu2(__vmaxu2(p.x & M, p.y & M), __vmaxu2(p.z & M, p.w & M));
    const uint32_t b = __vmaxu2(__vmaxu2(q.x & M, q.y & M), __vmaxu2(q.z & M, q.w & M));
    const uint32_t m = __vmaxu2(a, b);
    return max(m & 0xFFFFu, m >> 16);
}

// Stage one unit (raw = its 32 fp16 values as four 16-byte vectors) into 16 words and four constants; returns true
// when the unit holds an inf or a nan.
template <int F>
__device__ __forceinline__ bool stage_regs(const uint4 (&raw)[4], uint32_t (&st)[16], float (&c)[NXC]) {
    float sg[2], inv[2];
    bool bad = false;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t mb = half_max_bits(raw[2 * h], raw[2 * h + 1]);
        const bool nf = mb >= 0x7C00u;
        bad |= nf;
        const float s = __fmul_rn(h2f_bits(uint16_t(nf ? 0u : mb)), 1.0f / 32767.0f);
        sg[h] = nf ? __int_as_float(0x7FC00000) : s;
        inv[h] = (nf || mb == 0u) ? 0.f : __frcp_rn(s);
    }
    const uint32_t hx[16] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w, raw[1].x, raw[1].y, raw[1].z, raw[1].w,
                             raw[2].x, raw[2].y, raw[2].z, raw[2].w, raw[3].x, raw[3].y, raw[3].z, raw[3].w};
    constexpr float RND = 12582912.0f;                          // 1.5 * 2^23, bits 0x4B400000
    uint32_t xb[32];                                            // 0x4B400000 + xi (a nan pattern in a non-finite half)
    uint32_t s0 = 0u - 16u * 0x4B400000u, s1 = s0;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&hx[e]));
        xb[2 * e] = __float_as_uint(fmaf(v.x, inv[e >> 3], RND));
        xb[2 * e + 1] = __float_as_uint(fmaf(v.y, inv[e >> 3], RND));
        if (e < 8) s0 += xb[2 * e] + xb[2 * e + 1]; else s1 += xb[2 * e] + xb[2 * e + 1];
    }
#pragma unroll
    for (int a = 0; a < 16; ++a) st[a] = __byte_perm(xb[dp_elem<F>(a, 0)], xb[dp_elem<F>(a, 1)], 0x5410u);
    // s0, s1 = the sums of the 16 integers of each half (exact modulo 2^32; |sum| <= 16 * 32767)
    if constexpr (F == FMT_Q2S) {
        c[0] = float(int32_t(s0)) * sg[0]; c[1] = float(int32_t(s1)) * sg[1]; c[2] = sg[0]; c[3] = sg[1];
    } else if constexpr (F == FMT_Q5S) {
        c[0] = float(int32_t(s0)) * sg[0] + float(int32_t(s1)) * sg[1]; c[1] = sg[0]; c[2] = sg[1]; c[3] = 0.f;
    } else {
        constexpr int32_t OFS = F == FMT_Q4G32A ? -16 : -128;
        constexpr float PS = kInt4<F> ? 0.0625f : F == FMT_Q3S ? 0.03125f : 0.25f;
        c[0] = __int_as_float(OFS * int32_t(s0)); c[1] = __int_as_float(OFS * int32_t(s1));
        c[2] = sg[0] * PS; c[3] = sg[1] * PS;
    }
    return bad;
}

// Staged unit u of one activation row in shared memory: its 16 words as four 16-byte vectors at vector index
// t * U + u (consecutive lanes read consecutive vectors), its constants as one 16-byte vector at cst[u].
template <int F>
__device__ __forceinline__ bool stage_unit(const uint4 (&raw)[4], uint4 *xs, float4 *cst, uint32_t U, uint32_t u) {
    uint32_t st[16];
    float c[NXC];
    const bool bad = stage_regs<F>(raw, st, c);
#pragma unroll
    for (int t = 0; t < 4; ++t) xs[t * U + u] = make_uint4(st[4 * t], st[4 * t + 1], st[4 * t + 2], st[4 * t + 3]);
    cst[u] = make_float4(c[0], c[1], c[2], c[3]);
    return bad;
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
// Thread 0 issues the first copies; every later copy is issued by the warp that releases a stage last. The 16
// warps consume every stage together: warp w handles row class rc = w / P (rows rc, rc + RC, ...: RW rows) over K
// part q = w % P of the chunk (32 units; lane l owns unit 32 q + l of every chunk).
// Every lane unpacks each of its unit-rows once (unpack_dp) and multiplies it against the MT staged activation rows
// (dot_dp), so every weight is read and unpacked once for the whole batch. Row sums accumulate over the chunks of a
// tile; then each warp reduces its lanes with shuffles and stores one partial per (row, activation row, part), and
// the P partials are summed in a fixed order (deterministic).
// ------------------------------------------------------------------------------------------------------------
constexpr int G1_CW = 16;                      // consumer warps
template <int F, int MT = 1> struct T1 {
    static constexpr int CHW = (F == FMT_Q5S || F == FMT_Q6S) ? 2048 : 4096;      // weights per K chunk
    static constexpr int UPC = CHW / 32;                                          // units per chunk
    static constexpr int P = UPC / 32;                                            // K parts of 32 units
    static constexpr int RC = G1_CW / P;                                          // row classes
    static constexpr int RW = MT > 4 ? 2 : MT > 2 ? 4 : MT == 2 ? 8 : (kInt4<F> ? 4 : (P == 4 ? 8 : 4)); // rows per warp and stage
    static constexpr int TR = RC * RW;                                            // rows per tile
    static constexpr int PR = MT > 1 ? (256 / MT > TR ? 256 / MT : TR) : 256;     // rows per partial-sum round
    static constexpr int CB = Fmt<F>::sb ? (CHW / 256) * Fmt<F>::bytes : CHW / 2; // code bytes per row chunk
    static constexpr int SE = F == FMT_Q4G32H ? 2 : 4;                            // INT4 group-scale element bytes
    static constexpr int SU = (F == FMT_Q4G16 || F == FMT_Q4G32A) ? 2 * SE : SE;  // INT4 scale bytes per 32-weight unit
    static constexpr int SB = Fmt<F>::sb ? 0 : (CHW / 32) * SU;                   // INT4 scale bytes per row chunk
    static constexpr int TX = TR * (CB + SB);                                     // bytes a stage receives
    static constexpr int STAGE = (TX + 127) / 128 * 128;
    static_assert(CB % 16 == 0 && CB / 8 <= 256 && SB / 8 <= 256, "tensor-map box limits");
    static_assert(PR % TR == 0 && RW * MT <= 32, "tile and reduction shapes");
};
constexpr int G1_THREADS = G1_CW * 32;          // 16 warps: up to 128 registers a thread
constexpr int G1_MAXNS = 16;                   // stages in the ring at most
constexpr int G1_PRE = 1;                      // shared-memory staging: fills issued before the activations are staged
constexpr int G1_PRE_XR = 1;                   // register staging, CTAs whose stages fit the ring: the same
constexpr uint32_t G1_HDR = 256;               // mbarriers and release counters

struct G1Plan {
    uint32_t off_part, off_xs, off_cst, off_xraw, off_stages, smem;
    int ns;
    int xt;   // batch 1, long streams: x arrives by one bulk copy queued ahead of the rest of the ring (see launch_split)
};

// XR = 0: the activations are staged once per CTA in shared memory (any K, any MT). XR = 1 or 2 (batch 1, rows of
// at most XR K chunks): every lane stages the units it owns (one per chunk) in its own registers straight from
// global memory, so no barrier and no shared-memory round trip stand between the activations and the first stage.
template <int F, int MT, int XR>
__global__ void __launch_bounds__(G1_THREADS, 1)
    gemv1_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_scales,
                 GemvArgs a, G1Plan pl) {
    static_assert(XR == 0 || MT == 1, "register staging is a batch-1 path");
    using T = T1<F, MT>;
    constexpr int P = T::P, RC = T::RC, RW = T::RW, TR = T::TR, CB = T::CB, SB = T::SB, UPC = T::UPC, PR = T::PR;
    constexpr uint32_t NT = G1_CW * 32;
    extern __shared__ __align__(1024) uint8_t smem_g1[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t N = uint32_t(a.N), K = uint32_t(a.K), U = K / 32;
    const uint32_t Mg = uint32_t(a.M);                     // activation rows of this launch (<= MT)
    // this CTA's rows: a contiguous range; the row counts of any two CTAs differ by at most one
    const uint32_t rq = N / gridDim.x, rm = N % gridDim.x, b = blockIdx.x;
    const uint32_t rbeg = b * rq + min(b, rm), nrows = rq + (b < rm ? 1u : 0u);
    const uint32_t nch = (U + UPC - 1) / UPC;              // K chunks per row (<= XR when XR > 0)
    const uint32_t nit = (nrows + TR - 1) / TR * nch;      // stages of this CTA: tiles x chunks
    const uint32_t NS = uint32_t(pl.ns);

    uint64_t *full = reinterpret_cast<uint64_t *>(smem_g1);                  // [NS] stage filled
    uint32_t *rel = reinterpret_cast<uint32_t *>(smem_g1 + G1_MAXNS * 8);    // [NS] warps done with the stage
    float *part = reinterpret_cast<float *>(smem_g1 + pl.off_part);
    uint4 *xs = reinterpret_cast<uint4 *>(smem_g1 + pl.off_xs);              // [MT][4][U]
    float4 *cst = reinterpret_cast<float4 *>(smem_g1 + pl.off_cst);          // [MT][U]
    uint8_t *stages = smem_g1 + pl.off_stages;
    const bool xt = XR == 0 && MT == 1 && pl.xt != 0;
    uint64_t *xbar = reinterpret_cast<uint64_t *>(smem_g1 + G1_MAXNS * 12);   // raw x landed (xt)
    const uint4 *xraw = reinterpret_cast<const uint4 *>(smem_g1 + pl.off_xraw);

    if (tid == 0) {
        for (uint32_t s = 0; s < NS; ++s) { mbar_init(&full[s], 1); rel[s] = 0; }
        if (xt) mbar_init(xbar, 1);
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
        const int ck = int(a.kc0) + int(cj);
        tma_load_2d(st, &tm_codes, ck * (CB / 8), int(rbeg + tj * TR), &full[s], pol);
        if constexpr (SB > 0) tma_load_2d(st + TR * CB, &tm_scales, ck * (SB / 8), int(rbeg + tj * TR), &full[s], pol);
    };

    // Thread 0 issues the first fills now and the rest of the ring once the activations are staged; every later
    // fill is issued by the warp that releases a stage last. Packed weights are read before the previous grid has
    // finished only when the caller opted in (QPACK_OPT_WEIGHT_PREFETCH: weights are not written by the kernel just
    // before this one). Only the first fill goes out before the activations are staged: a deeper early prefetch
    // spreads the memory system over every stage of the CTA, so the first stage lands later and delays the first
    // compute (measured with either staging: 1 early fill beats 2, 3 or the whole ring).
    // A CTA with more stages than the ring holds (long streams) fills the whole ring at once instead: there the
    // stream's rate matters more than the first stage's arrival (register staging only; the shared-memory path gets
    // the same effect from its bulk-copied activations, pl.xt).
    const uint32_t PRE = XR > 0 ? (nit > NS ? NS : uint32_t(G1_PRE_XR)) : uint32_t(G1_PRE);
    if (tid == 0) {
        if (!a.weight_prefetch) pdl_wait();
        for (uint32_t j = 0; j < nit && j < NS && j < PRE; ++j) fill(j);
        if (xt) {
            // x by one bulk copy as soon as the previous grid is done, ahead of the rest of the ring in the copy queue
            if (a.weight_prefetch) pdl_wait();
            mbar_arrive_expect_tx(xbar, K * 2u);
            bulk_g2s(const_cast<uint4 *>(xraw), a.X, K * 2u, xbar, l2_evict_last_policy());
            for (uint32_t j = PRE; j < nit && j < NS; ++j) fill(j);
        }
    }

    // -------------------------------------- consumers --------------------------------------
    const uint32_t rc = uint32_t(warp) / P, q = uint32_t(warp) % P;
    const uint32_t uc = q * 32u + uint32_t(lane);           // this lane's unit within every chunk
    pdl_wait();                  // x (and y) may belong to the previous grid
    bool xlost = false;
    constexpr int XRN = XR > 0 ? XR : 1;
    uint32_t xr[XRN][16];        // XR > 0: this lane's staged units, one per chunk
    float cr[XRN][NXC];
    if constexpr (XR > 0) {
        const uint4 *xg = reinterpret_cast<const uint4 *>(a.X);
        uint4 raw[XR][4];
#pragma unroll
        for (int cc = 0; cc < XR; ++cc) {
            const uint32_t u = uint32_t(cc) * UPC + uc;
#pragma unroll
            for (int t = 0; t < 4; ++t) raw[cc][t] = make_uint4(0u, 0u, 0u, 0u);
            if (u < U) {
#pragma unroll
                for (int t = 0; t < 4; ++t) raw[cc][t] = __ldg(xg + 4 * u + t);
            }
        }
        bool bad = false;
#pragma unroll
        for (int cc = 0; cc < XR; ++cc) bad |= stage_regs<F>(raw[cc], xr[cc], cr[cc]);
        if (bad) atomicOr(&g_fault_gemv, FAULT_NONFINITE_X);
        if (tid == 0)
            for (uint32_t j = PRE; j < nit && j < NS; ++j) fill(j);
    } else {
        if (xt) {
            if (!mbar_wait_bounded(xbar, 0u)) { xlost = true; if (tid == 0) atomicOr(&g_fault_gemv, FAULT_WAIT_FULL); }
        }
        const uint4 *xg = reinterpret_cast<const uint4 *>(a.X);
        // Thread t stages items t, t + NT, ... (item i = unit u of activation row m, i = m * U + u), each unit on its
        // own, so no unit waits for another; the loads of XD items go out before any of them is staged.
        constexpr int XD = 2;
        const uint32_t items = uint32_t(MT) * U;
        bool bad = false;
        for (uint32_t i0 = uint32_t(tid); i0 < items; i0 += XD * NT) {
            uint4 raw[XD][4];
#pragma unroll
            for (int d = 0; d < XD; ++d) {
                const uint32_t it = i0 + d * NT, m = it / U, u = it - m * U;
#pragma unroll
                for (int t = 0; t < 4; ++t) raw[d][t] = make_uint4(0u, 0u, 0u, 0u);
                if (it < items && m < Mg) {
                    if (xt) {
#pragma unroll
                        for (int t = 0; t < 4; ++t) raw[d][t] = xraw[4 * u + t];
                    } else {
                        const uint4 *xrow = xg + (int64_t(m) * a.ldx) / 8 + 4 * u;
#pragma unroll
                        for (int t = 0; t < 4; ++t) raw[d][t] = __ldg(xrow + t);
                    }
                }
            }
#pragma unroll
            for (int d = 0; d < XD; ++d) {
                const uint32_t it = i0 + d * NT, m = it / U, u = it - m * U;
                if (it < items) bad |= stage_unit<F>(raw[d], xs + m * 4 * U, cst + m * U, U, u);
            }
        }
        if (bad) atomicOr(&g_fault_gemv, FAULT_NONFINITE_X);
        // every consumer meets here: masked lanes read the last unit's staged activations, whichever part staged it
        named_bar_sync(1, G1_CW * 32);
        if (!xt && tid == 0)
            for (uint32_t j = PRE; j < nit && j < NS; ++j) fill(j);
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
            const uint8_t *sp = st + TR * CB + rc * SB + uc * T::SU;   // INT4: this lane's group scale(s) of row rc
            const uint32_t u = c * UPC + uc;
            const bool uv = u < U;
            const uint32_t uu = uv ? u : U - 1;
            const bool full_tile = rows == uint32_t(TR) && (last_full || c + 1 < nch);
            if constexpr (MT == 1) {
                uint32_t xv[16];
                float cv[NXC];
                if constexpr (XR == 1) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) xv[i] = xr[0][i];
#pragma unroll
                    for (int i = 0; i < NXC; ++i) cv[i] = cr[0][i];
                } else if constexpr (XR == 2) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) xv[i] = c ? xr[1][i] : xr[0][i];
#pragma unroll
                    for (int i = 0; i < NXC; ++i) cv[i] = c ? cr[1][i] : cr[0][i];
                } else {
                    load_xp(xs, U, uu, xv);
                    const float4 c4 = cst[uu];
                    cv[0] = c4.x; cv[1] = c4.y; cv[2] = c4.z; cv[3] = c4.w;
                }
                if (full_tile) {
#pragma unroll
                    for (int i = 0; i < RW; ++i) {
                        DRow dr;
                        unpack_dp<F>(ub + i * RC * CB, sp + i * RC * SB, geo, true, dr);
                        dot_dp<F>(dr, xv, cv, acc[i]);
                    }
                } else {
                    // ragged tile or chunk: rows past the tile's end are skipped (uniform branches), lanes past K masked
#pragma unroll
                    for (int i = 0; i < RW; ++i)
                        if (rc + uint32_t(RC * i) < rows) {
                            DRow dr;
                            unpack_dp<F>(ub + i * RC * CB, sp + i * RC * SB, geo, uv, dr);
                            dot_dp<F>(dr, xv, cv, acc[i]);
                        }
                }
            } else if constexpr (MT == 2) {
                // both activation rows stay in registers; each unit-row is unpacked once and used twice
                uint32_t xv0[16], xv1[16];
                load_xp(xs, U, uu, xv0);
                load_xp(xs + 4 * U, U, uu, xv1);
                const float4 c40 = cst[uu], c41 = cst[U + uu];
                const float cv0[NXC] = {c40.x, c40.y, c40.z, c40.w}, cv1[NXC] = {c41.x, c41.y, c41.z, c41.w};
#pragma unroll
                for (int i = 0; i < RW; ++i) {
                    if (full_tile || rc + uint32_t(RC * i) < rows) {
                        DRow ur;
                        unpack_dp<F>(ub + i * RC * CB, sp + i * RC * SB, geo, full_tile || uv, ur);
                        dot_dp<F>(ur, xv0, cv0, acc[2 * i]);
                        dot_dp<F>(ur, xv1, cv1, acc[2 * i + 1]);
                    }
                }
            } else {
                // each unit-row unpacked once, then multiplied against every activation row
                DRow ur[RW];
#pragma unroll
                for (int i = 0; i < RW; ++i)
                    unpack_dp<F>(ub + i * RC * CB, sp + i * RC * SB, geo,
                                  full_tile || (uv && rc + uint32_t(RC * i) < rows), ur[i]);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    uint32_t xv[16];
                    load_xp(xs + m * 4 * U, U, uu, xv);
                    const float4 c4 = cst[m * U + uu];
                    const float cv[NXC] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                    for (int i = 0; i < RW; ++i) dot_dp<F>(ur[i], xv, cv, acc[i * MT + m]);
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
                for (int pp = 0; pp < P; ++pp) yv += part[(r * MT + m) * P + pp];
                if (m < Mg) {
                    float *yp = a.Y + int64_t(m) * a.ldy + rbeg + base + r;
                    *yp = a.accumulate ? *yp + yv : yv;
                }
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
    if (xlost && tid == 0) mbar_wait_bounded(xbar, 0u);   // the activation copy too (xt)
}

// Shared-memory plan of one launch: returns false when two stages plus the staged activations do not fit `budget`.
// Register staging (xr) keeps no activations in shared memory.
template <int F, int MT>
static bool plan_gemv1(const GemvArgs &a, uint32_t budget, G1Plan *pl, bool xt = false, bool xr = false) {
    using T = T1<F, MT>;
    const uint32_t U = xr ? 0u : uint32_t(a.K / 32);
    pl->off_part = G1_HDR;
    pl->off_xs = pl->off_part + uint32_t(T::PR * MT * T::P * 4);
    pl->off_cst = pl->off_xs + uint32_t(round_up(int64_t(MT) * U * 64, 128));
    pl->off_xraw = uint32_t(round_up(pl->off_cst + int64_t(MT) * U * NXC * 4, 128));
    const int64_t xraw_bytes = (xt && !xr && MT == 1) ? round_up(int64_t(a.K) * 2, 128) : 0;
    pl->xt = (xt && !xr && MT == 1) ? 1 : 0;
    pl->off_stages = uint32_t(round_up(pl->off_xraw + xraw_bytes, 128));
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
template <int F, int MT, int XR>
static cudaError_t launch_gemv_mt(const GemvArgs &a, const G1Plan &pl, cudaStream_t st) {
    using T = T1<F, MT>;
    CUtensorMap tmc, tms;
    cudaError_t e = encode_rows(&tmc, a.packed, a.N, a.row_stride, uint32_t(T::CB / 8), uint32_t(T::TR));
    if (e != cudaSuccess) return e;
    if constexpr (T::SB > 0) {
        e = encode_rows(&tms, a.gscale, a.N, a.scale_stride * T::SE, uint32_t(T::SB / 8), uint32_t(T::TR));
        if (e != cudaSuccess) return e;
    } else {
        tms = tmc;
    }
    static int opted[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!opted[dev]) {
        e = cudaFuncSetAttribute(gemv1_kernel<F, MT, XR>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
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
    return cudaLaunchKernelEx(&cfg, gemv1_kernel<F, MT, XR>, tmc, tms, a, pl);
}

// All M <= MT activation rows in one group, K in splits of whole chunks: the widest split whose staged activations
// leave room for a ring of at least two stages (MT <= 2) or three (MT >= 4). Every split is one launch over its
// columns of the packed rows, so the weights are read once however long the rows are; the first split writes Y, the
// later ones add to it (stream order, so the sum over the splits is taken in a fixed order). Batch-1 rows of one
// chunk, and rows of two chunks whose CTAs' stages all fit the ring, stage their activations in registers (one
// launch); longer streams do better with the bulk-copied shared staging (measured: 70B-shaped INT4 28672x8192
// reaches 85% of HBM peak with register staging, 91% without).
template <int F, int MT>
static cudaError_t launch_split(const GemvArgs &a, cudaStream_t s) {
    constexpr uint32_t BUDGET = 227u * 1024u;
    constexpr int64_t CW = T1<F, MT>::CHW;
    const int min_ns = MT <= 2 ? 2 : 3;
    const int64_t nchunks = (a.K + CW - 1) / CW;
    if constexpr (MT == 1) {
        if (nchunks <= 2) {
            G1Plan pl;
            GemvArgs h = a;
            h.kc0 = 0;
            h.accumulate = 0;
            if (!plan_gemv1<F, MT>(h, BUDGET, &pl, false, true)) return cudaErrorInvalidValue;
            using T = T1<F, MT>;
            const int64_t grid = num_sms() < h.N ? num_sms() : h.N;
            const int64_t nit = (((h.N + grid - 1) / grid) + T::TR - 1) / T::TR * nchunks;
            if (nchunks == 1) return launch_gemv_mt<F, MT, 1>(h, pl, s);
            if (nit <= pl.ns) return launch_gemv_mt<F, MT, 2>(h, pl, s);
        }
    }
    for (int64_t parts = 1; parts <= nchunks; ++parts) {
        const int64_t ks = (nchunks + parts - 1) / parts * CW;
        GemvArgs g = a;
        g.K = ks < a.K ? ks : a.K;
        G1Plan pl;
        if (!plan_gemv1<F, MT>(g, BUDGET, &pl) || (pl.ns < min_ns && parts < nchunks)) continue;
        for (int64_t k0 = 0; k0 < a.K; k0 += ks) {
            GemvArgs h = a;
            h.K = ks < a.K - k0 ? ks : a.K - k0;
            h.X = a.X + k0;
            h.kc0 = k0 / CW;
            h.accumulate = k0 > 0 ? 1 : 0;
            if (!plan_gemv1<F, MT>(h, BUDGET, &pl)) return cudaErrorInvalidValue;
            if constexpr (MT == 1) {
                // Batch 1 with more stages per CTA than the ring holds: x by a bulk copy queued right behind the first
                // fill and the whole ring filled at once beats staging x first (measured; with a ring that holds all
                // of a CTA's stages the early fills only delay x, and a raw x buffer that costs the ring stages
                // below four loses more than it gains).
                using T = T1<F, MT>;
                const int64_t grid = num_sms() < h.N ? num_sms() : h.N;
                const int64_t rows = (h.N + grid - 1) / grid;
                const int64_t nit = (rows + T::TR - 1) / T::TR * ((h.K + T::CHW - 1) / T::CHW);
                G1Plan px;
                if (plan_gemv1<F, MT>(h, BUDGET, &px, true) && nit > px.ns && px.ns >= (pl.ns < 4 ? pl.ns : 4)) pl = px;
            }
            const cudaError_t e = launch_gemv_mt<F, MT, 0>(h, pl, s);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    return cudaErrorInvalidValue;
}

template <int F>
static cudaError_t launch_fmt(const GemvArgs &a, cudaStream_t s) {
    if (a.M <= 1) return launch_split<F, 1>(a, s);
    if (a.M <= 2) return launch_split<F, 2>(a, s);
    if (a.M <= 4) return launch_split<F, 4>(a, s);
    if (a.M <= 8) return launch_split<F, 8>(a, s);
    return launch_split<F, 16>(a, s);
}

cudaError_t launch_gemv(int fmt, const GemvArgs &a, cudaStream_t s) {
    switch (fmt) {
        case FMT_Q4G32: return launch_fmt<FMT_Q4G32>(a, s);
        case FMT_Q4G32H: return launch_fmt<FMT_Q4G32H>(a, s);
        case FMT_Q4G16: return launch_fmt<FMT_Q4G16>(a, s);
        case FMT_Q4G32A: return launch_fmt<FMT_Q4G32A>(a, s);
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
