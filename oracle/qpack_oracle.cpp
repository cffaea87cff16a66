// qpack oracle — TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, obviously correct CPU implementation of what the qpack hot path computes: the five weight
// formats' quantizers, bit packing and unpacking, dequantization, and fp64-accumulated matrix-vector /
// matrix-matrix products. It exists so that tests and the benchmark's CPU-baseline leg can check and time
// the CUDA kernels. Nothing in the product path may call it; it shares no code, header or table with the
// CUDA sources.
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -fPIC -shared (no -ffast-math; default rounding mode, so
// std::nearbyint rounds half to even).
//
// Sources. P1 = the 2/3/5/6-bit quantization article (lpnh.cn/news/2857666); P2 = the DBHOO-CIM INT4 CPU
// inference article (pwwt.cn/news/4452170). Where a page leaves a choice open, the comment of the function that
// makes the choice states the reading it follows.
//
// Pins: every function is pinned by tests under tests/ that do not re-derive it from itself (hand-computed
// fixtures, exact lattices, one-hot products, exhaustive converter checks, round trips).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ----------------------------------------------------------------------------------------------------------
// fp16 / bf16 <-> fp32, round-to-nearest-even, written out bit by bit from the IEEE 754 binary16 definition.
// ----------------------------------------------------------------------------------------------------------

uint32_t f32_bits(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }
float bits_f32(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }

// Round-to-nearest-even of an unsigned integer `v` shifted right by `s` bits (s >= 1).
uint64_t shift_rne(uint64_t v, int s) {
    if (s >= 64) return 0;
    uint64_t q = v >> s;
    uint64_t rem = v - (q << s);
    uint64_t half = uint64_t(1) << (s - 1);
    if (rem > half || (rem == half && (q & 1))) q += 1;
    return q;
}

uint16_t f32_to_f16(float f) {
    uint32_t x = f32_bits(f);
    uint16_t sign = uint16_t((x >> 16) & 0x8000u);
    uint32_t exp = (x >> 23) & 0xFFu;
    uint32_t man = x & 0x7FFFFFu;
    if (exp == 0xFF) {                       // inf or NaN
        if (man == 0) return uint16_t(sign | 0x7C00u);
        return uint16_t(sign | 0x7E00u | (man >> 13));   // quiet NaN, keep top payload bits
    }
    if (exp == 0 && man == 0) return sign;   // signed zero
    // value = m * 2^(e) with m an integer mantissa
    int e;            // unbiased exponent of the leading bit
    uint64_t m;       // 24-bit significand (with hidden bit) for normals
    if (exp == 0) {   // fp32 subnormal: far below fp16 range, rounds to zero
        return sign;
    }
    e = int(exp) - 127;
    m = (uint64_t(1) << 23) | man;           // value = m * 2^(e - 23)
    if (e > 15) return uint16_t(sign | 0x7C00u);          // overflow to inf (|v| >= 2^16)
    if (e >= -14) {
        // fp16 normal range: keep 10 fraction bits -> shift by 13
        uint64_t r = shift_rne(m, 13);       // r in [2^10, 2^11]
        int he = e + 15;
        if (r == (uint64_t(1) << 11)) { r >>= 1; he += 1; }
        if (he >= 31) return uint16_t(sign | 0x7C00u);
        return uint16_t(sign | (uint16_t(he) << 10) | uint16_t(r & 0x3FFu));
    }
    // fp16 subnormal: value = r * 2^-24 with r = round(m * 2^(e - 23 + 24))
    int s = 13 + (-14 - e);                  // shift so that units are 2^-24
    uint64_t r = shift_rne(m, s);            // r in [0, 2^10]
    // r == 2^10 becomes the smallest normal, which the bit pattern encodes naturally.
    return uint16_t(sign | uint16_t(r));
}

float f16_to_f32(uint16_t h) {
    uint32_t sign = uint32_t(h & 0x8000u) << 16;
    uint32_t exp = (h >> 10) & 0x1Fu;
    uint32_t man = h & 0x3FFu;
    if (exp == 0x1F) return bits_f32(sign | 0x7F800000u | (man << 13));
    if (exp == 0) {
        // subnormal or zero: man * 2^-24, exact in fp32
        float v = float(man) * std::ldexp(1.0f, -24);
        return sign ? -v : v;
    }
    return bits_f32(sign | ((exp - 15 + 127) << 23) | (man << 13));
}

uint16_t f32_to_bf16(float f) {
    uint32_t x = f32_bits(f);
    if ((x & 0x7F800000u) == 0x7F800000u && (x & 0x7FFFFFu)) return uint16_t((x >> 16) | 0x40u);  // NaN
    uint32_t lower = x & 0xFFFFu;
    uint32_t upper = x >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;   // carries into exp: correct
    return uint16_t(upper);
}

float bf16_to_f32(uint16_t b) { return bits_f32(uint32_t(b) << 16); }

// ----------------------------------------------------------------------------------------------------------
// Format descriptions (P1 §2.3 byte table; P2 §3.2 / §4.1 for INT4).
// ----------------------------------------------------------------------------------------------------------

enum { Q4G32 = 0, Q2S = 1, Q3S = 2, Q5S = 3, Q6S = 4, Q4G32H = 5, Q4G16 = 6, Q4G32A = 7 };

// Weights per INT4 group: 32, or 16 for Q4G16.
int int4_group(int fmt) { return fmt == Q4G16 ? 16 : 32; }
bool is_int4(int fmt) { return fmt == Q4G32 || fmt == Q4G32H || fmt == Q4G16 || fmt == Q4G32A; }

struct SbFormat {
    int bits;      // code width b
    int nsub;      // sub-blocks per super-block
    int sublen;    // weights per sub-block
    int lmax;      // largest sub-scale integer
    bool asym;     // has a minimum (dmin, M_j)
    int bytes;     // bytes per 256-weight super-block
};

bool sb_format(int fmt, SbFormat *f) {
    switch (fmt) {
        case Q2S: *f = {2, 16, 16, 15, true, 84}; return true;
        case Q3S: *f = {3, 16, 16, 63, false, 110}; return true;
        case Q5S: *f = {5, 8, 32, 63, true, 176}; return true;
        case Q6S: *f = {6, 16, 16, 127, false, 210}; return true;
        default: return false;
    }
}

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

float clampf(float v, float lo, float hi) { return v < lo ? lo : (v > hi ? hi : v); }

// ----------------------------------------------------------------------------------------------------------
// Bit runs. Every packed field of the super-block formats (P1 §2.2 cross-byte codes, §2.3 bit planes and sub-block
// scale fields) is a "run": consecutive fields of one width w laid end to end in a little-endian bit string, field
// i taking bits w*i .. w*i + w - 1, where bit b of the string is bit (b mod 8) of byte b / 8 (least significant bit
// first). The two functions below move one field in or out bit by bit through that global bit index; the format
// layouts further down are nothing but (run start, width, field index) triples.
// ----------------------------------------------------------------------------------------------------------

void run_put(uint8_t *run, int w, int64_t i, uint32_t v) {
    for (int k = 0; k < w; ++k) {
        const int64_t b = int64_t(w) * i + k;                 // global bit index of bit k of field i
        const uint8_t bit = uint8_t(1u << (b % 8));
        if ((v >> k) & 1u) run[b / 8] |= bit; else run[b / 8] &= uint8_t(~bit);
    }
}
uint32_t run_get(const uint8_t *run, int w, int64_t i) {
    uint32_t v = 0;
    for (int k = 0; k < w; ++k) {
        const int64_t b = int64_t(w) * i + k;
        v |= uint32_t((run[b / 8] >> (b % 8)) & 1u) << k;
    }
    return v;
}

uint16_t rd16(const uint8_t *p) { return uint16_t(p[0] | (p[1] << 8)); }
void wr16(uint8_t *p, uint16_t v) { p[0] = uint8_t(v); p[1] = uint8_t(v >> 8); }

// ----------------------------------------------------------------------------------------------------------
// Quantizers.
// ----------------------------------------------------------------------------------------------------------

// INT4 symmetric group quantizer, P2 §3.1: scale = max|w| / 8 floored at 1e-12, q = clamp(round(w/scale),-8,7).
// P2 §3.1 for a group of G weights (G = 32; G = 16 is P2 §5.1's remedy for layers with many outlier weights).
void quantize_int4_row(const float *w, int64_t K, int G, int8_t *q, float *scales) {
    for (int64_t g = 0; g < K / G; ++g) {
        const float *wg = w + G * g;
        float amax = 0.0f;
        for (int i = 0; i < G; ++i) amax = std::fmax(amax, std::fabs(wg[i]));
        float scale = amax / 8.0f;
        if (scale < 1e-12f) scale = 1e-12f;
        for (int i = 0; i < G; ++i) {
            float t = std::nearbyint(wg[i] / scale);
            q[G * g + i] = int8_t(clampf(t, -8.0f, 7.0f));
        }
        scales[g] = scale;
    }
}

// INT4 group-32 with an fp16 group scale (P1 §2.1: an fp16 scale per 32 weights costs 0.5 bpw, so 4.5 bpw). Reading
// (the P2 rule with the scale stored in fp16, used rounded as the super-block formats use d): s = max|w| / 8 in
// fp32, s16 = fp16(s), D = s16 as fp32; q = D > 0 ? clamp(rint(w / D), -8, 7) : 0 (no 1e-12 floor: a scale that
// rounds to 0 gives zero codes). Returns the RANGE flag if s16 overflows.
int quantize_q4g32h_row(const float *w, int64_t K, int8_t *q, uint16_t *scales) {
    int flags = 0;
    for (int64_t g = 0; g < K / 32; ++g) {
        const float *wg = w + 32 * g;
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) amax = std::fmax(amax, std::fabs(wg[i]));
        const uint16_t s16 = f32_to_f16(amax / 8.0f);
        const float D = f16_to_f32(s16);
        if ((s16 & 0x7FFFu) == 0x7C00u) flags |= 1;
        for (int i = 0; i < 32; ++i) {
            float t = 0.0f;
            if (D > 0.0f) t = clampf(std::nearbyint(wg[i] / D), -8.0f, 7.0f);
            q[32 * g + i] = int8_t(t);
        }
        scales[g] = s16;
    }
    return flags;
}

// Asymmetric INT4, group 32 (P2 §5.1: a layer whose weight maxima stand out gets asymmetric quantization). P1 §2.1
// defines the asymmetric form: q = rint(w / s) + z, w' = s * (q - z), with an integer zero point z. Reading (the
// pages give no rule for s and z): the group range widened to contain 0, lo = min(0, min w), hi = max(0, max w);
// s = max((hi - lo) / 15, 1e-12f) (the floor of P2's symmetric rule); z = clamp(rint(-lo / s), 0, 15);
// q = clamp(rint(w / s) + z, 0, 15); dequant w' = s * (float)(q - z), so a zero weight comes back exactly as 0.
// The group's pair goes to sm[2g] = s, sm[2g + 1] = (float)z.
void quantize_q4g32a_row(const float *w, int64_t K, int8_t *q, float *sm) {
    for (int64_t g = 0; g < K / 32; ++g) {
        const float *wg = w + 32 * g;
        float lo = 0.0f, hi = 0.0f;
        for (int i = 0; i < 32; ++i) {
            lo = std::fmin(lo, wg[i]);
            hi = std::fmax(hi, wg[i]);
        }
        float s = (hi - lo) / 15.0f;
        if (s < 1e-12f) s = 1e-12f;
        const int z = int(clampf(std::nearbyint(-lo / s), 0.0f, 15.0f));
        for (int i = 0; i < 32; ++i)
            q[32 * g + i] = int8_t(clampf(std::nearbyint(wg[i] / s) + float(z), 0.0f, 15.0f));
        sm[2 * g] = s;
        sm[2 * g + 1] = float(z);
    }
}

// Two-level round-to-nearest super-block quantizer (P1 §2.1: fp16 super-block scale, then low-bit sub-block
// scales, then the weights; byte budget from P1 §2.3). The pages print no algorithm for it. Reading: each
// sub-block's own scale s_j (symmetric: max |w| / 2^(b-1); asymmetric: (max w - min(0, min w)) / (2^b - 1), with
// minimum m_j = 0 - min(0, min w)); d = fp16(max_j s_j / Lmax) (dmin likewise from the m_j), used rounded; the
// sub-block integers L_j = clamp(rint(s_j / d), 0, Lmax) (M_j likewise); the codes against the rounded sub-block
// scale e = d * L_j: symmetric clamp(rint(w / e), -2^(b-1), 2^(b-1) - 1), asymmetric clamp(rint((w + dmin * M_j) / e),
// 0, 2^b - 1); a zero scale gives zero integers. Returns the RANGE flag if fp16(d) or fp16(dmin) overflows.
int quantize_sb_row(const SbFormat &F, const float *w, int64_t K, int8_t *q, uint8_t *sub_scale,
                    uint8_t *sub_min, uint16_t *d_out, uint16_t *dmin_out) {
    int flags = 0;
    const int64_t nb = K / 256;
    for (int64_t b = 0; b < nb; ++b) {
        const float *ws = w + 256 * b;
        float s[16], m[16];
        if (!F.asym) {
            const float half_range = float(1 << (F.bits - 1));           // 2^(b-1)
            for (int j = 0; j < F.nsub; ++j) {
                float amax = 0.0f;
                for (int i = 0; i < F.sublen; ++i) amax = std::fmax(amax, std::fabs(ws[j * F.sublen + i]));
                s[j] = amax / half_range;
            }
            float smax = 0.0f;
            for (int j = 0; j < F.nsub; ++j) smax = std::fmax(smax, s[j]);
            float d = smax / float(F.lmax);
            uint16_t d16 = f32_to_f16(d);
            if ((d16 & 0x7FFFu) == 0x7C00u) flags |= 1;
            float D = f16_to_f32(d16);
            d_out[b] = d16;
            for (int j = 0; j < F.nsub; ++j) {
                float L = 0.0f;
                if (D > 0.0f) L = clampf(std::nearbyint(s[j] / D), 0.0f, float(F.lmax));
                sub_scale[b * F.nsub + j] = uint8_t(int(L));
                float e = D * L;
                for (int i = 0; i < F.sublen; ++i) {
                    float t = 0.0f;
                    if (e > 0.0f) t = clampf(std::nearbyint(ws[j * F.sublen + i] / e), -half_range, half_range - 1.0f);
                    q[256 * b + j * F.sublen + i] = int8_t(t);
                }
            }
        } else {
            const float levels = float((1 << F.bits) - 1);                // 2^b - 1
            for (int j = 0; j < F.nsub; ++j) {
                float lo = 0.0f, hi = -INFINITY;
                for (int i = 0; i < F.sublen; ++i) {
                    float v = ws[j * F.sublen + i];
                    lo = std::fmin(lo, v);
                    hi = std::fmax(hi, v);
                }
                s[j] = (hi - lo) / levels;
                m[j] = 0.0f - lo;          // -lo, written as a subtraction so that it is never -0
            }
            float smax = 0.0f, mmax = 0.0f;
            for (int j = 0; j < F.nsub; ++j) { smax = std::fmax(smax, s[j]); mmax = std::fmax(mmax, m[j]); }
            float d = smax / float(F.lmax);
            float dmin = mmax / float(F.lmax);
            uint16_t d16 = f32_to_f16(d), dm16 = f32_to_f16(dmin);
            if ((d16 & 0x7FFFu) == 0x7C00u || (dm16 & 0x7FFFu) == 0x7C00u) flags |= 1;
            float D = f16_to_f32(d16), Dm = f16_to_f32(dm16);
            d_out[b] = d16;
            dmin_out[b] = dm16;
            for (int j = 0; j < F.nsub; ++j) {
                float L = 0.0f, M = 0.0f;
                if (D > 0.0f) L = clampf(std::nearbyint(s[j] / D), 0.0f, float(F.lmax));
                if (Dm > 0.0f) M = clampf(std::nearbyint(m[j] / Dm), 0.0f, float(F.lmax));
                sub_scale[b * F.nsub + j] = uint8_t(int(L));
                sub_min[b * F.nsub + j] = uint8_t(int(M));
                float es = D * L;
                float em = Dm * M;
                for (int i = 0; i < F.sublen; ++i) {
                    float t = 0.0f;
                    if (es > 0.0f) {
                        float shifted = ws[j * F.sublen + i] + em;
                        t = clampf(std::nearbyint(shifted / es), 0.0f, levels);
                    }
                    q[256 * b + j * F.sublen + i] = int8_t(t);
                }
            }
        }
    }
    return flags;
}

// ----------------------------------------------------------------------------------------------------------
// Packing and unpacking of one super-block (P1 §2.2 / §2.3; bit orders little-endian, weight i at the lowest free
// bit, as each function states) and of one INT4 row (P2 §3.2).
// ----------------------------------------------------------------------------------------------------------

// Layouts: Q2S codes = run of 2-bit fields at byte 0, sub-block nibbles L_j, M_j = fields 2j, 2j + 1 of a 4-bit run
// at byte 64, d at 80, dmin at 82. Q3S codes (offset q + 4) = 3-bit run at 0 (so a 3-byte group holds 8 codes,
// P1 §2.2), L_j = 6-bit run at 96 (four fields per 3 bytes), d at 108. Q5S low nibbles = 4-bit run at 0, fifth bits
// = 1-bit run at 128 in the order q5s_hbit gives, fields L_0..7, M_0..7 = 6-bit run at 160, d at 172, dmin at 174.
// Q6S (offset q + 32) low nibbles = 4-bit run at 0, top two bits = 2-bit run at 128, int8 L_j at 192, d at 208.
// fp16 values are stored little-endian.

// Position, in the Q5S high-bit run (P1 §2.3 gives it 32 B and no bit order), of the fifth bit of weight i. The run
// is read as one 32-bit little-endian word per 32 weights; weight 32c + 8j + 2b + e (j, b in 0..3, e in 0..1) takes
// bit 8b + 4 + j of word c when e = 0 and bit 8((b + 1) mod 4) + j when e = 1. Every bit of the word is used once.
int64_t q5s_hbit(int64_t i) {
    const int64_t c = i >> 5;
    const int t = int(i & 31), j = t >> 3, b = (t >> 1) & 3, e = t & 1;
    return 32 * c + (e == 0 ? 8 * b + 4 + j : 8 * ((b + 1) & 3) + j);
}
void pack_sb(int fmt, const int8_t *q, const uint8_t *L, const uint8_t *M, uint16_t d, uint16_t dmin, uint8_t *p) {
    SbFormat F;
    sb_format(fmt, &F);
    std::memset(p, 0, size_t(F.bytes));
    switch (fmt) {
        case Q2S:
            for (int i = 0; i < 256; ++i) run_put(p, 2, i, uint8_t(q[i]));
            for (int j = 0; j < 16; ++j) { run_put(p + 64, 4, 2 * j, L[j]); run_put(p + 64, 4, 2 * j + 1, M[j]); }
            wr16(p + 80, d); wr16(p + 82, dmin);
            break;
        case Q3S:
            for (int i = 0; i < 256; ++i) run_put(p, 3, i, uint32_t(q[i] + 4));
            for (int j = 0; j < 16; ++j) run_put(p + 96, 6, j, L[j]);
            wr16(p + 108, d);
            break;
        case Q5S:
            for (int i = 0; i < 256; ++i) {
                const uint32_t u = uint8_t(q[i]);
                run_put(p, 4, i, u % 16);
                run_put(p + 128, 1, q5s_hbit(i), u / 16);
            }
            for (int j = 0; j < 8; ++j) { run_put(p + 160, 6, j, L[j]); run_put(p + 160, 6, 8 + j, M[j]); }
            wr16(p + 172, d); wr16(p + 174, dmin);
            break;
        case Q6S:
            for (int i = 0; i < 256; ++i) {
                const uint32_t u = uint32_t(q[i] + 32);
                run_put(p, 4, i, u % 16);
                run_put(p + 128, 2, i, u / 16);
            }
            for (int j = 0; j < 16; ++j) p[192 + j] = L[j];
            wr16(p + 208, d);
            break;
    }
}

void unpack_sb(int fmt, const uint8_t *p, int8_t *q, uint8_t *L, uint8_t *M, uint16_t *d, uint16_t *dmin) {
    switch (fmt) {
        case Q2S:
            for (int i = 0; i < 256; ++i) q[i] = int8_t(run_get(p, 2, i));
            for (int j = 0; j < 16; ++j) { L[j] = uint8_t(run_get(p + 64, 4, 2 * j)); M[j] = uint8_t(run_get(p + 64, 4, 2 * j + 1)); }
            *d = rd16(p + 80); *dmin = rd16(p + 82);
            break;
        case Q3S:
            for (int i = 0; i < 256; ++i) q[i] = int8_t(int(run_get(p, 3, i)) - 4);
            for (int j = 0; j < 16; ++j) L[j] = uint8_t(run_get(p + 96, 6, j));
            *d = rd16(p + 108);
            break;
        case Q5S:
            for (int i = 0; i < 256; ++i) q[i] = int8_t(run_get(p, 4, i) + 16 * run_get(p + 128, 1, q5s_hbit(i)));
            for (int j = 0; j < 8; ++j) { L[j] = uint8_t(run_get(p + 160, 6, j)); M[j] = uint8_t(run_get(p + 160, 6, 8 + j)); }
            *d = rd16(p + 172); *dmin = rd16(p + 174);
            break;
        case Q6S:
            for (int i = 0; i < 256; ++i) q[i] = int8_t(int(run_get(p, 4, i) + 16 * run_get(p + 128, 2, i)) - 32);
            for (int j = 0; j < 16; ++j) L[j] = p[192 + j];
            *d = rd16(p + 208);
            break;
    }
}

// Dequantize one super-block from its unpacked parts: w' = (d * L_j) * q (symmetric) or (d * L_j) * q - dmin * M_j
// (asymmetric), each product and difference an fp32 rounding, no FMA.
void dequant_sb(const SbFormat &F, int fmt, const int8_t *q, const uint8_t *L, const uint8_t *M, uint16_t d,
                uint16_t dmin, float *out) {
    float D = f16_to_f32(d);
    float Dm = F.asym ? f16_to_f32(dmin) : 0.0f;
    for (int j = 0; j < F.nsub; ++j) {
        // Q6S sub-scales are int8; the others are unsigned fields.
        float Lj = (fmt == Q6S) ? float(int8_t(L[j])) : float(L[j]);
        float es = D * Lj;
        float em = F.asym ? Dm * float(M[j]) : 0.0f;
        for (int i = 0; i < F.sublen; ++i) {
            float v = es * float(q[j * F.sublen + i]);
            if (F.asym) v = v - em;
            out[j * F.sublen + i] = v;
        }
    }
}

// Dequantize row r of a packed matrix into out[K].
void dequant_row(int fmt, const uint8_t *packed, const float *gs, int64_t K, int64_t r, int64_t row_stride,
                 int64_t scale_stride, float *out) {
    if (is_int4(fmt)) {
        const uint8_t *row = packed + r * row_stride;
        const uint16_t *gs16 = reinterpret_cast<const uint16_t *>(gs);
        const int G = int4_group(fmt);
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = row[k >> 1];
            int u = (k & 1) ? (byte >> 4) : (byte & 15);
            if (fmt == Q4G32A) {
                const float s = gs[r * scale_stride + 2 * (k / 32)];
                const int z = int(gs[r * scale_stride + 2 * (k / 32) + 1]);
                out[k] = s * float(u - z);
                continue;
            }
            float s = fmt == Q4G32H ? f16_to_f32(gs16[r * scale_stride + k / G]) : gs[r * scale_stride + k / G];
            out[k] = s * float(u - 8);
        }
        return;
    }
    SbFormat F;
    sb_format(fmt, &F);
    const uint8_t *row = packed + r * row_stride;
    for (int64_t b = 0; b < K / 256; ++b) {
        int8_t q[256]; uint8_t L[16], M[16] = {0}; uint16_t d = 0, dmin = 0;
        unpack_sb(fmt, row + b * F.bytes, q, L, M, &d, &dmin);
        dequant_sb(F, fmt, q, L, M, d, dmin, out + 256 * b);
    }
}

bool shape_ok(int fmt, int64_t N, int64_t K) {
    if (N < 0 || K < 0) return false;
    if (is_int4(fmt)) return K % 32 == 0;   // Q4G16 too: rows of whole 32-weight units
    SbFormat F;
    if (!sb_format(fmt, &F)) return false;
    return K % 256 == 0;
}

}  // namespace

extern "C" {

// ---- converters (exported for the exhaustive converter pins) ----
void orc_f32_to_f16(const float *x, uint16_t *y, int64_t n) { for (int64_t i = 0; i < n; ++i) y[i] = f32_to_f16(x[i]); }
void orc_f16_to_f32(const uint16_t *x, float *y, int64_t n) { for (int64_t i = 0; i < n; ++i) y[i] = f16_to_f32(x[i]); }
void orc_f32_to_bf16(const float *x, uint16_t *y, int64_t n) { for (int64_t i = 0; i < n; ++i) y[i] = f32_to_bf16(x[i]); }
void orc_bf16_to_f32(const uint16_t *x, float *y, int64_t n) { for (int64_t i = 0; i < n; ++i) y[i] = bf16_to_f32(x[i]); }

// ---- bit runs (P1 §2.2), exported for the round-trip pins: n fields of width w ----
void orc_run_pack(const uint8_t *f, int w, int64_t n, uint8_t *p) {
    std::memset(p, 0, size_t((int64_t(w) * n + 7) / 8));
    for (int64_t i = 0; i < n; ++i) run_put(p, w, i, f[i]);
}
void orc_run_unpack(const uint8_t *p, int w, int64_t n, uint8_t *f) {
    for (int64_t i = 0; i < n; ++i) f[i] = uint8_t(run_get(p, w, i));
}

// Layout: out[0] = packed row stride (bytes), out[1] = packed bytes, out[2] = INT4 scale row stride (elements:
// fp32 for Q4G32, fp16 for Q4G32H, rows padded to 16 bytes; 0 otherwise), out[3] = INT4 scale bytes (0
// otherwise), out[4] = super-block bytes (0 for the INT4 formats).
// Returns 0, or -2 for a shape the format does not accept.
int orc_layout(int fmt, int64_t N, int64_t K, int64_t *out) {
    if (!shape_ok(fmt, N, K)) return -2;
    if (fmt == Q4G32) {
        out[0] = K / 2;
        out[1] = N * (K / 2);
        out[2] = round_up(K / 32, 4);
        out[3] = N * out[2] * 4;
        out[4] = 0;
        return 0;
    }
    if (fmt == Q4G32H) {
        out[0] = K / 2;
        out[1] = N * (K / 2);
        out[2] = round_up(K / 32, 8);
        out[3] = N * out[2] * 2;
        out[4] = 0;
        return 0;
    }
    if (fmt == Q4G16 || fmt == Q4G32A) {     // Q4G32A: one (scale, zero point) fp32 pair per 32-group
        out[0] = K / 2;
        out[1] = N * (K / 2);
        out[2] = round_up(K / 16, 4);
        out[3] = N * out[2] * 4;
        out[4] = 0;
        return 0;
    }
    SbFormat F;
    sb_format(fmt, &F);
    out[0] = round_up((K / 256) * F.bytes, 16);
    out[1] = N * out[0];
    out[2] = 0;
    out[3] = 0;
    out[4] = F.bytes;
    return 0;
}

// Quantize W (fp32, [N][K]) into unpacked parts. Q4G32 writes q and gscale [N][K/32]; Q4G32H writes q and its
// fp16 group scales into d [N][K/32]; super-block formats
// write q, sub_scale [N][nb*nsub], sub_min (asymmetric only), d and dmin [N][nb]. Returns flags (1 = RANGE)
// or -2 for a bad shape.
int orc_quantize(int fmt, const float *W, int64_t N, int64_t K, int8_t *q, float *gscale, uint8_t *sub_scale,
                 uint8_t *sub_min, uint16_t *d, uint16_t *dmin) {
    if (!shape_ok(fmt, N, K)) return -2;
    int flags = 0;
    if (fmt == Q4G32) {
        for (int64_t r = 0; r < N; ++r) quantize_int4_row(W + r * K, K, 32, q + r * K, gscale + r * (K / 32));
        return 0;
    }
    if (fmt == Q4G16) {
        for (int64_t r = 0; r < N; ++r) quantize_int4_row(W + r * K, K, 16, q + r * K, gscale + r * (K / 16));
        return 0;
    }
    if (fmt == Q4G32A) {
        for (int64_t r = 0; r < N; ++r) quantize_q4g32a_row(W + r * K, K, q + r * K, gscale + r * (K / 16));
        return 0;
    }
    if (fmt == Q4G32H) {
        for (int64_t r = 0; r < N; ++r) flags |= quantize_q4g32h_row(W + r * K, K, q + r * K, d + r * (K / 32));
        return flags;
    }
    SbFormat F;
    sb_format(fmt, &F);
    const int64_t nb = K / 256;
    for (int64_t r = 0; r < N; ++r)
        flags |= quantize_sb_row(F, W + r * K, K, q + r * K, sub_scale + r * nb * F.nsub,
                                 F.asym ? sub_min + r * nb * F.nsub : nullptr, d + r * nb,
                                 F.asym ? dmin + r * nb : nullptr);
    return flags;
}

// Pack unpacked parts into the format's bytes (and the padded Q4G32 scale array).
int orc_pack(int fmt, int64_t N, int64_t K, const int8_t *q, const float *gscale, const uint8_t *sub_scale,
             const uint8_t *sub_min, const uint16_t *d, const uint16_t *dmin, uint8_t *packed, float *group_scales) {
    int64_t lay[5];
    if (orc_layout(fmt, N, K, lay)) return -2;
    std::memset(packed, 0, size_t(lay[1]));
    if (is_int4(fmt)) {
        uint16_t *gs16 = reinterpret_cast<uint16_t *>(group_scales);
        const int64_t ng = fmt == Q4G32A ? K / 16 : K / int4_group(fmt);   // scale-array entries per row
        const int off = fmt == Q4G32A ? 0 : 8;                              // stored nibble u = q + off
        for (int64_t r = 0; r < N; ++r) {
            uint8_t *row = packed + r * lay[0];
            for (int64_t j = 0; j < K / 2; ++j) {
                uint8_t u0 = uint8_t(q[r * K + 2 * j] + off), u1 = uint8_t(q[r * K + 2 * j + 1] + off);
                row[j] = uint8_t((u0 & 15u) | ((u1 & 15u) << 4));
            }
            for (int64_t g = 0; g < lay[2]; ++g) {
                if (fmt == Q4G32H) gs16[r * lay[2] + g] = (g < ng) ? d[r * ng + g] : uint16_t(0);
                else group_scales[r * lay[2] + g] = (g < ng) ? gscale[r * ng + g] : 0.0f;
            }
        }
        return 0;
    }
    SbFormat F;
    sb_format(fmt, &F);
    const int64_t nb = K / 256;
    uint8_t zeros[16] = {0};
    for (int64_t r = 0; r < N; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            int64_t sb = r * nb + b;
            pack_sb(fmt, q + r * K + 256 * b, sub_scale + sb * F.nsub, F.asym ? sub_min + sb * F.nsub : zeros,
                    d[sb], F.asym ? dmin[sb] : uint16_t(0), packed + r * lay[0] + b * F.bytes);
        }
    return 0;
}

// Inverse of orc_pack (padding is ignored).
int orc_unpack(int fmt, int64_t N, int64_t K, const uint8_t *packed, const float *group_scales, int8_t *q,
               float *gscale, uint8_t *sub_scale, uint8_t *sub_min, uint16_t *d, uint16_t *dmin) {
    int64_t lay[5];
    if (orc_layout(fmt, N, K, lay)) return -2;
    if (is_int4(fmt)) {
        const uint16_t *gs16 = reinterpret_cast<const uint16_t *>(group_scales);
        const int64_t ng = fmt == Q4G32A ? K / 16 : K / int4_group(fmt);
        const int off = fmt == Q4G32A ? 0 : 8;
        for (int64_t r = 0; r < N; ++r) {
            const uint8_t *row = packed + r * lay[0];
            for (int64_t k = 0; k < K; ++k) {
                uint8_t byte = row[k >> 1];
                uint8_t u = (k & 1) ? uint8_t(byte >> 4) : uint8_t(byte & 15u);
                q[r * K + k] = int8_t(int(u) - off);
            }
            for (int64_t g = 0; g < ng; ++g) {
                if (fmt == Q4G32H) d[r * ng + g] = gs16[r * lay[2] + g];
                else gscale[r * ng + g] = group_scales[r * lay[2] + g];
            }
        }
        return 0;
    }
    SbFormat F;
    sb_format(fmt, &F);
    const int64_t nb = K / 256;
    for (int64_t r = 0; r < N; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            int64_t sb = r * nb + b;
            uint8_t M[16] = {0};
            uint16_t dm = 0;
            unpack_sb(fmt, packed + r * lay[0] + b * F.bytes, q + r * K + 256 * b, sub_scale + sb * F.nsub, M,
                      d + sb, &dm);
            if (F.asym) {
                for (int j = 0; j < F.nsub; ++j) sub_min[sb * F.nsub + j] = M[j];
                dmin[sb] = dm;
            }
        }
    return 0;
}

// Dequantize rows [r0, r0 + nrows) of a packed matrix into out[nrows][K] (fp32).
int orc_dequant_rows(int fmt, int64_t N, int64_t K, const uint8_t *packed, const float *group_scales, int64_t r0,
                     int64_t nrows, float *out) {
    int64_t lay[5];
    if (orc_layout(fmt, N, K, lay)) return -2;
    if (r0 < 0 || nrows < 0 || r0 + nrows > N) return -1;
    for (int64_t i = 0; i < nrows; ++i) dequant_row(fmt, packed, group_scales, K, r0 + i, lay[0], lay[2], out + i * K);
    return 0;
}

// Y[m][r] = sum_k w'[r,k] * X[m,k] in fp64, X given as fp16 bits [M][ldx]; rows [r0, r0 + nrows) only,
// written to Y[m][r - r0] (row stride nrows). Rows are split over `nthreads` std::threads.
int orc_gemm_rows(int fmt, int64_t N, int64_t K, const uint8_t *packed, const float *group_scales, int64_t M,
                  const uint16_t *X, int64_t ldx, int64_t r0, int64_t nrows, double *Y, int nthreads) {
    int64_t lay[5];
    if (orc_layout(fmt, N, K, lay)) return -2;
    if (r0 < 0 || nrows < 0 || r0 + nrows > N || M < 0) return -1;
    std::vector<double> xd(size_t(M * K));
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) xd[size_t(m * K + k)] = double(f16_to_f32(X[m * ldx + k]));
    if (nthreads < 1) nthreads = 1;
    auto work = [&](int64_t a, int64_t b) {
        std::vector<float> w(static_cast<size_t>(K));
        for (int64_t i = a; i < b; ++i) {
            dequant_row(fmt, packed, group_scales, K, r0 + i, lay[0], lay[2], w.data());
            for (int64_t m = 0; m < M; ++m) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) acc += double(w[size_t(k)]) * xd[size_t(m * K + k)];
                Y[m * nrows + i] = acc;
            }
        }
    };
    if (nthreads == 1 || nrows < 2) {
        work(0, nrows);
    } else {
        std::vector<std::thread> th;
        int64_t per = (nrows + nthreads - 1) / nthreads;
        for (int t = 0; t < nthreads; ++t) {
            int64_t a = t * per, b = std::min(nrows, a + per);
            if (a < b) th.emplace_back(work, a, b);
        }
        for (auto &t : th) t.join();
    }
    return 0;
}

// Prefill reference for sampled outputs: out[i] = sum_k bf16(X[m_i,k]) * v(w'[n_i,k]) in fp64, where v rounds
// the dequantized weight to bf16 when round_w != 0 and keeps it fp32 otherwise. X is bf16 bits [M][ldx].
int orc_prefill_sample(int fmt, int64_t N, int64_t K, const uint8_t *packed, const float *group_scales,
                       const uint16_t *X, int64_t ldx, int64_t M, const int64_t *ms, const int64_t *ns,
                       int64_t count, int round_w, double *out) {
    int64_t lay[5];
    if (orc_layout(fmt, N, K, lay)) return -2;
    std::vector<float> w(static_cast<size_t>(K));
    int64_t last_row = -1;
    for (int64_t i = 0; i < count; ++i) {
        if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N) return -1;
        if (ns[i] != last_row) {
            dequant_row(fmt, packed, group_scales, K, ns[i], lay[0], lay[2], w.data());
            last_row = ns[i];
        }
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double wv = round_w ? double(bf16_to_f32(f32_to_bf16(w[size_t(k)]))) : double(w[size_t(k)]);
            acc += double(bf16_to_f32(X[ms[i] * ldx + k])) * wv;
        }
        out[i] = acc;
    }
    return 0;
}

// ---------------------------------------------------------------------------------------------------------
// 8-bit KV cache. The 2/3/5/6-bit article (§4.1) quantizes the KV cache to 8 bits with every 32 elements sharing
// one fp16 scale (about 1.06 bytes per element, half the fp16 size); the Mix-Quant article (§2.3) dequantizes such
// an int8 cache back to fp16. Reading (plainest, the super-block rules at 8 bits): groups of 32 consecutive
// elements, d = max|v| / 127 in fp32 rounded to fp16 and used rounded from there on, q = clamp(rint(v / d), -127,
// 127) (0 when d is 0), dequant v' = fp16(d * q). Inputs are fp16 and finite.
// ---------------------------------------------------------------------------------------------------------
int orc_kv_quantize(const uint16_t *v, int64_t n, int8_t *q, uint16_t *scales) {
    if (n < 0 || n % 32 != 0) return -1;
    for (int64_t g = 0; g < n / 32; ++g) {
        float a = 0.0f;
        for (int i = 0; i < 32; ++i) {
            const float x = std::fabs(f16_to_f32(v[32 * g + i]));
            if (x > a) a = x;
        }
        const uint16_t d16 = f32_to_f16(a / 127.0f);
        const float d = f16_to_f32(d16);
        scales[g] = d16;
        for (int i = 0; i < 32; ++i) {
            float t = 0.0f;
            if (d > 0.0f) {
                t = std::nearbyint(f16_to_f32(v[32 * g + i]) / d);
                if (t > 127.0f) t = 127.0f;
                if (t < -127.0f) t = -127.0f;
            }
            q[32 * g + i] = int8_t(t);
        }
    }
    return 0;
}

int orc_kv_dequant(const int8_t *q, const uint16_t *scales, int64_t n, uint16_t *out) {
    if (n < 0 || n % 32 != 0) return -1;
    for (int64_t g = 0; g < n / 32; ++g) {
        const float d = f16_to_f32(scales[g]);
        for (int i = 0; i < 32; ++i) out[32 * g + i] = f32_to_f16(d * float(q[32 * g + i]));
    }
    return 0;
}

}  // extern "C"
