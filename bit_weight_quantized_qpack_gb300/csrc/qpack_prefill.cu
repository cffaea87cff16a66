// qpack_prefill.cu — prefill dequant GEMM on the 5th-generation tensor cores (sm_103a):
//   Y[m, n] = sum_k bf16(X[m, k]) * bf16(w'[n, k]),  fp32 accumulation in tensor memory, Y rounded to bf16.
//
// Prefill is a dense [tokens, hidden] x [hidden, hidden] contraction (2/3/5/6-bit article,
// lpnh.cn/news/2857666, §1.2), so it belongs on the tensor cores; the packed weights are still read in their
// compact form and dequantized on chip (DBHOO-CIM article, pwwt.cn/news/4452170, §3.3: no fp32 weight array).
//
// Two kernels. The pair kernel (prefill_pair_kernel, further below) spreads each tensor-core instruction over a
// cluster of two CTAs on two SMs (512 tokens x 256 or 224 weight rows per pair) and is the default for every format.
// The single-CTA kernel (prefill_kernel) serves the tile heights 112 and 128 when they are asked for.
//
// Single-CTA kernel: one CTA computes a 512 x 128 block of Y (four 128-token sub-tiles x 128 weight rows):
//   warp 9      TMA producer: per 64-wide K step, four 2-D tensor copies bring the 4 x (128 x 64) bf16 X tiles into
//               shared memory already in the 128-byte-swizzled K-major layout the MMA reads.
//   warps 0..7  weight producers: per K step, each thread dequantizes one 32-weight unit of one of the 128 weight
//               rows (the exact fp32 dequantized value, from aligned global loads issued three K steps ahead,
//               then bf16 round-to-nearest-even) into the swizzled 128 x 64 weight tile, the two threads of a row
//               side by side in a warp; afterwards they are the epilogue warps (tcgen05.ld of their TMEM lane
//               quarter, bf16 conversion, global stores).
//   warp 8      allocates all 512 TMEM columns (four fp32 128 x 128 accumulators); lane 0 issues the tcgen05.mma
//               instructions (M=128, N=128, K=16; both operands from shared-memory descriptors) and commits them to
//               mbarriers that free the stage and, at the end, publish the accumulators.
// Each weight tile is dequantized once for 512 tokens (the dequantization is the CUDA-core cost of this path).
// Every wait is bounded; on a timeout the kernel records a fault bit, skips the remaining work, still frees its
// TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "qpack_dev.cuh"
#include "qpack_launch.h"

namespace qpack {

__device__ int g_fault_prefill = 0;

namespace {

constexpr int BMS = 128, NSUB = 4, BM = BMS * NSUB;   // tokens per sub-tile, sub-tiles, tokens per CTA
constexpr int BNMAX = 128, BK = 64;                // weight rows per CTA (at most), K per stage
constexpr int STAGES = 2;
constexpr int PD = 3;                              // K steps the packed-weight loads run ahead of the dequantization
constexpr int A_BYTES = BMS * BK * 2;              // 16 KB per X sub-tile
// Per weight-tile height BN (128, or 112 when that fills the GPU's SMs better): the BN x 64 bf16 weight tile and
// one stage (four X sub-tiles + the weight tile; a multiple of 1024 bytes since BN is a multiple of 8).
template <int BN> constexpr int kBBytes = BN * BK * 2;
template <int BN> constexpr int kStageBytes = NSUB * A_BYTES + kBBytes<BN>;
constexpr int NDQW = 8;                            // dequant / epilogue warps
constexpr int NPROD = NDQW * 32;
constexpr int THREADS = NPROD + 64;                // + MMA warp + TMA warp
constexpr uint32_t TMEM_COLS = 512;
template <int BN> constexpr int kSmemBytes = 1024 /*alignment slack*/ + STAGES * kStageBytes<BN> + 256 /*barriers*/;

// ------------------------------------------------------------------------------------------------------------
// tcgen05 / TMEM wrappers (PTX ISA, tcgen05 family)
// ------------------------------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] x B[smem desc]^T, kind::f16 (bf16 inputs per the instruction descriptor).
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive (once) on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row core-matrix groups 1024 bytes apart.
//   bits [0,14) start address >> 4, [16,30) leading byte offset >> 4 (unused for swizzled K-major, set to 1),
//   [32,46) stride byte offset >> 4 (1024 B), [46,48) descriptor version 1, [61,64) layout 2 = 128B swizzle.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= uint64_t((smem_addr >> 4) & 0x3FFFu);
    d |= uint64_t(1) << 16;
    d |= uint64_t(1024 >> 4) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;
    return d;
}
// Instruction descriptor, kind::f16: D fp32 (bit 4), A bf16 (bits 7-9 = 1), B bf16 (bits 10-12 = 1), both
// K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
template <int BN>
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(BMS >> 4) << 24);

// Byte offset of the 16-byte chunk c (K elements 8c..8c+7) of row r inside a 128B-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t c) {
    return (r >> 3) * 1024u + (r & 7u) * 128u + ((c ^ (r & 7u)) << 4);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    return lo | (hi << 16);
}

__device__ __forceinline__ uint32_t ldg32(const uint8_t *p) { return __ldg(reinterpret_cast<const uint32_t *>(p)); }
__device__ __forceinline__ uint32_t ldg16(const uint8_t *p) { return __ldg(reinterpret_cast<const uint16_t *>(p)); }
// n consecutive 32-bit words starting at a 2-byte aligned global address (aligned loads plus funnel shifts).
template <int n>
__device__ __forceinline__ void ldg_words_a2(const uint8_t *p, uint32_t *w) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t *base = reinterpret_cast<const uint32_t *>(a & ~uintptr_t(3));
    const uint32_t sh = uint32_t(a & 3u) * 8u;   // 0 or 16
    uint32_t r[n + 1];
#pragma unroll
    for (int i = 0; i <= n; ++i) r[i] = __ldg(base + i);
#pragma unroll
    for (int i = 0; i < n; ++i) w[i] = __funnelshift_r(r[i], r[i + 1], sh);
}

// Dequantization of one 32-weight unit u of a packed row, in two steps so that the loads of the next K step can be in
// flight while the current one is converted: load_raw gathers the unit's bytes with aligned global loads,
// unit_bf16 turns them into 16 bf16x2 words. The values are exactly the dequantized weights of the format (the
// sub-block scale d * L first, then its product with the code, minus dmin * M; every step an fp32 rounding) rounded
// to bf16.
struct RawUnit {
    uint32_t c[5];      // code words (formats differ in how many they use)
    uint32_t e[4];      // high-bit planes / scale fields / super-block scales
};
template <int F>
__device__ __forceinline__ void load_raw(const uint8_t *row, const uint8_t *gs_row, uint32_t u, RawUnit &r) {
    if constexpr (kInt4<F>) {
        const uint4 c = __ldg(reinterpret_cast<const uint4 *>(row + 16 * u));
        r.c[0] = c.x; r.c[1] = c.y; r.c[2] = c.z; r.c[3] = c.w;
        // the group scale as fp32 bits: stored fp32 (Q4G32) or fp16 widened exactly (Q4G32H)
        if constexpr (F == FMT_Q4G32) {
            r.e[0] = __float_as_uint(__ldg(reinterpret_cast<const float *>(gs_row) + u));
        } else if constexpr (F == FMT_Q4G32H) {
            r.e[0] = __float_as_uint(h2f_bits(uint16_t(ldg16(gs_row + 2 * u))));
        } else {    // Q4G16: the scales of weights 0-15 and 16-31 of the unit; Q4G32A: the pair (s, z)
            const float2 s2 = __ldg(reinterpret_cast<const float2 *>(gs_row) + u);
            r.e[0] = __float_as_uint(s2.x);
            r.e[1] = __float_as_uint(s2.y);
        }
    } else {
        const uint32_t b = u >> 3, su = u & 7u;
        const uint8_t *blk = row + b * Fmt<F>::bytes;
        if constexpr (F == FMT_Q2S) {
            r.c[0] = ldg32(blk + 8 * su); r.c[1] = ldg32(blk + 8 * su + 4);
            r.e[0] = ldg16(blk + 64 + 2 * su);
            r.e[1] = ldg32(blk + 80);
        } else if constexpr (F == FMT_Q3S) {
            ldg_words_a2<3>(blk + 12 * su, r.c);
            // the 12 bits of L_{2su}, L_{2su+1}: bits 12 (su & 1) .. +11 of the 24-bit field group su >> 1, read as
            // two bytes that stay inside the super-block
            const uint32_t fb = 96u + 3u * (su >> 1) + (su & 1u);
            r.e[0] = uint32_t(__ldg(blk + fb)) | (uint32_t(__ldg(blk + fb + 1)) << 8);
            r.e[1] = ldg16(blk + 108);
        } else if constexpr (F == FMT_Q5S) {
            const uint4 c = __ldg(reinterpret_cast<const uint4 *>(blk + 16 * su));
            r.c[0] = c.x; r.c[1] = c.y; r.c[2] = c.z; r.c[3] = c.w;
            r.c[4] = ldg32(blk + 128 + 4 * su);
            const uint4 fl = __ldg(reinterpret_cast<const uint4 *>(blk + 160));
            r.e[0] = fl.x; r.e[1] = fl.y; r.e[2] = fl.z; r.e[3] = fl.w;
        } else {
            ldg_words_a2<4>(blk + 16 * su, r.c);
            ldg_words_a2<2>(blk + 128 + 8 * su, r.e);
            r.e[2] = ldg16(blk + 192 + 2 * su);
            r.e[3] = ldg16(blk + 208);
        }
    }
}
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}
// Codes are unpacked four at a time into the bytes of 32-bit words, each byte one code shifted left inside it by a
// known bit class p (the byte holds q * 2^p). A byte becomes a float with no conversion instruction: placed in the
// low mantissa bits of 2^23 it reads 2^23 + q * 2^p, and subtracting 2^23 + off * 2^p leaves (q - off) * 2^p
// exactly. The scale is taken times 2^-p (exact), so every product is the same real number as scale * (q - off),
// rounded once: the weights are bit for bit those of the formats' dequantization rule.
__device__ __forceinline__ float byte_f(uint32_t v, int b) {                  // 2^23 + byte b of v
    return __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7540u | uint32_t(b)));
}
constexpr float TWO23 = 8388608.0f;

template <int F>
__device__ __forceinline__ void unit_bf16(const RawUnit &r, uint32_t u, uint32_t out[16]) {
    float w[32];
    if constexpr (kInt4<F>) {
        // weight 8j + 2b: low nibble of byte b of code word j (class 0); weight 8j + 2b + 1: its high nibble (class 4)
        const float sc0 = __uint_as_float(r.e[0]), sc1 = F == FMT_Q4G16 ? __uint_as_float(r.e[1]) : sc0;
        const float z = F == FMT_Q4G32A ? __uint_as_float(r.e[1]) : 8.0f;   // the code offset, or the zero point
        const float off0 = __fadd_rn(TWO23, z), off4 = __fadd_rn(TWO23, 16.0f * z);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float sc = j < 2 ? sc0 : sc1, sc4 = sc * 0.0625f;
            const uint32_t lo = r.c[j] & 0x0F0F0F0Fu, hi = r.c[j] & 0xF0F0F0F0u;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                w[8 * j + 2 * b] = __fmul_rn(sc, __fsub_rn(byte_f(lo, b), off0));
                w[8 * j + 2 * b + 1] = __fmul_rn(sc4, __fsub_rn(byte_f(hi, b), off4));
            }
        }
    } else if constexpr (F == FMT_Q2S) {
        // weight 4b + k of a sub-block: bits 2k of byte b of its code word (class 2k)
        const float D = h2f_bits(uint16_t(r.e[1] & 0xFFFFu)), Dm = h2f_bits(uint16_t(r.e[1] >> 16));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t l = (r.e[0] >> (8 * h)) & 0xFFu;
            const float es = __fmul_rn(D, float(l & 15u)), em = __fmul_rn(Dm, float(l >> 4));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t v = r.c[h] & (0x03030303u << (2 * k));
                const float sk = es * (k == 0 ? 1.0f : k == 1 ? 0.25f : k == 2 ? 0.0625f : 0.015625f);
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    w[16 * h + 4 * b + k] = __fsub_rn(__fmul_rn(sk, __fsub_rn(byte_f(v, b), TWO23)), em);
            }
        }
    } else if constexpr (F == FMT_Q3S) {
        // per sub-block (two 3-byte groups b0 b1 b2 | b3 b4 b5, code t of a group at bits 3t, weights t and 8 + t):
        // byte permutes P = (b0 b3 b2 b5), Q = (b1 b4 b1 b4), R = (b0 b1 b3 b4), S = (b1 b2 b4 b5), then
        //   P & 0x1C1C0707: weights 0, 8 (class 0), 6, 14 (class 2);  P & 0xE0E03838: 1, 9 (3), 7, 15 (5)
        //   Q & 0x70700E0E: 3, 11 (1), 4, 12 (4);  the codes straddling bytes (2, 5, 10, 13) from R and S, class 0
        const uint32_t su = u & 7u;
        const uint32_t fsh = 4u * (su & 1u);
        const float D = h2f_bits(uint16_t(r.e[1]));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float es = __fmul_rn(D, float((r.e[0] >> (fsh + 6 * h)) & 63u));
            const uint32_t wa = r.c[h], wb = r.c[h + 1], o = h == 0 ? 0u : 0x2222u;   // bytes 6h .. 6h + 5
            const uint32_t P = __byte_perm(wa, wb, 0x5230u + o), Q = __byte_perm(wa, wb, 0x4141u + o);
            const uint32_t R = __byte_perm(wa, wb, 0x4310u + o), S = __byte_perm(wa, wb, 0x5421u + o);
            const uint32_t v[4] = {P & 0x1C1C0707u, P & 0xE0E03838u, Q & 0x70700E0Eu,
                                   ((R >> 6) & 0x00070007u) | ((S << 1) & 0x07000700u)};
            constexpr int wi[4][4] = {{0, 8, 6, 14}, {1, 9, 7, 15}, {3, 11, 4, 12}, {2, 5, 10, 13}};
            constexpr int cl[4][4] = {{0, 0, 2, 2}, {3, 3, 5, 5}, {1, 1, 4, 4}, {0, 0, 0, 0}};
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const float p2 = float(1 << cl[k][b]);                      // 2^p, exact
                    w[16 * h + wi[k][b]] =
                        __fmul_rn(es * (1.0f / p2), __fsub_rn(byte_f(v[k], b), TWO23 + 4.0f * p2));
                }
        }
    } else if constexpr (F == FMT_Q5S) {
        // weight 8j + 2b (+1): the low (high) nibble of byte b of code word j with its fifth bit from bit lane j of the
        // unit's high-bit word (bit 8b + 4, or bit 8((b + 1) & 3) for the odd weight): one select for the even codes,
        // a select and a funnel shift by 4 for the odd ones
        const uint32_t su = u & 7u;
        const uint64_t lo64 = (uint64_t(r.e[1]) << 32) | r.e[0], hi64 = (uint64_t(r.e[2]) << 32) | r.e[1];
        const float D = h2f_bits(uint16_t(r.e[3] & 0xFFFFu)), Dm = h2f_bits(uint16_t(r.e[3] >> 16));
        const float es = __fmul_rn(D, float(uint32_t(lo64 >> (6 * su)) & 63u));
        const float em = __fmul_rn(Dm, float(uint32_t(hi64 >> (16 + 6 * su)) & 63u));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t hj = (r.c[4] >> j) & 0x11111111u;
            const uint32_t ve = lop3_sel(r.c[j], hj, 0x0F0F0F0Fu);
            const uint32_t vo = __funnelshift_r(lop3_sel(r.c[j], hj, 0xF0F0F0F0u), hj, 4);
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                w[8 * j + 2 * b] = __fsub_rn(__fmul_rn(es, __fsub_rn(byte_f(ve, b), TWO23)), em);
                w[8 * j + 2 * b + 1] = __fsub_rn(__fmul_rn(es, __fsub_rn(byte_f(vo, b), TWO23)), em);
            }
        }
    } else {
        // per sub-block: low-4 plane words A (weights 0-7), B (8-15), high-2 plane H (weight 4b + k at bits 2k of
        // byte b). Word k holds weight 4b + k in byte b: k even at class 0 (nibble | high bits << 4), k odd at class 2.
        const float D = h2f_bits(uint16_t(r.e[3]));
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const float es = __fmul_rn(D, float(int(int8_t(uint8_t(r.e[2] >> (8 * hh)))))), es2 = es * 0.25f;
            const uint32_t A = r.c[2 * hh], B = r.c[2 * hh + 1], H = r.e[hh];
            const uint32_t P0 = __byte_perm(A, B, 0x6420u), P1 = __byte_perm(A, B, 0x7531u), Hs = H << 4;
            const uint32_t v[4] = {(P0 & 0x0F0F0F0Fu) | (Hs & 0x30303030u), ((P0 >> 2) & 0x3C3C3C3Cu) | (Hs & 0xC0C0C0C0u),
                                   (P1 & 0x0F0F0F0Fu) | (H & 0x30303030u), ((P1 >> 2) & 0x3C3C3C3Cu) | (H & 0xC0C0C0C0u)};
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    w[16 * hh + 4 * b + k] = (k & 1) ? __fmul_rn(es2, __fsub_rn(byte_f(v[k], b), TWO23 + 128.0f))
                                                     : __fmul_rn(es, __fsub_rn(byte_f(v[k], b), TWO23 + 32.0f));
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = bf16x2_rn(w[2 * i], w[2 * i + 1]);
}

// 2-D tensor copy global -> shared (box at coordinates {x, y}), completion on `bar` as bytes.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}


// ------------------------------------------------------------------------------------------------------------
// CTA-pair (cluster of two) building blocks for the pair kernel below (PTX ISA: tcgen05 with .cta_group::2,
// mapa, cluster-scope mbarrier arrive / try_wait, barrier.cluster).
// ------------------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t cta_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(cta_addr), "r"(rank));
    return r;
}
// Arrive on an mbarrier anywhere in the cluster, releasing this thread's prior writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait on a local mbarrier whose arrivals may come from the peer CTA (false after `limit` polls).
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t *bar, uint32_t parity, uint32_t limit = (1u << 22)) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// TMEM allocation for a CTA pair: one warp of each of the two CTAs executes these together.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D (both CTAs' TMEM) (+)= A (M/2 rows in each CTA's shared memory) x B (N/2 rows in each)^T, issued by one
// thread of the even CTA.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the mbarrier at `bar`'s offset in every CTA of `cta_mask` when the pair MMAs issued so far are done.
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(smem_u32(bar)), "h"(cta_mask)
        : "memory");
}
}  // namespace

template <int F, int BN>
__global__ void __launch_bounds__(THREADS, 1) prefill_kernel(const __grid_constant__ CUtensorMap tm_x, PrefillArgs a) {
    static_assert(BN % 16 == 0 && BN <= BNMAX, "MMA N: a multiple of 16, at most 128 (one TMEM quarter per sub-tile)");
    constexpr int STAGE_BYTES = kStageBytes<BN>;
    constexpr uint32_t IDESC = kIdesc<BN>;
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;           // 1024-aligned operand area
    uint8_t *sm = smem_raw + (base - smem_u32(smem_raw));
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + STAGES * STAGE_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *accum = empty + STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum + 1);

    const int64_t M = a.M, N = a.N, K = a.K;
    const int64_t n0 = int64_t(blockIdx.x) * BN, m0 = int64_t(blockIdx.y) * BM;
    const int nk = int(K / BK);
    const int nsub = int((M - m0 + BMS - 1) / BMS < NSUB ? (M - m0 + BMS - 1) / BMS : NSUB);   // sub-tiles with tokens

    if (tid == 0) {
        for (int st = 0; st < STAGES; ++st) { mbar_init(&full[st], NDQW + 1); mbar_init(&empty[st], 1); }
        mbar_init(accum, 1);
        fence_mbar_init();
    }
    if (warp == NDQW) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot;
    bool dead = false;

    if (warp < NDQW) {
        // ------------------------------ weight producers ------------------------------
        // weight row and K half of the stage: the two lanes of a row pair up in the warp, so that each warp-wide
        // load of packed bytes touches 16 rows (the two units of a row are adjacent) instead of 32
        const int r = 16 * warp + (lane >> 1), h = lane & 1;
        const bool rin = r < BN;                                            // rows past a short tile stay idle
        const int64_t n = n0 + r;
        const uint8_t *row = a.packed + n * a.row_stride;
        constexpr int64_t SE = F == FMT_Q4G32H ? 2 : 4;                   // INT4 group-scale element bytes
        const uint8_t *gs_row = a.gscale ? reinterpret_cast<const uint8_t *>(a.gscale) + n * a.scale_stride * SE : nullptr;
        // The raw bytes of step k + PD are loaded while step k is converted and stored: PD + 1 register slots in
        // fixed roles (the loop is unrolled by PD + 1), so no slot is copied while its loads are in flight.
        RawUnit S[PD + 1] = {};
        if (rin && n < N) {
#pragma unroll
            for (int i = 0; i < PD; ++i)
                if (i < nk) load_raw<F>(row, gs_row, uint32_t(2 * i + h), S[i]);
        }
        auto step = [&](int kt, const RawUnit &use, RawUnit &into) {
            if (kt >= nk || dead) return;
            const int st = kt % STAGES;
            if (rin && n < N && kt + PD < nk) load_raw<F>(row, gs_row, uint32_t(2 * (kt + PD) + h), into);
            if (kt >= STAGES && !mbar_wait_bounded(&empty[st], uint32_t((kt / STAGES) - 1) & 1u)) {
                atomicOr(&g_fault_prefill, FAULT_WAIT_EMPTY);
                dead = true;
                return;
            }
            uint8_t *Bs = sm + st * STAGE_BYTES + NSUB * A_BYTES;
            uint4 v[4];
            if (n < N) {
                uint32_t o[16];
                unit_bf16<F>(use, uint32_t(2 * kt + h), o);
#pragma unroll
                for (int c = 0; c < 4; ++c) v[c] = make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) v[c] = make_uint4(0u, 0u, 0u, 0u);
            }
            if (rin) {
#pragma unroll
                for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4 *>(Bs + sw128_off(uint32_t(r), uint32_t(4 * h + c))) = v[c];
            }
            fence_proxy_async_smem();      // make the generic-proxy stores visible to the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[st]);
        };
#pragma unroll 1
        for (int kt = 0; kt < nk && !dead; kt += PD + 1) {
#pragma unroll
            for (int i = 0; i <= PD; ++i) step(kt + i, S[i], S[(i + PD) % (PD + 1)]);
        }
        // ---------------------------------- epilogue ----------------------------------
        {
            // warp-uniform decision: the phase is complete if any lane observed it (tcgen05.ld is .sync.aligned)
            const bool seen = dead ? false : mbar_wait_bounded(accum, 0u);
            const bool ok = __any_sync(0xffffffffu, seen);
            if (!ok && lane == 0) atomicOr(&g_fault_prefill, FAULT_WAIT_MMA);
            dead = !ok;
        }
        tc_fence_after();
        if (!dead) {
            // warp w reads TMEM lanes 32 (w % 4) .. +31 (its lane quarter) of sub-tiles 2 (w / 4) and 2 (w / 4) + 1
            const int qw = warp & 3, half = warp >> 2;
#pragma unroll 1
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * half + jj;
                if (j >= nsub) break;
                const int64_t m = m0 + int64_t(BMS) * j + 32 * qw + lane;
                const uint32_t lane_base = tmem_d + (uint32_t(32 * qw) << 16) + uint32_t(BNMAX * j);
#pragma unroll 1
                for (int cc = 0; cc < (BN + 31) / 32; ++cc) {
                    uint32_t rr[32];
                    tmem_ld32(lane_base + uint32_t(32 * cc), rr);   // columns past BN are read, never stored
                    tmem_ld_wait();
                    const int w = BN - 32 * cc < 32 ? BN - 32 * cc : 32;   // columns of this chunk (16 or 32)
                    const int64_t nc = n0 + 32 * cc;
                    if (m < M && nc < N) {
                        uint16_t *dst = a.Y + m * a.ldy + nc;
                        if (nc + w <= N && a.vec_y) {
                            uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                if (8 * q < w)
                                    d4[q] = make_uint4(pack_bf16x2(__uint_as_float(rr[8 * q]), __uint_as_float(rr[8 * q + 1])),
                                                       pack_bf16x2(__uint_as_float(rr[8 * q + 2]), __uint_as_float(rr[8 * q + 3])),
                                                       pack_bf16x2(__uint_as_float(rr[8 * q + 4]), __uint_as_float(rr[8 * q + 5])),
                                                       pack_bf16x2(__uint_as_float(rr[8 * q + 6]), __uint_as_float(rr[8 * q + 7])));
                        } else {
#pragma unroll
                            for (int q = 0; q < 32; ++q)
                                if (q < w && nc + q < N)
                                    dst[q] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(rr[q])));
                        }
                    }
                }
            }
        }
    } else if (warp == NDQW) {
        // ------------------------------------ MMA issuer ------------------------------------
        if (lane == 0) {
            for (int kt = 0; kt < nk; ++kt) {
                const int st = kt % STAGES;
                if (!mbar_wait_bounded(&full[st], uint32_t(kt / STAGES) & 1u)) {
                    atomicOr(&g_fault_prefill, FAULT_WAIT_FULL);
                    dead = true;
                    break;
                }
                tc_fence_after();
                const uint32_t As = base + uint32_t(st * STAGE_BYTES), Bs = As + uint32_t(NSUB * A_BYTES);
                for (int j = 0; j < nsub; ++j) {
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_bf16(tmem_d + uint32_t(BNMAX * j), sw128_kmajor_desc(As + uint32_t(j * A_BYTES) + 32u * k),
                                  sw128_kmajor_desc(Bs + 32u * k), IDESC, (kt > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit(&empty[st]);                // the stage may be refilled once these MMAs have read it
            }
            umma_commit(accum);                         // accumulators complete (also on the failure path)
        }
        __syncwarp();
    } else {
        // ------------------------------------ X producer ------------------------------------
        if (lane == 0) {
            for (int kt = 0; kt < nk; ++kt) {
                const int st = kt % STAGES;
                if (kt >= STAGES && !mbar_wait_bounded(&empty[st], uint32_t((kt / STAGES) - 1) & 1u)) {
                    atomicOr(&g_fault_prefill, FAULT_WAIT_EMPTY);
                    break;
                }
                uint8_t *As = sm + st * STAGE_BYTES;
                mbar_arrive_expect_tx(&full[st], uint32_t(nsub * A_BYTES));
                for (int j = 0; j < nsub; ++j)
                    tma_load_2d(As + j * A_BYTES, &tm_x, kt * BK, int(m0 + int64_t(BMS) * j), &full[st]);
            }
        }
        __syncwarp();
    }

    // ---- teardown: every TMEM read is finished; free the accumulators ----
    tc_fence_before();
    __syncthreads();
    if (warp == NDQW) {
        tc_fence_after();
        if (lane == 0 && dead) {
            // On the failure path wait (bounded) for the MMAs already issued before freeing their TMEM.
            (void)mbar_wait_bounded(accum, 0u, 1u << 16);
        }
        __syncwarp();
        tmem_dealloc(tmem_d, TMEM_COLS);
    }
}


// ------------------------------------------------------------------------------------------------------------
// Pair kernel: a cluster of two CTAs on two SMs computes a 512 x 2 PR block of Y with tcgen05.mma.cta_group::2
// (M = 256 tokens, N = 2 PR weight rows per instruction; PR = 128, or 112 to spread a 4096-row matrix over more
// SMs). CTA r of the pair holds, per 64-wide K step,
//   A: two 128 x 64 bf16 X tiles (tokens m0 + 256 j + 128 r .. +127 of token sub-tile j = 0, 1), by TMA,
//   B: the PR x 64 bf16 weight tile of its own weight rows np + PR r .. +PR-1, dequantized by its warps 0..7,
// and its TMEM receives the 128 x 2 PR fp32 accumulators of its own tokens for both sub-tiles (256 columns each).
// Each SM thus reads 8 KB of operands per 256 x 256 x 16 MMA instead of the 8 KB per 128 x 128 x 16 of the
// single-CTA kernel, and still dequantizes each weight once per 512 tokens.
//   warps 0..7    dequant (arriving on the local wfull barrier), then epilogue (tcgen05.ld of their TMEM lane
//                 quarter, bf16 stores)
//   warp 8        TMEM allocation (both CTAs, together); lane 0 of the even CTA issues the MMAs
//   warp 9        lane 0: X tiles by TMA into this CTA's stage (completion on the local xfull barrier)
//   warps 10..13  lane 0 of warp 10 + st forwards stage st: once this CTA's xfull[st] and wfull[st] phases have
//                 completed, one cluster-scope release-arrive on the even CTA's full[st]
// The even CTA's full[st] completes with the two CTAs' forwarding arrivals. A cluster-scope release costs ~0.6 us
// (measured with globaltimer stamps), so it is made by threads with no loads in flight, one warp per ring stage so
// that the releases of consecutive stages overlap (one forwarding thread for all stages, or the dequant warps
// arriving across the cluster themselves, held the kernel below the single-CTA one). The MMA commits arrive on
// empty[st] and, at the end, on accum in both CTAs (multicast).
// ------------------------------------------------------------------------------------------------------------
namespace {
constexpr int P2_NSUB = 2;                                 // token sub-tiles (pair MMAs of M = 256)
constexpr int P2_ROWS = 128;                               // weight rows per CTA at most (shared-memory tile height)
constexpr int P2_STAGES = 4;
constexpr int P2_STAGE = P2_NSUB * A_BYTES + P2_ROWS * BK * 2;     // 48 KB
constexpr int P2_NFWD = P2_STAGES;                         // forwarding warps: stage st is forwarded by warp NDQW + 2 + st
constexpr int P2_THREADS = NPROD + 64 + 32 * P2_NFWD;      // + MMA warp, TMA warp, forwarding warps
constexpr int P2_SMEM = 1024 + P2_STAGES * P2_STAGE + 256;
// kind::f16 instruction descriptor: D fp32, A and B bf16, both K-major, N = 2 PR weight rows over the pair (N >> 3 at
// bits 17-22), M = 256 (M >> 4 at bits 24-28).
template <int PR>
constexpr uint32_t kIdescPair = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(2 * PR >> 3) << 17) | (uint32_t(256 >> 4) << 24);
}  // namespace

// PR = weight rows per CTA: 128, or 112 (pair N = 224), which covers more of the SMs on 4096-row matrices.
template <int F, int PR>
__global__ void __launch_bounds__(P2_THREADS, 1) prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_x, PrefillArgs a) {
    static_assert(PR == 112 || PR == 128, "pair tiles of 112 or 128 weight rows per CTA");
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;           // 1024-aligned operand area
    uint8_t *sm = smem_raw + (base - smem_u32(smem_raw));
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + P2_STAGES * P2_STAGE);   // used in the even CTA
    uint64_t *empty = full + P2_STAGES;
    uint64_t *xfull = empty + P2_STAGES;
    uint64_t *wfull = xfull + P2_STAGES;                                     // this CTA's weight tile stored
    uint64_t *accum = wfull + P2_STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum + 1);

    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int64_t M = a.M, N = a.N, K = a.K;
    const int64_t np = int64_t(blockIdx.x >> 1) * (2 * PR);                  // the pair's first weight row
    const int64_t n0 = np + int64_t(rank) * PR;                              // this CTA's weight rows
    const int64_t m0 = int64_t(blockIdx.y) * (2 * P2_NSUB * BMS);            // the pair's first token
    const int nk = int(K / BK);
    // sub-tiles with any token in the pair, and this CTA's own 128 tokens of sub-tile j start at m0 + 256 j + 128 r
    const int nsub = int((M - m0 + 2 * BMS - 1) / (2 * BMS) < P2_NSUB ? (M - m0 + 2 * BMS - 1) / (2 * BMS) : P2_NSUB);
    auto own_tok0 = [&](int j) { return m0 + int64_t(2 * BMS) * j + int64_t(BMS) * rank; };
    int nload = 0;                                                           // this CTA's sub-tiles with tokens
    for (int j = 0; j < nsub; ++j) nload += own_tok0(j) < M ? 1 : 0;

    if (tid == 0) {
        for (int st = 0; st < P2_STAGES; ++st) {
            mbar_init(&full[st], 2);                     // the two CTAs' forwarding arrivals
            mbar_init(&empty[st], 1);
            mbar_init(&xfull[st], 1);
            mbar_init(&wfull[st], NDQW);
        }
        mbar_init(accum, 1);
        fence_mbar_init();
    }
    if (warp == NDQW) {
        tmem_alloc_pair(tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();            // both CTAs: barriers initialised and TMEM allocated before any cross-CTA use
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot;
    const uint32_t full0_leader = mapa_shared(smem_u32(&full[0]), 0);      // the even CTA's full[0], cluster address
    bool dead = false;

    if (warp < NDQW) {
        // ------------------------------ weight producers ------------------------------
        // weight row and K half of the stage, the two lanes of a row side by side (see prefill_kernel); PR / 8 rows
        // per warp (with 112 rows lanes 28..31 are idle)
        const int r = (PR / 8) * warp + (lane >> 1), h = lane & 1;
        const bool live = (lane >> 1) < PR / 8;
        const int64_t n = live ? n0 + r : N;
        const uint8_t *row = a.packed + n * a.row_stride;
        constexpr int64_t SE = F == FMT_Q4G32H ? 2 : 4;
        const uint8_t *gs_row = a.gscale ? reinterpret_cast<const uint8_t *>(a.gscale) + n * a.scale_stride * SE : nullptr;
        RawUnit S[PD + 1] = {};
        if (n < N) {
#pragma unroll
            for (int i = 0; i < PD; ++i)
                if (i < nk) load_raw<F>(row, gs_row, uint32_t(2 * i + h), S[i]);
        }
        auto step = [&](int kt, const RawUnit &use, RawUnit &into) {
            if (kt >= nk || dead) return;
            const int st = kt % P2_STAGES;
            if (n < N && kt + PD < nk) load_raw<F>(row, gs_row, uint32_t(2 * (kt + PD) + h), into);
            if (kt >= P2_STAGES && !mbar_wait_cluster_bounded(&empty[st], uint32_t((kt / P2_STAGES) - 1) & 1u)) {
                atomicOr(&g_fault_prefill, FAULT_WAIT_EMPTY);
                dead = true;
                return;
            }
            uint8_t *Bs = sm + st * P2_STAGE + P2_NSUB * A_BYTES;
            uint4 v[4];
            if (n < N) {
                uint32_t o[16];
                unit_bf16<F>(use, uint32_t(2 * kt + h), o);
#pragma unroll
                for (int c = 0; c < 4; ++c) v[c] = make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) v[c] = make_uint4(0u, 0u, 0u, 0u);
            }
            if (live) {
#pragma unroll
                for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4 *>(Bs + sw128_off(uint32_t(r), uint32_t(4 * h + c))) = v[c];
            }
            // the generic-proxy stores, visible to the tensor cores; this CTA's forwarding warp passes the stage on
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&wfull[st]);
        };
#pragma unroll 1
        for (int kt = 0; kt < nk && !dead; kt += PD + 1) {
#pragma unroll
            for (int i = 0; i <= PD; ++i) step(kt + i, S[i], S[(i + PD) % (PD + 1)]);
        }
        // ---------------------------------- epilogue ----------------------------------
        {
            const bool seen = dead ? false : mbar_wait_cluster_bounded(accum, 0u);
            const bool ok = __any_sync(0xffffffffu, seen);
            if (!ok && lane == 0) atomicOr(&g_fault_prefill, FAULT_WAIT_MMA);
            dead = !ok;
        }
        tc_fence_after();
        // warp w reads TMEM lanes 32 (w % 4) .. +31 (its lane quarter: this CTA's tokens) of sub-tile w / 4
        const int qw = warp & 3, j = warp >> 2;
        if (!dead && j < nsub) {
            const int64_t m = own_tok0(j) + 32 * qw + lane;
            const uint32_t lane_base = tmem_d + (uint32_t(32 * qw) << 16) + uint32_t(256 * j);
#pragma unroll 1
            for (int cc = 0; cc < 2 * PR / 32; ++cc) {
                uint32_t rr[32];
                tmem_ld32(lane_base + uint32_t(32 * cc), rr);
                tmem_ld_wait();
                const int64_t nc = np + 32 * cc;
                if (m < M && nc < N) {
                    uint16_t *dst = a.Y + m * a.ldy + nc;
                    if (nc + 32 <= N && a.vec_y) {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            d4[q] = make_uint4(pack_bf16x2(__uint_as_float(rr[8 * q]), __uint_as_float(rr[8 * q + 1])),
                                               pack_bf16x2(__uint_as_float(rr[8 * q + 2]), __uint_as_float(rr[8 * q + 3])),
                                               pack_bf16x2(__uint_as_float(rr[8 * q + 4]), __uint_as_float(rr[8 * q + 5])),
                                               pack_bf16x2(__uint_as_float(rr[8 * q + 6]), __uint_as_float(rr[8 * q + 7])));
                    } else {
#pragma unroll
                        for (int q = 0; q < 32; ++q)
                            if (nc + q < N) dst[q] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(rr[q])));
                    }
                }
            }
        }
    } else if (warp == NDQW) {
        // ------------------------------------ MMA issuer (even CTA) ------------------------------------
        if (leader && lane == 0) {
            for (int kt = 0; kt < nk; ++kt) {
                const int st = kt % P2_STAGES;
                if (!mbar_wait_cluster_bounded(&full[st], uint32_t(kt / P2_STAGES) & 1u)) {
                    atomicOr(&g_fault_prefill, FAULT_WAIT_FULL);
                    dead = true;
                    break;
                }
                tc_fence_after();
                const uint32_t As = base + uint32_t(st * P2_STAGE), Bs = As + uint32_t(P2_NSUB * A_BYTES);
                for (int j = 0; j < nsub; ++j) {
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_bf16_pair(tmem_d + uint32_t(256 * j), sw128_kmajor_desc(As + uint32_t(j * A_BYTES) + 32u * k),
                                       sw128_kmajor_desc(Bs + 32u * k), kIdescPair<PR>, (kt > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit_pair(&empty[st], uint16_t(0x3));   // both CTAs may refill the stage once these MMAs are done
            }
            umma_commit_pair(accum, uint16_t(0x3));             // accumulators complete (also on the failure path)
        }
        __syncwarp();
    } else if (warp == NDQW + 1) {
        // ------------------------------------ X producer ------------------------------------
        if (lane == 0) {
            for (int kt = 0; kt < nk; ++kt) {
                const int st = kt % P2_STAGES;
                if (kt >= P2_STAGES && !mbar_wait_cluster_bounded(&empty[st], uint32_t((kt / P2_STAGES) - 1) & 1u)) {
                    atomicOr(&g_fault_prefill, FAULT_WAIT_EMPTY);
                    break;
                }
                uint8_t *As = sm + st * P2_STAGE;
                mbar_arrive_expect_tx(&xfull[st], uint32_t(nload * A_BYTES));
                for (int j = 0; j < nsub; ++j)
                    if (own_tok0(j) < M) tma_load_2d(As + j * A_BYTES, &tm_x, kt * BK, int(own_tok0(j)), &xfull[st]);
            }
        }
        __syncwarp();
    } else {
        // --------------------- forward "X landed" to the even CTA's full barrier ---------------------
        if (lane == 0) {
            for (int kt = warp - (NDQW + 2); kt < nk; kt += P2_NFWD) {
                const int st = kt % P2_STAGES;
                if (!mbar_wait_bounded(&xfull[st], uint32_t(kt / P2_STAGES) & 1u) ||
                    !mbar_wait_bounded(&wfull[st], uint32_t(kt / P2_STAGES) & 1u)) {
                    atomicOr(&g_fault_prefill, FAULT_WAIT_FULL);
                    break;
                }
                mbar_arrive_cluster(full0_leader + uint32_t(st) * 8u);
            }
        }
        __syncwarp();
    }

    // ---- teardown: both CTAs' TMEM reads and the pair's MMAs are finished before the TMEM is freed ----
    tc_fence_before();
    __syncthreads();
    if (warp == NDQW && leader && lane == 0 && dead) (void)mbar_wait_cluster_bounded(accum, 0u, 1u << 16);
    __syncwarp();
    cluster_sync_all();
    if (warp == NDQW) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_d, TMEM_COLS);
    }
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

// Tensor map over X [M][ldx] bf16: boxes of 64 K x 128 tokens, 128-byte swizzle (the K-major operand layout of the
// MMA); tokens past M read as zeros.
static cudaError_t encode_x(CUtensorMap *m, const PrefillArgs &a) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {cuuint64_t(a.K), cuuint64_t(a.M)};
    const cuuint64_t strides[1] = {cuuint64_t(a.ldx) * 2};
    const cuuint32_t box[2] = {uint32_t(BK), uint32_t(BMS)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(a.X), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int F, int BN>
static cudaError_t launch_prefill_bn(const PrefillArgs &a, const CUtensorMap &tmx, cudaStream_t s) {
    static int opted[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!opted[dev]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<F, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes<BN>);
        if (e != cudaSuccess) return e;
        opted[dev] = 1;
    }
    dim3 grid(unsigned((a.N + BN - 1) / BN), unsigned((a.M + BM - 1) / BM));
    if (grid.y > 65535u) return cudaErrorInvalidValue;
    prefill_kernel<F, BN><<<grid, THREADS, kSmemBytes<BN>, s>>>(tmx, a);
    return cudaGetLastError();
}

// Weight-tile height of the single-CTA kernel: 128 rows, or 112 when that takes fewer waves of CTAs per row of
// weight tiles than 128 does in proportion to the tile (one CTA per SM; time per CTA about proportional to its rows).
static int prefill_bn(const PrefillArgs &a) {
    const int64_t sms = num_sms(), mt = (a.M + BM - 1) / BM;
    auto cost = [&](int64_t bn) { return ((a.N + bn - 1) / bn * mt + sms - 1) / sms * bn; };
    return cost(112) < cost(128) ? 112 : 128;
}

// The pair kernel halves the operand reads each SM's shared memory serves to the tensor cores; on the prefill
// workload's matrices (M = 2048, 14336x4096 and 4096x14336) it is faster than the single-CTA kernel for every format
// (measured once the two lanes of a weight row share a warp's packed-weight loads).
template <int F> constexpr bool kPairPrefill = true;

// The CTA-pair kernel: clusters of two CTAs, each pair a 512-token x 2 PR-weight-row block of Y.
template <int F, int PR>
static cudaLaunchConfig_t pair_config(const PrefillArgs &a, cudaStream_t s, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    const int64_t gx = 2 * ((a.N + 2 * PR - 1) / (2 * PR)), gy = (a.M + 2 * P2_NSUB * BMS - 1) / (2 * P2_NSUB * BMS);
    cfg.gridDim = dim3(unsigned(gx > 0x7FFFFFFF ? 0 : gx), unsigned(gy > 65535 ? 0 : gy));
    cfg.blockDim = dim3(unsigned(P2_THREADS));
    cfg.dynamicSmemBytes = P2_SMEM;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int F, int PR>
static cudaError_t pair_opt_in() {
    static int opted[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!opted[dev]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_pair_kernel<F, PR>, cudaFuncAttributeMaxDynamicSharedMemorySize, P2_SMEM);
        if (e != cudaSuccess) return e;
        opted[dev] = 1;
    }
    return cudaSuccess;
}

template <int F, int PR>
static cudaError_t launch_prefill_pair(const PrefillArgs &a, const CUtensorMap &tmx, cudaStream_t s) {
    const cudaError_t e = pair_opt_in<F, PR>();
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pair_config<F, PR>(a, s, attr);
    if (cfg.gridDim.x == 0 || cfg.gridDim.y == 0) return cudaErrorInvalidValue;
    return cudaLaunchKernelEx(&cfg, prefill_pair_kernel<F, PR>, tmx, a);
}

// Weight rows per CTA of the pair kernel: 128, or 112 when that takes fewer waves of clusters than 128 does in
// proportion to the tile. The clusters that fit at once come from the occupancy query, as a pair of CTAs must sit
// on two SMs of one GPC. A cluster's time is set by its K steps more than by its rows (each step waits on the same
// round trip), so on a 4096-row matrix at M = 2048 the 112-row pairs (76 clusters instead of 64) gain only 0.5-2%,
// and lose ~1% for Q3S, which keeps 128.
template <int F>
static int prefill_pair_rows(const PrefillArgs &a, cudaStream_t s) {
    if (F == FMT_Q3S) return 128;
    static int fit[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 128;
    if (!fit[dev]) {
        int n = 0;
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = pair_config<F, 112>(a, s, attr);
        cfg.gridDim = dim3(2u, 1u);                       // one cluster: the query does not depend on the grid
        if (pair_opt_in<F, 112>() != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&n, prefill_pair_kernel<F, 112>, &cfg) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            n = num_sms() / 2;
        }
        fit[dev] = n;
    }
    const int64_t mt = (a.M + 2 * P2_NSUB * BMS - 1) / (2 * P2_NSUB * BMS), c = fit[dev];
    auto cost = [&](int64_t pr) { return ((a.N + 2 * pr - 1) / (2 * pr) * mt + c - 1) / c * pr; };
    return cost(112) < cost(128) ? 112 : 128;
}

template <int F>
static cudaError_t launch_prefill_f(const PrefillArgs &a, cudaStream_t s) {
    CUtensorMap tmx;
    const cudaError_t e = encode_x(&tmx, a);
    if (e != cudaSuccess) return e;
    const int forced = prefill_tile_rows();
    if (forced == 256) return launch_prefill_pair<F, 128>(a, tmx, s);
    if (forced == 224) return launch_prefill_pair<F, 112>(a, tmx, s);
    if (forced == 0 && kPairPrefill<F>)
        return prefill_pair_rows<F>(a, s) == 112 ? launch_prefill_pair<F, 112>(a, tmx, s) : launch_prefill_pair<F, 128>(a, tmx, s);
    const int bn = forced ? forced : prefill_bn(a);
    return bn == 112 ? launch_prefill_bn<F, 112>(a, tmx, s) : launch_prefill_bn<F, 128>(a, tmx, s);
}

cudaError_t launch_prefill(int fmt, const PrefillArgs &a, cudaStream_t s) {
    switch (fmt) {
        case FMT_Q4G32: return launch_prefill_f<FMT_Q4G32>(a, s);
        case FMT_Q4G32H: return launch_prefill_f<FMT_Q4G32H>(a, s);
        case FMT_Q4G16: return launch_prefill_f<FMT_Q4G16>(a, s);
        case FMT_Q4G32A: return launch_prefill_f<FMT_Q4G32A>(a, s);
        case FMT_Q2S: return launch_prefill_f<FMT_Q2S>(a, s);
        case FMT_Q3S: return launch_prefill_f<FMT_Q3S>(a, s);
        case FMT_Q5S: return launch_prefill_f<FMT_Q5S>(a, s);
        default: return launch_prefill_f<FMT_Q6S>(a, s);
    }
}

cudaError_t fetch_fault_prefill(int32_t *flags) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_fault_prefill, sizeof(int));
    if (e != cudaSuccess) return e;
    *flags |= v;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_fault_prefill, &zero, sizeof(int));
}

}  // namespace qpack
