/*
 * qpack.h — C ABI of libqpack: group-quantized low-bit weights with dequantization fused into the
 * decode-phase matrix-vector product (and the small-batch and prefill matrix products), for one NVIDIA
 * GB300 (sm_103a).
 *
 * Sources. P1 = the 2/3/5/6-bit quantization article (lpnh.cn/news/2857666); P2 = the DBHOO-CIM INT4 CPU
 * inference article (pwwt.cn/news/4452170). Where the pages leave a bit order open, fields are little-endian
 * with weight i at the lowest free bit.
 *
 * Conventions shared by every entry point:
 *  - W is row-major [N, K]: N output features (rows), K input features. Groups and super-blocks run along K.
 *  - All data pointers are DEVICE pointers owned by the caller; the library never allocates device memory
 *    and never frees caller memory. Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *  - fp16 and bf16 data are passed as their 16-bit patterns (uint16_t).
 *  - Argument errors are detected on the host before anything is launched and returned as a negative
 *    qpack_status; a failed launch returns QPACK_ERR_CUDA. Data-dependent conditions are reported through a
 *    device status word (qpack_quantize*) and never trap.
 *  - N == 0 (or M == 0) is accepted and launches nothing.
 */
#ifndef QPACK_H_
#define QPACK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *qpack_stream_t; /* identical to cudaStream_t */

/* Weight formats. Q4G32: INT4 symmetric, group 32, fp32 group scales (P2 §3.1–§3.2, §4.1).
 * Q2S/Q3S/Q5S/Q6S: 256-weight super-blocks of 84/110/176/210 bytes (P1 §2.3 byte table).
 * Q4G32H: the INT4 codes of Q4G32 with fp16 group scales, used rounded (4.5 bpw, P1 §2.1).
 * Q4G16: the INT4 rule of Q4G32 with groups of 16 weights, fp32 scales (6 bpw, P2 §5.1); K a
 * multiple of 32.
 * Q4G32A: INT4 asymmetric, group 32 (P2 §5.1; P1 §2.1's zero-point form w' = s*(q - z)): unsigned codes 0..15,
 * one fp32 pair (s, z) per group with z an integer value 0..15 (6 bpw): lo = min(0, min w), hi = max(0, max w),
 * s = max((hi - lo) / 15, 1e-12), z = clamp(rint(-lo / s), 0, 15), q = clamp(rint(w / s) + z, 0, 15). */
typedef enum {
    QPACK_Q4G32 = 0,
    QPACK_Q2S = 1,
    QPACK_Q3S = 2,
    QPACK_Q5S = 3,
    QPACK_Q6S = 4,
    QPACK_Q4G32H = 5,
    QPACK_Q4G16 = 6,
    QPACK_Q4G32A = 7
} qpack_format;

typedef enum { QPACK_F32 = 0, QPACK_F16 = 1, QPACK_BF16 = 2 } qpack_dtype;

typedef enum {
    QPACK_OK = 0,
    QPACK_ERR_ARG = -1,        /* null pointer where one is required, bad enum, negative size */
    QPACK_ERR_SHAPE = -2,      /* K not a multiple of the format's group (32) or super-block (256), M out of range */
    QPACK_ERR_ALIGN = -3,      /* a pointer or leading dimension breaks the stated alignment */
    QPACK_ERR_RANGE = -4,      /* reserved: data-dependent range failure reported synchronously */
    QPACK_ERR_CUDA = -5,       /* a CUDA runtime call or kernel launch failed */
    QPACK_ERR_UNSUPPORTED = -6 /* format / path combination not provided */
} qpack_status;

/* Bit OR-ed into the device status word when a super-block's fp16 d or dmin, or a Q4G32H fp16 group scale,
 * overflows to infinity (P1 §2.3 warns about fp16 super-scale overflow). */
#define QPACK_FLAG_RANGE 1

/* Sizes of the packed representation (host-only, no GPU work).
 *  row_stride    bytes between consecutive packed rows (super-block formats: rows padded to 16 B, P1 §3.3)
 *  packed_bytes  N * row_stride
 *  scale_stride  INT4 formats: elements between consecutive rows of the separate group-scale array (fp32 for
 *                Q4G32 / Q4G16 / Q4G32A, fp16 for Q4G32H; K/32 (K/16 for Q4G16 and for Q4G32A's (s, z) pairs)
 *                rounded up so that rows are 16 bytes, P2 §4.1); 0 otherwise
 *  scale_bytes   INT4 formats: N * scale_stride * (4 or 2); 0 otherwise
 *  block_bytes   bytes per 256-weight super-block (84/110/176/210, P1 §2.3); 0 for the INT4 formats
 *  nsub          sub-blocks per super-block (16, or 8 for Q5S); for the INT4 formats the groups per row
 *  weight_bytes  packed_bytes + scale_bytes: the bytes one product call streams from memory
 * Returns QPACK_OK, QPACK_ERR_ARG (bad format, negative size, null out) or QPACK_ERR_SHAPE. */
typedef struct {
    int64_t row_stride;
    int64_t packed_bytes;
    int64_t scale_stride;
    int64_t scale_bytes;
    int64_t block_bytes;
    int64_t nsub;
    int64_t weight_bytes;
} qpack_layout_t;
int qpack_layout(int fmt, int64_t N, int64_t K, qpack_layout_t *out);

/* Quantize W into unpacked parts (P2 §3.1 for Q4G32; two-level round-to-nearest for the super-block formats,
 * following P1 §2.1's fp16 super-scale -> sub-block scale -> weight structure: each sub-block's own scale, fp16 d
 * (and dmin) used rounded, integer sub-block scales against it, codes against the rounded sub-block scale).
 *  W          [N, K] of dtype wdt (F32, F16 or BF16), 16-byte aligned
 *  codes      [N, K] int8: the integer q (Q4G32/Q4G32H/Q4G16 -8..7, Q4G32A 0..15, Q3S -4..3, Q6S -32..31,
 *             Q2S 0..3, Q5S 0..31)
 *  gscale     Q4G32: [N, K/32], Q4G16: [N, K/16] fp32 group scales; Q4G32A: [N, K/16] fp32, the pair (s, z) of
 *             group g at 2g, 2g + 1; NULL for other formats
 *  sub_scale  super-block formats: [N, K/256 * nsub] uint8 sub-block scale integers L_j; NULL for the INT4 formats
 *  sub_min    Q2S/Q5S: [N, K/256 * nsub] uint8 sub-block minimum integers M_j; NULL otherwise
 *  d, dmin    super-block formats: [N, K/256] fp16 bits of d; dmin for Q2S/Q5S only (NULL otherwise).
 *             Q4G32H: d holds the [N, K/32] fp16 group scales (2-byte aligned), dmin NULL
 *  status     device int32 (may be NULL): QPACK_FLAG_RANGE is OR-ed in; the caller clears it.
 * The results are bit-identical to the IEEE fp32 definition (round to nearest even, true division, no FMA). */
int qpack_quantize(int fmt, const void *W, int wdt, int64_t N, int64_t K, int8_t *codes, float *gscale,
                   uint8_t *sub_scale, uint8_t *sub_min, uint16_t *d, uint16_t *dmin, int32_t *status,
                   qpack_stream_t stream);

/* Pack unpacked parts (layouts as produced by qpack_quantize) into the format's bytes: P2 §3.2 nibble
 * packing (low nibble = even index) for Q4G32; P1 §2.2 cross-byte packing and §2.3 bit planes for the
 * super-block formats (little-endian fields, weight i at the lowest free bit).
 *  packed        [N, row_stride] bytes, 16-byte aligned; padding bytes are written as zero
 *  group_scales  Q4G32, Q4G16, Q4G32A: [N, scale_stride] fp32, Q4G32H: [N, scale_stride] fp16; 16-byte aligned,
 *                padding written as zero; NULL for the super-block formats. Q4G32A pairs are copied bit for bit;
 *                the products and qpack_dequant read z as an integer 0..15 */
int qpack_pack(int fmt, int64_t N, int64_t K, const int8_t *codes, const float *gscale, const uint8_t *sub_scale,
               const uint8_t *sub_min, const uint16_t *d, const uint16_t *dmin, uint8_t *packed,
               void *group_scales, qpack_stream_t stream);

/* Fused quantize + pack: W straight to packed bytes (and INT4 group scales) in one pass over W.
 * Arguments as qpack_quantize (W, wdt, status) and qpack_pack (packed, group_scales). */
int qpack_quantize_pack(int fmt, const void *W, int wdt, int64_t N, int64_t K, uint8_t *packed,
                        void *group_scales, int32_t *status, qpack_stream_t stream);

/* Inverse of qpack_pack: packed bytes back to unpacked parts (same pointer conventions). */
int qpack_unpack(int fmt, int64_t N, int64_t K, const uint8_t *packed, const void *group_scales, int8_t *codes,
                 float *gscale, uint8_t *sub_scale, uint8_t *sub_min, uint16_t *d, uint16_t *dmin,
                 qpack_stream_t stream);

/* Dequantize a packed matrix to fp32 out [N, K] (the page's self-check path, P1 §3.4): Q4G32 w' = s*q,
 * Q4G32H w' = fp32(s16)*q; Q4G32A w' = s*(q - z);
 * symmetric super-blocks w' = (d*L_j)*q; asymmetric w' = (d*L_j)*q - (dmin*M_j), each step an fp32 rounding,
 * no FMA. out must be 16-byte aligned. */
int qpack_dequant(int fmt, int64_t N, int64_t K, const uint8_t *packed, const void *group_scales, float *out,
                  qpack_stream_t stream);

/* Fused dequant-GEMV (decode, batch 1; P1 §1.2 and §3.3, P2 §3.3 "fused dequantization"):
 *   y[r] = sum_k w'[r,k] * x[k],  r < N
 * packed weights are read exactly once and unpacked in registers. x is rounded once to 16-bit integers per
 * 16-element half of each 32-element unit: step sigma = m / 32767 (m = the half's largest |x|), so every staged
 * value is within m / 65000 of x and the half's largest element is exact to 2.4e-7 relative; code x activation sums
 * are exact int32 within a half, fp32 across halves. Worst case over all finite fp16 x, the staging moves y[r] by at
 * most sqrt(15) / 65000 * ||w'_r||_2 * ||x||_2 = 6.0e-5 * ||w'_r||_2 * ||x||_2.
 *  packed, group_scales  as produced by qpack_pack (group_scales NULL except the INT4 formats), 16-byte aligned
 *  x                     [K] fp16, 16-byte aligned
 *  y                     [N] fp32, 4-byte aligned
 *  K                     any multiple of the format's group (rows longer than one SM's shared memory can stage go
 *                        in K splits whose products are added to y in split order)
 * Parity bound against an fp64 sum: |y[r] - y_ref[r]| <= 1e-4 * ||w'_r||_2 * ||x||_2 for every finite x.
 * Non-finite activations: if x holds an inf or a nan, every y[r] is nan and QPACK_FAULT_NONFINITE_X is set in the
 * fault word (qpack_fetch_fault_flags); the IEEE sum would be nan or +-inf, and the call refuses to pick one. */
int qgemv(int fmt, const uint8_t *packed, const void *group_scales, int64_t N, int64_t K, const uint16_t *x,
          float *y, qpack_stream_t stream);

/* Small-batch decode GEMM (P2 §5.2 decode vs prefill; batch up to 16):
 *   Y[m, r] = sum_k w'[r,k] * X[m,k],  m < M, r < N,  1 <= M <= 16
 * each packed weight is read once and reused across the M activation rows; activations and sums as in qgemv
 * (a non-finite activation makes every output of its row nan and sets QPACK_FAULT_NONFINITE_X).
 *  X  [M, ldx] fp16, 16-byte aligned, ldx >= K and ldx a multiple of 8
 *  Y  [M, ldy] fp32, ldy >= N
 * Same parity bound as qgemv, per element. */
int qgemm_small(int fmt, const uint8_t *packed, const void *group_scales, int64_t N, int64_t K, int M,
                const uint16_t *X, int64_t ldx, float *Y, int64_t ldy, qpack_stream_t stream);

/* Prefill dequant GEMM on the tensor cores (P1 §1.2: prefill is a dense [tokens, hidden] x [hidden, hidden]
 * contraction):
 *   Y[m, n] = sum_k bf16(X[m,k]) * bf16(w'[n,k]),  fp32 accumulation, Y rounded to bf16
 * Weight tiles are dequantized to bf16 in shared memory and fed to tcgen05 MMA with TMEM accumulators; by
 * default two CTAs on two SMs share each MMA (see QPACK_OPT_PREFILL_TILE_ROWS).
 *  formats  the INT4 formats (K a multiple of 64) and the super-block formats (K a multiple of 256)
 *  X        [M, ldx] bf16, 16-byte aligned, ldx >= K, ldx a multiple of 8
 *  Y        [M, ldy] bf16, 2-byte aligned, ldy >= N (16-byte aligned rows with ldy % 8 == 0 store fastest)
 * Parity bound: ||Y - Y_ref||_2 / ||Y_ref||_2 <= 2e-2 with Y_ref in fp64.
 * No workspace argument: accumulators live in TMEM and tiles in shared memory, and Y is written directly. */
int qgemm_prefill(int fmt, const uint8_t *packed, const void *group_scales, int64_t N, int64_t K, int64_t M,
                  const uint16_t *X, int64_t ldx, uint16_t *Y, int64_t ldy, qpack_stream_t stream);

/* 8-bit KV cache (2/3/5/6-bit article §4.1: the KV cache in 8 bits with one fp16 scale per 32 elements, about
 * 1.06 bytes per element instead of 2). Groups are 32 consecutive elements of the flat array.
 *   d = fp16_rn(max|v| / 127) (fp32 division; the rounded d is the one used), q = clamp(rint(v / d), -127, 127),
 *   q = 0 when d == 0.
 *  v       [n] fp16 keys or values, 16-byte aligned; finite (non-finite inputs give unspecified codes, no fault)
 *  codes   [n] int8 out, 8-byte aligned
 *  scales  [n / 32] fp16 out, 2-byte aligned
 *  n       a multiple of 32 (QPACK_ERR_SHAPE otherwise); 0 launches nothing
 * Codes and scales are bit-identical to the oracle's. The caller owns every buffer. */
int qpack_kv_quantize(const uint16_t *v, int64_t n, int8_t *codes, uint16_t *scales, qpack_stream_t stream);

/* Inverse of qpack_kv_quantize (the Mix-Quant article §2.3: the int8 cache dequantized to fp16 in bulk):
 *   out[i] = fp16_rn(d_g * q_i), g = i / 32 (the product is exact in fp32).
 *  codes 8-byte aligned, scales 2-byte aligned, out [n] fp16 16-byte aligned; n a multiple of 32. */
int qpack_kv_dequant(const int8_t *codes, const uint16_t *scales, int64_t n, uint16_t *out, qpack_stream_t stream);

/* Human-readable name of a qpack_status value. Never NULL. */
const char *qpack_status_string(int status);

/* Device-side fault record: bounded waits inside the kernels that give up OR a bit into a per-device word
 * instead of hanging, and the decode products OR in QPACK_FAULT_NONFINITE_X when an activation was inf or nan.
 * Copies the current device's word to *flags (synchronous) and clears it.
 * Returns QPACK_OK or QPACK_ERR_CUDA. A non-zero *flags means some kernel result is invalid. */
#define QPACK_FAULT_NONFINITE_X 16
int qpack_fetch_fault_flags(int32_t *flags);

/* Per-device options (the device current at the call).
 *  QPACK_OPT_WEIGHT_PREFETCH (default 0): when 1, qgemv / qgemm_small launch as programmatic dependents of the
 *  previous kernel in the stream and start streaming their packed weights before that kernel has finished
 *  (activations are still read only after it has finished, and outputs written after). The caller guarantees
 *  that the packed weights and scales of a product are not written by the kernel launched just before it on
 *  that stream (true for a decode loop over resident weights).
 *  QPACK_OPT_PREFILL_TILE_ROWS (default 0): the qgemm_prefill tiling. 256 or 224: pairs of CTAs on two SMs (a
 *  cluster of two), each pair a 512-token x 256- or 224-weight-row block of Y computed by tcgen05 MMAs of M = 256
 *  tokens and N = 256 or 224 weight rows spread over the pair. 112 or 128: one CTA per 512-token x 112- or
 *  128-row block (MMAs of M = 128, N = 112 or 128). 0 (the default) takes the pairs for every format, of 224 rows
 *  where they fill more of the SMs at once (not for Q3S), else of 256. All of them meet the prefill bound.
 * Returns QPACK_OK, QPACK_ERR_ARG (unknown option or value) or QPACK_ERR_CUDA (no current device). Host-only. */
#define QPACK_OPT_WEIGHT_PREFETCH 1
#define QPACK_OPT_PREFILL_TILE_ROWS 2
int qpack_set_option(int option, int value);

/* Library version: major * 10000 + minor * 100 + patch. */
int qpack_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QPACK_H_ */
