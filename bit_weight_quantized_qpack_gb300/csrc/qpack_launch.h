// qpack_launch.h — host-side interface between the C ABI (qpack_api.cu) and the kernel translation units.
// Argument validation happens in the C ABI layer; these launchers assume valid arguments.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace qpack {

// Arguments of the per-256-weight-block kernels (quantize / pack / unpack / dequant). Unused pointers are null.
struct BlockArgs {
    const void *W;            // quantize input [N, K] (f32 / f16 / bf16)
    int64_t N, K;
    int64_t nbk;              // 256-weight blocks per row (ceil(K / 256))
    int64_t row_stride;       // packed bytes per row
    int64_t scale_stride;     // Q4G32 packed scale floats per row
    int8_t *codes;            // [N, K] signed codes (written by quantize/unpack, read by pack)
    float *gscale;            // Q4G32 [N, K/32]
    uint8_t *sub_scale;       // [N, nbk * nsub]
    uint8_t *sub_min;         // [N, nbk * nsub] (asymmetric formats)
    uint16_t *d;              // [N, nbk]
    uint16_t *dmin;           // [N, nbk] (asymmetric formats)
    uint8_t *packed;          // packed output
    float *gs_out;            // Q4G32 packed scale output [N, scale_stride]
    const uint8_t *packed_in; // packed input (unpack / dequant)
    const float *gs_in;       // Q4G32 packed scale input
    float *out;               // dequant output [N, K]
    int32_t *status;          // RANGE flag word (quantize modes), may be null
};

// mode: 0 quantize->parts, 1 quantize->packed, 2 parts->packed, 3 packed->parts, 4 packed->fp32
cudaError_t launch_block_op(int fmt, int mode, int wdt, const BlockArgs &a, cudaStream_t s);

// Arguments of the streaming products (qgemv / qgemm_small).
struct GemvArgs {
    const uint8_t *packed;
    const float *gscale;      // Q4G32 packed scales, else null
    int64_t N, K;
    int64_t row_stride;       // bytes
    int64_t scale_stride;     // floats (Q4G32)
    const uint16_t *X;        // [M, ldx] fp16
    int64_t ldx;
    float *Y;                 // [M, ldy] fp32
    int64_t ldy;
    int M;
    int weight_prefetch;      // 1: launched as a programmatic dependent of the previous kernel and allowed to
                              //    stream packed weights before that kernel has finished (caller's opt-in)
    int64_t kc0;              // first K chunk of this launch: it covers columns [kc0 * chunk, kc0 * chunk + K) of
                              //    the packed rows (X already points at column kc0 * chunk)
    int accumulate;           // 1: add the products to Y (a later K split), 0: overwrite Y
};
cudaError_t launch_gemv(int fmt, const GemvArgs &a, cudaStream_t s);

// Arguments of the tensor-core prefill GEMM.
struct PrefillArgs {
    const uint8_t *packed;
    const float *gscale;
    int64_t N, K, M;
    int64_t row_stride;
    int64_t scale_stride;
    const uint16_t *X;        // bf16 [M, ldx]
    int64_t ldx;
    uint16_t *Y;              // bf16 [M, ldy]
    int64_t ldy;
    int vec_y;                // 1 when Y rows allow 16-byte stores (Y 16-byte aligned, ldy % 8 == 0)
};
cudaError_t launch_prefill(int fmt, const PrefillArgs &a, cudaStream_t s);

// Per-translation-unit device fault words (bounded waits that gave up). Read and cleared synchronously.
// 8-bit KV cache (qpack_kv.cu); n a positive multiple of 32, pointers checked by the caller.
cudaError_t launch_kv_quantize(const uint16_t *v, int64_t n, int8_t *q, uint16_t *scales, cudaStream_t s);
cudaError_t launch_kv_dequant(const int8_t *q, const uint16_t *scales, int64_t n, uint16_t *out, cudaStream_t s);
cudaError_t fetch_fault_gemv(int32_t *flags);
cudaError_t fetch_fault_prefill(int32_t *flags);

int num_sms();
int weight_prefetch_enabled();   // per-device option QPACK_OPT_WEIGHT_PREFETCH
int prefill_tile_rows();         // per-device option QPACK_OPT_PREFILL_TILE_ROWS (0: chosen per launch)

}  // namespace qpack
