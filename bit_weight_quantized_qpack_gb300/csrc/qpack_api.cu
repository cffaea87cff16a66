// qpack_api.cu — the extern "C" entry points of libqpack (declared in include/qpack.h).
//
// Every entry point validates its arguments on the host (null pointers, enum values, shapes, alignment) and
// returns a negative qpack_status without launching anything when they are wrong; otherwise it launches the
// kernels asynchronously on the caller's stream and returns QPACK_OK, or QPACK_ERR_CUDA if a launch failed.
// There is no host fallback: every computation runs in the kernels of this library.
#include <cuda_runtime.h>

#include <mutex>

#include "qpack.h"
#include "qpack_dev.cuh"
#include "qpack_launch.h"

namespace qpack {

int set_weight_prefetch(int v);
int set_prefill_tile_rows(int v);

int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

static int g_weight_prefetch[64] = {0};

int weight_prefetch_enabled() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    return g_weight_prefetch[dev];
}

int set_weight_prefetch(int v) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    g_weight_prefetch[dev] = v ? 1 : 0;
    return 0;
}

static int g_prefill_rows[64] = {0};

int prefill_tile_rows() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    return g_prefill_rows[dev];
}

int set_prefill_tile_rows(int v) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    g_prefill_rows[dev] = v;
    return 0;
}

}  // namespace qpack

namespace {

using namespace qpack;

bool fmt_ok(int fmt) { return fmt >= QPACK_Q4G32 && fmt <= QPACK_Q4G32A; }
bool is_int4_fmt(int fmt) {
    return fmt == QPACK_Q4G32 || fmt == QPACK_Q4G32H || fmt == QPACK_Q4G16 || fmt == QPACK_Q4G32A;
}
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct FmtInfo { int bytes, nsub; bool asym; };
FmtInfo info(int fmt) {
    switch (fmt) {
        case QPACK_Q2S: return {84, 16, true};
        case QPACK_Q3S: return {110, 16, false};
        case QPACK_Q5S: return {176, 8, true};
        case QPACK_Q6S: return {210, 16, false};
        default: return {0, 0, false};
    }
}

int layout(int fmt, int64_t N, int64_t K, qpack_layout_t *o) {
    if (!fmt_ok(fmt) || N < 0 || K < 0 || !o) return QPACK_ERR_ARG;
    if (is_int4_fmt(fmt)) {
        if (K == 0 || K % 32) return QPACK_ERR_SHAPE;
        const int64_t es = fmt == QPACK_Q4G32H ? 2 : 4;   // fp16 or fp32 group scales, rows padded to 16 bytes
        const int64_t g = fmt == QPACK_Q4G16 ? 16 : 32;    // weights per group
        const int64_t epg = fmt == QPACK_Q4G32A ? 2 : 1;   // scale-array entries per group: Q4G32A keeps (s, z)
        o->row_stride = K / 2;
        o->packed_bytes = N * o->row_stride;
        o->scale_stride = round_up(epg * (K / g), 16 / es);
        o->scale_bytes = N * o->scale_stride * es;
        o->block_bytes = 0;
        o->nsub = K / g;
    } else {
        if (K == 0 || K % 256) return QPACK_ERR_SHAPE;
        const FmtInfo f = info(fmt);
        o->row_stride = round_up((K / 256) * f.bytes, 16);
        o->packed_bytes = N * o->row_stride;
        o->scale_stride = 0;
        o->scale_bytes = 0;
        o->block_bytes = f.bytes;
        o->nsub = f.nsub;
    }
    o->weight_bytes = o->packed_bytes + o->scale_bytes;
    return QPACK_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? QPACK_OK : QPACK_ERR_CUDA; }

BlockArgs base_args(int64_t N, int64_t K, const qpack_layout_t &L) {
    BlockArgs a = {};
    a.N = N;
    a.K = K;
    a.nbk = (K + 255) / 256;
    a.row_stride = L.row_stride;
    a.scale_stride = L.scale_stride;
    return a;
}

// Checks shared by the quantize-output / pack-input part pointers.
int check_parts(int fmt, const void *codes, const void *gscale, const void *sub_scale, const void *sub_min,
                const void *d, const void *dmin) {
    if (!codes || !aligned(codes, 16)) return codes ? QPACK_ERR_ALIGN : QPACK_ERR_ARG;
    if (fmt == QPACK_Q4G32 || fmt == QPACK_Q4G16 || fmt == QPACK_Q4G32A) {
        if (!gscale) return QPACK_ERR_ARG;
        if (!aligned(gscale, 4)) return QPACK_ERR_ALIGN;
    } else if (fmt == QPACK_Q4G32H) {                      // the fp16 group scales travel in d
        if (!d) return QPACK_ERR_ARG;
        if (!aligned(d, 2)) return QPACK_ERR_ALIGN;
    } else {
        const FmtInfo f = info(fmt);
        if (!sub_scale || !d) return QPACK_ERR_ARG;
        if (f.asym && (!sub_min || !dmin)) return QPACK_ERR_ARG;
        if (!aligned(d, 2) || (f.asym && !aligned(dmin, 2))) return QPACK_ERR_ALIGN;
    }
    return QPACK_OK;
}

int check_packed(int fmt, const void *packed, const void *gs) {
    if (!packed) return QPACK_ERR_ARG;
    if (!aligned(packed, 16)) return QPACK_ERR_ALIGN;
    if (is_int4_fmt(fmt)) {
        if (!gs) return QPACK_ERR_ARG;
        if (!aligned(gs, 16)) return QPACK_ERR_ALIGN;
    }
    return QPACK_OK;
}

}  // namespace

extern "C" {

int qpack_layout(int fmt, int64_t N, int64_t K, qpack_layout_t *out) { return layout(fmt, N, K, out); }

int qpack_quantize(int fmt, const void *W, int wdt, int64_t N, int64_t K, int8_t *codes, float *gscale,
                   uint8_t *sub_scale, uint8_t *sub_min, uint16_t *d, uint16_t *dmin, int32_t *status,
                   qpack_stream_t stream) {
    qpack_layout_t L;
    int rc = layout(fmt, N, K, &L);
    if (rc) return rc;
    if (wdt < QPACK_F32 || wdt > QPACK_BF16) return QPACK_ERR_ARG;
    if ((rc = check_parts(fmt, codes, gscale, sub_scale, sub_min, d, dmin))) return rc;
    if (!W) return QPACK_ERR_ARG;
    if (!aligned(W, 16) || (status && !aligned(status, 4))) return QPACK_ERR_ALIGN;
    if (N == 0) return QPACK_OK;
    BlockArgs a = base_args(N, K, L);
    a.W = W;
    a.codes = codes;
    a.gscale = gscale;
    a.sub_scale = sub_scale;
    a.sub_min = sub_min;
    a.d = d;
    a.dmin = dmin;
    a.status = status;
    return cuda_status(launch_block_op(fmt, 0, wdt, a, reinterpret_cast<cudaStream_t>(stream)));
}

int qpack_pack(int fmt, int64_t N, int64_t K, const int8_t *codes, const float *gscale, const uint8_t *sub_scale,
               const uint8_t *sub_min, const uint16_t *d, const uint16_t *dmin, uint8_t *packed,
               void *group_scales, qpack_stream_t stream) {
    qpack_layout_t L;
    int rc = layout(fmt, N, K, &L);
    if (rc) return rc;
    if ((rc = check_parts(fmt, codes, gscale, sub_scale, sub_min, d, dmin))) return rc;
    if ((rc = check_packed(fmt, packed, group_scales))) return rc;
    if (N == 0) return QPACK_OK;
    BlockArgs a = base_args(N, K, L);
    a.codes = const_cast<int8_t *>(codes);
    a.gscale = const_cast<float *>(gscale);
    a.sub_scale = const_cast<uint8_t *>(sub_scale);
    a.sub_min = const_cast<uint8_t *>(sub_min);
    a.d = const_cast<uint16_t *>(d);
    a.dmin = const_cast<uint16_t *>(dmin);
    a.packed = packed;
    a.gs_out = static_cast<float *>(group_scales);
    return cuda_status(launch_block_op(fmt, 2, QPACK_F32, a, reinterpret_cast<cudaStream_t>(stream)));
}

int qpack_quantize_pack(int fmt, const void *W, int wdt, int64_t N, int64_t K, uint8_t *packed,
                        void *group_scales, int32_t *status, qpack_stream_t stream) {
    qpack_layout_t L;
    int rc = layout(fmt, N, K, &L);
    if (rc) return rc;
    if (wdt < QPACK_F32 || wdt > QPACK_BF16 || !W) return QPACK_ERR_ARG;
    if ((rc = check_packed(fmt, packed, group_scales))) return rc;
    if (!aligned(W, 16) || (status && !aligned(status, 4))) return QPACK_ERR_ALIGN;
    if (N == 0) return QPACK_OK;
    BlockArgs a = base_args(N, K, L);
    a.W = W;
    a.packed = packed;
    a.gs_out = static_cast<float *>(group_scales);
    a.status = status;
    return cuda_status(launch_block_op(fmt, 1, wdt, a, reinterpret_cast<cudaStream_t>(stream)));
}

int qpack_unpack(int fmt, int64_t N, int64_t K, const uint8_t *packed, const void *group_scales, int8_t *codes,
                 float *gscale, uint8_t *sub_scale, uint8_t *sub_min, uint16_t *d, uint16_t *dmin,
                 qpack_stream_t stream) {
    qpack_layout_t L;
    int rc = layout(fmt, N, K, &L);
    if (rc) return rc;
    if ((rc = check_packed(fmt, packed, group_scales))) return rc;
    if ((rc = check_parts(fmt, codes, gscale, sub_scale, sub_min, d, dmin))) return rc;
    if (N == 0) return QPACK_OK;
    BlockArgs a = base_args(N, K, L);
    a.packed_in = packed;
    a.gs_in = static_cast<const float *>(group_scales);
    a.codes = codes;
    a.gscale = gscale;
    a.sub_scale = sub_scale;
    a.sub_min = sub_min;
    a.d = d;
    a.dmin = dmin;
    return cuda_status(launch_block_op(fmt, 3, QPACK_F32, a, reinterpret_cast<cudaStream_t>(stream)));
}

int qpack_dequant(int fmt, int64_t N, int64_t K, const uint8_t *packed, const void *group_scales, float *out,
                  qpack_stream_t stream) {
    qpack_layout_t L;
    int rc = layout(fmt, N, K, &L);
    if (rc) return rc;
    if ((rc = check_packed(fmt, packed, group_scales))) return rc;
    if (!out) return QPACK_ERR_ARG;
    if (!aligned(out, 16)) return QPACK_ERR_ALIGN;
    if (N == 0) return QPACK_OK;
    BlockArgs a = base_args(N, K, L);
    a.packed_in = packed;
    a.gs_in = static_cast<const float *>(group_scales);
    a.out = out;
    return cuda_status(launch_block_op(fmt, 4, QPACK_F32, a, reinterpret_cast<cudaStream_t>(stream)));
}

int qgemm_small(int fmt, const uint8_t *packed, const void *group_scales, int64_t N, int64_t K, int M,
                const uint16_t *X, int64_t ldx, float *Y, int64_t ldy, qpack_stream_t stream) {
    qpack_layout_t L;
    int rc = layout(fmt, N, K, &L);
    if (rc) return rc;
    if ((rc = check_packed(fmt, packed, group_scales))) return rc;
    if (M < 0 || M > 16) return QPACK_ERR_SHAPE;
    if (!X || !Y) return QPACK_ERR_ARG;
    if (ldx < K || ldy < N) return QPACK_ERR_SHAPE;
    if (!aligned(X, 16) || (ldx % 8) || !aligned(Y, 4)) return QPACK_ERR_ALIGN;
    if (N == 0 || M == 0) return QPACK_OK;
    GemvArgs a = {};
    a.packed = packed;
    a.gscale = static_cast<const float *>(group_scales);
    a.N = N;
    a.K = K;
    a.row_stride = L.row_stride;
    a.scale_stride = L.scale_stride;
    a.X = X;
    a.ldx = ldx;
    a.Y = Y;
    a.ldy = ldy;
    a.M = M;
    a.weight_prefetch = weight_prefetch_enabled();
    return cuda_status(launch_gemv(fmt, a, reinterpret_cast<cudaStream_t>(stream)));
}

int qgemv(int fmt, const uint8_t *packed, const void *group_scales, int64_t N, int64_t K, const uint16_t *x,
          float *y, qpack_stream_t stream) {
    return qgemm_small(fmt, packed, group_scales, N, K, 1, x, K, y, N, stream);
}

int qgemm_prefill(int fmt, const uint8_t *packed, const void *group_scales, int64_t N, int64_t K, int64_t M,
                  const uint16_t *X, int64_t ldx, uint16_t *Y, int64_t ldy, qpack_stream_t stream) {
    qpack_layout_t L;
    int rc = layout(fmt, N, K, &L);
    if (rc) return rc;
    if ((rc = check_packed(fmt, packed, group_scales))) return rc;
    if (M < 0) return QPACK_ERR_SHAPE;
    if (is_int4_fmt(fmt) && K % 64) return QPACK_ERR_SHAPE;
    if (!X || !Y) return QPACK_ERR_ARG;
    if (ldx < K || ldy < N) return QPACK_ERR_SHAPE;
    if (!aligned(X, 16) || (ldx % 8) || !aligned(Y, 2)) return QPACK_ERR_ALIGN;
    if (N == 0 || M == 0) return QPACK_OK;
    PrefillArgs a = {};
    a.packed = packed;
    a.gscale = static_cast<const float *>(group_scales);
    a.N = N;
    a.K = K;
    a.M = M;
    a.row_stride = L.row_stride;
    a.scale_stride = L.scale_stride;
    a.X = X;
    a.ldx = ldx;
    a.Y = Y;
    a.ldy = ldy;
    a.vec_y = (aligned(Y, 16) && ldy % 8 == 0) ? 1 : 0;
    const cudaError_t e = launch_prefill(fmt, a, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return QPACK_ERR_UNSUPPORTED;
    return cuda_status(e);
}

int qpack_kv_quantize(const uint16_t *v, int64_t n, int8_t *codes, uint16_t *scales, qpack_stream_t stream) {
    if (n < 0 || n % 32 != 0) return QPACK_ERR_SHAPE;
    if (n == 0) return QPACK_OK;
    if (!v || !codes || !scales) return QPACK_ERR_ARG;
    if (!aligned(v, 16) || !aligned(codes, 8) || !aligned(scales, 2)) return QPACK_ERR_ALIGN;
    return cuda_status(launch_kv_quantize(v, n, codes, scales, reinterpret_cast<cudaStream_t>(stream)));
}

int qpack_kv_dequant(const int8_t *codes, const uint16_t *scales, int64_t n, uint16_t *out, qpack_stream_t stream) {
    if (n < 0 || n % 32 != 0) return QPACK_ERR_SHAPE;
    if (n == 0) return QPACK_OK;
    if (!codes || !scales || !out) return QPACK_ERR_ARG;
    if (!aligned(codes, 8) || !aligned(scales, 2) || !aligned(out, 16)) return QPACK_ERR_ALIGN;
    return cuda_status(launch_kv_dequant(codes, scales, n, out, reinterpret_cast<cudaStream_t>(stream)));
}

const char *qpack_status_string(int status) {
    switch (status) {
        case QPACK_OK: return "QPACK_OK";
        case QPACK_ERR_ARG: return "QPACK_ERR_ARG: null pointer, bad enum or negative size";
        case QPACK_ERR_SHAPE: return "QPACK_ERR_SHAPE: K not a multiple of the group / super-block, or M out of range";
        case QPACK_ERR_ALIGN: return "QPACK_ERR_ALIGN: pointer or leading dimension misaligned";
        case QPACK_ERR_RANGE: return "QPACK_ERR_RANGE: value out of the format's range";
        case QPACK_ERR_CUDA: return "QPACK_ERR_CUDA: a CUDA call or kernel launch failed";
        case QPACK_ERR_UNSUPPORTED: return "QPACK_ERR_UNSUPPORTED: path not provided for this format / size";
        default: return "unknown qpack status";
    }
}

int qpack_fetch_fault_flags(int32_t *flags) {
    if (!flags) return QPACK_ERR_ARG;
    *flags = 0;
    cudaError_t e = fetch_fault_gemv(flags);
    if (e == cudaSuccess) e = fetch_fault_prefill(flags);
    return cuda_status(e);
}

int qpack_set_option(int option, int value) {
    if (option == QPACK_OPT_WEIGHT_PREFETCH) return set_weight_prefetch(value) == 0 ? QPACK_OK : QPACK_ERR_CUDA;
    if (option == QPACK_OPT_PREFILL_TILE_ROWS) {
        if (value != 0 && value != 112 && value != 128 && value != 224 && value != 256) return QPACK_ERR_ARG;
        return set_prefill_tile_rows(value) == 0 ? QPACK_OK : QPACK_ERR_CUDA;
    }
    return QPACK_ERR_ARG;
}

int qpack_version(void) { return 1 * 10000 + 0 * 100 + 0; }

}  // extern "C"
