// qpack_prefill.cu — prefill dequant GEMM on the 5th-generation tensor cores (sm_103a):
//   Y[m, n] = sum_k bf16(X[m, k]) * bf16(w'[n, k]),  fp32 accumulation in tensor memory, Y rounded to bf16.
//
// Prefill is a dense [tokens, hidden] x [hidden, hidden] contraction (2/3/5/6-bit article,
// lpnh.cn/news/2857666, §1.2), so it belongs on the tensor cores; the packed weights are still read in their
// compact form and dequantized on chip (DBHOO-CIM article, pwwt.cn/news/4452170, §3.3: no fp32 weight array).
//
// One CTA computes a 128 x 256 tile of Y:
//   warps 0..3  producers: per 64-wide K step, stage the 128 x 64 bf16 X tile and dequantize the 256 x 64 weight
//               tile (exact fp32 dequant of FORMATS.md, then bf16 round-to-nearest-even) into shared memory in
//               the 128-byte-swizzled K-major layout the MMA reads; afterwards they are the epilogue warps
//               (tcgen05.ld of their 32 TMEM lanes, bf16 conversion, global stores).
//   warp 4      allocates 256 TMEM columns (the fp32 128 x 256 accumulator); lane 0 issues the tcgen05.mma
//               instructions (M=128, N=256, K=16 each, both operands from shared-memory descriptors) and commits
//               them to mbarriers that free the stage and, at the end, publish the accumulator.
// Every wait is bounded; on a timeout the kernel records a fault bit, skips the remaining work, still frees its
// TMEM and returns.
#include <cuda_runtime.h>

#include "qpack_dev.cuh"
#include "qpack_launch.h"

namespace qpack {

__device__ int g_fault_prefill = 0;

namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int STAGES = 3;
constexpr int A_BYTES = BM * BK * 2;               // 16 KB
constexpr int B_BYTES = BN * BK * 2;               // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;     // 48 KB (multiple of 1024)
constexpr int NPROD = 128;                         // producer / epilogue threads
constexpr int THREADS = NPROD + 32;
constexpr uint32_t TMEM_COLS = 256;
constexpr int SMEM_BYTES = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + 256 /*barriers*/;

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
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

// Byte offset of the 16-byte chunk c (K elements 8c..8c+7) of row r inside a 128B-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t c) {
    return (r >> 3) * 1024u + (r & 7u) * 128u + ((c ^ (r & 7u)) << 4);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    return lo | (hi << 16);
}

__device__ __forceinline__ uint32_t ldg_u8(const uint8_t *p) { return __ldg(p); }
__device__ __forceinline__ uint32_t ldg_u16(const uint8_t *p) { return uint32_t(__ldg(p)) | (uint32_t(__ldg(p + 1)) << 8); }
__device__ __forceinline__ uint32_t ldg_u24(const uint8_t *p) { return ldg_u16(p) | (uint32_t(__ldg(p + 2)) << 16); }

// Dequantize 64 consecutive weights (k0 .. k0+63, k0 a multiple of 64) of one packed row to fp32, exactly as
// FORMATS.md (the same roundings as the dequant kernel and the CPU reference).
template <int F>
__device__ __forceinline__ void dequant64(const uint8_t *row, const float *gs_row, uint32_t k0, float w[64]) {
    if constexpr (F == FMT_Q4G32) {
        const uint4 *cp = reinterpret_cast<const uint4 *>(row + k0 / 2);
        const float s0 = __ldg(gs_row + k0 / 32), s1 = __ldg(gs_row + k0 / 32 + 1);
#pragma unroll
        for (int v = 0; v < 2; ++v) {
            const uint4 c = __ldg(cp + v);
            const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
            const float s = v ? s1 : s0;
#pragma unroll
            for (int i = 0; i < 32; ++i) w[32 * v + i] = __fmul_rn(s, float(int((cw[i >> 3] >> (4 * (i & 7))) & 15u) - 8));
        }
    } else {
        const uint32_t b = k0 / 256, j = (k0 % 256) / 64;      // super-block, quarter within it
        const uint8_t *blk = row + b * Fmt<F>::bytes;
        if constexpr (F == FMT_Q2S) {
            const float D = h2f_bits(uint16_t(ldg_u16(blk + 80))), Dm = h2f_bits(uint16_t(ldg_u16(blk + 82)));
#pragma unroll
            for (int sbi = 0; sbi < 4; ++sbi) {
                const uint32_t lm = ldg_u8(blk + 64 + 4 * j + sbi);
                const float es = __fmul_rn(D, float(lm & 15u)), em = __fmul_rn(Dm, float(lm >> 4));
                const uint32_t cw = ldg_u8(blk + 16 * j + 4 * sbi) | (ldg_u8(blk + 16 * j + 4 * sbi + 1) << 8) |
                                    (ldg_u8(blk + 16 * j + 4 * sbi + 2) << 16) | (ldg_u8(blk + 16 * j + 4 * sbi + 3) << 24);
#pragma unroll
                for (int i = 0; i < 16; ++i) w[16 * sbi + i] = __fsub_rn(__fmul_rn(es, float((cw >> (2 * i)) & 3u)), em);
            }
        } else if constexpr (F == FMT_Q3S) {
            const float D = h2f_bits(uint16_t(ldg_u16(blk + 108)));
            const uint32_t f = ldg_u24(blk + 96 + 3 * j);          // L_{4j .. 4j+3}
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const uint32_t v = ldg_u24(blk + 24 * j + 3 * g);
                const float es = __fmul_rn(D, float((f >> (6 * (g >> 1))) & 63u));
#pragma unroll
                for (int t = 0; t < 8; ++t) w[8 * g + t] = __fmul_rn(es, float(int((v >> (3 * t)) & 7u) - 4));
            }
        } else if constexpr (F == FMT_Q5S) {
            const float D = h2f_bits(uint16_t(ldg_u16(blk + 172))), Dm = h2f_bits(uint16_t(ldg_u16(blk + 174)));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t sub = 2 * j + h;                    // sub-block of 32
                const uint32_t fl = ldg_u24(blk + 160 + 3 * (sub >> 2)), fm = ldg_u24(blk + 166 + 3 * (sub >> 2));
                const float es = __fmul_rn(D, float((fl >> (6 * (sub & 3))) & 63u));
                const float em = __fmul_rn(Dm, float((fm >> (6 * (sub & 3))) & 63u));
                const uint32_t H = ldg_u8(blk + 128 + 4 * sub) | (ldg_u8(blk + 129 + 4 * sub) << 8) |
                                   (ldg_u8(blk + 130 + 4 * sub) << 16) | (ldg_u8(blk + 131 + 4 * sub) << 24);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const uint32_t lo = (ldg_u8(blk + 16 * sub + (i >> 1)) >> (4 * (i & 1))) & 15u;
                    const uint32_t u = lo | (((H >> i) & 1u) << 4);
                    w[32 * h + i] = __fsub_rn(__fmul_rn(es, float(u)), em);
                }
            }
        } else {
            const float D = h2f_bits(uint16_t(ldg_u16(blk + 208)));
#pragma unroll
            for (int sbi = 0; sbi < 4; ++sbi) {
                const uint32_t sub = 4 * j + sbi;                  // sub-block of 16
                const float es = __fmul_rn(D, float(int8_t(ldg_u8(blk + 192 + sub))));
                const uint32_t hw = ldg_u8(blk + 128 + 4 * sub) | (ldg_u8(blk + 129 + 4 * sub) << 8) |
                                    (ldg_u8(blk + 130 + 4 * sub) << 16) | (ldg_u8(blk + 131 + 4 * sub) << 24);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint32_t ii = 16 * sub + i;
                    const uint32_t lo = (ldg_u8(blk + (ii >> 1)) >> (4 * (ii & 1))) & 15u;
                    const uint32_t u = lo | (((hw >> (2 * i)) & 3u) << 4);
                    w[16 * sbi + i] = __fmul_rn(es, float(int(u) - 32));
                }
            }
        }
    }
}

}  // namespace

template <int F>
__global__ void __launch_bounds__(THREADS, 1) prefill_kernel(PrefillArgs a) {
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

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], NPROD); mbar_init(&empty[s], 1); }
        mbar_init(accum, 1);
        fence_mbar_init();
    }
    if (warp == 4) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot;
    bool dead = false;

    if (warp < 4) {
        // ---------------------------------- producers ----------------------------------
        const int t = tid;                                                  // 0..127
        for (int kt = 0; kt < nk && !dead; ++kt) {
            const int s = kt % STAGES;
            if (kt >= STAGES && !mbar_wait_bounded(&empty[s], uint32_t((kt / STAGES) - 1) & 1u)) {
                atomicOr(&g_fault_prefill, FAULT_WAIT_EMPTY);
                dead = true;
                break;
            }
            uint8_t *As = sm + s * STAGE_BYTES;
            uint8_t *Bs = As + A_BYTES;
            const int64_t k0 = int64_t(kt) * BK;
            // X tile: row t of the 128 x 64 bf16 tile, eight 16-byte chunks
            {
                const int64_t m = m0 + t;
                uint4 v[8];
                if (m < M) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(a.X + m * a.ldx + k0);
#pragma unroll
                    for (int c = 0; c < 8; ++c) v[c] = __ldg(src + c);
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c) v[c] = make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(As + sw128_off(uint32_t(t), uint32_t(c))) = v[c];
            }
            // weight tile: rows t and t + 128 of the 256 x 64 bf16 tile
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                const uint32_t r = uint32_t(t + 128 * h);
                const int64_t n = n0 + r;
                uint4 v[8];
                if (n < N) {
                    float w[64];
                    dequant64<F>(a.packed + n * a.row_stride, a.gscale ? a.gscale + n * a.scale_stride : nullptr,
                                 uint32_t(k0), w);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        v[c] = make_uint4(pack_bf16x2(w[8 * c], w[8 * c + 1]), pack_bf16x2(w[8 * c + 2], w[8 * c + 3]),
                                          pack_bf16x2(w[8 * c + 4], w[8 * c + 5]), pack_bf16x2(w[8 * c + 6], w[8 * c + 7]));
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c) v[c] = make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(Bs + sw128_off(r, uint32_t(c))) = v[c];
            }
            fence_proxy_async_smem();      // make the generic-proxy stores visible to the tensor core
            mbar_arrive(&full[s]);
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
            const int64_t m = m0 + 32 * warp + lane;
            const uint32_t lane_base = tmem_d + (uint32_t(32 * warp) << 16);
#pragma unroll 1
            for (int cc = 0; cc < BN / 32; ++cc) {
                uint32_t r[32];
                tmem_ld32(lane_base + uint32_t(32 * cc), r);
                tmem_ld_wait();
                const int64_t nc = n0 + 32 * cc;
                if (m < M && nc < N) {
                    uint16_t *dst = a.Y + m * a.ldy + nc;
                    if (nc + 32 <= N && a.vec_y) {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            d4[q] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * q]), __uint_as_float(r[8 * q + 1])),
                                               pack_bf16x2(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3])),
                                               pack_bf16x2(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5])),
                                               pack_bf16x2(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7])));
                    } else {
                        for (int q = 0; q < 32 && nc + q < N; ++q)
                            dst[q] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[q])));
                    }
                }
            }
        }
    } else {
        // ------------------------------------ MMA issuer ------------------------------------
        if (lane == 0) {
            for (int kt = 0; kt < nk; ++kt) {
                const int s = kt % STAGES;
                if (!mbar_wait_bounded(&full[s], uint32_t(kt / STAGES) & 1u)) {
                    atomicOr(&g_fault_prefill, FAULT_WAIT_FULL);
                    dead = true;
                    break;
                }
                tc_fence_after();
                const uint32_t As = base + uint32_t(s * STAGE_BYTES), Bs = As + A_BYTES;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_bf16(tmem_d, sw128_kmajor_desc(As + 32u * k), sw128_kmajor_desc(Bs + 32u * k), IDESC,
                              (kt > 0 || k > 0) ? 1u : 0u);
                umma_commit(&empty[s]);                 // the stage may be refilled once these MMAs have read it
            }
            umma_commit(accum);                         // accumulator complete (also on the failure path)
        }
        __syncwarp();
    }

    // ---- teardown: every TMEM read is finished; free the accumulator ----
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        if (lane == 0 && dead) {
            // On the failure path wait (bounded) for the MMAs already issued before freeing their TMEM.
            (void)mbar_wait_bounded(accum, 0u, 1u << 16);
        }
        __syncwarp();
        tmem_dealloc(tmem_d, TMEM_COLS);
    }
}

template <int F>
static cudaError_t launch_prefill_f(const PrefillArgs &a, cudaStream_t s) {
    static int opted[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!opted[dev]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        opted[dev] = 1;
    }
    dim3 grid(unsigned((a.N + BN - 1) / BN), unsigned((a.M + BM - 1) / BM));
    if (grid.y > 65535u) return cudaErrorInvalidValue;
    prefill_kernel<F><<<grid, THREADS, SMEM_BYTES, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_prefill(int fmt, const PrefillArgs &a, cudaStream_t s) {
    switch (fmt) {
        case FMT_Q4G32: return launch_prefill_f<FMT_Q4G32>(a, s);
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
