// qpack_prefill.cu — tensor-core prefill dequant GEMM (placeholder until the tcgen05 kernel lands).
#include <cuda_runtime.h>

#include "qpack_dev.cuh"
#include "qpack_launch.h"

namespace qpack {

__device__ int g_fault_prefill = 0;

cudaError_t launch_prefill(int, const PrefillArgs &, cudaStream_t) { return cudaErrorNotSupported; }

cudaError_t fetch_fault_prefill(int32_t *flags) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_fault_prefill, sizeof(int));
    if (e != cudaSuccess) return e;
    *flags |= v;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_fault_prefill, &zero, sizeof(int));
}

}  // namespace qpack
