// bqg_gemm.cu -- prefill GEMM (M = 512) on the sm_103a tensor cores.
#include "bqg_common.cuh"

namespace bqg {

// Error word set by bounded device-side waits (0 = none).
__device__ int g_gemm_error;

int gemm_read_error(cudaStream_t stream, int *out)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess) return BQG_ERR_CUDA;
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(int)) != cudaSuccess) return BQG_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(int)) != cudaSuccess) return BQG_ERR_CUDA;
    *out = v;
    return BQG_OK;
}

size_t gemm_workspace(int, int64_t, int64_t) { return 0; }

int gemm_q4_0_bf16(const void *, const void *, float *, int, int64_t, int64_t, cudaStream_t, int)
{
    return BQG_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace bqg
