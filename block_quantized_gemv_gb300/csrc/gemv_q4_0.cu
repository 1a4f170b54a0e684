// gemv_q4_0.cu -- instantiations of the skinny-GEMV kernel for W_Q4_0 weights x X_BF16 activations.
#include "bqg_gemv.cuh"
#include "bqg_gemv_mma.cuh"

namespace bqg {
cudaError_t gemv_run_q4_0(const GemvParams &p, int M, int C, dim3 grid, int threads, size_t smem,
                        cudaStream_t stream, bool pdl, int *occupancy)
{
    return gemv_dispatch<W_Q4_0, X_BF16>(p, M, C, grid, threads, smem, stream, pdl, occupancy);
}
cudaError_t gemv_error_q4_0(int *out) { return gemv_take_error(out); }
cudaError_t gemv_lpr_run_q4_0(const GemvParams &p, int M, dim3 grid, int threads, size_t smem, cudaStream_t stream,
                            bool pdl, int *occupancy)
{
    return gemv_lpr_dispatch<W_Q4_0, X_BF16>(p, M, grid, threads, smem, stream, pdl, occupancy);
}
int gemv_x_stage_bytes_q4_0(int nc, int nb, int bf16) { return bf16 ? x_stage_row_bytes<W_Q4_0, X_BF16>(nc, nb) : x_stage_row_bytes<W_Q4_0, X_F32>(nc, nb); }
cudaError_t gemv_mma_run_q4_0(const CUtensorMap &wmap, const CUtensorMap &smap, const MmaParams &p, int M, dim3 grid, int threads, size_t smem,
                            cudaStream_t stream, bool pdl, int *occupancy)
{
    return gemv_mma_launch<W_Q4_0, X_BF16>(wmap, smap, p, M, grid, threads, smem, stream, pdl, occupancy);
}
}  // namespace bqg
