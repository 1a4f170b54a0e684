// gemv_q4_0_q8_1.cu -- instantiations of the skinny-GEMV kernel for W_Q4_0 weights x X_Q8_1 activations.
#include "bqg_gemv.cuh"
#include "bqg_gemv_mma.cuh"

namespace bqg {
// The check instantiation of the q4_0 x q8_1 kernel at M = 1 (every rows-per-
// lane choice the planner can make for it): same staging, stream and dot
// routine as the GEMV, plus the integer block dots in p.dots.  With
// `occupancy` set it only prepares the kernel (its shared-memory limit) and
// reports its occupancy.
static cudaError_t gemv_lpr_dots_dispatch(const GemvParams &p, dim3 grid, int threads, size_t smem,
                                                   cudaStream_t stream, int *occupancy)
{
    if (p.rl == 1) return gemv_lpr_launch_one<W_Q4_0, X_Q8_1, 1, 1, true>(p, grid, threads, smem, stream, false, occupancy);
    if (p.rl == 2) return gemv_lpr_launch_one<W_Q4_0, X_Q8_1, 1, 2, true>(p, grid, threads, smem, stream, false, occupancy);
    if (p.rl == 4) return gemv_lpr_launch_one<W_Q4_0, X_Q8_1, 1, 4, true>(p, grid, threads, smem, stream, false, occupancy);
    return cudaErrorInvalidValue;
}

cudaError_t gemv_run_q4_0_q8_1(const GemvParams &p, int M, int C, dim3 grid, int threads, size_t smem,
                        cudaStream_t stream, bool pdl, int *occupancy)
{
    return gemv_dispatch<W_Q4_0, X_Q8_1>(p, M, C, grid, threads, smem, stream, pdl, occupancy);
}
cudaError_t gemv_error_q4_0_q8_1(int *out) { return gemv_take_error(out); }
cudaError_t gemv_lpr_run_q4_0_q8_1(const GemvParams &p, int M, dim3 grid, int threads, size_t smem, cudaStream_t stream,
                            bool pdl, int *occupancy)
{
    return gemv_lpr_dispatch<W_Q4_0, X_Q8_1>(p, M, grid, threads, smem, stream, pdl, occupancy);
}
cudaError_t gemv_lpr_dots_run_q4_0_q8_1(const GemvParams &p, dim3 grid, int threads, size_t smem, cudaStream_t stream,
                                        int *occupancy)
{
    return gemv_lpr_dots_dispatch(p, grid, threads, smem, stream, occupancy);
}
int gemv_x_stage_bytes_q4_0_q8_1(int nc, int nb, int) { return x_stage_row_bytes<W_Q4_0, X_Q8_1>(nc, nb); }
cudaError_t gemv_mma_run_q4_0_q8_1(const CUtensorMap &wmap, const CUtensorMap &smap, const MmaParams &p, int M, dim3 grid,
                                  int threads, size_t smem, cudaStream_t stream, bool pdl, int *occupancy)
{
    return gemv_mma_launch<W_Q4_0, X_Q8_1>(wmap, smap, p, M, grid, threads, smem, stream, pdl, occupancy);
}
}  // namespace bqg
