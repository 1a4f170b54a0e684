// bqg_quant.cu -- block encoders, the load-time repack and the block-dot
// debug export.
//
// Encoders (one warp per 32-element block, lane i = element i):
//   q8_0 / q8_1 : d = fp16_rn(amax / 127), q = round_half_away(x / d) in
//                 IEEE fp32, clamped to [-127, 127]; d == 0 gives q = 0;
//                 q8_1 also stores s = fp16_rn(d * sum q) (exact product).
//   q4_0        : m = first element of largest |x|, d = fp16_rn(m / -8),
//                 q = clamp(round_half_away(x / d) + 8, 0, 15); d == 0 gives 8.
// The formats are the llama.cpp-style blocks the pages rely on ("MI50
// megakernel": 18-byte q4_0 blocks; "rx-6700xt-llama2-decode": Q8_1
// activations of the integer-dot matvec).  Divisions use __fdiv_rn so the
// result does not depend on fast-math flags.
#include "bqg_gemv.cuh"

namespace bqg {


__device__ __forceinline__ float load_act(const void *x, int x_f32, int64_t i)
{
    if (x_f32) return reinterpret_cast<const float *>(x)[i];
    const uint16_t b = reinterpret_cast<const uint16_t *>(x)[i];
    return __uint_as_float((uint32_t)b << 16);
}


// M x K activations -> M x K/32 q8_1 blocks (36 B)
__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const void *__restrict__ x, int x_f32,
                                                            uint8_t *__restrict__ xq, int64_t nblocks,
                                                            int nb, int64_t K)
{
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (blk >= nblocks) return;
    const int64_t m = blk / nb, b = blk - (blk / nb) * nb;
    q8_1_encode_warp(load_act(x, x_f32, m * K + b * QK + lane), lane, xq + blk * Q8_1_BYTES);
}

// Fused RMSNorm -> q8_1, one CTA per activation row ("MI50 megakernel",
// hypothesis ledger: neighbouring steps fused into one dispatch; the Q8_1
// activation of "rx-6700xt-llama2-decode").  s = sum x^2 is accumulated in
// fp64, which is exact for bf16 inputs whatever the order (each square has
// 16 significant bits), r = fp32(1 / sqrt(s / K + eps)) in fp64, then
// y = fp32(fp32(x * r) * gamma) goes through the q8_1 encoder, one warp per
// block.
__global__ void __launch_bounds__(256) rmsnorm_q8_1_kernel(const void *__restrict__ x, int x_f32,
                                                           const float *__restrict__ gamma, float eps,
                                                           uint8_t *__restrict__ xq, int nb, int64_t K)
{
    __shared__ double part[8];
    __shared__ float s_r;
    pdl_wait();
    pdl_launch_dependents();
    const int64_t m = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    double s = 0.0;
    for (int64_t k = tid; k < K; k += 256) {
        const double v = (double)load_act(x, x_f32, m * K + k);
        s += v * v;                                   // exact square (<= 48 bits)
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) part[warp] = s;
    __syncthreads();
    if (tid == 0) {
        double t = 0.0;
        for (int w = 0; w < 8; w++) t += part[w];
        s_r = (float)(1.0 / sqrt(t / (double)K + (double)eps));
    }
    __syncthreads();
    const float r = s_r;
    for (int b = warp; b < nb; b += 8) {
        const int64_t k = (int64_t)b * QK + lane;
        float y = __fmul_rn(load_act(x, x_f32, m * K + k), r);
        if (gamma) y = __fmul_rn(y, gamma[k]);
        q8_1_encode_warp(y, lane, xq + (m * nb + b) * Q8_1_BYTES);
    }
}

// N x K fp32 weights -> canonical q8_0 (34 B) or q4_0 (18 B) blocks
__global__ void __launch_bounds__(256) quantize_weights_kernel(const float *__restrict__ W, int fmt,
                                                               uint8_t *__restrict__ dst, int64_t nblocks,
                                                               int nb, int64_t K)
{
    const int lane = threadIdx.x & 31;
    const int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (blk >= nblocks) return;
    const int64_t n = blk / nb, b = blk - (blk / nb) * nb;
    const float v = W[n * K + b * QK + lane];
    if (fmt == BQG_Q8_0) {
        const float amax = warp_max(fabsf(v));
        const __half dh = __float2half_rn(__fdiv_rn(amax, 127.0f));
        const int q = q8_code(v, __half2float(dh));
        uint8_t *out = dst + blk * Q8_0_BYTES;
        out[2 + lane] = (uint8_t)(int8_t)q;
        if (lane == 0) *reinterpret_cast<uint16_t *>(out) = __half_as_ushort(dh);
    } else {
        // signed element of largest magnitude, lowest lane on ties
        float bv = v, ba = fabsf(v);
        int bi = lane;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const float oa = __shfl_xor_sync(0xffffffffu, ba, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oa > ba || (oa == ba && oi < bi)) { bv = ov; ba = oa; bi = oi; }
        }
        const __half dh = __float2half_rn(__fdiv_rn(bv, -8.0f));
        const float d = __half2float(dh);
        int q = 8;
        if (d != 0.0f) q = (int)fminf(fmaxf(roundf(__fdiv_rn(v, d)) + 8.0f, 0.0f), 15.0f);
        const int qhi = __shfl_down_sync(0xffffffffu, q, 16);
        uint8_t *out = dst + blk * Q4_0_BYTES;
        if (lane < 16) out[2 + lane] = (uint8_t)(q | (qhi << 4));
        if (lane == 0) *reinterpret_cast<uint16_t *>(out) = __half_as_ushort(dh);
    }
}

// Canonical -> repacked (include/bqgemv.h).  One thread per (row, tile slot);
// slots past the last block are zero-filled.  Canonical blocks are only
// 2-byte aligned, so they are read as 16-bit words.
__global__ void __launch_bounds__(256) repack_kernel(int fmt, const uint8_t *__restrict__ src,
                                                     uint8_t *__restrict__ dst, int64_t N, int nb, int T)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t slots = (int64_t)T * 32;
    if (i >= N * slots) return;
    const int64_t n = i / slots;
    const int js = (int)(i - n * slots);
    const int t = js >> 5, s = js & 31, b = js;
    if (fmt == BQG_Q4_0) {
        uint8_t *tile = dst + (n * T + t) * Q4_0_TILE;
        uint32_t w[4] = {0, 0, 0, 0};
        uint16_t d = 0;
        if (b < nb) {
            const uint16_t *blk = reinterpret_cast<const uint16_t *>(src + (n * nb + b) * Q4_0_BYTES);
            d = blk[0];
            for (int k = 0; k < 4; k++) w[k] = (uint32_t)blk[1 + 2 * k] | ((uint32_t)blk[2 + 2 * k] << 16);
        }
        *reinterpret_cast<uint4 *>(tile + 16 * s) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint16_t *>(tile + 512 + 2 * s) = d;
    } else {
        uint8_t *tile = dst + (n * T + t) * Q8_0_TILE;
        uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        uint16_t d = 0;
        if (b < nb) {
            const uint16_t *blk = reinterpret_cast<const uint16_t *>(src + (n * nb + b) * Q8_0_BYTES);
            d = blk[0];
            for (int k = 0; k < 8; k++) w[k] = (uint32_t)blk[1 + 2 * k] | ((uint32_t)blk[2 + 2 * k] << 16);
        }
        *reinterpret_cast<uint4 *>(tile + 16 * s) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4 *>(tile + 512 + 16 * s) = make_uint4(w[4], w[5], w[6], w[7]);
        *reinterpret_cast<uint16_t *>(tile + 1024 + 2 * s) = d;
    }
}

__global__ void __launch_bounds__(256) copy_u16_kernel(const uint16_t *__restrict__ src, uint16_t *__restrict__ dst,
                                                       int64_t n)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

// The exact per-block integer dots of q4_0 x q8_1 (one activation row),
// computed with the GEMV's own device routine (q4_0_q8_1_sumi).
__global__ void __launch_bounds__(256) block_dots_kernel(const uint8_t *__restrict__ Wp, const uint8_t *__restrict__ Xq,
                                                         int32_t *__restrict__ dots, int64_t N, int nb, int64_t row_bytes,
                                                         int K)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N * nb) return;
    const int64_t n = i / nb;
    const int b = (int)(i - n * nb);
    GemvParams p = {};
    p.X = Xq; p.nb = nb; p.K = K;
    XSlice<W_Q4_0, X_Q8_1> xs;
    load_x<W_Q4_0, X_Q8_1>(xs, p, 0, b, true);
    WChunk<W_Q4_0> wc;
    load_w<W_Q4_0>(wc, Wp + n * row_bytes, b, true);
    dots[i] = q4_0_q8_1_sumi(wc.c, xs);
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
cudaError_t launch_quantize_q8_1(const void *x, int x_f32, void *xq, int M, int64_t K, cudaStream_t s, bool pdl)
{
    const int nb = (int)(K / QK);
    const int64_t nblocks = (int64_t)M * nb;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((nblocks + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel, x, x_f32, (uint8_t *)xq, nblocks, nb, K);
}

cudaError_t launch_rmsnorm_q8_1(const void *x, int x_f32, const float *gamma, float eps, void *xq, int M, int64_t K,
                               cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)M);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, rmsnorm_q8_1_kernel, x, x_f32, gamma, eps, (uint8_t *)xq, (int)(K / QK), K);
}

cudaError_t launch_quantize_weights(int fmt, const float *W, void *dst, int64_t N, int64_t K, cudaStream_t s)
{
    const int nb = (int)(K / QK);
    const int64_t nblocks = N * nb;
    quantize_weights_kernel<<<(unsigned)((nblocks + 7) / 8), 256, 0, s>>>(W, fmt, (uint8_t *)dst, nblocks, nb, K);
    return cudaGetLastError();
}

cudaError_t launch_repack(int fmt, const void *src, void *dst, int64_t N, int64_t K, cudaStream_t s)
{
    if (fmt == BQG_BF16) {
        const int64_t n = N * K;
        const int64_t blocks = std::min<int64_t>((n + 255) / 256, 65536);
        copy_u16_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint16_t *)src, (uint16_t *)dst, n);
        return cudaGetLastError();
    }
    const int nb = (int)(K / QK), T = (nb + 31) / 32;
    const int64_t total = N * T * 32;
    repack_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(fmt, (const uint8_t *)src, (uint8_t *)dst, N, nb, T);
    return cudaGetLastError();
}

cudaError_t launch_block_dots(const void *Wp, const void *Xq, int32_t *dots, int64_t N, int64_t K, int64_t row_bytes,
                              cudaStream_t s)
{
    const int nb = (int)(K / QK);
    const int64_t total = N * nb;
    block_dots_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>((const uint8_t *)Wp, (const uint8_t *)Xq, dots, N,
                                                                        nb, row_bytes, (int)K);
    return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const GemvParams &p, int M, int splits, int final_epi, cudaStream_t s, bool pdl)
{
    const int64_t n = (final_epi == EPI_SWIGLU) ? (int64_t)M * (p.Nv >> 1) : (int64_t)M * p.Nv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((n + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_splitk_reduce, p, M, splits, final_epi);
}

}  // namespace bqg
