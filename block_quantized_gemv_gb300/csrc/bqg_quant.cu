// bqg_quant.cu -- block encoders, the load-time repack, the block-dot
// debug export and the SM-driven copy (activations in, outputs out over the
// coherent CPU-GPU link without a copy-engine transfer).
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
#include <algorithm>

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

// Knuth's TwoSum: s + e == a + b exactly (round-to-nearest, no contraction).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Sum of squares as an unevaluated pair hi + lo of fp32 values, plus an fp64
// part for magnitudes whose square or its rounding error would leave the
// normal fp32 range.  Each square is exact as p + e (e = fma(v, v, -p); zero
// for bf16 inputs), hi takes the exact TwoSum of p, lo the rest.
struct SumSq {
    float hi = 0.f, lo = 0.f;
    double wide = 0.0;
    __device__ __forceinline__ void add(float v)
    {
        const uint32_t ex = (__float_as_uint(v) >> 23) & 0xFFu;
        if (ex - 77u <= 176u - 77u) {                 // 2^-50 <= |v| < 2^50
            const float p = __fmul_rn(v, v);
            const float ep = fmaf(v, v, -p);
            float t;
            two_sum(hi, p, hi, t);
            lo = __fadd_rn(lo, __fadd_rn(t, ep));
        } else if (v != 0.f) {
            wide = fma((double)v, (double)v, wide);   // exact square in fp64
        }
    }
    __device__ __forceinline__ void merge(float ohi, float olo)
    {
        float t;
        two_sum(hi, ohi, hi, t);
        lo = __fadd_rn(lo, __fadd_rn(olo, t));
    }
};

// r = 1 / sqrt(s / K + eps) rounded once to fp32, from s = sh + sl, without
// fp64: u = s / K + eps is formed as an fp32 pair (q1 = RN(sh / K), whose
// remainder sh - q1 K an fma gives exactly), then y = rsqrtf(u) is refined by
// one Newton step for u^-1/2 with its second-order term,
// y (1 + d/2 + 3 d^2 / 8), d = 1 - u y^2, the products split exactly by fma.
// Before the last rounding the value is within about 2^-44 of the exact one.
__device__ __forceinline__ float rms_recip_pair(float sh, float sl, float Kf, float eps)
{
    const float q1 = __fdiv_rn(sh, Kf);
    const float rem = fmaf(-q1, Kf, sh);
    const float q2 = __fdiv_rn(__fadd_rn(rem, sl), Kf);
    float uh, ul;
    two_sum(q1, eps, uh, ul);
    ul = __fadd_rn(ul, q2);
    const float t = __fadd_rn(uh, ul);                 // renormalise (|uh| >= |ul|)
    ul = __fsub_rn(ul, __fsub_rn(t, uh));
    uh = t;
    const float y = rsqrtf(uh);
    const float p = __fmul_rn(y, y), pe = fmaf(y, y, -p);
    const float wh = __fmul_rn(uh, p), we = fmaf(uh, p, -wh);
    const float d = __fsub_rn(__fsub_rn(__fsub_rn(1.0f, wh), we), fmaf(uh, pe, __fmul_rn(ul, p)));
    return __fadd_rn(y, __fmul_rn(y, __fmul_rn(d, fmaf(0.375f, d, 0.5f))));
}

// Fused RMSNorm -> q8_1 ("MI50 megakernel", hypothesis ledger: neighbouring
// steps fused into one dispatch; the Q8_1 activation of "rx-6700xt-llama2-
// decode").  Grid: blockIdx.y = activation row, blockIdx.x = a slice of its
// blocks.  Every CTA of a row computes s = sum x^2 (the same value in each, in
// the same order) to about 2^-44 relative: squares exact, accumulated as
// fp32 pairs with error-free sums.  Then r = 1 / sqrt(s / K + eps) to about
// 2^-44 relative, rounded once to fp32 (in fp64 when an input or s leaves the
// range the pair arithmetic covers), and its warps encode
// y = fp32(fp32(x * r) * gamma) of their blocks with the q8_1 encoder.
// fp64 arithmetic is kept off the common path: its rate, and the issue time
// of one warp's fp64 instruction, are a small fraction of fp32's on this part.
__global__ void __launch_bounds__(256) rmsnorm_q8_1_kernel(const void *__restrict__ x, int x_f32, int vec,
                                                           const float *__restrict__ gamma, float eps,
                                                           uint8_t *__restrict__ xq, int nb, int64_t K)
{
    __shared__ float part_hi[8], part_lo[8];
    __shared__ double part_w[8];
    __shared__ float s_r;
    pdl_wait();
    pdl_launch_dependents();
    const int64_t m = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // this warp's first block, loaded beside the sum so that its L2 trip overlaps
    const int bfirst = blockIdx.x * 8 + warp;
    float x0 = 0.f, g0 = 1.f;
    if (bfirst < nb) {
        const int64_t k = (int64_t)bfirst * QK + lane;
        x0 = load_act(x, x_f32, m * K + k);
        if (gamma) g0 = gamma[k];
    }
    SumSq acc;
    if (vec && x_f32) {
        const float4 *row = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) + m * K);
        for (int64_t i = tid; i < K / 4; i += 256) {
            const float4 q = row[i];
            acc.add(q.x); acc.add(q.y); acc.add(q.z); acc.add(q.w);
        }
    } else if (vec) {
        const uint4 *row = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(x) + m * K);
        for (int64_t i = tid; i < K / 8; i += 256) {
            const uint4 q = row[i];
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; j++) {
                acc.add(__uint_as_float(w[j] << 16));
                acc.add(__uint_as_float(w[j] & 0xFFFF0000u));
            }
        }
    } else {
        for (int64_t k = tid; k < K; k += 256) acc.add(load_act(x, x_f32, m * K + k));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        acc.merge(__shfl_xor_sync(0xffffffffu, acc.hi, o), __shfl_xor_sync(0xffffffffu, acc.lo, o));
    if (__any_sync(0xffffffffu, acc.wide != 0.0)) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc.wide += __shfl_xor_sync(0xffffffffu, acc.wide, o);
    }
    if (lane == 0) {
        part_hi[warp] = acc.hi;
        part_lo[warp] = acc.lo;
        part_w[warp] = acc.wide;
    }
    __syncthreads();
    if (warp == 0) {
        SumSq tot;
        if (lane < 8) {
            tot.hi = part_hi[lane];
            tot.lo = part_lo[lane];
            tot.wide = part_w[lane];
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1)
            tot.merge(__shfl_xor_sync(0xffffffffu, tot.hi, o), __shfl_xor_sync(0xffffffffu, tot.lo, o));
        const bool wide = __any_sync(0xffffffffu, tot.wide != 0.0);
        if (lane == 0) {
            // pair path: s and s / K well inside the normal fp32 range
            if (!wide && tot.hi >= 0x1p-60f && tot.hi <= 0x1p100f && eps >= 0.f && K < (1 << 24)) {
                s_r = rms_recip_pair(tot.hi, tot.lo, (float)K, eps);
            } else {
                double t = 0.0;
                for (int w = 0; w < 8; w++) t += ((double)part_hi[w] + (double)part_lo[w]) + part_w[w];
                s_r = (float)(1.0 / sqrt(t / (double)K + (double)eps));
            }
        }
    }
    __syncthreads();
    const float r = s_r;
    for (int b = bfirst; b < nb; b += gridDim.x * 8) {
        const int64_t k = (int64_t)b * QK + lane;
        const bool first = (b == bfirst);
        float y = __fmul_rn(first ? x0 : load_act(x, x_f32, m * K + k), r);
        if (gamma) y = __fmul_rn(y, first ? g0 : gamma[k]);
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

// n pieces of 16 B from src to dst, copied by the SMs.  Either side may be
// page-locked host memory mapped into the device's address space: each load
// then crosses the CPU-GPU link, so every thread issues four before its
// first store and the link's latency is paid about once per thread.  With
// programmatic dependent launch the copy waits for the previous kernel
// before it reads or writes anything.
__global__ void __launch_bounds__(256) copy_sm_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                      int64_t n)
{
    pdl_wait();
    pdl_launch_dependents();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; u++) v[u] = src[i + u * stride];
#pragma unroll
        for (int u = 0; u < 4; u++) dst[i + u * stride] = v[u];
    }
    for (; i < n; i += stride) dst[i] = src[i];
}

// The exact per-block integer dots of q4_0 x q8_1 (one activation row),
// computed with the K-slice kernel's routine (q4_0_q8_1_sumi on the
// operands as that kernel loads them: the q8_1 block through load_x, the
// code chunk of the repacked row).
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

cudaError_t launch_copy_sm(void *dst, const void *src, int64_t bytes, int sms, cudaStream_t s, bool pdl)
{
    const int64_t n = bytes / 16;
    // one 16-byte piece per thread up to four resident waves of CTAs, then grid-stride
    const int64_t ctas = std::min<int64_t>((n + 255) / 256, (int64_t)sms * 4);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::max<int64_t>(ctas, 1));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, copy_sm_kernel, reinterpret_cast<const uint4 *>(src),
                              reinterpret_cast<uint4 *>(dst), n);
}

cudaError_t launch_rmsnorm_q8_1(const void *x, int x_f32, const float *gamma, float eps, void *xq, int M, int64_t K,
                               cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    const int nb = (int)(K / QK);
    cfg.gridDim = dim3((unsigned)std::min((nb + 7) / 8, 64), (unsigned)M);   // up to 64 CTAs per row
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const int vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0;   // rows are then 16-byte aligned too
    return cudaLaunchKernelEx(&cfg, rmsnorm_q8_1_kernel, x, x_f32, vec, gamma, eps, (uint8_t *)xq, (int)(K / QK), K);
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
