// bqg_gemv.cuh -- the skinny-GEMV kernels (M = 1, 2, 4, 8).
//
// Y[m, n] = sum_k W[n, k] X[m, k] for the memory-bound decode shape of
// "The Shape That Actually Matters" (M = 1, K = 4096, N = 12288 and the
// rest of the decode projections).  Design for sm_103a:
//
//  * Weights are the only large stream.  They are read once from the
//    repacked layout (include/bqgemv.h): runs of whole consecutive rows are
//    single cp.async.bulk copies into shared memory, and inside a tile lane
//    s of a warp owns block (or 16-byte chunk) s, so every warp-wide shared
//    load covers 512 contiguous bytes and a block's fp16 scale sits in the
//    same tile ("Rounds 1-3" of that page: the layout and the load width,
//    not the byte count, decided the bandwidth).
//  * The activation rows are staged once per CTA in shared memory, in the
//    same per-lane layout, so every activation load serves the RL rows a
//    warp works on ("MI50 megakernel", microbenchmark ladder: re-loading the
//    activation was three of five memory instructions per iteration).
//  * gemv_lpr_kernel (the lanes-per-row kernel, every M): each warp streams
//    its own groups of RL rows through its own shared-memory slots, all 32
//    lanes on each row, one warp shuffle reduction per output; no producer
//    warp and no cross-warp coupling.
//  * gemv_kernel (the K-slice kernel): each thread owns a fixed slice of K
//    held in registers; serves the shapes whose staged activations would
//    not fit beside the weight stages.
//  * Each CTA owns a contiguous range of rows; the grid is sized from the
//    SM count and the measured occupancy.  Split-K (grid.y > 1) writes
//    partial sums to a workspace reduced by gemv_splitk_reduce.
//  * q4_0 x q8_1 multiplies codes with dp4a: per block the integer dot
//    sum (qw - 8) qx is exact ("rx-6700xt-llama2-decode": integer-dot
//    Q4_0 x Q8_1 matvec), scaled by d_w d_x in fp32.
#pragma once

#include "bqg_common.cuh"

namespace bqg {

enum WFmt { W_BF16 = 0, W_Q8_0 = 1, W_Q4_0 = 2 };
enum XFmt { X_BF16 = 0, X_Q8_1 = 1, X_F32 = 2 };   // X_F32: bf16 input held as fp32 in registers
enum Epi { EPI_STORE = 0, EPI_SWIGLU = 1, EPI_PARTIAL = 2 };

// elements covered by one chunk (one 16-byte code load)
template <int WF> struct ChunkTraits;
template <> struct ChunkTraits<W_BF16> { static constexpr int E = 8; };
template <> struct ChunkTraits<W_Q8_0> { static constexpr int E = 16; };
template <> struct ChunkTraits<W_Q4_0> { static constexpr int E = 32; };

struct GemvParams {
    // up to three weight matrices in one "virtual" row space
    const uint8_t *W[3];
    float *Y[3];
    int64_t rows[3];        // rows of each matrix
    int nmat;               // 1, 2 (gate/up, rows interleaved g0 u0 g1 u1 ...) or 3 (q, k, v)
    int epi;                // Epi
    const uint8_t *X;       // bf16 [M][K] or q8_1 [M][K/32]
    float *ws;              // split-K partials [splits][M][Nv]
    int64_t Nv;             // virtual rows
    int64_t row_bytes;      // bytes of one repacked row
    int K;
    int nb;                 // K / 32
    int nc;                 // chunks per row (chunk index space, may contain holes)
    int TPR;                // threads per row group (multiple of 32)
    int RG;                 // row groups per CTA
    int64_t rows_per_cta;   // virtual rows per CTA (multiple of 2 for gate/up)
    int chunks_per_split;   // chunk range of one split (grid.y)
    // shared-memory pipeline
    int nstages;            // NS stages in the ring
    int stage_rows;         // S rows per stage (RG * rows per group per stage)
    int row_stride;         // bytes of one staged row (largest split range, multiple of 16)
    int win_stages;         // stages per partial-sum window
    int part_off;           // byte offset of the partial sums
    int bar_off;            // byte offset of the mbarriers (8-byte aligned)
    int ctas;               // CTAs along grid.x (rows are split evenly over them)
    // lanes-per-row kernel
    int L;                  // lanes that share one row (8, 16 or 32)
    int wg;                 // warps per stage group
    int ng;                 // stage groups
    int x_off;              // byte offset of the staged activations
    int x_row_bytes;        // staged bytes of one activation row
    int xraw_off;           // byte offset of the raw activation copy (lanes-per-row kernel)
    int early;              // stages per warp requested before waiting for the previous grid
    int rl;                 // rows per lane (lanes-per-row kernel: 1, 2 or 4)
    int piece_chunks;       // chunks per K-piece (lanes-per-row kernel)
    int x_bf16s;            // lanes-per-row kernel at M = 1: bf16 activations staged as bf16
    int rows_kernel;        // lanes-per-row plan served by gemv_lpr_rows_kernel (one matrix, whole rows,
                            // no split, plain store)
    // SwiGLU with a q8_1 output: the blocks go to hq (M x rows[0]/32 blocks);
    // Y[0] is then an fp32 staging row set and cnt one arrival counter per
    // block (zero between calls)
    uint8_t *hq;
    int *cnt;
    // check instantiation only (q4_0 x q8_1, one activation row, one matrix):
    // the integer block dots the kernel computes, rows x nb int32, row-major
    int32_t *dots;
};

// One decode layer's three projection groups in one persistent launch
// (bqg_layer.cu; the entry point validates and plans it).
struct LayerParams {
    GemvParams qkv;         // phase 1, CTAs [0, cq): nmat 3, whole rows, K = model width
    GemvParams gu;          // phase 1, CTAs [cq, grid): nmat 2 (gate/up interleaved), SwiGLU -> q8_1
    GemvParams dn;          // phase 2, every CTA: nmat 1, K = Nff, activations = gu.hq
    const void *xa, *xb;    // activation rows of qkv and gate/up (K values each)
    int x_f32;              // activations fp32 (else bf16)
    int cq;                 // phase-1 CTAs given to qkv
    int slot_bytes;         // per-warp slot (largest stage of the two phases)
    int x_off;              // staged activations (room for the larger phase)
    int xraw_off;           // phase 1's q8_1 blocks before staging
    int bar_off;            // one mbarrier per warp
    unsigned long long *gbar;   // grid barrier word in the workspace: generation << 32 | arrivals
};

// Error word set when a bounded wait gives up (one per translation unit).
static __device__ int g_gemv_error;

// ---------------------------------------------------------------------------
// SwiGLU epilogue with a q8_1 output.  The 32 outputs of a block are finished
// by different warps and CTAs, so each output is stored in fp32 and counted
// at its block (the store is made visible first); the arrival that completes
// the block encodes it from L2 and re-arms the counter for the next call.
// Nothing waits on another CTA.
// ---------------------------------------------------------------------------
// warp-wide: encode block b of activation row m
__device__ __forceinline__ void swiglu_encode_block_warp(const GemvParams &p, int m, int64_t b, int lane)
{
    __threadfence();
    const int64_t blk = (int64_t)m * (p.rows[0] / 32) + b;
    const float v = __ldcg(p.Y[0] + (int64_t)m * p.rows[0] + b * 32 + lane);
    q8_1_encode_warp(v, lane, p.hq + blk * Q8_1_BYTES);
    if (lane == 0) p.cnt[blk] = 0;
}

// Virtual row -> (matrix, row in matrix)
__device__ __forceinline__ void map_row(const GemvParams &p, int64_t v, int &mat, int64_t &r)
{
    if (p.nmat == 2) { mat = (int)(v & 1); r = v >> 1; return; }
    mat = 0; r = v;
    if (p.nmat == 3) {
        if (r >= p.rows[0]) { r -= p.rows[0]; mat = 1;
            if (r >= p.rows[1]) { r -= p.rows[1]; mat = 2; } }
    }
}

// Is chunk c of a row a real chunk (not a hole in a partly used last tile)?
template <int WF>
__device__ __forceinline__ bool chunk_valid(int c, int nb, int nc)
{
    if (c >= nc) return false;
    if (WF == W_Q8_0) return (c >> 6) * 32 + (c & 31) < nb;
    if (WF == W_Q4_0) return c < nb;
    return true;
}

// Byte offset of chunk c's codes within a repacked row, and of its scale.
template <int WF>
__device__ __forceinline__ int64_t chunk_code_off(int c)
{
    if (WF == W_BF16) return 16ll * c;
    if (WF == W_Q8_0) return (int64_t)(c >> 6) * Q8_0_TILE + ((c >> 5) & 1) * 512 + 16 * (c & 31);
    return (int64_t)(c >> 5) * Q4_0_TILE + 16 * (c & 31);
}
template <int WF>
__device__ __forceinline__ int64_t chunk_scale_off(int c)
{
    if (WF == W_Q8_0) return (int64_t)(c >> 6) * Q8_0_TILE + 1024 + 2 * (c & 31);
    return (int64_t)(c >> 5) * Q4_0_TILE + 512 + 2 * (c & 31);
}
// First element of chunk c along K.
template <int WF>
__device__ __forceinline__ int chunk_elem0(int c)
{
    if (WF == W_BF16) return 8 * c;
    if (WF == W_Q8_0) return 32 * ((c >> 6) * 32 + (c & 31)) + 16 * ((c >> 5) & 1);
    return 32 * c;
}

// ---------------------------------------------------------------------------
// per-thread activation slice
// ---------------------------------------------------------------------------
template <int WF, int XF> struct XSlice;
// bf16 activations: E bf16 values per chunk, kept packed (E/2 words)
template <int WF> struct XSlice<WF, X_BF16> {
    static constexpr int WORDS = ChunkTraits<WF>::E / 2;
    uint32_t w[WORDS];
};
// bf16 activations converted once to fp32 (E values per chunk)
template <int WF> struct XSlice<WF, X_F32> {
    float f[ChunkTraits<WF>::E];
};
// q8_1 activations (q4_0 weights only): 32 codes, d, and the exact sum of codes
template <> struct XSlice<W_Q4_0, X_Q8_1> {
    int32_t q[8];
    float d;
    int32_t sum;
};

template <int WF, int XF>
__device__ __forceinline__ void load_x(XSlice<WF, XF> &xs, const GemvParams &p, int m, int c, bool valid)
{
    if constexpr (XF == X_F32) {
        constexpr int E = ChunkTraits<WF>::E;
        if (!valid) {
#pragma unroll
            for (int i = 0; i < E; i++) xs.f[i] = 0.f;
            return;
        }
        const uint8_t *src = p.X + ((int64_t)m * p.K + chunk_elem0<WF>(c)) * 2;
#pragma unroll
        for (int i = 0; i < E / 8; i++) {
            const uint4 v = ldg_v4(src + 16 * i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; k++) {
                xs.f[8 * i + 2 * k] = bf16_lo(w[k]);
                xs.f[8 * i + 2 * k + 1] = bf16_hi(w[k]);
            }
        }
    } else if constexpr (XF == X_BF16) {
        constexpr int WORDS = XSlice<WF, XF>::WORDS;
        if (!valid) {
#pragma unroll
            for (int i = 0; i < WORDS; i++) xs.w[i] = 0;
            return;
        }
        const uint8_t *src = p.X + ((int64_t)m * p.K + chunk_elem0<WF>(c)) * 2;
#pragma unroll
        for (int i = 0; i < WORDS / 4; i++) {
            uint4 v = ldg_v4(src + 16 * i);
            xs.w[4 * i + 0] = v.x; xs.w[4 * i + 1] = v.y; xs.w[4 * i + 2] = v.z; xs.w[4 * i + 3] = v.w;
        }
    } else {
        if (!valid) {
#pragma unroll
            for (int i = 0; i < 8; i++) xs.q[i] = 0;
            xs.d = 0.f; xs.sum = 0;
            return;
        }
        // q8_1 block: fp16 d | fp16 s | int8 q[32]; rows of 36-byte blocks are
        // only 4-byte aligned, so read words.
        const uint32_t *blk = reinterpret_cast<const uint32_t *>(p.X + ((int64_t)m * p.nb + c) * Q8_1_BYTES);
        uint32_t ds = __ldg(blk);
        xs.d = half_bits_to_float(ds & 0xffffu);
        int s = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            xs.q[i] = (int32_t)__ldg(blk + 1 + i);
            s = __dp4a(xs.q[i], 0x01010101, s);    // exact sum of the 32 codes
        }
        xs.sum = s;
    }
}

// ---------------------------------------------------------------------------
// per-thread weight chunk
// ---------------------------------------------------------------------------
template <int WF> struct WChunk { uint4 c; uint32_t s; };

template <int WF>
__device__ __forceinline__ void load_w(WChunk<WF> &w, const uint8_t *row, int c, bool valid)
{
    if (!valid) { w.c = make_uint4(0, 0, 0, 0); w.s = 0; return; }
    w.c = ldg_stream_v4(row + chunk_code_off<WF>(c));
    if constexpr (WF != W_BF16) w.s = ldg_stream_u16(row + chunk_scale_off<WF>(c));
    else w.s = 0;
}

// Chunk c from a row staged in shared memory starting at byte `base` of the row.
template <int WF>
__device__ __forceinline__ void lds_w(WChunk<WF> &w, const uint8_t *srow, int64_t base, int c)
{
    w.c = *reinterpret_cast<const uint4 *>(srow + (chunk_code_off<WF>(c) - base));
    if constexpr (WF != W_BF16) w.s = *reinterpret_cast<const uint16_t *>(srow + (chunk_scale_off<WF>(c) - base));
    else w.s = 0;
}

// Byte range [off, off + bytes) of a row that holds chunks [cbeg, cend).
template <int WF>
__device__ __host__ __forceinline__ void chunk_range_bytes(int cbeg, int cend, int64_t &off, int64_t &bytes)
{
    if (WF == W_BF16) { off = 16ll * cbeg; bytes = 16ll * (cend - cbeg); return; }
    const int per_tile = (WF == W_Q8_0) ? 64 : 32;
    const int64_t tb = (WF == W_Q8_0) ? Q8_0_TILE : Q4_0_TILE;
    const int64_t t0 = cbeg / per_tile, t1 = (cend + per_tile - 1) / per_tile;
    off = t0 * tb;
    bytes = (t1 - t0) * tb;
}

// Exact per-block integer dot of a q4_0 code chunk with a q8_1 block:
// sum_i (qw_i - 8) qx_i.  Word i of the codes holds elements 4i..4i+3 in its
// low nibbles and 16+4i..16+4i+3 in its high nibbles; x.q[i] holds codes
// 4i..4i+3.  |result| <= 32 * 8 * 127.
__device__ __forceinline__ int q4_0_q8_1_sumi(const uint4 &c, const XSlice<W_Q4_0, X_Q8_1> &x)
{
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    int s = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) s = __dp4a((int)(cw[i] & 0x0f0f0f0fu), x.q[i], s);
#pragma unroll
    for (int i = 0; i < 4; i++) s = __dp4a((int)((cw[i] >> 4) & 0x0f0f0f0fu), x.q[4 + i], s);
    return s - 8 * x.sum;
}

// dot(chunk, activation slice) in fp32
template <int WF, int XF>
__device__ __forceinline__ float chunk_dot(const WChunk<WF> &w, const XSlice<WF, XF> &x)
{
    const uint32_t cw[4] = {w.c.x, w.c.y, w.c.z, w.c.w};
    if constexpr (XF == X_F32 && WF == W_BF16) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < 4; i++) ffma2(a0, a1, bf16_lo(cw[i]), bf16_hi(cw[i]), x.f[2 * i], x.f[2 * i + 1]);
        return a0 + a1;
    } else if constexpr (XF == X_F32 && WF == W_Q8_0) {
        // codes are int8 q; byte ^ 0x80 = q + 128; pairs of elements go through
        // one packed subtract and one packed FMA
        constexpr float OFF = 8388608.0f + 128.0f;
        float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t u = cw[i] ^ 0x80808080u;
            float e0 = byte_plus_2p23<0>(u), e1 = byte_plus_2p23<1>(u);
            float e2 = byte_plus_2p23<2>(u), e3 = byte_plus_2p23<3>(u);
            fadd2(e0, e1, -OFF);
            fadd2(e2, e3, -OFF);
            ffma2(a0, a1, e0, e1, x.f[4 * i], x.f[4 * i + 1]);
            ffma2(b0, b1, e2, e3, x.f[4 * i + 2], x.f[4 * i + 3]);
        }
        return ((a0 + a1) + (b0 + b1)) * half_bits_to_float(w.s);
    } else if constexpr (XF == X_F32 && WF == W_Q4_0) {
        // q4_0 codes against fp32 activations: low nibbles of word i are
        // elements 4i..4i+3, high nibbles 16+4i..16+4i+3
        constexpr float OFF = 8388608.0f + 8.0f;
        float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t lo = cw[i] & 0x0f0f0f0fu;
            const uint32_t hi = (cw[i] >> 4) & 0x0f0f0f0fu;
            float l0 = byte_plus_2p23<0>(lo), l1 = byte_plus_2p23<1>(lo);
            float l2 = byte_plus_2p23<2>(lo), l3 = byte_plus_2p23<3>(lo);
            float h0 = byte_plus_2p23<0>(hi), h1 = byte_plus_2p23<1>(hi);
            float h2 = byte_plus_2p23<2>(hi), h3 = byte_plus_2p23<3>(hi);
            fadd2(l0, l1, -OFF);
            fadd2(l2, l3, -OFF);
            fadd2(h0, h1, -OFF);
            fadd2(h2, h3, -OFF);
            ffma2(a0, a1, l0, l1, x.f[4 * i], x.f[4 * i + 1]);
            ffma2(b0, b1, l2, l3, x.f[4 * i + 2], x.f[4 * i + 3]);
            ffma2(a0, a1, h0, h1, x.f[16 + 4 * i], x.f[16 + 4 * i + 1]);
            ffma2(b0, b1, h2, h3, x.f[16 + 4 * i + 2], x.f[16 + 4 * i + 3]);
        }
        return ((a0 + a1) + (b0 + b1)) * half_bits_to_float(w.s);
    } else if constexpr (WF == W_BF16) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            a0 = fmaf(bf16_lo(cw[i]), bf16_lo(x.w[i]), a0);
            a1 = fmaf(bf16_hi(cw[i]), bf16_hi(x.w[i]), a1);
        }
        return a0 + a1;
    } else if constexpr (WF == W_Q8_0) {
        // codes are int8 q; byte ^ 0x80 = q + 128 as an unsigned byte
        constexpr float OFF = 8388608.0f + 128.0f;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t u = cw[i] ^ 0x80808080u;
            a0 = fmaf(byte_plus_2p23<0>(u) - OFF, bf16_lo(x.w[2 * i]), a0);
            a1 = fmaf(byte_plus_2p23<1>(u) - OFF, bf16_hi(x.w[2 * i]), a1);
            a0 = fmaf(byte_plus_2p23<2>(u) - OFF, bf16_lo(x.w[2 * i + 1]), a0);
            a1 = fmaf(byte_plus_2p23<3>(u) - OFF, bf16_hi(x.w[2 * i + 1]), a1);
        }
        return (a0 + a1) * half_bits_to_float(w.s);
    } else if constexpr (XF == X_BF16) {
        // q4_0 x bf16: word i holds elements 4i..4i+3 (low nibbles) and
        // 16+4i..16+4i+3 (high nibbles); x.w[k] holds elements 2k, 2k+1.
        constexpr float OFF = 8388608.0f + 8.0f;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t lo = cw[i] & 0x0f0f0f0fu;
            const uint32_t hi = (cw[i] >> 4) & 0x0f0f0f0fu;
            a0 = fmaf(byte_plus_2p23<0>(lo) - OFF, bf16_lo(x.w[2 * i]), a0);
            a1 = fmaf(byte_plus_2p23<1>(lo) - OFF, bf16_hi(x.w[2 * i]), a1);
            a0 = fmaf(byte_plus_2p23<2>(lo) - OFF, bf16_lo(x.w[2 * i + 1]), a0);
            a1 = fmaf(byte_plus_2p23<3>(lo) - OFF, bf16_hi(x.w[2 * i + 1]), a1);
            a0 = fmaf(byte_plus_2p23<0>(hi) - OFF, bf16_lo(x.w[8 + 2 * i]), a0);
            a1 = fmaf(byte_plus_2p23<1>(hi) - OFF, bf16_hi(x.w[8 + 2 * i]), a1);
            a0 = fmaf(byte_plus_2p23<2>(hi) - OFF, bf16_lo(x.w[8 + 2 * i + 1]), a0);
            a1 = fmaf(byte_plus_2p23<3>(hi) - OFF, bf16_hi(x.w[8 + 2 * i + 1]), a1);
        }
        return (a0 + a1) * half_bits_to_float(w.s);
    } else {
        // q4_0 x q8_1: exact integer dot, then one fp32 scale
        return (half_bits_to_float(w.s) * x.d) * (float)q4_0_q8_1_sumi(w.c, x);
    }
}

__device__ __forceinline__ void named_barrier(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// The SwiGLU q8_1 output of a CTA, once its fp32 outputs [o0, o1) of every
// activation row are stored by the `nwarps` warps that meet at barrier
// `bar`: one fence and barrier, then per (block, row) one counted arrival
// carrying the number of outputs this CTA gave the block.  A block wholly
// inside the range is complete at once and skips the counter.
__device__ __forceinline__ void swiglu_q8_1_finish(const GemvParams &p, int M, int64_t o0, int64_t o1, int bar,
                                                   int warp, int nwarps, int lane)
{
    __threadfence();
    named_barrier(bar, nwarps * 32);
    if (o1 <= o0) return;
    const int64_t b0 = o0 / 32;
    const int nbm = (int)((o1 - 1) / 32 - b0 + 1) * M;
    for (int i = warp; i < nbm; i += nwarps) {
        const int64_t b = b0 + i / M;
        const int m = i - (i / M) * M;
        const int c = (int)(min(o1, 32 * (b + 1)) - max(o0, 32 * b));
        bool last = true;
        if (c < 32) {
            int prev = 0;
            if (lane == 0) prev = atomicAdd(p.cnt + (int64_t)m * (p.rows[0] / 32) + b, c);
            last = (__shfl_sync(0xffffffffu, prev, 0) + c == 32);
        }
        if (last) swiglu_encode_block_warp(p, m, b, lane);
    }
}

// rows each group takes from a stage (per pass); V = RPS * M values per warp reduction
template <int M> struct RowsPerStage { static constexpr int value = (M == 8) ? 1 : 4 / M; };

// This CTA's virtual rows [v0, v1): an even split of Nv over p.ctas CTAs
// (in pairs when gate and up rows alternate).
__device__ __forceinline__ void cta_rows(const GemvParams &p, int64_t &v0, int64_t &v1)
{
    const int64_t unit = (p.nmat == 2) ? 2 : 1;
    const int64_t units = p.Nv / unit;
    v0 = (int64_t)blockIdx.x * units / p.ctas * unit;
    v1 = (int64_t)(blockIdx.x + 1) * units / p.ctas * unit;
}

// Virtual row held by staged row r of a stage that starts at virtual row vs.
// With gate/up pairs a stage of S rows holds S/2 gate rows then the S/2 up
// rows of the same outputs, so each half is one contiguous run in memory.
__device__ __forceinline__ int64_t staged_vrow(const GemvParams &p, int64_t vs, int S, int r)
{
    if (p.nmat == 2) {
        const int half = S >> 1;
        return (r < half) ? vs + 2 * r : vs + 2 * (r - half) + 1;
    }
    return vs + r;
}

// Fill one stage: the staged rows of the stage that starts at virtual row vs
// (those below v1), one cp.async.bulk per run of consecutive rows of one
// matrix, all completing on `bar`, which is told the byte count first.
template <int WF>
__device__ __forceinline__ void issue_stage(const GemvParams &p, uint32_t dst, uint32_t bar, int64_t vs, int S,
                                            int64_t v1, int64_t roff, int64_t rbytes)
{
    const bool whole_rows = (roff == 0 && rbytes == p.row_bytes);
    int nvalid = 0;
    for (int r = 0; r < S; r++) nvalid += staged_vrow(p, vs, S, r) < v1;
    mbar_arrive_expect_tx(bar, (uint32_t)(nvalid * rbytes));
    for (int r = 0; r < S;) {
        const int64_t v = staged_vrow(p, vs, S, r);
        if (v >= v1) { r++; continue; }
        int mat; int64_t rr;
        map_row(p, v, mat, rr);
        int len = 1;
        while (whole_rows && r + len < S) {
            const int64_t vn = staged_vrow(p, vs, S, r + len);
            if (vn >= v1) break;
            int mn; int64_t rn;
            map_row(p, vn, mn, rn);
            if (mn != mat || rn != rr + len) break;
            len++;
        }
        bulk_g2s(dst + r * p.row_stride, p.W[mat] + rr * p.row_bytes + roff, (uint32_t)(len * rbytes), bar);
        r += len;
    }
}

// The producer lane of the K-slice kernel: streams stages [0, nst) of this
// CTA's rows into the ring.  The first NS stages are requested before
// waiting for the previous grid on the stream: weights do not depend on it
// (the documented contract of programmatic dependent launch), so this call's
// weight stream overlaps the previous kernel's tail.
template <int WF>
__device__ __forceinline__ void produce_stages(const GemvParams &p, uint8_t *smem, uint32_t bar0, int64_t v0,
                                               int64_t v1, int64_t roff, int64_t rbytes, int nst, int *s_abort)
{
    const int S = p.stage_rows;
    const int NS = p.nstages;
    const int stage_bytes = S * p.row_stride;
    int s = 0;
    uint32_t ph = 0;
    int issued = 0;
    for (int j = 0; j < nst; j++) {
        if (j == NS) { pdl_wait(); pdl_launch_dependents(); }
        if (j >= NS && !mbar_wait_bounded(bar0 + 8 * (NS + s), ph ^ 1)) {
            atomicExch(&g_gemv_error, 1);
            *s_abort = 1;
            break;
        }
        if (*(volatile int *)s_abort) break;
        issue_stage<WF>(p, smem_u32(smem) + (uint32_t)(s * stage_bytes), bar0 + 8 * s, v0 + (int64_t)j * S, S, v1,
                        roff, rbytes);
        issued = j + 1;
        if (++s == NS) { s = 0; ph ^= 1; }
    }
    if (nst <= NS) { pdl_wait(); pdl_launch_dependents(); }
    // do not leave while copies into this CTA's shared memory are in flight
    for (int j = max(0, issued - NS); j < issued; j++)
        mbar_wait_bounded(bar0 + 8 * (j % NS), (uint32_t)((j / NS) & 1));
}

// ---------------------------------------------------------------------------
// the kernel: one producer warp streams the CTA's rows into a ring of
// shared-memory stages with cp.async.bulk (one copy per contiguous run of
// rows); RG x TPR consumer threads read their K-slice of each staged row
// against activations held in registers.  Per-row partial sums of each warp
// go to shared memory and are combined (in warp order, so results are
// deterministic) once per window of rows.  Every wait on an mbarrier is
// bounded; on a timeout the kernel records an error in g_gemv_error and
// finishes without reading stale data.
// ---------------------------------------------------------------------------
template <int WF, int XF, int M, int C>
__global__ void __launch_bounds__(544, (M == 1) ? 2 : 1) gemv_kernel(const GemvParams p)
{
    constexpr int RPS = RowsPerStage<M>::value;
    constexpr int V = RPS * M;
    using WR = WarpReduce<V>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int ncons = p.RG * p.TPR;                // consumer threads (a multiple of 32)
    const int S = p.stage_rows;                    // SUB * RG * RPS
    const int NS = p.nstages;
    const int stage_bytes = S * p.row_stride;
    uint8_t *stages = smem;
    float *part = reinterpret_cast<float *>(smem + p.part_off);
    const uint32_t bar0 = smem_u32(smem + p.bar_off);   // full[NS] then empty[NS]

    int64_t v0, v1;
    cta_rows(p, v0, v1);
    const int split = blockIdx.y;
    const int cbeg = split * p.chunks_per_split;
    const int cend = min(p.nc, cbeg + p.chunks_per_split);
    int64_t roff, rbytes;
    chunk_range_bytes<WF>(cbeg, cend, roff, rbytes);
    const int nrows = (int)(v1 - v0);
    const int nst = (nrows + S - 1) / S;            // stages this CTA streams

    if (tid == 0) {
        for (int i = 0; i < NS; i++) {
            mbar_init(bar0 + 8 * i, 1);                       // full: producer's arrive + bytes
            mbar_init(bar0 + 8 * (NS + i), ncons / 32);       // empty: one arrive per consumer warp
        }
        s_abort = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (tid >= ncons) {
        if (lane == 0) produce_stages<WF>(p, smem, bar0, v0, v1, roff, rbytes, nst, &s_abort);
        return;
    }

    // ---------------- consumers ----------------
    pdl_wait();
    pdl_launch_dependents();
    const int g = tid / p.TPR;             // row group
    const int tau = tid - g * p.TPR;       // thread in group
    const int wig = tau >> 5;              // warp in group
    const int WPG = p.TPR >> 5;
    const int SUB = S / (p.RG * RPS);      // passes over a stage

    int coff[C], soff[C];
    bool cval[C];
    XSlice<WF, XF> xs[C][M];
#pragma unroll
    for (int i = 0; i < C; i++) {
        const int c = cbeg + tau + i * p.TPR;
        cval[i] = c < cend && chunk_valid<WF>(c, p.nb, p.nc);
        coff[i] = (int)(chunk_code_off<WF>(c) - roff);
        soff[i] = (WF == W_BF16) ? 0 : (int)(chunk_scale_off<WF>(c) - roff);
#pragma unroll
        for (int m = 0; m < M; m++) load_x<WF, XF>(xs[i][m], p, m, c, cval[i]);
    }

    const int64_t WIN = (int64_t)p.win_stages * S;
    int64_t win0 = v0;
    int s = 0, wstage = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int j = 0; j < nst; j++) {
        if (ok && !mbar_wait_bounded(bar0 + 8 * s, ph)) {
            atomicExch(&g_gemv_error, 1);
            s_abort = 1;
        }
        ok = ok && !*(volatile int *)&s_abort;
        const int64_t vs = v0 + (int64_t)j * S;
        const bool full = ok && (vs + S <= v1);
        const uint8_t *stage = stages + s * stage_bytes;
        for (int sub = 0; sub < SUB; sub++) {
            float acc[V];
#pragma unroll
            for (int rr = 0; rr < RPS; rr++) {
                const int r = (sub * RPS + rr) * p.RG + g;
                const bool rv = full || (ok && staged_vrow(p, vs, S, r) < v1);
                const uint8_t *srow = stage + r * p.row_stride;
                WChunk<WF> wc[C];
#pragma unroll
                for (int i = 0; i < C; i++) {
                    if (rv && cval[i]) {
                        wc[i].c = *reinterpret_cast<const uint4 *>(srow + coff[i]);
                        wc[i].s = (WF == W_BF16) ? 0u : (uint32_t)*reinterpret_cast<const uint16_t *>(srow + soff[i]);
                    } else {
                        wc[i].c = make_uint4(0, 0, 0, 0);
                        wc[i].s = 0;
                    }
                }
#pragma unroll
                for (int m = 0; m < M; m++) {
                    float a = 0.f;
#pragma unroll
                    for (int i = 0; i < C; i++) a += chunk_dot<WF, XF>(wc[i], xs[i][m]);
                    acc[rr * M + m] = a;
                }
            }
            if (sub == SUB - 1) {
                __syncwarp();
                if (lane == 0) mbar_arrive(bar0 + 8 * (NS + s));   // this warp is done with stage s
            }
            const float tot = WR::run(acc, lane);
            if (WR::is_holder(lane)) {
                const int idx = WR::index_of_lane(lane);
                const int rr = idx / M, m = idx - (idx / M) * M;
                const int64_t v = staged_vrow(p, vs, S, (sub * RPS + rr) * p.RG + g);
                if (v < v1) part[((int)(v - win0) * WPG + wig) * M + m] = tot;
            }
        }
        if (++s == NS) { s = 0; ph ^= 1; }

        // window complete: combine the warps' partials (warp order) and store
        if (++wstage == p.win_stages || j + 1 == nst) {
            wstage = 0;
            named_barrier(1, ncons);
            const int nrw = (int)min(WIN, v1 - win0);
            if (p.epi == EPI_SWIGLU) {
                for (int t = tid; t < (nrw >> 1) * M; t += ncons) {
                    const int pr = t / M;
                    const int m = t - pr * M;
                    float gs = 0.f, us = 0.f;
                    for (int w = 0; w < WPG; w++) {
                        gs += part[((2 * pr) * WPG + w) * M + m];
                        us += part[((2 * pr + 1) * WPG + w) * M + m];
                    }
                    const int64_t o = (win0 >> 1) + pr;
                    p.Y[0][(int64_t)m * p.rows[0] + o] = silu(gs) * us;
                }
            } else {
                for (int t = tid; t < nrw * M; t += ncons) {
                    const int row = t / M;
                    const int m = t - row * M;
                    float sum = 0.f;
                    for (int w = 0; w < WPG; w++) sum += part[(row * WPG + w) * M + m];
                    const int64_t v = win0 + row;
                    if (p.epi == EPI_PARTIAL) {
                        p.ws[((int64_t)split * M + m) * p.Nv + v] = sum;
                    } else {
                        int mat; int64_t rr;
                        map_row(p, v, mat, rr);
                        p.Y[mat][(int64_t)m * p.rows[mat] + rr] = sum;
                    }
                }
            }
            named_barrier(1, ncons);
            win0 += WIN;
        }
    }
    if (p.epi == EPI_SWIGLU && p.hq) swiglu_q8_1_finish(p, M, v0 >> 1, v1 >> 1, 1, tid >> 5, ncons >> 5, lane);
}

// ---------------------------------------------------------------------------
// Staged activations for the lanes-per-row kernel.  Chunk c of activation
// row m is P pieces of 16 bytes; piece p of chunks 32u .. 32u+31 is one run
// of 512 bytes, so lanes reading consecutive chunks hit distinct banks.
// Pieces hold eight bf16 (X_BF16, the default for bf16 activations) or four
// fp32 (X_F32, bf16 activations at M <= 2 when bf16 staging is off).  q8_1
// rows add, per block, (d as float, exact sum of codes) after the runs.
// ---------------------------------------------------------------------------
template <int WF, int XF> struct XPieces {
    static constexpr int P = ChunkTraits<WF>::E / ((XF == X_BF16) ? 8 : 4);
};
template <> struct XPieces<W_Q4_0, X_Q8_1> { static constexpr int P = 2; };                    // 32 codes

template <int WF, int XF>
__host__ __device__ __forceinline__ int x_stage_row_bytes(int nc, int nb)
{
    const int runs = (nc + 31) / 32;
    return runs * XPieces<WF, XF>::P * 512 + ((XF == X_Q8_1) ? nb * 8 : 0);
}

// Bytes of one activation row as the caller passes it: q8_1 blocks, or bf16
// (staged as bf16 or fp32).
template <int XF>
__device__ __forceinline__ int64_t x_src_row_bytes(const GemvParams &p)
{
    return (XF == X_Q8_1) ? (int64_t)p.nb * Q8_1_BYTES : (int64_t)p.K * 2;
}

// Build the staged layout from a raw copy of the M activation rows in
// shared memory (`raw` points at X[0]): bf16 become fp32; q8_1 blocks give
// their codes and a (d, exact sum of codes) pair.
template <int WF, int XF>
__device__ __forceinline__ void expand_x(const GemvParams &p, const uint8_t *raw, uint8_t *xs, int M, int tid, int nthr)
{
    constexpr int P = XPieces<WF, XF>::P;
    const int runs = (p.nc + 31) / 32;
    for (int m = 0; m < M; m++) {
        uint8_t *xr = xs + (size_t)m * p.x_row_bytes;
        for (int i = tid; i < p.nc * P; i += nthr) {
            const int c = i / P, pc = i - (i / P) * P;
            if (!chunk_valid<WF>(c, p.nb, p.nc)) continue;
            uint4 v;
            if constexpr (XF == X_Q8_1) {
                const uint32_t *blk = reinterpret_cast<const uint32_t *>(raw + ((int64_t)m * p.nb + c) * Q8_1_BYTES);
                v = make_uint4(blk[1 + 4 * pc], blk[2 + 4 * pc], blk[3 + 4 * pc], blk[4 + 4 * pc]);
                if (pc == 0) {
                    int sum = 0;
#pragma unroll
                    for (int k = 0; k < 8; k++) sum = __dp4a((int)blk[1 + k], 0x01010101, sum);
                    const float2 ds = make_float2(half_bits_to_float(blk[0] & 0xffffu), __int_as_float(sum));
                    *reinterpret_cast<float2 *>(xr + (size_t)runs * P * 512 + (size_t)c * 8) = ds;
                }
            } else {
                // four consecutive bf16 -> fp32
                const uint2 w = *reinterpret_cast<const uint2 *>(raw + ((int64_t)m * p.K + chunk_elem0<WF>(c) + 4 * pc) * 2);
                v = make_uint4(w.x << 16, w.x & 0xffff0000u, w.y << 16, w.y & 0xffff0000u);
            }
            *reinterpret_cast<uint4 *>(xr + ((size_t)(c >> 5) * P + pc) * 512 + (c & 31) * 16) = v;
        }
    }
}

// bf16 activation rows copied as they are (row m at m * x_row_bytes) into
// the staged bf16 layout, in place: for 32-element blocks (q8_0, q4_0
// weights) piece j (elements 8j .. 8j+7) of block s of tile t moves from
// t * 2048 + s * 64 + j * 16 to t * 2048 + j * 512 + s * 16.  A tile's
// 2 KiB map onto themselves, so each warp permutes whole tiles alone.  For
// bf16 weights (one piece per chunk) the copied rows are already staged.
template <int WF>
__device__ __forceinline__ void permute_x_bf16(const GemvParams &p, uint8_t *xs, int M, int warp, int nwarps, int lane)
{
    if constexpr (WF != W_BF16) {
        const int T = (p.nb + 31) / 32;
        for (int r = warp; r < M * T; r += nwarps) {
            uint8_t *base = xs + (size_t)(r / T) * p.x_row_bytes + (size_t)(r - (r / T) * T) * 2048;
            uint4 v[4];
#pragma unroll
            for (int k = 0; k < 4; k++) v[k] = *reinterpret_cast<const uint4 *>(base + lane * 64 + k * 16);
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; k++) *reinterpret_cast<uint4 *>(base + k * 512 + lane * 16) = v[k];
            __syncwarp();
        }
    }
}

template <int WF, int XF>
__device__ __forceinline__ void lds_x(XSlice<WF, XF> &x, const uint8_t *xr, int c, int runs)
{
    constexpr int P = XPieces<WF, XF>::P;
    const uint8_t *base = xr + (size_t)(c >> 5) * P * 512 + (c & 31) * 16;
    if constexpr (XF == X_Q8_1) {
        const uint4 a = *reinterpret_cast<const uint4 *>(base);
        const uint4 b = *reinterpret_cast<const uint4 *>(base + 512);
        x.q[0] = a.x; x.q[1] = a.y; x.q[2] = a.z; x.q[3] = a.w;
        x.q[4] = b.x; x.q[5] = b.y; x.q[6] = b.z; x.q[7] = b.w;
        const float2 ds = *reinterpret_cast<const float2 *>(xr + (size_t)runs * P * 512 + (size_t)c * 8);
        x.d = ds.x;
        x.sum = __float_as_int(ds.y);
    } else {
#pragma unroll
        for (int pc = 0; pc < P; pc++) {
            const float4 f = *reinterpret_cast<const float4 *>(base + pc * 512);
            x.f[4 * pc] = f.x; x.f[4 * pc + 1] = f.y; x.f[4 * pc + 2] = f.z; x.f[4 * pc + 3] = f.w;
        }
    }
}

// ---------------------------------------------------------------------------
// Tile loops of the lanes-per-row kernel.  A "tile" is 32 lane units of a
// row: 32 q8_0 / q4_0 blocks (one repacked tile) or 32 chunks of 8 bf16.
// Lane `sub` owns unit `sub` of every tile, so all its addresses inside a
// tile are fixed offsets from the tile's base; the staged activations use
// the matching layout (16-byte piece pc of unit s of tile t at
// t * TX + pc * 512 + s * 16), which keeps every warp-wide shared load
// conflict-free.  Sums go to two fp32 partials per output (acc[i][m][0..1]).
// ---------------------------------------------------------------------------
template <int WF> struct TileTraits;
template <> struct TileTraits<W_BF16> { static constexpr int CPT = 32, TW = 512; };    // chunks, weight bytes
template <> struct TileTraits<W_Q8_0> { static constexpr int CPT = 64, TW = Q8_0_TILE; };
template <> struct TileTraits<W_Q4_0> { static constexpr int CPT = 32, TW = Q4_0_TILE; };
// staged activation bytes of one tile
template <int WF, int XF> struct TileX {
    static constexpr int TX = ((WF == W_BF16) ? 1024 : 4096) / ((XF == X_BF16) ? 2 : 1);
};
template <> struct TileX<W_Q4_0, X_Q8_1> { static constexpr int TX = 1024; };

// sum over the 16 int8 codes of c of q * x (x: 16 fp32 in four float4), into
// four running partials
__device__ __forceinline__ void q8x16(const uint4 &c, const float4 *x, float &a0, float &a1, float &b0, float &b1)
{
    constexpr float OFF = 8388608.0f + 128.0f;     // codes enter as 2^23 + (q + 128)
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const uint32_t u = cw[k] ^ 0x80808080u;
        float e0 = byte_plus_2p23<0>(u), e1 = byte_plus_2p23<1>(u);
        float e2 = byte_plus_2p23<2>(u), e3 = byte_plus_2p23<3>(u);
        fadd2(e0, e1, -OFF);
        fadd2(e2, e3, -OFF);
        ffma2(a0, a1, e0, e1, x[k].x, x[k].y);
        ffma2(b0, b1, e2, e3, x[k].z, x[k].w);
    }
}

// sum over 32 q4_0 codes (16 bytes: word k = elements 4k..4k+3 in its low
// nibbles, 16+4k..16+4k+3 in its high nibbles) of (q - 8) * x, x: 32 fp32
__device__ __forceinline__ float q4x32(const uint4 &c, const float4 *x)
{
    constexpr float OFF = 8388608.0f + 8.0f;
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const uint32_t lo = cw[k] & 0x0f0f0f0fu;
        const uint32_t hi = (cw[k] >> 4) & 0x0f0f0f0fu;
        float l0 = byte_plus_2p23<0>(lo), l1 = byte_plus_2p23<1>(lo);
        float l2 = byte_plus_2p23<2>(lo), l3 = byte_plus_2p23<3>(lo);
        float h0 = byte_plus_2p23<0>(hi), h1 = byte_plus_2p23<1>(hi);
        float h2 = byte_plus_2p23<2>(hi), h3 = byte_plus_2p23<3>(hi);
        fadd2(l0, l1, -OFF);
        fadd2(l2, l3, -OFF);
        fadd2(h0, h1, -OFF);
        fadd2(h2, h3, -OFF);
        ffma2(a0, a1, l0, l1, x[k].x, x[k].y);
        ffma2(b0, b1, l2, l3, x[k].z, x[k].w);
        ffma2(a0, a1, h0, h1, x[4 + k].x, x[4 + k].y);
        ffma2(b0, b1, h2, h3, x[4 + k].z, x[4 + k].w);
    }
    return (a0 + a1) + (b0 + b1);
}

// four unsigned bytes of a times four signed bytes of b, plus c
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// exact sum over 32 q4_0 codes of (q - 8) * qx: low nibbles against codes
// 0..15 of the q8_1 block, high nibbles (kept as 16 h, unsigned) against
// codes 16..31; the second sum is a multiple of 16 and divides exactly
__device__ __forceinline__ int q4q8_sumi(const uint4 &c, const uint4 &xlo, const uint4 &xhi, int xsum)
{
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    const int xl[4] = {(int)xlo.x, (int)xlo.y, (int)xlo.z, (int)xlo.w};
    const int xh[4] = {(int)xhi.x, (int)xhi.y, (int)xhi.z, (int)xhi.w};
    int a = 0, b = 0;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        a = __dp4a((int)(cw[k] & 0x0f0f0f0fu), xl[k], a);
        b = dp4a_us(cw[k] & 0xf0f0f0f0u, xh[k], b);
    }
    return a + (b >> 4) - 8 * xsum;
}

// acc[i][m] += dot(row i of the stage, activation row m) over tiles
// [0, nt) of the stage (global tile tg + t); in the last tile only lanes
// below `tail` hold a unit.  DOTS (q4_0 x q8_1 check instantiation): the
// integer dot of block b of stage row i < dots_rows is also stored at
// dots[i * nb + b].
template <int WF, int XF, int M, int RL, bool DOTS = false>
__device__ __forceinline__ void lpr_tiles(float (&acc)[RL][M][2], const uint8_t *stage, int row_stride,
                                          const uint8_t *xs, int x_row_bytes, int ds_off, int tg, int nt, int tail,
                                          int sub, int32_t *dots = nullptr, int dots_rows = 0, int nb = 0)
{
    constexpr int TW = TileTraits<WF>::TW;
    constexpr int TX = TileX<WF, XF>::TX;
    const uint8_t *w0 = stage + 16 * sub;
    const uint8_t *x0 = xs + (int64_t)tg * TX + 16 * sub;
    auto body = [&](int t) {
        const uint8_t *wt = w0 + t * TW;
        const uint8_t *xt = x0 + t * TX;
        if constexpr (WF == W_BF16 && XF == X_BF16) {
            // weights converted once, each activation piece (8 bf16) once per row m
            float w[RL][8];
#pragma unroll
            for (int i = 0; i < RL; i++) {
                const uint4 c = *reinterpret_cast<const uint4 *>(wt + i * row_stride);
                bf16x8_to_f32(c, w[i]);
            }
#pragma unroll
            for (int m = 0; m < M; m++) {
                float x[8];
                bf16x8_to_f32(*reinterpret_cast<const uint4 *>(xt + m * x_row_bytes), x);
#pragma unroll
                for (int i = 0; i < RL; i++)
#pragma unroll
                    for (int k = 0; k < 8; k += 2) ffma2(acc[i][m][0], acc[i][m][1], w[i][k], w[i][k + 1], x[k], x[k + 1]);
            }
        } else if constexpr (WF == W_BF16) {
            uint4 c[RL];
#pragma unroll
            for (int i = 0; i < RL; i++) c[i] = *reinterpret_cast<const uint4 *>(wt + i * row_stride);
#pragma unroll
            for (int m = 0; m < M; m++) {
                const float4 xa = *reinterpret_cast<const float4 *>(xt + m * x_row_bytes);
                const float4 xb = *reinterpret_cast<const float4 *>(xt + m * x_row_bytes + 512);
#pragma unroll
                for (int i = 0; i < RL; i++) {
                    float &s0 = acc[i][m][0], &s1 = acc[i][m][1];
                    ffma2(s0, s1, bf16_lo(c[i].x), bf16_hi(c[i].x), xa.x, xa.y);
                    ffma2(s0, s1, bf16_lo(c[i].y), bf16_hi(c[i].y), xa.z, xa.w);
                    ffma2(s0, s1, bf16_lo(c[i].z), bf16_hi(c[i].z), xb.x, xb.y);
                    ffma2(s0, s1, bf16_lo(c[i].w), bf16_hi(c[i].w), xb.z, xb.w);
                }
            }
        } else if constexpr (WF == W_Q8_0 && XF == X_BF16) {
            // unit = block sub; codes dequantized once per 8-element piece,
            // each activation piece loaded once per row m
            constexpr float OFF = 8388608.0f + 128.0f;
            uint4 c0[RL], c1[RL];
            float d[RL];
#pragma unroll
            for (int i = 0; i < RL; i++) {
                c0[i] = *reinterpret_cast<const uint4 *>(wt + i * row_stride);
                c1[i] = *reinterpret_cast<const uint4 *>(wt + i * row_stride + 512);
                d[i] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(wt + i * row_stride + 1024 - 14 * sub));
            }
            float sm[RL][M][2];
#pragma unroll
            for (int i = 0; i < RL; i++)
#pragma unroll
                for (int m = 0; m < M; m++) sm[i][m][0] = sm[i][m][1] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                float e[RL][8];
#pragma unroll
                for (int i = 0; i < RL; i++) {
                    const uint32_t wa = (j == 0) ? c0[i].x : (j == 1) ? c0[i].z : (j == 2) ? c1[i].x : c1[i].z;
                    const uint32_t wb = (j == 0) ? c0[i].y : (j == 1) ? c0[i].w : (j == 2) ? c1[i].y : c1[i].w;
                    const uint32_t ua = wa ^ 0x80808080u, ub = wb ^ 0x80808080u;
                    e[i][0] = byte_plus_2p23<0>(ua); e[i][1] = byte_plus_2p23<1>(ua);
                    e[i][2] = byte_plus_2p23<2>(ua); e[i][3] = byte_plus_2p23<3>(ua);
                    e[i][4] = byte_plus_2p23<0>(ub); e[i][5] = byte_plus_2p23<1>(ub);
                    e[i][6] = byte_plus_2p23<2>(ub); e[i][7] = byte_plus_2p23<3>(ub);
#pragma unroll
                    for (int k = 0; k < 8; k += 2) fadd2(e[i][k], e[i][k + 1], -OFF);
                }
#pragma unroll
                for (int m = 0; m < M; m++) {
                    float x[8];
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(xt + m * x_row_bytes + j * 512), x);
#pragma unroll
                    for (int i = 0; i < RL; i++)
#pragma unroll
                        for (int k = 0; k < 8; k += 2) ffma2(sm[i][m][0], sm[i][m][1], e[i][k], e[i][k + 1], x[k], x[k + 1]);
                }
            }
#pragma unroll
            for (int i = 0; i < RL; i++)
#pragma unroll
                for (int m = 0; m < M; m++) acc[i][m][0] = fmaf(sm[i][m][0] + sm[i][m][1], d[i], acc[i][m][0]);
        } else if constexpr (WF == W_Q8_0) {
            // unit = block sub: codes 0..15 at +0, 16..31 at +512, scale at 1024 + 2 sub
            uint4 c0[RL], c1[RL];
            float d[RL];
#pragma unroll
            for (int i = 0; i < RL; i++) {
                c0[i] = *reinterpret_cast<const uint4 *>(wt + i * row_stride);
                c1[i] = *reinterpret_cast<const uint4 *>(wt + i * row_stride + 512);
                d[i] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(wt + i * row_stride + 1024 - 14 * sub));
            }
#pragma unroll
            for (int m = 0; m < M; m++) {
                float4 x[8];
#pragma unroll
                for (int pc = 0; pc < 8; pc++) x[pc] = *reinterpret_cast<const float4 *>(xt + m * x_row_bytes + pc * 512);
#pragma unroll
                for (int i = 0; i < RL; i++) {
                    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
                    q8x16(c0[i], x, a0, a1, b0, b1);
                    q8x16(c1[i], x + 4, a0, a1, b0, b1);
                    acc[i][m][0] = fmaf((a0 + a1) + (b0 + b1), d[i], acc[i][m][0]);
                }
            }
        } else if constexpr (XF == X_Q8_1) {
            // unit = block sub: codes at +0, scale at 512 + 2 sub; q8_1 codes at +0 / +512, (d, sum) at ds_off
            uint4 c[RL];
            float d[RL];
#pragma unroll
            for (int i = 0; i < RL; i++) {
                c[i] = *reinterpret_cast<const uint4 *>(wt + i * row_stride);
                d[i] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(wt + i * row_stride + 512 - 14 * sub));
            }
#pragma unroll
            for (int m = 0; m < M; m++) {
                const uint4 xl = *reinterpret_cast<const uint4 *>(xt + m * x_row_bytes);
                const uint4 xh = *reinterpret_cast<const uint4 *>(xt + m * x_row_bytes + 512);
                const float2 ds = *reinterpret_cast<const float2 *>(xs + m * x_row_bytes + ds_off +
                                                                    ((tg + t) * 32 + sub) * 8);
#pragma unroll
                for (int i = 0; i < RL; i++) {
                    const int sumi = q4q8_sumi(c[i], xl, xh, __float_as_int(ds.y));
                    if constexpr (DOTS) {
                        if (m == 0 && i < dots_rows) dots[(int64_t)i * nb + (tg + t) * 32 + sub] = sumi;
                    }
                    acc[i][m][0] = fmaf(d[i] * ds.x, (float)sumi, acc[i][m][0]);
                }
            }
        } else if constexpr (XF == X_BF16) {
            // q4_0 against bf16 activations: unit = block sub; piece j
            // (elements 8j .. 8j+7) is the low (j < 2) or high nibbles of
            // words 2(j&1), 2(j&1)+1
            constexpr float OFF = 8388608.0f + 8.0f;
            uint4 c[RL];
            float d[RL];
#pragma unroll
            for (int i = 0; i < RL; i++) {
                c[i] = *reinterpret_cast<const uint4 *>(wt + i * row_stride);
                d[i] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(wt + i * row_stride + 512 - 14 * sub));
            }
            float sm[RL][M][2];
#pragma unroll
            for (int i = 0; i < RL; i++)
#pragma unroll
                for (int m = 0; m < M; m++) sm[i][m][0] = sm[i][m][1] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                float e[RL][8];
#pragma unroll
                for (int i = 0; i < RL; i++) {
                    const uint32_t w0 = (j & 1) ? c[i].z : c[i].x;
                    const uint32_t w1 = (j & 1) ? c[i].w : c[i].y;
                    const uint32_t ua = ((j < 2) ? w0 : (w0 >> 4)) & 0x0f0f0f0fu;
                    const uint32_t ub = ((j < 2) ? w1 : (w1 >> 4)) & 0x0f0f0f0fu;
                    e[i][0] = byte_plus_2p23<0>(ua); e[i][1] = byte_plus_2p23<1>(ua);
                    e[i][2] = byte_plus_2p23<2>(ua); e[i][3] = byte_plus_2p23<3>(ua);
                    e[i][4] = byte_plus_2p23<0>(ub); e[i][5] = byte_plus_2p23<1>(ub);
                    e[i][6] = byte_plus_2p23<2>(ub); e[i][7] = byte_plus_2p23<3>(ub);
#pragma unroll
                    for (int k = 0; k < 8; k += 2) fadd2(e[i][k], e[i][k + 1], -OFF);
                }
#pragma unroll
                for (int m = 0; m < M; m++) {
                    float x[8];
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(xt + m * x_row_bytes + j * 512), x);
#pragma unroll
                    for (int i = 0; i < RL; i++)
#pragma unroll
                        for (int k = 0; k < 8; k += 2) ffma2(sm[i][m][0], sm[i][m][1], e[i][k], e[i][k + 1], x[k], x[k + 1]);
                }
            }
#pragma unroll
            for (int i = 0; i < RL; i++)
#pragma unroll
                for (int m = 0; m < M; m++) acc[i][m][0] = fmaf(sm[i][m][0] + sm[i][m][1], d[i], acc[i][m][0]);
        } else {
            // q4_0 against fp32 activations: unit = block sub
            uint4 c[RL];
            float d[RL];
#pragma unroll
            for (int i = 0; i < RL; i++) {
                c[i] = *reinterpret_cast<const uint4 *>(wt + i * row_stride);
                d[i] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(wt + i * row_stride + 512 - 14 * sub));
            }
#pragma unroll
            for (int m = 0; m < M; m++) {
                float4 x[8];
#pragma unroll
                for (int pc = 0; pc < 8; pc++) x[pc] = *reinterpret_cast<const float4 *>(xt + m * x_row_bytes + pc * 512);
#pragma unroll
                for (int i = 0; i < RL; i++) acc[i][m][0] = fmaf(q4x32(c[i], x), d[i], acc[i][m][0]);
            }
        }
    };
    int t = 0;
#pragma unroll 2
    for (; t + 1 < nt; t++) body(t);
    if (nt > 0 && sub < tail) body(nt - 1);
}

// ---------------------------------------------------------------------------
// Lanes-per-row kernel (M = 1, 2, 4, 8).  There is no producer warp: each of the
// CTA's NW warps streams its own work.  The CTA's rows are cut into blocks
// of RL consecutive rows (a gate/up block holds RL/2 gate rows, then the
// matching up rows), and block b belongs to warp b % NW.  A block is
// streamed in K-pieces of whole tiles: stage (b, piece) holds that piece of
// the block's rows, one bulk copy per run of rows.  Each warp owns D
// shared-memory slots and uses them in turn.  Lane 0 requests the warp's
// first stages before the grid waits for the previous kernel on the stream
// (weights do not depend on it) and refills a slot with the warp's stage D
// places later as soon as the warp has read it.  A slot is only ever filled
// and read by its own warp, in order, so each full barrier is waited on once
// per phase and no empty barrier is needed.
//
// All 32 lanes of the warp work on every row of the block (lpr_tiles): each
// activation load serves the RL rows.  Sums carry across the pieces of a
// block; after its last piece one warp shuffle reduction per output
// finishes the block, which lane 0 stores.
// ---------------------------------------------------------------------------
// M = 4, 8: at most eight warps, so that two rows per lane (half the
// shared-memory activation reads per weight) fit in registers
template <int M> struct LprThreads { static constexpr int value = (M >= 4) ? 256 : 384; };

// DOTS: the check instantiation (q4_0 x q8_1, M = 1, one matrix) that also
// stores every integer block dot in p.dots and writes no output.
template <int WF, int XF, int M, int RL, bool DOTS = false>
__global__ void __launch_bounds__(LprThreads<M>::value, 2) gemv_lpr_kernel(const GemvParams p)
{
    static_assert(!DOTS || (WF == W_Q4_0 && XF == X_Q8_1 && M == 1), "block dots: q4_0 x q8_1, one row");
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort;
    constexpr int CPT = TileTraits<WF>::CPT;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int NW = p.ng;                           // warps
    const int D = p.nstages;                       // slots per warp
    const int PCS = p.piece_chunks;                // chunks per K-piece (whole tiles)
    const int row_stride = p.row_stride;           // bytes of one row's piece
    const int stage_bytes = RL * row_stride;
    uint8_t *xs = smem + p.x_off;
    const uint32_t bar0 = smem_u32(smem + p.bar_off);      // full barriers (NW * D), then the activation copy's

    int64_t v0, v1;
    cta_rows(p, v0, v1);
    const int split = blockIdx.y;
    const int cbeg = split * p.chunks_per_split;
    const int cend = min(p.nc, cbeg + p.chunks_per_split);
    const int npc = (cend - cbeg + PCS - 1) / PCS;           // pieces per block
    const int nrows = (int)(v1 - v0);
    const int nrb = (nrows + RL - 1) / RL;
    const int my_blocks = (warp < nrb) ? (nrb - warp + NW - 1) / NW : 0;
    const int my_stages = my_blocks * npc;
    const uint32_t slot0 = smem_u32(smem) + (uint32_t)(warp * D * stage_bytes);
    const uint32_t wbar = bar0 + 8 * warp * D;
    const uint32_t xbar = bar0 + 8 * NW * D;
    // units (blocks, or chunks of bf16) of a row: the last tile may be partial
    const int units = (WF == W_BF16) ? p.nc : p.nb;

    // stage t of this warp: block warp + NW * (t / npc), piece t % npc
    // one matrix, whole rows: a stage is RL consecutive rows, one copy
    const bool simple = (p.nmat == 1 && npc == 1 && cbeg == 0 && cend == p.nc);
    const uint8_t *wrow0 = p.W[0] + v0 * p.row_bytes;
    auto issue = [&](int t, int slot) {
        if (simple) {
            const int r = (warp + NW * t) * RL;                  // first row of the stage, from v0
            const uint32_t n = (uint32_t)min(RL, nrows - r) * (uint32_t)p.row_bytes;
            mbar_arrive_expect_tx(wbar + 8 * slot, n);
            bulk_g2s(slot0 + slot * stage_bytes, wrow0 + (int64_t)r * p.row_bytes, n, wbar + 8 * slot);
            return;
        }
        const int bl = t / npc, pc = t - (t / npc) * npc;
        const int ca = cbeg + pc * PCS;
        int64_t poff, pbytes;
        chunk_range_bytes<WF>(ca, min(cend, ca + PCS), poff, pbytes);
        issue_stage<WF>(p, slot0 + slot * stage_bytes, wbar + 8 * slot, v0 + (int64_t)(warp + NW * bl) * RL, RL, v1,
                        poff, pbytes);
    };

    if (tid == 0) {
        for (int i = 0; i < NW * D; i++) mbar_init(bar0 + 8 * i, 1);   // lane 0's arrive + bytes
        mbar_init(xbar, 1);
        s_abort = 0;
        mbar_fence_init();
    }
    __syncthreads();

    // the warp's first stages, requested before the previous grid completes
    int issued = 0;
    const int first = min(D, my_stages);
    const int early = min(first, p.early);
    if (lane == 0)
        for (; issued < early; issued++) issue(issued, issued);

    // The activation rows may still be written by the previous grid, so they
    // are read only after the wait below; but their lines can be brought into
    // L2 now.  L2 is the point of coherence for the SMs' writes, so a line
    // fetched early still returns the previous grid's data after the wait,
    // and the copy after the wait then costs an L2 hit instead of a loaded
    // HBM round trip (measured: -0.2 to -0.4 us per call for the quantized
    // formats; nothing for bf16 weights, which skip it).  The span is the
    // 16-byte-aligned one the copy below reads.
    const uintptr_t xa = reinterpret_cast<uintptr_t>(p.X);
    const int xoff = (int)(xa & 15);
    if constexpr (WF != W_BF16) {
        if (tid == 32)
            prefetch_l2_bulk(reinterpret_cast<const void *>(xa - xoff),
                             (uint32_t)((xoff + M * x_src_row_bytes<XF>(p) + 15) & ~15ll));
    }
    pdl_wait();
    pdl_launch_dependents();
    // The activation rows come in one bulk copy, requested before the rest of
    // the weight stream so that they do not queue behind it.  The copy covers
    // the 16-byte-aligned span around X (at most 15 bytes either side, which
    // never crosses a page), as bulk copies need 16-byte alignment.
    if constexpr (XF == X_BF16) {
        // bf16 rows (16-byte aligned) straight into their staged rows
        if (tid == 0) {
            const uint32_t rb = (uint32_t)p.K * 2;
            mbar_arrive_expect_tx(xbar, (uint32_t)M * rb);
            for (int m = 0; m < M; m++)
                bulk_g2s(smem_u32(xs + (size_t)m * p.x_row_bytes), p.X + (size_t)m * rb, rb, xbar);
        }
    } else {
        const uint32_t xcopy = (uint32_t)((xoff + M * x_src_row_bytes<XF>(p) + 15) & ~15ll);
        if (tid == 0) {
            mbar_arrive_expect_tx(xbar, xcopy);
            bulk_g2s(smem_u32(smem + p.xraw_off), reinterpret_cast<const void *>(xa - xoff), xcopy, xbar);
        }
    }
    __syncthreads();
    if (lane == 0)
        for (; issued < first; issued++) issue(issued, issued);
    const bool xok = mbar_wait_bounded(xbar, 0);
    if (!xok) {
        atomicExch(&g_gemv_error, 1);
        s_abort = 1;
    }
    if constexpr (XF == X_BF16)
        permute_x_bf16<WF>(p, xs, M, warp, NW, lane);
    else
        expand_x<WF, XF>(p, smem + p.xraw_off + xoff, xs, M, tid, blockDim.x);
    __syncthreads();

    const int ds_off = ((p.nc + 31) / 32) * XPieces<WF, XF>::P * 512;   // q8_1 (d, sum) table
    const bool swiglu = (p.epi == EPI_SWIGLU);
    const int x_row_bytes = p.x_row_bytes;

    int d = 0;                                     // slot of the warp's next stage
    uint32_t ph = 0;
    int waited = 0;                                // stages whose bytes lane 0 has seen land
    bool ok = !*(volatile int *)&s_abort;
    float acc[RL][M][2];
#pragma unroll
    for (int i = 0; i < RL; i++)
#pragma unroll
        for (int m = 0; m < M; m++) acc[i][m][0] = acc[i][m][1] = 0.f;
    int bl = 0, pc = 0;                            // block (of this warp) and piece of stage t
    for (int t = 0; t < my_stages; t++) {
        if (ok) {
            if (mbar_wait_bounded(wbar + 8 * d, ph)) {
                waited++;
            } else {
                atomicExch(&g_gemv_error, 1);
                s_abort = 1;
            }
        }
        ok = ok && !*(volatile int *)&s_abort;
        if (ok) {
            const int ca = cbeg + pc * PCS;
            const int cb = min(cend, ca + PCS);
            const int tg = ca / CPT;                                 // first tile (global) of the piece
            const int nt = (cb - ca + CPT - 1) / CPT;
            const int tail = min(32, units - 32 * (tg + nt - 1));   // units in the piece's last tile
            if constexpr (DOTS) {
                const int64_t vb = v0 + (int64_t)(warp + NW * bl) * RL;      // first row of the stage
                lpr_tiles<WF, XF, M, RL, true>(acc, smem + (warp * D + d) * stage_bytes, row_stride, xs, x_row_bytes,
                                               ds_off, tg, nt, tail, lane, p.dots + vb * p.nb,
                                               (int)(v1 - vb < RL ? v1 - vb : RL), p.nb);
            } else {
                lpr_tiles<WF, XF, M, RL>(acc, smem + (warp * D + d) * stage_bytes, row_stride, xs, x_row_bytes, ds_off,
                                         tg, nt, tail, lane);
            }
        }
        // the warp is done with this slot: refill it with the warp's stage t + D
        __syncwarp();
        if (lane == 0 && ok && t + D < my_stages) {
            fence_proxy_async_smem();
            issue(t + D, d);
            issued++;
        }
        if (++d == D) { d = 0; ph ^= 1; }
        if (++pc < npc) continue;

        // the block's last piece: finish its outputs over the warp (fixed butterfly order)
        pc = 0;
        const int64_t vb = v0 + (int64_t)(warp + NW * bl) * RL;
        bl++;
        float tot[RL][M];
#pragma unroll
        for (int i = 0; i < RL; i++)
#pragma unroll
            for (int m = 0; m < M; m++) {
                float a = acc[i][m][0] + acc[i][m][1];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
                tot[i][m] = a;
                acc[i][m][0] = acc[i][m][1] = 0.f;
            }
        if (swiglu) {
            // rows 0 .. RL/2-1 are gates, RL/2 .. RL-1 the matching ups
#pragma unroll
            for (int k = 0; k < RL / 2; k++) {
                const int64_t v = staged_vrow(p, vb, RL, k);
                const bool valid = ok && v < v1;
#pragma unroll
                for (int m = 0; m < M; m++)
                    if (lane == 0 && valid) p.Y[0][(int64_t)m * p.rows[0] + (v >> 1)] = silu(tot[k][m]) * tot[RL / 2 + k][m];
            }
            continue;
        }
        if (lane != 0 || !ok) continue;
        if constexpr (!DOTS) {
#pragma unroll
            for (int i = 0; i < RL; i++) {
                const int64_t v = staged_vrow(p, vb, RL, i);
                if (v >= v1) continue;
#pragma unroll
                for (int m = 0; m < M; m++) {
                    if (p.epi == EPI_PARTIAL) {
                        p.ws[((int64_t)split * M + m) * p.Nv + v] = tot[i][m];
                    } else {
                        int mat; int64_t rr;
                        map_row(p, v, mat, rr);
                        p.Y[mat][(int64_t)m * p.rows[mat] + rr] = tot[i][m];
                    }
                }
            }
        }
    }
    // after a timeout: do not leave while this CTA's copies are in flight
    if (lane == 0) {
        for (int t = waited; t < issued; t++)
            mbar_wait_bounded(wbar + 8 * (t % D), (uint32_t)((t / D) & 1));
    }
    if (tid == 0 && !xok) mbar_wait_bounded(xbar, 0);
    if (swiglu && p.hq) swiglu_q8_1_finish(p, M, v0 >> 1, v1 >> 1, 0, warp, NW, lane);
}

// ---------------------------------------------------------------------------
// Lanes-per-row kernel, common case: one matrix, whole rows in every stage,
// no split of K, plain store of the outputs (every single-matrix GEMV whose
// staged rows fit a stage, which includes the decode and sweep shapes).  It
// is gemv_lpr_kernel with the general paths taken out at compile time:
// stage t of a warp is its block t (RL consecutive rows, one bulk copy), the
// tiles of a stage are the same for every stage, and each block's outputs
// are finished by a recursive-halving warp reduction whose holder lanes
// store them.  Measured on the decode shapes, the bookkeeping of the general
// kernel (piece arithmetic per stage, matrix and epilogue branches per row)
// was a quarter to a half of all instructions issued.
// DOTS: the check instantiation (q4_0 x q8_1, M = 1) that also stores every
// integer block dot in p.dots and writes no output.
// ---------------------------------------------------------------------------
template <int WF, int XF, int M, int RL, bool DOTS = false>
__global__ void __launch_bounds__(LprThreads<M>::value, 2) gemv_lpr_rows_kernel(const GemvParams p)
{
    static_assert(!DOTS || (WF == W_Q4_0 && XF == X_Q8_1 && M == 1), "block dots: q4_0 x q8_1, one row");
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort;
    constexpr int CPT = TileTraits<WF>::CPT;
    constexpr int V = RL * M;                      // outputs a warp finishes per block
    using WR = WarpReduce<V>;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int NW = p.ng;                           // warps
    const int D = p.nstages;                       // slots per warp
    const uint32_t row_bytes = (uint32_t)p.row_bytes;
    const uint32_t stage_bytes = RL * row_bytes;   // a stage is RL whole rows
    uint8_t *xs = smem + p.x_off;
    const uint32_t bar0 = smem_u32(smem + p.bar_off);

    int64_t v0, v1;
    cta_rows(p, v0, v1);
    const int nrows = (int)(v1 - v0);
    const int nrb = (nrows + RL - 1) / RL;
    const int my_blocks = (warp < nrb) ? (nrb - 1 - warp) / NW + 1 : 0;
    const uint32_t slot0 = smem_u32(smem) + (uint32_t)warp * (uint32_t)D * stage_bytes;
    const uint32_t wbar = bar0 + 8 * warp * D;
    const uint32_t xbar = bar0 + 8 * NW * D;
    const uint8_t *wrow0 = p.W[0] + v0 * p.row_bytes;
    // block b of this warp: rows r = (warp + NW b) RL .. + RL of the CTA's range
    auto issue = [&](int b, int slot) {
        const int r = (warp + NW * b) * RL;
        const uint32_t n = (uint32_t)min(RL, nrows - r) * row_bytes;
        mbar_arrive_expect_tx(wbar + 8 * slot, n);
        bulk_g2s(slot0 + slot * stage_bytes, wrow0 + (int64_t)r * row_bytes, n, wbar + 8 * slot);
    };

    if (tid == 0) {
        for (int i = 0; i < NW * D; i++) mbar_init(bar0 + 8 * i, 1);
        mbar_init(xbar, 1);
        s_abort = 0;
        mbar_fence_init();
    }
    __syncthreads();

    int issued = 0;
    const int first = min(D, my_blocks);
    const int early = min(first, p.early);
    if (lane == 0)
        for (; issued < early; issued++) issue(issued, issued);
    const uintptr_t xa = reinterpret_cast<uintptr_t>(p.X);
    const int xoff = (int)(xa & 15);
    if constexpr (WF != W_BF16) {
        // see gemv_lpr_kernel: the activation lines enter L2 before the wait
        if (tid == 32)
            prefetch_l2_bulk(reinterpret_cast<const void *>(xa - xoff),
                             (uint32_t)((xoff + M * x_src_row_bytes<XF>(p) + 15) & ~15ll));
    }
    pdl_wait();
    pdl_launch_dependents();
    if constexpr (XF == X_BF16) {
        if (tid == 0) {
            const uint32_t rb = (uint32_t)p.K * 2;
            mbar_arrive_expect_tx(xbar, (uint32_t)M * rb);
            for (int m = 0; m < M; m++)
                bulk_g2s(smem_u32(xs + (size_t)m * p.x_row_bytes), p.X + (size_t)m * rb, rb, xbar);
        }
    } else {
        const uint32_t xcopy = (uint32_t)((xoff + M * x_src_row_bytes<XF>(p) + 15) & ~15ll);
        if (tid == 0) {
            mbar_arrive_expect_tx(xbar, xcopy);
            bulk_g2s(smem_u32(smem + p.xraw_off), reinterpret_cast<const void *>(xa - xoff), xcopy, xbar);
        }
    }
    __syncthreads();
    if (lane == 0)
        for (; issued < first; issued++) issue(issued, issued);
    const bool xok = mbar_wait_bounded(xbar, 0);
    if (!xok) {
        atomicExch(&g_gemv_error, 1);
        s_abort = 1;
    }
    if constexpr (XF == X_BF16)
        permute_x_bf16<WF>(p, xs, M, warp, NW, lane);
    else
        expand_x<WF, XF>(p, smem + p.xraw_off + xoff, xs, M, tid, blockDim.x);
    __syncthreads();

    // the same tiles in every stage: tiles 0 .. nt-1 of the row, the last one
    // holding `tail` units
    const int nt = (p.nc + CPT - 1) / CPT;
    const int units = (WF == W_BF16) ? p.nc : p.nb;
    const int tail = units - 32 * (nt - 1);
    const int ds_off = ((p.nc + 31) / 32) * XPieces<WF, XF>::P * 512;
    const int x_row_bytes = p.x_row_bytes;
    const int64_t N = p.rows[0];
    float *const ycta = p.Y[0] + v0;

    int d = 0;
    uint32_t ph = 0;
    int waited = 0;
    bool ok = !*(volatile int *)&s_abort;
    for (int b = 0; b < my_blocks && ok; b++) {
        if (mbar_wait_bounded(wbar + 8 * d, ph)) {
            waited++;
        } else {
            atomicExch(&g_gemv_error, 1);
            s_abort = 1;
        }
        ok = !*(volatile int *)&s_abort;
        if (!ok) break;
        const int r0 = (warp + NW * b) * RL;           // first row of the block, from v0
        float acc[RL][M][2];
#pragma unroll
        for (int i = 0; i < RL; i++)
#pragma unroll
            for (int m = 0; m < M; m++) acc[i][m][0] = acc[i][m][1] = 0.f;
        const uint8_t *stage = smem + (warp * D + d) * stage_bytes;
        if constexpr (DOTS) {
            lpr_tiles<WF, XF, M, RL, true>(acc, stage, (int)row_bytes, xs, x_row_bytes, ds_off, 0, nt, tail, lane,
                                           p.dots + (v0 + r0) * p.nb, min(RL, nrows - r0), p.nb);
        } else {
            lpr_tiles<WF, XF, M, RL>(acc, stage, (int)row_bytes, xs, x_row_bytes, ds_off, 0, nt, tail, lane);
        }
        // the warp is done with this slot: refill it with its block b + D
        __syncwarp();
        if (lane == 0 && b + D < my_blocks) {
            fence_proxy_async_smem();
            issue(b + D, d);
            issued++;
        }
        if (++d == D) { d = 0; ph ^= 1; }
        if constexpr (!DOTS) {
            // value i * M + m is row r0 + i, activation row m
            float v[V];
#pragma unroll
            for (int i = 0; i < RL; i++)
#pragma unroll
                for (int m = 0; m < M; m++) v[i * M + m] = acc[i][m][0] + acc[i][m][1];
            const float tot = WR::run(v, lane);
            if (WR::is_holder(lane)) {
                const int idx = WR::index_of_lane(lane);
                const int i = idx / M, m = idx - (idx / M) * M;
                if (r0 + i < nrows) ycta[(int64_t)m * N + r0 + i] = tot;
            }
        }
    }
    // after a timeout: do not leave while this CTA's copies are in flight
    if (lane == 0) {
        for (int t = waited; t < issued; t++)
            mbar_wait_bounded(wbar + 8 * (t % D), (uint32_t)((t / D) & 1));
    }
    if (tid == 0 && !xok) mbar_wait_bounded(xbar, 0);
}

// Allow `kern` the largest dynamic shared memory (opt-in limit minus its
// static shared memory); error if `smem` does not fit.
template <typename Kern>
__host__ cudaError_t lpr_allow_smem(Kern kern, size_t smem)
{
    int dev = 0, optin = 0;
    cudaFuncAttributes fa;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
    if (e == cudaSuccess && smem + fa.sharedSizeBytes > (size_t)optin) return cudaErrorInvalidValue;
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
    return e;
}

// With `occupancy` set: prepare both lanes-per-row kernels of this
// instantiation (their shared-memory limit) and report the smaller of their
// occupancies; else launch the one p.rows_kernel selects.
template <int WF, int XF, int M, int RL, bool DOTS = false>
__host__ cudaError_t gemv_lpr_launch_one(const GemvParams &p, dim3 grid, int threads, size_t smem,
                                         cudaStream_t stream, bool pdl, int *occupancy)
{
    auto general = gemv_lpr_kernel<WF, XF, M, RL, DOTS>;
    auto rows = gemv_lpr_rows_kernel<WF, XF, M, RL, DOTS>;
    auto kern = p.rows_kernel ? rows : general;
    if (occupancy) {
        cudaError_t e = lpr_allow_smem(general, smem);
        if (e == cudaSuccess) e = lpr_allow_smem(rows, smem);
        int o1 = 0, o2 = 0;
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o1, general, threads, smem);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o2, rows, threads, smem);
        if (e != cudaSuccess) return e;
        *occupancy = min(o1, o2);
        return cudaSuccess;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int WF, int XF>
__host__ cudaError_t gemv_lpr_dispatch(const GemvParams &p, int M, dim3 grid, int threads, size_t smem,
                                       cudaStream_t stream, bool pdl, int *occupancy)
{
    // The staging the plan chose (bf16 pieces, fp32, or q8_1) selects the
    // instantiation; a combination without one is an error, never a kernel
    // that expects another staging.
    const int rl = p.rl;
#define BQG_LPR(XX, MM, RR) \
    if (M == MM && rl == RR) return gemv_lpr_launch_one<WF, XX, MM, RR>(p, grid, threads, smem, stream, pdl, occupancy);
    if constexpr (XF == X_BF16) {
        if (p.x_bf16s) {
            BQG_LPR(X_BF16, 1, 1) BQG_LPR(X_BF16, 1, 2) BQG_LPR(X_BF16, 2, 1) BQG_LPR(X_BF16, 2, 2)
            BQG_LPR(X_BF16, 4, 1) BQG_LPR(X_BF16, 4, 2) BQG_LPR(X_BF16, 8, 1) BQG_LPR(X_BF16, 8, 2)
            return cudaErrorInvalidValue;
        }
        BQG_LPR(X_F32, 1, 1) BQG_LPR(X_F32, 1, 2) BQG_LPR(X_F32, 1, 4) BQG_LPR(X_F32, 2, 1) BQG_LPR(X_F32, 2, 2)
    } else {
        BQG_LPR(XF, 1, 1) BQG_LPR(XF, 1, 2) BQG_LPR(XF, 1, 4) BQG_LPR(XF, 2, 1) BQG_LPR(XF, 2, 2)
        BQG_LPR(XF, 4, 1) BQG_LPR(XF, 4, 2) BQG_LPR(XF, 8, 1) BQG_LPR(XF, 8, 2)
    }
#undef BQG_LPR
    return cudaErrorInvalidValue;
}

// Split-K finish: Y = sum over splits (in split order) of the partials,
// then the same epilogue as the single-pass kernel.
static __global__ void __launch_bounds__(256) gemv_splitk_reduce(const GemvParams p, int M, int splits, int final_epi)
{
    pdl_wait();
    pdl_launch_dependents();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (final_epi == EPI_SWIGLU) {
        const int64_t np = p.Nv >> 1;
        if (i >= (int64_t)M * np) return;
        const int64_t m = i / np, pr = i - (i / np) * np;
        float gs = 0.f, us = 0.f;
        for (int s = 0; s < splits; s++) {
            gs += p.ws[((int64_t)s * M + m) * p.Nv + 2 * pr];
            us += p.ws[((int64_t)s * M + m) * p.Nv + 2 * pr + 1];
        }
        const float h = silu(gs) * us;
        if (p.hq) {
            // np % 32 == 0: the warp holds exactly block i / 32 of row m
            q8_1_encode_warp(h, threadIdx.x & 31, p.hq + (i / 32) * Q8_1_BYTES);
        } else {
            p.Y[0][m * p.rows[0] + pr] = h;
        }
    } else {
        if (i >= (int64_t)M * p.Nv) return;
        const int64_t m = i / p.Nv, v = i - (i / p.Nv) * p.Nv;
        float s = 0.f;
        for (int k = 0; k < splits; k++) s += p.ws[((int64_t)k * M + m) * p.Nv + v];
        int mat; int64_t rr;
        map_row(p, v, mat, rr);
        p.Y[mat][m * p.rows[mat] + rr] = s;
    }
}

// ---------------------------------------------------------------------------
// host-side launch helpers (one instantiation set per translation unit)
// ---------------------------------------------------------------------------
template <int WF, int XF, int M, int C>
__host__ cudaError_t gemv_launch_one(const GemvParams &p, dim3 grid, int threads, size_t smem,
                                     cudaStream_t stream, bool pdl, int *occupancy)
{
    auto kern = gemv_kernel<WF, XF, M, C>;
    if (occupancy) {
        // allow the largest dynamic shared memory (opt-in limit minus static), then ask for this size
        int dev = 0, optin = 0;
        cudaFuncAttributes fa;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
        if (e == cudaSuccess && smem + fa.sharedSizeBytes > (size_t)optin) return cudaErrorInvalidValue;
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occupancy, kern, threads, smem);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// Reads and clears this translation unit's error word.
__host__ inline cudaError_t gemv_take_error(int *out)
{
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(int));
    if (e != cudaSuccess) return e;
    *out = v;
    return v ? cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(int)) : cudaSuccess;
}

// bf16 activations are held as fp32 in registers where that costs few
// registers (it saves one conversion per element per output row).
template <int WF, int XF, int M> struct ActRep {
    static constexpr int value =
        (XF == X_BF16 && ((WF == W_BF16 && M <= 4) || (WF == W_Q8_0 && M <= 2))) ? X_F32 : XF;
};

template <int WF, int XF>
__host__ cudaError_t gemv_dispatch(const GemvParams &p, int M, int C, dim3 grid, int threads, size_t smem,
                                   cudaStream_t stream, bool pdl, int *occupancy)
{
#define BQG_CASE(MM, CC)                                                                 \
    if (M == MM && C == CC)                                                              \
        return gemv_launch_one<WF, ActRep<WF, XF, MM>::value, MM, CC>(p, grid, threads, smem, stream, pdl, occupancy);
    BQG_CASE(1, 1) BQG_CASE(1, 2) BQG_CASE(1, 4)
    BQG_CASE(2, 1) BQG_CASE(2, 2) BQG_CASE(2, 4)
    BQG_CASE(4, 1) BQG_CASE(4, 2) BQG_CASE(4, 4)
    BQG_CASE(8, 1) BQG_CASE(8, 2) BQG_CASE(8, 4)
#undef BQG_CASE
    return cudaErrorInvalidValue;
}

}  // namespace bqg
