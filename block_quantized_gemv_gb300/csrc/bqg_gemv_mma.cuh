// bqg_gemv_mma.cuh -- the skinny GEMV on the tensor cores, M = 4 and 8.
//
// Y[m, n] = sum_k W[n, k] X[m, k] for M activation rows.  The lanes-per-row
// kernels pay the activation's conversion and one FMA per weight and per
// activation row, so at M = 4 and 8 they are bound by that arithmetic ("The
// Shape That Actually Matters", Round 4: the kernel built for M = 8 and the
// one for M = 1 differ in what each weight costs).  Here the products go to
// the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate): per weight
// the cost is its conversion to bf16, whatever M is.
//
//  * The weights are the MMA's A operand: a unit is 16 weight rows.  The
//    activation rows are its B operand (8 columns, the first M real, the
//    rest zero).  Lane (g, t) of a warp holds weight rows g and g + 8 and
//    activation row g.  The K order inside one MMA is free as long as A and
//    B agree: of each 32 values (one q8_0 / q4_0 block) lane t takes values
//    4t .. 4t + 3 for the first MMA and 16 + 4t .. 16 + 4t + 3 for the
//    second -- one 32-bit word of q8_0 codes from each half of the block,
//    the low and high nibbles of one q4_0 word, 8 bytes of each bf16 half.
//    The activation rows are staged permuted to match (16 bytes per lane
//    and block: one shared-memory load feeds both MMAs).
//  * The conversion is exact: a q8_0 code (|q| <= 128) and a q4_0 value q - 8
//    are small integers, exact in bf16, and bf16 x bf16 products are exact in
//    fp32.  A q8_0 / q4_0 block's two MMAs (K = 32) accumulate into a fresh
//    fragment, which is then scaled by the block's fp16 scale d into the fp32
//    sum: y += d * sum_k q x, the order the lanes-per-row kernels use.  bf16
//    weights accumulate in the fragment.
//  * A stage is part of one tile of the repacked layout for the unit's 16
//    rows: a whole tile for bf16 (256 values, 512 B per row) and q4_0 (32
//    blocks, 576 B), half a tile for q8_0 (16 blocks: three copies, the low
//    codes, the high codes and the scales).  Each copy is a 2-D tensor copy
//    whose box is 16 (bf16: 32) bytes wider than the data, so that the 8
//    rows of a fragment load sit in distinct banks.
//  * A CTA takes a contiguous range of units; their stages (unit-major) are
//    split evenly over its warp groups, each streaming its own stages
//    through its own slots.  A warp's sums for one unit are a partial record
//    in shared memory; the records of a unit are added in warp order
//    (deterministic) and stored once.
#pragma once

#include <cuda.h>

#include "bqg_gemv.cuh"

namespace bqg {

struct MmaParams {
    const uint8_t *X;       // bf16 [M][K], or q8_1 blocks [M][K/32] (q4_0 weights)
    float *Y;               // [M][N]
    int64_t N;              // weight rows
    int K;
    int nb;                 // K / 32
    int T;                  // stages per row
    int64_t units;          // ceil(N / 16)
    int nw;                 // warps per CTA (at most 16)
    int gw;                 // warps per group (sharing each stage): 1 or 2
    int D;                  // slots per group
    int early;              // stages per group requested before the previous grid completes
    int rmax;               // partial records per warp
    int x_pitch;            // staged activation row pitch: round_up(2K, 128) + 64
    int x_off, rec_off, bar_off;  // shared-memory offsets
    int xd_off;             // q8_1 activations: their block scales d, [K/32][8] floats
};

// Stage geometry per weight format: row pitch in the slot, blocks of 32
// values per stage, slot bytes, and the tensor copies' boxes (8-byte units).
template <int WF> struct MmaGeom;
template <> struct MmaGeom<W_BF16> {
    static constexpr int PITCH = 544, SB = 8, SLOT = 16 * PITCH, BOX = PITCH / 8, STAGE_X = 512 / 8;
};
template <> struct MmaGeom<W_Q4_0> {
    static constexpr int PITCH = 592, SB = 32, SLOT = 16 * PITCH, BOX = PITCH / 8, STAGE_X = Q4_0_TILE / 8;
    static constexpr int SC = 512, SC_PITCH = PITCH;           // scales: row r at r * PITCH + 512
};
template <> struct MmaGeom<W_Q8_0> {
    // half a tile: low codes (16 x 272 B), high codes (16 x 272 B), scales (16 x 32 B)
    static constexpr int PITCH = 272, SB = 16, HI = 16 * PITCH, SC = 32 * PITCH, SC_PITCH = 32;
    static constexpr int SLOT = SC + 16 * SC_PITCH, BOX = PITCH / 8, SC_BOX = SC_PITCH / 8;
};

// d (fp32 accumulator fragment) += A (16 x 16 bf16) * B (16 x 8 bf16)
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void tma_load_2d_mma(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// The four q8_0 codes of w as two exact bf16 pairs: lo = (q0, q1), hi = (q2, q3).
__device__ __forceinline__ void q8_word_bf16(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    constexpr float OFF = 8388608.0f + 128.0f;
    const uint32_t u = w ^ 0x80808080u;                           // q + 128 as unsigned bytes
    float f0 = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7440));   // 2^23 + q + 128
    float f1 = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7441));
    float f2 = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7442));
    float f3 = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7443));
    fadd2(f0, f1, -OFF);                                          // q, exact
    fadd2(f2, f3, -OFF);
    lo = pack_bf16x2_rn(f0, f1);                                  // |q| <= 128: exact in bf16
    hi = pack_bf16x2_rn(f2, f3);
}

// The eight q4_0 values q - 8 of w (byte j: element j in the low nibble,
// element j + 16 in the high one) as exact bf16 pairs: l01 = (e0, e1),
// l23 = (e2, e3), h01 = (e16, e17), h23 = (e18, e19).  The bf16 pattern
// 0x43 n is 128 + n.
__device__ __forceinline__ void q4_word_bf16(uint32_t w, uint32_t &l01, uint32_t &l23, uint32_t &h01, uint32_t &h23)
{
    const uint32_t lo = w & 0x0f0f0f0fu, hi = (w >> 4) & 0x0f0f0f0fu;
    l01 = __byte_perm(lo, 0x43434343u, 0x4140);
    l23 = __byte_perm(lo, 0x43434343u, 0x4342);
    h01 = __byte_perm(hi, 0x43434343u, 0x4140);
    h23 = __byte_perm(hi, 0x43434343u, 0x4342);
    asm("sub.rn.bf16x2 %0, %0, %1;" : "+r"(l01) : "r"(0x43084308u));     // - 136: q - 8, exact
    asm("sub.rn.bf16x2 %0, %0, %1;" : "+r"(l23) : "r"(0x43084308u));
    asm("sub.rn.bf16x2 %0, %0, %1;" : "+r"(h01) : "r"(0x43084308u));
    asm("sub.rn.bf16x2 %0, %0, %1;" : "+r"(h23) : "r"(0x43084308u));
}

// (a0, a1) *= (b0, b1), one packed multiply
__device__ __forceinline__ void fmul2x(float &a0, float &a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 ra, rb;\n\t"
        "mov.b64 ra, {%0, %1};\n\t"
        "mov.b64 rb, {%2, %3};\n\t"
        "mul.rn.f32x2 ra, ra, rb;\n\t"
        "mov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(b0), "f"(b1));
}

// fp16 scale i (0..7) of eight packed in s
__device__ __forceinline__ float scale_of(const uint4 &s, int i)
{
    const uint32_t w = (i < 2) ? s.x : (i < 4) ? s.y : (i < 6) ? s.z : s.w;
    return half_bits_to_float((i & 1) ? (w >> 16) : (w & 0xffffu));
}

// One block of 32 values (bf16: two 16-value chunks) of the lane's weight
// rows g and g + 8 against its 16 activation bytes xq, added into cb (for
// q8_0 / q4_0 a fresh fragment, scaled afterwards).  st: the slot; s: the
// block's index in the stage.
template <int WF>
__device__ __forceinline__ void mma_block(const uint8_t *st, int g, int t, int s, const uint4 &xq, float (&cb)[4])
{
    using G = MmaGeom<WF>;
    if constexpr (WF == W_BF16) {
        const uint8_t *r0 = st + g * G::PITCH + 64 * s + 8 * t;
        const uint8_t *r8 = r0 + 8 * G::PITCH;
        const uint2 wa = *reinterpret_cast<const uint2 *>(r0);       // values 4t .. 4t + 3
        const uint2 wb = *reinterpret_cast<const uint2 *>(r8);
        const uint2 wc = *reinterpret_cast<const uint2 *>(r0 + 32);  // values 16 + 4t ..
        const uint2 wd = *reinterpret_cast<const uint2 *>(r8 + 32);
        mma_bf16_16816(cb, wa.x, wb.x, wa.y, wb.y, xq.x, xq.y);
        mma_bf16_16816(cb, wc.x, wd.x, wc.y, wd.y, xq.z, xq.w);
    } else if constexpr (WF == W_Q8_0) {
        const uint8_t *r0 = st + g * G::PITCH + 16 * s + 4 * t;
        const uint8_t *r8 = r0 + 8 * G::PITCH;
        uint32_t a0, a1, a2, a3;
        q8_word_bf16(*reinterpret_cast<const uint32_t *>(r0), a0, a2);
        q8_word_bf16(*reinterpret_cast<const uint32_t *>(r8), a1, a3);
        mma_bf16_16816(cb, a0, a1, a2, a3, xq.x, xq.y);
        q8_word_bf16(*reinterpret_cast<const uint32_t *>(r0 + G::HI), a0, a2);
        q8_word_bf16(*reinterpret_cast<const uint32_t *>(r8 + G::HI), a1, a3);
        mma_bf16_16816(cb, a0, a1, a2, a3, xq.z, xq.w);
    } else {
        const uint8_t *r0 = st + g * G::PITCH + 16 * s + 4 * t;
        uint32_t l0, l2, h0, h2, l1, l3, h1, h3;
        q4_word_bf16(*reinterpret_cast<const uint32_t *>(r0), l0, l2, h0, h2);
        q4_word_bf16(*reinterpret_cast<const uint32_t *>(r0 + 8 * G::PITCH), l1, l3, h1, h3);
        mma_bf16_16816(cb, l0, l1, l2, l3, xq.x, xq.y);
        mma_bf16_16816(cb, h0, h1, h2, h3, xq.z, xq.w);
    }
}

// One CTA: units [u0, u1) (an even split of ceil(N / 16) units over the
// grid); their S = (u1 - u0) T stages, unit-major, split into contiguous
// ranges over p.nw / p.gw groups of p.gw warps.  The warps of a group share
// each stage's slot, warp `sub` taking its sub-th share of the stage's
// blocks.  wmap: the repacked rows (8-byte units); smap: the same rows with
// the q8_0 scales' box.
//
// q8_1 activations (q4_0 weights): the codes are staged as exact bf16 values
// and each block's scale d_x in a table; a block's MMA sum is then the exact
// integer sum_i (q_w - 8) q_x of the integer-dot kernels (|sum| < 2^15, so
// exact in fp32 whatever the order of the tensor core's additions), and
// y += (d_w d_x) sum, in their order of rounding.
template <int WF, int XF, int M>
__global__ void __launch_bounds__(512, 1)
    gemv_mma_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap smap, const MmaParams p)
{
    static_assert(M == 2 || M == 4 || M == 8, "tensor-core GEMV: M = 2, 4 or 8");
    static_assert(XF == X_BF16 || (XF == X_Q8_1 && WF == W_Q4_0), "tensor-core GEMV: bf16 activations, or q8_1 with q4_0");
    using G = MmaGeom<WF>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_abort;
    __shared__ int s_first[16], s_last[16];        // per warp: first and last unit of its records
    // tensor copies land on 128-byte boundaries (the launch adds 128 bytes of
    // slack); an offset from the shared array keeps the accesses shared-space
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int g = lane >> 2;                       // fragment group: weight rows g, g + 8; activation row g
    const int t = lane & 3;                        // fragment column pair
    const int NW = p.nw, GW = p.gw, D = p.D, T = p.T;
    const int NG = NW / GW;
    const int grp = warp / GW, sub = warp - grp * GW;
    const bool leader = sub == 0 && lane == 0;     // issues the group's copies
    const int64_t u0 = (int64_t)blockIdx.x * p.units / gridDim.x;
    const int64_t u1 = (int64_t)(blockIdx.x + 1) * p.units / gridDim.x;
    const int S = (int)(u1 - u0) * T;
    const int a = grp * S / NG;                    // S * NG < 2^30 (host check)
    const int nst = (grp + 1) * S / NG - a;        // the group's stages a .. a + nst - 1
    const int ul_first = a / T;                    // its first unit (CTA-local)
    const int nbx = p.K / 32;                      // blocks of 32 values per row
    const uint32_t bar0 = smem_u32(smem + p.bar_off);
    const uint32_t wbar = bar0 + 8 * grp * D;
    const uint32_t slot0 = smem_u32(smem) + (uint32_t)(grp * D * G::SLOT);
    uint8_t *xs = smem + p.x_off;
    float *rec = reinterpret_cast<float *>(smem + p.rec_off);

    auto issue = [&](int q, int slot) {            // leader: the group's stage q into `slot`
        const int j = a + q;
        const int ul = j / T;
        const int ts = j - ul * T;
        const int y = (int)((u0 + ul) * 16);
        const uint32_t dst = slot0 + slot * G::SLOT, bar = wbar + 8 * slot;
        mbar_arrive_expect_tx(bar, (uint32_t)G::SLOT);
        if constexpr (WF == W_Q8_0) {
            const int x0 = (ts >> 1) * (Q8_0_TILE / 8) + (ts & 1) * 32;    // half ts & 1 of tile ts >> 1
            tma_load_2d_mma(dst, &wmap, x0, y, bar);                        // low codes
            tma_load_2d_mma(dst + G::HI, &wmap, x0 + 64, y, bar);           // high codes
            tma_load_2d_mma(dst + G::SC, &smap, (ts >> 1) * (Q8_0_TILE / 8) + 128 + (ts & 1) * 4, y, bar);
        } else {
            tma_load_2d_mma(dst, &wmap, ts * G::STAGE_X, y, bar);
        }
    };
    // the group's warps are done reading a slot
    auto group_sync = [&]() {
        if (GW == 1)
            __syncwarp();
        else
            asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(32 * GW) : "memory");
    };
    // v of any thread of the group, the same answer in all of them
    auto group_any = [&](bool v) -> bool {
        if (GW == 1) return __any_sync(0xffffffffu, v);
        uint32_t r;
        asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                     "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                     : "=r"(r)
                     : "r"((uint32_t)v), "r"(1 + grp), "r"(32 * GW)
                     : "memory");
        return r != 0;
    };

    // the activation rows: into L2 first (ahead of the weight copies in the
    // SM's copy queue; each CTA its 1/grid share), into shared memory once
    // the previous grid has completed (it may be their producer)
    if (tid == 32) {
        // the 16-byte-aligned span around X (q8_1 rows are only 4-byte aligned)
        const uintptr_t xa = reinterpret_cast<uintptr_t>(p.X);
        const uint32_t xoff = (uint32_t)(xa & 15);
        const uint32_t xb = (xoff + (uint32_t)((XF == X_BF16) ? M * p.K * 2 : M * nbx * Q8_1_BYTES) + 15) & ~15u;
        const uint32_t ch = ((xb + gridDim.x - 1) / gridDim.x + 15) & ~15u;
        const uint32_t at = blockIdx.x * ch;
        if (at < xb) prefetch_l2_bulk(reinterpret_cast<const uint8_t *>(xa - xoff) + at, min(ch, xb - at));
    }
    if (tid == 0) {
        for (int i = 0; i < NG * D; i++) mbar_init(bar0 + 8 * i, 1);
        s_abort = 0;
        mbar_fence_init();
    }
    if (lane == 0) {
        s_first[warp] = nst > 0 ? ul_first : 1;
        s_last[warp] = nst > 0 ? (a + nst - 1) / T : 0;
    }
    __syncthreads();
    int issued = 0;                                // the leader's count
    const int first = min(D, nst);
    if (leader)
        for (; issued < min(first, p.early); issued++) issue(issued, issued);
    pdl_wait();
    pdl_launch_dependents();
    if (leader)
        for (; issued < first; issued++) issue(issued, issued);
    // The activation rows by plain loads (they would queue behind the weight
    // copies in the tensor-copy unit), all of a thread's loads in flight at
    // once, permuted on the way in: of each 32 values, lane t's 16 bytes
    // (values 4t .. 4t + 3 and 16 + 4t .. 16 + 4t + 3) at 16 t.  Thread i
    // writes staged chunk i (consecutive threads, consecutive chunks: no
    // bank conflicts) from its two 8-byte source pieces.  Every CTA reads all
    // of X: each starts at its own offset, so that at any moment the CTAs
    // ask different L2 lines for it.
    if constexpr (XF == X_BF16) {
        constexpr int XU = 8;                      // chunks per thread and round
        const int n16 = M * nbx * 4;
        const int rot = (int)(((int64_t)blockIdx.x * 389) % n16);
        const uint2 *src = reinterpret_cast<const uint2 *>(p.X);
        for (int i0 = tid; i0 < n16; i0 += XU * (int)blockDim.x) {
            uint2 lo[XU], hi[XU];
#pragma unroll
            for (int k = 0; k < XU; k++) {
                int i = i0 + k * (int)blockDim.x + rot;
                i -= (i >= n16) ? n16 : 0;
                if (i0 + k * (int)blockDim.x < n16) {
                    const int blk = i >> 2, c = i & 3;          // rows are contiguous: block blk of X
                    lo[k] = src[(size_t)blk * 8 + c];
                    hi[k] = src[(size_t)blk * 8 + 4 + c];
                }
            }
#pragma unroll
            for (int k = 0; k < XU; k++) {
                int i = i0 + k * (int)blockDim.x + rot;
                i -= (i >= n16) ? n16 : 0;
                if (i0 + k * (int)blockDim.x < n16) {
                    const int blk = i >> 2, c = i & 3;
                    const int m = blk / nbx, b = blk - m * nbx;
                    *reinterpret_cast<uint4 *>(xs + m * p.x_pitch + b * 64 + 16 * c) =
                        make_uint4(lo[k].x, lo[k].y, hi[k].x, hi[k].y);
                }
            }
        }
    } else {
        // q8_1 blocks (36 B: d, s, 32 codes; 4-byte aligned): thread i stages
        // chunk i, lane c's codes 4c .. 4c + 3 and 16 + 4c .. 16 + 4c + 3 as
        // exact bf16 values, and the block's d into the scale table
        constexpr int XU = 8;
        const int n16 = M * nbx * 4;
        const int rot = (int)(((int64_t)blockIdx.x * 389) % n16);
        const uint32_t *src = reinterpret_cast<const uint32_t *>(p.X);     // 9 words per block
        float *xd = reinterpret_cast<float *>(smem + p.xd_off);
        for (int i0 = tid; i0 < n16; i0 += XU * (int)blockDim.x) {
            uint32_t lo[XU], hi[XU], dw[XU];
#pragma unroll
            for (int k = 0; k < XU; k++) {
                int i = i0 + k * (int)blockDim.x + rot;
                i -= (i >= n16) ? n16 : 0;
                if (i0 + k * (int)blockDim.x < n16) {
                    const int blk = i >> 2, c = i & 3;          // rows are contiguous: block blk of X
                    lo[k] = src[(size_t)blk * 9 + 1 + c];
                    hi[k] = src[(size_t)blk * 9 + 5 + c];
                    dw[k] = (c == 0) ? src[(size_t)blk * 9] : 0u;
                }
            }
#pragma unroll
            for (int k = 0; k < XU; k++) {
                int i = i0 + k * (int)blockDim.x + rot;
                i -= (i >= n16) ? n16 : 0;
                if (i0 + k * (int)blockDim.x < n16) {
                    const int blk = i >> 2, c = i & 3;
                    const int m = blk / nbx, b = blk - m * nbx;
                    uint32_t l0, l1, h0, h1;
                    q8_word_bf16(lo[k], l0, l1);
                    q8_word_bf16(hi[k], h0, h1);
                    *reinterpret_cast<uint4 *>(xs + m * p.x_pitch + b * 64 + 16 * c) = make_uint4(l0, l1, h0, h1);
                    if (c == 0) xd[b * 8 + m] = half_bits_to_float(dw[k] & 0xffffu);
                }
            }
        }
        for (int i = tid; i < nbx * (8 - M); i += blockDim.x)   // the zero columns' scales
            xd[(i / (8 - M)) * 8 + M + i % (8 - M)] = 0.f;
    }
    __syncthreads();

    const bool xreal = g < M;                      // B columns g >= M are zero
    const uint8_t *xrow = xs + (xreal ? g : 0) * p.x_pitch + 16 * t;
    float c[4] = {0.f, 0.f, 0.f, 0.f};            // (row g, act 2t), (g, 2t + 1), (g + 8, 2t), (g + 8, 2t + 1)
    int d = 0;
    uint32_t ph = 0;
    int waited = 0;
    for (int q = 0; q < nst; q++) {
        const bool bad = !mbar_wait_bounded(wbar + 8 * d, ph);
        if (group_any(bad)) {                      // the whole group leaves
            if (bad) {
                atomicExch(&g_gemv_error, 1);
                s_abort = 1;
            }
            break;
        }
        waited++;
        const int j = a + q;
        const int ul = j / T;
        const int ts = j - ul * T;
        const uint8_t *st = smem + (grp * D + d) * G::SLOT;
        const int nbs = min(G::SB, nbx - ts * G::SB);              // blocks in this stage
        const int s0 = sub * G::SB / GW, s1 = min(nbs, (sub + 1) * G::SB / GW);
        const uint8_t *xk = xrow + ts * G::SB * 64;
        auto xload = [&](int s) {
            return xreal ? *reinterpret_cast<const uint4 *>(xk + 64 * s) : make_uint4(0u, 0u, 0u, 0u);
        };
        if constexpr (WF == W_BF16) {
#pragma unroll 4
            for (int s = s0; s < s1; s++) mma_block<WF>(st, g, t, s, xload(s), c);
        } else {
            // scales of rows g and g + 8, eight blocks at a time
            const uint8_t *sg = st + G::SC + g * G::SC_PITCH;
            auto qblock = [&](int s, float d0, float d8) {
                float cb[4] = {0.f, 0.f, 0.f, 0.f};
                mma_block<WF>(st, g, t, s, xload(s), cb);
                if constexpr (XF == X_Q8_1) {
                    // columns 2t, 2t + 1 have their own d_x: (d_w d_x) sum
                    const float2 dx = *reinterpret_cast<const float2 *>(
                        reinterpret_cast<const float *>(smem + p.xd_off) + (ts * G::SB + s) * 8 + 2 * t);
                    float e0 = d0, e1 = d0, e2 = d8, e3 = d8;
                    fmul2x(e0, e1, dx.x, dx.y);
                    fmul2x(e2, e3, dx.x, dx.y);
                    ffma2(c[0], c[1], e0, e1, cb[0], cb[1]);
                    ffma2(c[2], c[3], e2, e3, cb[2], cb[3]);
                } else {
                    ffma2(c[0], c[1], cb[0], cb[1], d0, d0);
                    ffma2(c[2], c[3], cb[2], cb[3], d8, d8);
                }
            };
            for (int s8 = s0; s8 < s1; s8 += 8) {
                const uint4 sc0 = *reinterpret_cast<const uint4 *>(sg + 2 * s8);
                const uint4 sc8 = *reinterpret_cast<const uint4 *>(sg + 8 * G::SC_PITCH + 2 * s8);
                if (s1 - s8 >= 8) {
#pragma unroll
                    for (int i = 0; i < 8; i++) qblock(s8 + i, scale_of(sc0, i), scale_of(sc8, i));
                } else {
                    for (int i = 0; i < s1 - s8; i++) qblock(s8 + i, scale_of(sc0, i), scale_of(sc8, i));
                }
            }
        }
        // the group is done with this slot: refill it with its stage q + D
        group_sync();
        if (leader && q + D < nst) {
            fence_proxy_async_smem();
            issue(q + D, d);
            issued++;
        }
        if (++d == D) { d = 0; ph ^= 1; }
        if (ts == T - 1 || q == nst - 1) {
            // this warp's part of unit ul: a record of 128 floats, lane l's
            // four sums (rows g, g + 8 x activation columns 2t, 2t + 1) at
            // floats 4l .. 4l + 3
            reinterpret_cast<float4 *>(rec + (warp * p.rmax + ul - ul_first) * 128)[lane] =
                make_float4(c[0], c[1], c[2], c[3]);
            c[0] = c[1] = c[2] = c[3] = 0.f;
        }
    }
    // after a timeout: do not leave while the group's copies are in flight
    if (leader) {
        for (int q = waited; q < issued; q++)
            mbar_wait_bounded(wbar + 8 * (q % D), (uint32_t)((q / D) & 1));
    }
    __syncthreads();
    if (*(volatile int *)&s_abort) return;

    // Y[m, 16 (u0 + ul) + r]: the unit's records added in warp order.  Thread
    // o takes float o & 127 of unit o >> 7's records (consecutive words: no
    // bank conflicts) and parks the sum in the staged-activation area, from
    // where the rows of Y go out contiguous.
    const int U = (int)(u1 - u0);
    const int ypitch = U * 16 + 1;
    float *ys = reinterpret_cast<float *>(xs);     // M x ypitch floats (the activations are done)
    int wf[16], wl[16];                            // the warps' unit ranges, in registers
#pragma unroll
    for (int w = 0; w < 16; w++) {
        wf[w] = (w < NW) ? s_first[w] : 1;
        wl[w] = (w < NW) ? s_last[w] : 0;
    }
    for (int o = tid; o < U * 128; o += blockDim.x) {
        const int ul = o >> 7, idx = o & 127;
        const int l = idx >> 2, reg = idx & 3;     // the record's lane and register
        const int m = ((l & 3) << 1) | (reg & 1);
        const int r = (l >> 2) | ((reg >> 1) << 3);
        if (m >= M) continue;
        float part[16];
#pragma unroll
        for (int w = 0; w < 16; w++)               // independent loads, then the sum in warp order
            part[w] = (ul >= wf[w] && ul <= wl[w]) ? rec[(w * p.rmax + ul - wf[w]) * 128 + idx] : 0.f;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < 16; w++)
            if (ul >= wf[w] && ul <= wl[w]) sum += part[w];
        ys[m * ypitch + ul * 16 + r] = sum;
    }
    __syncthreads();
    const int64_t row0 = u0 * 16;
    const int nr = (int)(min(u1 * 16, p.N) - row0);
    for (int o = tid; o < M * nr; o += blockDim.x) {
        const int m = o / nr, r = o - m * nr;
        p.Y[(int64_t)m * p.N + row0 + r] = ys[m * ypitch + r];
    }
}

template <int WF, int XF>
__host__ cudaError_t gemv_mma_launch(const CUtensorMap &wmap, const CUtensorMap &smap, const MmaParams &p, int M,
                                     dim3 grid, int threads, size_t smem, cudaStream_t stream, bool pdl,
                                     int *occupancy)
{
    if (M != 2 && M != 4 && M != 8) return cudaErrorInvalidValue;
    auto kern = (M == 8) ? gemv_mma_kernel<WF, XF, 8> : gemv_mma_kernel<WF, XF, 4>;
    if constexpr (WF == W_Q4_0 && XF == X_BF16) {        // M = 2: q4_0 x bf16 only
        if (M == 2) kern = gemv_mma_kernel<WF, XF, 2>;
    } else {
        if (M == 2) return cudaErrorInvalidValue;
    }
    if (occupancy) {
        cudaError_t e = lpr_allow_smem(kern, smem);
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
    return cudaLaunchKernelEx(&cfg, kern, wmap, smap, p);
}

}  // namespace bqg
