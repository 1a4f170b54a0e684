// bqg_gemm.cu -- prefill GEMM Y[M x N] = X[M x K] W^T on the sm_103a tensor cores.
//
// The tiled prefill GEMM of "llama-3x-prompt-speed" ("the tile"): a weight
// tile is unpacked once and serves every activation row of the tile,
// instead of being unpacked once per row.  Here the unit of work is 128
// weight rows x 256 activation rows (a "big" unit, one MMA of N = 256 per
// K-step of 16) or 128 x 128 (a "small" unit).  On this part an MMA costs
// about 90 cycles beyond its N / 2 cycles of tensor work, so N = 256 runs
// 1.4x faster per flop than N = 128, and each dequantized weight tile then
// serves twice the activation rows.  Big units come first in the order;
// the big units of an incomplete last wave are split into two small units
// each when that keeps every SM busy (M = 512, N = 14336: 152 big units,
// then 144 small ones, on 152 SMs).  Per stage of 64 along K:
//   * warp 14, lane 0 stages the raw weight codes and scales of four stages
//     at a time (eight q4_0 blocks per row) into shared memory with two-dimensional TMA copies (128 rows
//     x 128 bytes of codes in the 128-byte swizzle, 128 rows x 16 bytes of
//     scales), so the weight stream is coalesced;
//   * warps 1-8 (one weight block of one weight row per thread) read their
//     block's codes and scale from there (conflict-free thanks to the
//     swizzle), dequantize it to (q - 8) d or q d rounded once to bf16
//     (q4_0: in packed bf16 arithmetic, the fp16 scale split exactly into two
//     bf16 parts so that one fused multiply-add rounds the exact product;
//     q8_0: in fp32) and store the 128 x 64 bf16 tile straight into tensor
//     memory (tcgen05.st: lane = weight row, two k per column), where the
//     MMA reads its A operand.  Shared memory then carries only the
//     activation tiles: with A staged there too, its bandwidth (dequant
//     writes, TMA writes and both MMA operands) bounded the loop at twice the
//     MMA time;
//   * warp 13, lane 0 loads the matching 128- or 256-row x 64 bf16
//     activation tile (one or two TMA copies of one 64-wide swizzle atom) as
//     soon as the stage is free;
//   * warp 0, lane 0 issues four tcgen05.mma.kind::f16 (A from tensor
//     memory, B from shared memory; M = 128 weight rows, N = 128 or 256
//     activations, K = 16) accumulating fp32 in tensor memory as soon as both
//     halves of the stage are in place; tcgen05.commit frees the stage.  It
//     never waits for its own MMAs, so the tensor core always has the next
//     K-step queued;
//   * warps 9-12 read the finished accumulator with tcgen05.ld (each warp
//     its 32 lanes = 32 weight rows) and store Y[m][n] coalesced along n.
// Tensor memory (512 columns): accumulator slot 0 (256 columns: a big unit,
// or a small one), the NSTAGE A slots, accumulator slot 1 (128 columns,
// small units), so the epilogue of one unit overlaps the MMAs of the next
// whenever the next one is small.  The kernel is persistent (one CTA per
// SM).  Every mbarrier wait is bounded: on a timeout the kernel sets
// g_gemm_error, stops issuing work, drains what it started and frees TMEM.
#include <algorithm>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "bqg_common.cuh"

namespace bqg {

// Error word set by bounded device-side waits (0 = none).
__device__ int g_gemm_error;

namespace {

constexpr int TM = 128;         // weight rows per unit (MMA M)
constexpr int TNS = 128;        // activation rows of a small unit, and of one TMA box
constexpr int TNB = 256;        // activation rows of a big unit
constexpr int TK = 64;          // K per stage: one 128-byte swizzle atom of bf16
constexpr int BOX_BYTES = TNS * TK * 2;       // 16 KiB: one 128-row activation box
constexpr int A_COLS = TK / 2;                // 32-bit columns of one bf16 A tile of a stage (two bf16 each)
constexpr int TMEM_COLS = 512;
constexpr int kGemmExactBelowK = 1024;        // K below which the weights are split into exact bf16 terms

// Pipeline shape per number of bf16 terms a dequantized weight is split
// into.  TERMS = 1: (q - 8) d or q d rounded once to bf16 (the prefill
// config's dequantization); big units allowed.  TERMS = 2 (q4_0) / 3 (q8_0):
// the weight written exactly as a sum of bf16 values (a 4-bit code times an
// fp16 scale has at most 14 significant bits, an 8-bit code times one at
// most 19, and bf16 holds 8), one MMA per term into the same fp32
// accumulator, so the GEMM is exact up to fp32 accumulation; small units
// only (two 128-column accumulators), fewer stages at three terms.
template <int TERMS> struct Pipe {
    static constexpr bool BIG = (TERMS == 1);
    static constexpr int NSTAGE = (TERMS == 3) ? 2 : 4;
    static constexpr int STAGE_BYTES = (BIG ? 2 : 1) * BOX_BYTES;
    static constexpr int SLOT_COLS = TERMS * A_COLS;      // one stage's A terms
    static constexpr int ACC0 = 0;                        // accumulator slot 0
    static constexpr int A_COL0 = 256;                    // first column of the A slots
    static constexpr int ACC1 = BIG ? A_COL0 + NSTAGE * SLOT_COLS : 128;   // accumulator slot 1
    static_assert(A_COL0 + NSTAGE * SLOT_COLS <= TMEM_COLS, "tensor memory budget");
    static_assert(!BIG || ACC1 + TNS <= TMEM_COLS, "tensor memory budget");
};
constexpr int DQ_WARPS = 8;                   // dequantizing warps (1..8)
constexpr int EPI_WARP0 = 1 + DQ_WARPS;       // epilogue warps 9..12
constexpr int TMA_WARP = EPI_WARP0 + 4;       // activation loads: warp 13
constexpr int RAW_WARP = TMA_WARP + 1;        // raw weight codes: warp 14
constexpr int NUM_THREADS = (RAW_WARP + 1) * 32;
constexpr int RAW_STEPS = 4;                  // stages per raw group: 8 blocks = 128 code bytes (q4_0)
constexpr int RAW_CODES = TM * 128;           // bytes of one 128-row x 128-byte code box
constexpr int RAW_SCALES = TM * 16;           // bytes of one 128-row x 16-byte scale box

// shared memory map (dynamic, 1024-byte aligned), per weight format and
// activation ring
template <int WF, int NSTAGE, int STAGE_BYTES> struct GemmSmem {
    static constexpr int CODE_BOXES = (WF == BQG_Q8_0) ? 2 : 1;   // q8_0: codes 0..15 and 16..31
    static constexpr int NRAW = (WF == BQG_Q8_0) ? 2 : 3;         // raw groups in flight
    static constexpr int RAW_GROUP = CODE_BOXES * RAW_CODES;
    static constexpr int OFF_STAGES = 0;
    static constexpr int OFF_RAW = NSTAGE * STAGE_BYTES;
    static constexpr int OFF_SCALES = OFF_RAW + NRAW * RAW_GROUP;
    static constexpr int OFF_BARS = OFF_SCALES + NRAW * RAW_SCALES;
    // fullW, fullX, empty per stage; acc full/empty x2; raw full/empty per group
    static constexpr int NBARS = 3 * NSTAGE + 4 + 2 * NRAW;
    static constexpr int OFF_TMEM_SLOT = OFF_BARS + NBARS * 8;
    static constexpr int OFF_FLAG = OFF_TMEM_SLOT + 8;
    static constexpr int SMEM_BYTES = OFF_FLAG + 8 + 1024;       // + slack for 1024-byte alignment
};
template <int WF, int TERMS> using SmemOf = GemmSmem<WF, Pipe<TERMS>::NSTAGE, Pipe<TERMS>::STAGE_BYTES>;

// instruction descriptor, kind::f16: D fp32, A bf16, B bf16, both K-major, M = 128; N per unit
constexpr uint32_t IDESC_BASE = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(TM >> 4) << 24);
__device__ __forceinline__ uint32_t idesc_n(int n) { return IDESC_BASE | ((uint32_t)(n >> 3) << 17); }

// K-major, 128-byte swizzle smem descriptor: rows of 128 bytes in atoms of
// 8 rows (1024 bytes); consecutive atoms along M/N are 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3fff);            // start address
    d |= (uint64_t)1 << 16;                            // leading byte offset (unused with swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;                  // stride byte offset: next 8-row atom
    d |= (uint64_t)1 << 46;                            // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                            // 128-byte swizzle
    return d;
}


__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(bar)
                 : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem descriptor]
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                             uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// 32 lanes x 16 columns of 32-bit words into tensor memory (this warp's lane
// quarter); tcgen05.wait::st makes them complete
__device__ __forceinline__ void tmem_st16_nowait(uint32_t taddr, const uint4 (&v)[4])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
                 ::"r"(taddr), "r"(v[0].x), "r"(v[0].y), "r"(v[0].z), "r"(v[0].w), "r"(v[1].x), "r"(v[1].y),
                   "r"(v[1].z), "r"(v[1].w), "r"(v[2].x), "r"(v[2].y), "r"(v[2].z), "r"(v[2].w), "r"(v[3].x),
                   "r"(v[3].y), "r"(v[3].z), "r"(v[3].w)
                 : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 32 lanes x 32 columns of fp32 from tensor memory (this warp's lane quarter)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

// two fp32 -> bf16x2, round to nearest even (lo in the low half)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Eight exact fp32 weights as TERMS bf16x2 quadruples: term 0 is each weight
// rounded to nearest-even bf16, every further term the same rounding of what
// is left (the subtraction is exact); with enough terms the sum of the terms
// is the weight exactly.
template <int TERMS>
__device__ __forceinline__ void bf16_terms(float (&f)[8], uint4 (&t)[TERMS])
{
#pragma unroll
    for (int j = 0; j < TERMS; j++) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            w[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
            if (j + 1 < TERMS) {
                f[2 * i] = __fsub_rn(f[2 * i], __uint_as_float(w[i] << 16));
                f[2 * i + 1] = __fsub_rn(f[2 * i + 1], __uint_as_float(w[i] & 0xffff0000u));
            }
        }
        t[j] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// 8 dequantized weights (q - 8) * d of one q4_0 word pair, as TERMS bf16x2
// quadruples.  w0, w1 hold code bytes 4i..4i+7; `shift` 0 takes the low
// nibbles (elements j), 4 the high nibbles (elements j + 16).
template <int TERMS>
__device__ __forceinline__ void dequant8(uint32_t w0, uint32_t w1, int shift, float d, uint4 (&t)[TERMS])
{
    constexpr float OFF = 8388608.0f + 8.0f;
    const uint32_t a = (w0 >> shift) & 0x0f0f0f0fu, b = (w1 >> shift) & 0x0f0f0f0fu;
    float f[8] = {byte_plus_2p23<0>(a), byte_plus_2p23<1>(a), byte_plus_2p23<2>(a), byte_plus_2p23<3>(a),
                  byte_plus_2p23<0>(b), byte_plus_2p23<1>(b), byte_plus_2p23<2>(b), byte_plus_2p23<3>(b)};
#pragma unroll
    for (int i = 0; i < 8; i += 2) {          // exact: 4-bit integer times an fp16 value
        fadd2(f[i], f[i + 1], -OFF);
        fmul2(f[i], f[i + 1], d);
    }
    bf16_terms<TERMS>(f, t);
}

// 8 dequantized q8_0 weights q * d of one word pair (bytes = codes 4i..4i+7),
// as TERMS bf16x2 quadruples
template <int TERMS>
__device__ __forceinline__ void dequant8_q8(uint32_t w0, uint32_t w1, float d, uint4 (&t)[TERMS])
{
    constexpr float OFF = 8388608.0f + 128.0f;
    const uint32_t a = w0 ^ 0x80808080u, b = w1 ^ 0x80808080u;   // q + 128 as unsigned bytes
    float f[8] = {byte_plus_2p23<0>(a), byte_plus_2p23<1>(a), byte_plus_2p23<2>(a), byte_plus_2p23<3>(a),
                  byte_plus_2p23<0>(b), byte_plus_2p23<1>(b), byte_plus_2p23<2>(b), byte_plus_2p23<3>(b)};
#pragma unroll
    for (int i = 0; i < 8; i += 2) {          // exact: 8-bit integer times an fp16 value
        fadd2(f[i], f[i + 1], -OFF);
        fmul2(f[i], f[i + 1], d);
    }
    bf16_terms<TERMS>(f, t);
}

// One q4_0 block (codes c: word i holds elements 4i..4i+3 in its low
// nibbles, 16+4i..16+4i+3 in its high ones) as 16 bf16x2 words, each weight
// (q - 8) d rounded once to bf16, in packed bf16 arithmetic.  The fp16 scale
// is split exactly as d = dh + dl with dh = bf16(d): the remainder has at
// most three significant bits (fp16 carries 11, bf16 8), so it is a bf16
// value too.  q - 8 is exact in bf16 (the pattern 0x43 n is 128 + n), the
// product (q - 8) dl has at most six significant bits and is exact, and one
// fused multiply-add (q - 8) dh + (q - 8) dl rounds the exact (q - 8) d once
// -- the same bf16 value as rounding the fp32 product (q - 8) d, which is
// exact.  fp16 scales stay far inside the bf16 range, so nothing overflows
// or goes subnormal.
__device__ __forceinline__ void dequant32_q4_bf16(const uint4 &c, float d, uint4 (&v)[4])
{
    uint32_t dh, dl;
    asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(dh) : "f"(d));
    const float rest = d - __uint_as_float(dh << 16);             // exact
    asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(dl) : "f"(rest));  // exact
    // four codes (one per byte, 0..15) -> two bf16x2 words of (q - 8) d
    auto four = [&](uint32_t nib, uint32_t &r0, uint32_t &r1) {
        uint32_t e0 = __byte_perm(nib, 0x43434343u, 0x4140), e1 = __byte_perm(nib, 0x43434343u, 0x4342);
        uint32_t p0, p1;
        asm("sub.rn.bf16x2 %0, %0, %1;" : "+r"(e0) : "r"(0x43084308u));   // - 136: q - 8
        asm("sub.rn.bf16x2 %0, %0, %1;" : "+r"(e1) : "r"(0x43084308u));
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(p0) : "r"(e0), "r"(dl));
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(p1) : "r"(e1), "r"(dl));
        asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r0) : "r"(e0), "r"(dh), "r"(p0));
        asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r1) : "r"(e1), "r"(dh), "r"(p1));
    };
    const uint32_t m = 0x0f0f0f0fu;
    four(c.x & m, v[0].x, v[0].y);
    four(c.y & m, v[0].z, v[0].w);
    four(c.z & m, v[1].x, v[1].y);
    four(c.w & m, v[1].z, v[1].w);
    four((c.x >> 4) & m, v[2].x, v[2].y);
    four((c.y >> 4) & m, v[2].z, v[2].w);
    four((c.z >> 4) & m, v[3].x, v[3].y);
    four((c.w >> 4) & m, v[3].z, v[3].w);
}

// A dequantizing thread's weight block, read from the raw group staged in
// shared memory: `codes` is the group's 128 x 128-byte box (128-byte swizzle:
// 16-byte chunk c of row r sits at chunk c ^ (r & 7)), b8 the block within
// the group (0..7), d its scale.  The scales come from the group's 128 x
// 16-byte scale box, each thread reading its row's 16 bytes in one load (a
// warp's 32 rows are then 512 contiguous bytes: no bank conflict, where one
// 2-byte load per block at a 16-byte row stride was a 4-way conflict).
template <int WF> struct BlockCodes;
template <> struct BlockCodes<BQG_Q4_0> {
    static constexpr int TILE = Q4_0_TILE, SCALE_OFF = 512;
    // block elements 0..31 -> v[term][0..3] (8 each): low nibbles are 0..15, high 16..31
    template <int TERMS>
    static __device__ __forceinline__ void dequant(const uint8_t *codes, float d, int r, int b8,
                                                   uint4 (&v)[TERMS][4])
    {
        const uint4 c = *reinterpret_cast<const uint4 *>(codes + r * 128 + ((b8 ^ (r & 7)) << 4));
        if constexpr (TERMS == 1) {
            dequant32_q4_bf16(c, d, v[0]);
            return;
        }
        uint4 t[4][TERMS];
        dequant8<TERMS>(c.x, c.y, 0, d, t[0]);
        dequant8<TERMS>(c.z, c.w, 0, d, t[1]);
        dequant8<TERMS>(c.x, c.y, 4, d, t[2]);
        dequant8<TERMS>(c.z, c.w, 4, d, t[3]);
#pragma unroll
        for (int j = 0; j < TERMS; j++)
#pragma unroll
            for (int g = 0; g < 4; g++) v[j][g] = t[g][j];
    }
};
template <> struct BlockCodes<BQG_Q8_0> {
    static constexpr int TILE = Q8_0_TILE, SCALE_OFF = 1024;
    // (q8_0 keeps one 2-byte scale load per block: measured faster for it, 73.9
    // against 75.6-77.5 us for the variants at M = 512 N = 14336 K = 4096)
    template <int TERMS>
    static __device__ __forceinline__ void dequant(const uint8_t *codes, const uint8_t *scales, int r, int b8,
                                                   uint4 (&v)[TERMS][4])
    {
        const int off = r * 128 + ((b8 ^ (r & 7)) << 4);
        const uint4 lo = *reinterpret_cast<const uint4 *>(codes + off);             // codes 0..15
        const uint4 hi = *reinterpret_cast<const uint4 *>(codes + RAW_CODES + off); // codes 16..31
        const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(scales + r * 16 + 2 * b8));
        uint4 t[4][TERMS];
        dequant8_q8<TERMS>(lo.x, lo.y, d, t[0]);
        dequant8_q8<TERMS>(lo.z, lo.w, d, t[1]);
        dequant8_q8<TERMS>(hi.x, hi.y, d, t[2]);
        dequant8_q8<TERMS>(hi.z, hi.w, d, t[3]);
#pragma unroll
        for (int j = 0; j < TERMS; j++)
#pragma unroll
            for (int g = 0; g < 4; g++) v[j][g] = t[g][j];
    }
};


struct GemmArgs {
    float *Y;               // M x N
    int M, N, K;
    int tiles_n;            // N / TM
    int n_big;              // big units kept whole: the first in the order
    int n_split;            // big units split into two small units each: next
    int m_single0;          // activation tile of the first single-tile units (the rest of the order)
    int units;              // n_big + 2 n_split + tiles_n (M / 128 - m_single0)
};

// Unit u of the order: weight tile tn, first activation row m0, rows 128 or
// 256.  Big unit b covers weight tile b % tiles_n and activation tiles
// 2 (b / tiles_n) and the one after it.
struct Unit { int tn, m0, rows; };
__device__ __forceinline__ Unit unit_of(const GemmArgs &a, int u)
{
    Unit r;
    if (u < a.n_big) {
        r.tn = u % a.tiles_n;
        r.m0 = 2 * (u / a.tiles_n) * TNS;
        r.rows = TNB;
    } else if (u < a.n_big + 2 * a.n_split) {
        const int j = u - a.n_big, b = a.n_big + (j >> 1);
        r.tn = b % a.tiles_n;
        r.m0 = (2 * (b / a.tiles_n) + (j & 1)) * TNS;
        r.rows = TNS;
    } else {
        const int j = u - a.n_big - 2 * a.n_split;
        r.tn = j % a.tiles_n;
        r.m0 = (a.m_single0 + j / a.tiles_n) * TNS;
        r.rows = TNS;
    }
    return r;
}

// Accumulator slot of this CTA's l-th unit (global unit u).  A CTA takes
// units blockIdx.x, + gridDim.x, ..., so its big units come first: they use
// slot 0; the small units after them alternate between slots 1 and 0.
__device__ __forceinline__ int slot_of(const GemmArgs &a, int l, int u)
{
    if (u < a.n_big) return 0;
    const int bx = blockIdx.x, g = gridDim.x;
    const int lb = (a.n_big > bx) ? (a.n_big - bx + g - 1) / g : 0;   // this CTA's big units
    return ((l - lb) & 1) ? 0 : 1;
}

template <int WF, int TERMS>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_bf16_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                   const __grid_constant__ CUtensorMap cmap,
                                                                   const __grid_constant__ CUtensorMap smap,
                                                                   const GemmArgs a)
{
    using PP = Pipe<TERMS>;
    constexpr int NSTAGE = PP::NSTAGE, A_COL0 = PP::A_COL0, SLOT_COLS = PP::SLOT_COLS;
    constexpr int STAGE_BYTES = PP::STAGE_BYTES;
    using SM = SmemOf<WF, TERMS>;
    constexpr int OFF_STAGES = SM::OFF_STAGES, OFF_BARS = SM::OFF_BARS, OFF_TMEM_SLOT = SM::OFF_TMEM_SLOT;
    constexpr int OFF_FLAG = SM::OFF_FLAG, NRAW = SM::NRAW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + OFF_BARS;
    auto bar_fullW = [&](int s) { return bars + 8 * s; };
    auto bar_fullX = [&](int s) { return bars + 8 * (NSTAGE + s); };
    auto bar_empty = [&](int s) { return bars + 8 * (2 * NSTAGE + s); };
    auto bar_accf = [&](int b) { return bars + 8 * (3 * NSTAGE + b); };
    auto bar_acce = [&](int b) { return bars + 8 * (3 * NSTAGE + 2 + b); };
    auto bar_rawf = [&](int j) { return bars + 8 * (3 * NSTAGE + 4 + j); };
    auto bar_rawe = [&](int j) { return bars + 8 * (3 * NSTAGE + 4 + NRAW + j); };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_FLAG);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = a.K / TK;                         // stages per unit (K % 64 == 0)

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; s++) {
            mbar_init(bar_fullW(s), DQ_WARPS);  // one arrive per dequantizing warp
            mbar_init(bar_fullX(s), 1);     // the TMA issuer's arrive + bytes
            mbar_init(bar_empty(s), 1);     // tcgen05.commit
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(bar_accf(b), 1);      // tcgen05.commit after a unit's last k-step
            mbar_init(bar_acce(b), 4);      // one arrive per epilogue warp
        }
        for (int j = 0; j < NRAW; j++) {
            mbar_init(bar_rawf(j), 1);      // the raw issuer's arrive + bytes
            mbar_init(bar_rawe(j), DQ_WARPS);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sbase + OFF_TMEM_SLOT),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + OFF_TMEM_SLOT);

    pdl_wait();
    pdl_launch_dependents();

    auto fail = [&]() {
        atomicExch(&g_gemm_error, 2);
        *abort_flag = 1;
    };

    if (warp == 0) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int it = 0;        // global k-step counter across units (ring position)
            int uses0 = 0, uses1 = 0;     // units that used accumulator slot 0 / 1
            bool ok = true;
            int l = 0;
            for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x, l++) {
                const Unit un = unit_of(a, u);
                const int b = slot_of(a, l, u);
                const int ub = b ? uses1 : uses0;
                // the slot's accumulator must have been read out (its previous unit)
                if (ub > 0 && !mbar_wait_spin(bar_acce(b), (ub - 1) & 1)) {
                    fail(); ok = false; break;
                }
                tc_fence_after();
                const uint32_t dacc = tmem + (b ? PP::ACC1 : PP::ACC0);
                const uint32_t idesc = idesc_n(un.rows);
                for (int k = 0; k < nk && ok; k++) {
                    const int step = it + k;
                    const int s = step % NSTAGE;
                    const uint32_t ph = (step / NSTAGE) & 1;
                    if (!mbar_wait_spin(bar_fullX(s), ph) || !mbar_wait_spin(bar_fullW(s), ph)) {
                        fail(); ok = false; break;
                    }
                    if (*abort_flag) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t aw = tmem + A_COL0 + s * SLOT_COLS;              // weights: MMA A (M = 128 rows)
                    const uint32_t bx = sbase + OFF_STAGES + s * STAGE_BYTES;       // activations: MMA B (N rows)
#pragma unroll
                    for (int kk = 0; kk < TK / 16; kk++) {
                        const uint64_t bdesc = sw128_desc(bx + kk * 32);
#pragma unroll
                        for (int j = 0; j < TERMS; j++)      // the weight's bf16 terms, one MMA each
                            umma_bf16_ts(dacc, aw + j * A_COLS + kk * 8, bdesc, idesc,
                                         (k > 0 || kk > 0 || j > 0) ? 1u : 0u);
                    }
                    umma_commit(bar_empty(s));               // stage s is free when these MMAs finish
                }
                if (ok) umma_commit(bar_accf(b));            // the unit's accumulator is complete
                if (b) uses1++; else uses0++;
                it += nk;
            }
            // drain: wait for the last MMAs before TMEM is released
            if (it > 0) mbar_wait_spin(bar_empty((it - 1) % NSTAGE), ((it - 1) / NSTAGE) & 1);
        }
        __syncwarp();
    } else if (warp == TMA_WARP) {
        // ---------------- activation tiles (TMA) ----------------
        if (lane == 0) {
            int it = 0;
            int issued = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
                const Unit un = unit_of(a, u);
                for (int k = 0; k < nk; k++) {
                    const int step = it + k;
                    const int s = step % NSTAGE;
                    if (step >= NSTAGE && !mbar_wait_spin(bar_empty(s), ((step / NSTAGE) - 1) & 1)) {
                        fail(); ok = false; break;
                    }
                    if (*abort_flag) { ok = false; break; }
                    const uint32_t dst = sbase + OFF_STAGES + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(bar_fullX(s), un.rows * TK * 2);
                    tma_load_2d(dst, &xmap, k * TK, un.m0, bar_fullX(s));
                    if (un.rows == TNB) tma_load_2d(dst + BOX_BYTES, &xmap, k * TK, un.m0 + TNS, bar_fullX(s));
                    issued++;
                }
                it += nk;
            }
            // do not leave while copies into shared memory are in flight (after an abort)
            for (int q = (issued > NSTAGE ? issued - NSTAGE : 0); q < issued; q++)
                mbar_wait_spin(bar_fullX(q % NSTAGE), (q / NSTAGE) & 1);
        }
        __syncwarp();
    } else if (warp == RAW_WARP) {
        // ---------------- raw weight codes and scales (TMA) ----------------
        if (lane == 0) {
            const int ng = (nk + RAW_STEPS - 1) / RAW_STEPS;   // raw groups per unit
            int gi = 0;                                        // global group counter (ring position)
            bool ok = true;
            for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
                const int tn = unit_of(a, u).tn;
                for (int g = 0; g < ng; g++, gi++) {
                    const int j = gi % NRAW;
                    if (gi >= NRAW && !mbar_wait_spin(bar_rawe(j), ((gi / NRAW) - 1) & 1)) {
                        fail(); ok = false; break;
                    }
                    if (*abort_flag) { ok = false; break; }
                    // blocks 8g .. 8g+7: tile t, slots s0 .. s0+7 (never past the row's last tile)
                    const int t = g >> 2, s0 = 8 * (g & 3);
                    const int x = t * BlockCodes<WF>::TILE + 16 * s0;
                    const uint32_t dst = sbase + SM::OFF_RAW + j * SM::RAW_GROUP;
                    mbar_arrive_expect_tx(bar_rawf(j), SM::RAW_GROUP + RAW_SCALES);
                    tma_load_2d(dst, &cmap, x, tn * TM, bar_rawf(j));
                    if (SM::CODE_BOXES == 2) tma_load_2d(dst + RAW_CODES, &cmap, x + 512, tn * TM, bar_rawf(j));
                    tma_load_2d(sbase + SM::OFF_SCALES + j * RAW_SCALES, &smap,
                                t * BlockCodes<WF>::TILE + BlockCodes<WF>::SCALE_OFF + 2 * s0, tn * TM, bar_rawf(j));
                }
            }
            // do not leave while copies into shared memory are in flight (after an abort)
            for (int q = (gi > NRAW ? gi - NRAW : 0); q < gi; q++) mbar_wait_spin(bar_rawf(q % NRAW), (q / NRAW) & 1);
        }
        __syncwarp();
    } else if (warp <= DQ_WARPS) {
        // ---------------- weight dequantization (warps 1-8) ----------------
        // a warp may only reach its lane quarter of tensor memory: warps 1-4 and
        // 5-8 each cover quarters 1, 2, 3, 0, for the stage's block 0 and 1
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;                   // weight row in the unit
        const int h = (warp - 1) >> 2;                       // which of the stage's two blocks
        const uint32_t arow = tmem + ((uint32_t)(quarter * 32) << 16) + A_COL0 + h * (A_COLS / 2);
        int it = 0;       // global k-step counter (A slot ring)
        int gi = 0;       // global raw-group counter (raw ring)
        bool ok = true;
        uint4 sc = make_uint4(0, 0, 0, 0);   // this row's eight fp16 scales of the current raw group
        for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
            for (int k = 0; k < nk && ok; k++) {
                const int kq = k % RAW_STEPS;
                const int j = gi % NRAW;
                if (kq == 0) {
                    const bool raw_ready = mbar_wait_spin(bar_rawf(j), (gi / NRAW) & 1);
                    if (!__all_sync(0xffffffffu, raw_ready)) { fail(); ok = false; break; }
                    if constexpr (WF == BQG_Q4_0)
                        sc = *reinterpret_cast<const uint4 *>(smem + SM::OFF_SCALES + j * RAW_SCALES + r * 16);
                }
                // block 2 kq + h of the raw group, dequantized before the A slot is free
                const int b8 = 2 * kq + h;
                const uint8_t *codes = smem + SM::OFF_RAW + j * SM::RAW_GROUP;
                uint4 v[TERMS][4];
                if constexpr (WF == BQG_Q4_0) {
                    const uint32_t sw = (kq == 0) ? sc.x : (kq == 1) ? sc.y : (kq == 2) ? sc.z : sc.w;
                    BlockCodes<WF>::template dequant<TERMS>(codes, half_bits_to_float(h ? (sw >> 16) : (sw & 0xffffu)),
                                                            r, b8, v);
                } else {
                    BlockCodes<WF>::template dequant<TERMS>(codes, smem + SM::OFF_SCALES + j * RAW_SCALES, r, b8, v);
                }
                const int step = it + k;
                const int s = step % NSTAGE;
                // the whole warp takes the same branch (tcgen05.st is warp-wide)
                const bool free_slot = step < NSTAGE || mbar_wait_spin(bar_empty(s), ((step / NSTAGE) - 1) & 1);
                if (!__all_sync(0xffffffffu, free_slot)) { fail(); ok = false; break; }
                if (*abort_flag) { ok = false; break; }
#pragma unroll
                for (int t = 0; t < TERMS; t++) tmem_st16_nowait(arow + s * SLOT_COLS + t * A_COLS, v[t]);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();                             // tensor-memory writes -> the MMA thread
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_fullW(s));
                if (kq == RAW_STEPS - 1 || k == nk - 1) {      // done with this raw group
                    if (lane == 0) mbar_arrive(bar_rawe(j));
                    gi++;
                }
            }
            it += nk;
        }
    } else {
        // ---------------- epilogue (warps 9-12: lane quarters 1, 2, 3, 0) ----------------
        const int quarter = warp & 3;
        int uses0 = 0, uses1 = 0;
        int l = 0;
        for (int u = blockIdx.x; u < a.units; u += gridDim.x, l++) {
            const Unit un = unit_of(a, u);
            const int b = slot_of(a, l, u);
            if (*abort_flag || !mbar_wait_spin(bar_accf(b), (b ? uses1 : uses0) & 1)) { fail(); break; }
            tc_fence_after();
            const int n = un.tn * TM + quarter * 32 + lane;   // weight row = output column
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (b ? PP::ACC1 : PP::ACC0);
#pragma unroll 1
            for (int c0 = 0; c0 < un.rows; c0 += 32) {
                float v[32];
                tmem_ld32(taddr + c0, v);
#pragma unroll
                for (int i = 0; i < 32; i++) a.Y[(int64_t)(un.m0 + c0 + i) * a.N + n] = v[i];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acce(b));
            if (b) uses1++; else uses0++;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
}

}  // namespace

// cuTensorMapEncodeTiled from the driver, looked up once (thread-safe); null
// when the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

int gemm_read_error(cudaStream_t stream, int *out)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess) return BQG_ERR_CUDA;
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(int)) != cudaSuccess) return BQG_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(int)) != cudaSuccess) return BQG_ERR_CUDA;
    *out = v;
    return BQG_OK;
}

size_t gemm_workspace(int, int64_t, int64_t) { return 0; }

// The order of units for `ctas` CTAs: big units (two activation tiles)
// where the pipeline allows them, in whole waves; the big units of a last,
// incomplete wave stay big when more than half the CTAs would take one, and
// are split into two small units each otherwise (a small unit costs about
// 0.7 of a big one, so two rounds of small units would cost more); then the
// single activation tile left over when M / 128 is odd.
void gemm_schedule(GemmArgs &a, int tiles_m, bool big, int ctas)
{
    const int pairs = big ? tiles_m / 2 : 0;
    const int nb = a.tiles_n * pairs;
    a.n_big = nb;
    a.n_split = 0;
    if (nb > 0) {
        const int rest = nb % ctas;
        if (2 * rest <= ctas) {
            a.n_big = nb - rest;
            a.n_split = rest;
        }
    }
    a.m_single0 = 2 * pairs;
    a.units = a.n_big + 2 * a.n_split + a.tiles_n * (tiles_m - 2 * pairs);
}

template <int WF, int TERMS>
int gemm_launch(const CUtensorMap &xmap, const CUtensorMap &cmap, const CUtensorMap &smap, GemmArgs a, int tiles_m,
                int sms, cudaStream_t stream)
{
    constexpr int smem = SmemOf<WF, TERMS>::SMEM_BYTES;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(gemm_bf16_kernel<WF, TERMS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr != cudaSuccess) return BQG_ERR_CUDA;
    gemm_schedule(a, tiles_m, Pipe<TERMS>::BIG, sms);
    const int grid = std::min(a.units, sms);
    gemm_bf16_kernel<WF, TERMS><<<grid, NUM_THREADS, smem, stream>>>(xmap, cmap, smap, a);
    return cudaGetLastError() == cudaSuccess ? BQG_OK : BQG_ERR_CUDA;
}

// M % 128 == 0, N % 128 == 0, K % 64 == 0 (checked by the caller); wf: BQG_Q4_0 or BQG_Q8_0
int gemm_bf16(int wf, const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K, cudaStream_t stream,
              int sms)
{
    auto enc = tensor_map_encoder();
    if (!enc) return BQG_ERR_CUDA;
    CUtensorMap map;
    const cuuint64_t gdim[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t gstride[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {TK, TNS};
    const cuuint32_t estride[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(X), gdim, gstride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return BQG_ERR_CUDA;
    // the repacked weights as a 2-D byte array (row_bytes x N): 128-row boxes
    // of 128 code bytes (128-byte swizzle) and of 16 scale bytes
    const int64_t nb = K / QK, T = (nb + 31) / 32;
    const int64_t row_bytes = T * (wf == BQG_Q8_0 ? Q8_0_TILE : Q4_0_TILE);
    CUtensorMap cmap, smap;
    const cuuint64_t wdim[2] = {(cuuint64_t)row_bytes, (cuuint64_t)N};
    const cuuint64_t wstride[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t cbox[2] = {128, TM}, sbox[2] = {16, TM};
    if (enc(&cmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(Wp), wdim, wstride, cbox, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&smap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(Wp), wdim, wstride, sbox, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return BQG_ERR_CUDA;
    GemmArgs a;
    a.Y = Y;
    a.M = M;
    a.N = (int)N;
    a.K = (int)K;
    a.tiles_n = (int)(N / TM);
    const int tiles_m = M / TNS;
    // Below K = 1024 a product of few terms can be dominated by one weight,
    // and the one bf16 rounding of (q - 8) d (relative error up to 2^-9) can
    // then exceed the parity bound 1e-3 sum |w x|; those calls split each
    // weight exactly into bf16 terms (two for q4_0, three for q8_0).  From
    // K = 1024 on, one rounding per weight (the config's bf16 dequantization).
    const bool exact = K < kGemmExactBelowK;
    if (wf == BQG_Q8_0)
        return exact ? gemm_launch<BQG_Q8_0, 3>(map, cmap, smap, a, tiles_m, sms, stream)
                     : gemm_launch<BQG_Q8_0, 1>(map, cmap, smap, a, tiles_m, sms, stream);
    return exact ? gemm_launch<BQG_Q4_0, 2>(map, cmap, smap, a, tiles_m, sms, stream)
                 : gemm_launch<BQG_Q4_0, 1>(map, cmap, smap, a, tiles_m, sms, stream);
}

}  // namespace bqg
