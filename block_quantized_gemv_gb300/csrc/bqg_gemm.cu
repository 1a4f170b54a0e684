// bqg_gemm.cu -- prefill GEMM Y[M x N] = X[M x K] W^T on the sm_103a tensor cores.
//
// The tiled prefill GEMM of "llama-3x-prompt-speed" ("the tile"): a weight
// tile is unpacked once and serves every activation row of the tile,
// instead of being unpacked once per row.  Here the unit of work is 128
// weight rows x 128 activation rows; per stage of 128 along K:
//   * warp 14, lane 0 stages the raw weight codes and scales of two stages
//     at a time (eight q4_0 blocks per row) into shared memory with two-dimensional TMA copies (128 rows
//     x 128 bytes of codes in the 128-byte swizzle, 128 rows x 16 bytes of
//     scales), so the weight stream is coalesced;
//   * warps 1-8 (one weight block of one weight row per thread) read their
//     block's codes and scale from there (conflict-free thanks to the
//     swizzle), dequantize q * d or (q - 8) * d exactly in fp32, round once to
//     bf16 and store the 128 x 128 bf16 tile straight into tensor memory
//     (tcgen05.st: lane = weight row, two k per column), where the MMA reads
//     its A operand.  Shared memory then carries only the
//     activation tiles: with A staged there too, its bandwidth (dequant
//     writes, TMA writes and both MMA operands, 64 KiB per k-step) bounded
//     the loop at twice the MMA time;
//   * warp 13, lane 0 loads the matching 128 x 128 bf16 activation tile with
//     two TMA copies of one 64-wide swizzle atom each as soon as the stage
//     is free (a trailing half stage when K % 128 == 64);
//   * warp 0, lane 0 issues eight tcgen05.mma.kind::f16 (A from tensor
//     memory, B from shared memory; M = 128 weight rows, N = 128
//     activations, K = 16) accumulating fp32 in tensor memory as soon as both
//     halves of the stage are in place; tcgen05.commit frees the stage.  It
//     never waits for its own MMAs, so the tensor core always has the next
//     K-step queued;
//   * warps 9-12 read the finished 128 x 128 fp32 accumulator with
//     tcgen05.ld (each warp its 32 lanes = 32 weight rows) and store
//     Y[m][n] coalesced along n.
// Tensor memory (512 columns): two 128-column accumulators, so the epilogue
// of one unit overlaps the MMAs of the next, then the NSTAGE A slots of 64
// columns.  The kernel is persistent (one
// CTA per SM).  Every mbarrier wait is bounded: on a timeout the kernel sets
// g_gemm_error, stops issuing work, drains what it started and frees TMEM.
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "bqg_common.cuh"

namespace bqg {

// Error word set by bounded device-side waits (0 = none).
__device__ int g_gemm_error;

namespace {

constexpr int TM = 128;         // weight rows per unit (MMA M)
constexpr int TN = 128;         // activation rows per unit (MMA N)
constexpr int TK = 128;         // K per stage: two 128-byte swizzle atoms of bf16
constexpr int XATOM = 64;       // K of one swizzle atom (one TMA box)
constexpr int ATOM_BYTES = TN * XATOM * 2;    // 16 KiB
constexpr int TILE_BYTES = TN * TK * 2;       // 32 KiB activation tile
constexpr int STAGE_BYTES = TILE_BYTES;
constexpr int ACC_COLS = TN;                  // fp32 columns per accumulator
constexpr int A_COLS = TK / 2;                // 32-bit columns of one bf16 A tile of a stage (two bf16 each)
constexpr int TMEM_COLS = 512;                // accumulators + NSTAGE A slots
constexpr int kGemmExactBelowK = 1024;        // K below which the weights are split into exact bf16 terms

// Pipeline shape per number of bf16 terms a dequantized weight is split
// into.  TERMS = 1: (q - 8) d or q d rounded once to bf16 (the prefill
// config's dequantization).  TERMS = 2 (q4_0) / 3 (q8_0): the weight written
// exactly as a sum of bf16 values (a 4-bit code times an fp16 scale has at
// most 14 significant bits, an 8-bit code times one at most 19, and bf16
// holds 8), one MMA per term into the same fp32 accumulator, so the GEMM is
// exact up to fp32 accumulation.  Each A slot holds the stage's terms; the
// tensor memory then allows fewer stages (and, at three terms, one
// accumulator).
template <int TERMS> struct Pipe {
    static constexpr int NSTAGE = (TERMS == 1) ? 4 : 2;
    static constexpr int NACC = (TERMS == 3) ? 1 : 2;
    static constexpr int A_COL0 = NACC * ACC_COLS;        // first column of the A slots
    static constexpr int SLOT_COLS = TERMS * A_COLS;      // one stage's A terms
    static_assert(A_COL0 + NSTAGE * SLOT_COLS <= TMEM_COLS, "tensor memory budget");
};
constexpr int DQ_WARPS = 8;                   // dequantizing warps (1..8)
constexpr int EPI_WARP0 = 1 + DQ_WARPS;       // epilogue warps 9..12
constexpr int TMA_WARP = EPI_WARP0 + 4;       // activation loads: warp 13
constexpr int RAW_WARP = TMA_WARP + 1;        // raw weight codes: warp 14
constexpr int NUM_THREADS = (RAW_WARP + 1) * 32;
constexpr int RAW_STEPS = 2;                  // stages per raw group: 8 blocks = 128 code bytes (q4_0)
constexpr int RAW_CODES = TM * 128;           // bytes of one 128-row x 128-byte code box
constexpr int RAW_SCALES = TM * 16;           // bytes of one 128-row x 16-byte scale box

// shared memory map (dynamic, 1024-byte aligned), per weight format and
// number of activation stages
template <int WF, int NSTAGE> struct GemmSmem {
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

// instruction descriptor, kind::f16: D fp32, A bf16, B bf16, both K-major, N, M
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(TN >> 3) << 17) |
                           ((uint32_t)(TM >> 4) << 24);

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
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(IDESC), "r"(accumulate)
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
    const uint8_t *W;       // repacked q4_0, N rows
    float *Y;               // M x N
    int64_t row_bytes;      // repacked bytes per weight row
    int M, N, K;
    int units;              // (N / TM) * (M / TN)
    int tiles_n;            // N / TM
};

template <int WF, int TERMS>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_bf16_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                   const __grid_constant__ CUtensorMap cmap,
                                                                   const __grid_constant__ CUtensorMap smap,
                                                                   const GemmArgs a)
{
    using PP = Pipe<TERMS>;
    constexpr int NSTAGE = PP::NSTAGE, NACC = PP::NACC, A_COL0 = PP::A_COL0, SLOT_COLS = PP::SLOT_COLS;
    using SM = GemmSmem<WF, NSTAGE>;
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
    const int nk = (a.K + TK - 1) / TK;              // stages per unit (a last one may hold K = 64)

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
            int ucount = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x, ucount++) {
                const int b = ucount % NACC;
                // the accumulator must have been read out (NACC units ago)
                if (ucount >= NACC && !mbar_wait_spin(bar_acce(b), ((ucount / NACC) - 1) & 1)) {
                    fail(); ok = false; break;
                }
                tc_fence_after();
                const uint32_t dacc = tmem + b * ACC_COLS;
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
                    const uint32_t bx = sbase + OFF_STAGES + s * STAGE_BYTES;       // activations: MMA B (N = 128)
                    // a last stage of K = 64 (K % 128 == 64) holds one atom
                    const int nkk = (k == nk - 1 && (a.K % TK) != 0) ? XATOM / 16 : TK / 16;
#pragma unroll
                    for (int kk = 0; kk < TK / 16; kk++) {
                        if (kk >= nkk) break;
                        const uint64_t bdesc = sw128_desc(bx + (kk >> 2) * ATOM_BYTES + (kk & 3) * 32);
#pragma unroll
                        for (int j = 0; j < TERMS; j++)      // the weight's bf16 terms, one MMA each
                            umma_bf16_ts(dacc, aw + j * A_COLS + kk * 8, bdesc, (k > 0 || kk > 0 || j > 0) ? 1u : 0u);
                    }
                    umma_commit(bar_empty(s));               // stage s is free when these MMAs finish
                }
                if (ok) umma_commit(bar_accf(b));            // the unit's accumulator is complete
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
                const int tm = u / a.tiles_n;                      // activation tile
                for (int k = 0; k < nk; k++) {
                    const int step = it + k;
                    const int s = step % NSTAGE;
                    if (step >= NSTAGE && !mbar_wait_spin(bar_empty(s), ((step / NSTAGE) - 1) & 1)) {
                        fail(); ok = false; break;
                    }
                    if (*abort_flag) { ok = false; break; }
                    const bool half = (k == nk - 1) && (a.K % TK) != 0;
                    mbar_arrive_expect_tx(bar_fullX(s), half ? ATOM_BYTES : TILE_BYTES);
                    tma_load_2d(sbase + OFF_STAGES + s * STAGE_BYTES, &xmap, k * TK, tm * TN, bar_fullX(s));
                    if (!half)
                        tma_load_2d(sbase + OFF_STAGES + s * STAGE_BYTES + ATOM_BYTES, &xmap, k * TK + XATOM, tm * TN,
                                    bar_fullX(s));
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
                const int tn = u % a.tiles_n;
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
        // 5-8 each cover quarters 1, 2, 3, 0, for the stage's blocks 0-1 and 2-3
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;                   // weight row in the unit
        const int h = (warp - 1) >> 2;                       // which pair of the stage's four blocks
        const uint32_t arow = tmem + ((uint32_t)(quarter * 32) << 16) + A_COL0 + h * (A_COLS / 2);
        auto store_terms = [&](uint32_t col, uint4 (&v)[TERMS][4]) {
#pragma unroll
            for (int j = 0; j < TERMS; j++) tmem_st16_nowait(col + j * A_COLS, v[j]);
        };
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
                const int step = it + k;
                const int s = step % NSTAGE;
                // the whole warp takes the same branch (tcgen05.st is warp-wide)
                const bool free_slot = step < NSTAGE || mbar_wait_spin(bar_empty(s), ((step / NSTAGE) - 1) & 1);
                if (!__all_sync(0xffffffffu, free_slot)) { fail(); ok = false; break; }
                if (*abort_flag) { ok = false; break; }
                // blocks 2h, 2h+1 of the stage are blocks 4 kq + 2h (+1) of the raw group:
                // 32 columns of the A slot (a last half stage has blocks 0-1 only)
                const bool half = (k == nk - 1) && (a.K % TK) != 0;
                if (!(half && h == 1)) {
                    const uint8_t *codes = smem + SM::OFF_RAW + j * SM::RAW_GROUP;
                    uint4 v[TERMS][4];
                    if constexpr (WF == BQG_Q4_0) {
                        // blocks 4 kq + 2h and + 1: the two halves of scale word 2 kq + h
                        const uint32_t sw = kq ? (h ? sc.w : sc.z) : (h ? sc.y : sc.x);
                        BlockCodes<WF>::template dequant<TERMS>(codes, half_bits_to_float(sw & 0xffffu), r,
                                                                4 * kq + 2 * h, v);
                        store_terms(arow + s * SLOT_COLS, v);
                        BlockCodes<WF>::template dequant<TERMS>(codes, half_bits_to_float(sw >> 16), r,
                                                                4 * kq + 2 * h + 1, v);
                    } else {
                        const uint8_t *scales = smem + SM::OFF_SCALES + j * RAW_SCALES;
                        BlockCodes<WF>::template dequant<TERMS>(codes, scales, r, 4 * kq + 2 * h, v);
                        store_terms(arow + s * SLOT_COLS, v);
                        BlockCodes<WF>::template dequant<TERMS>(codes, scales, r, 4 * kq + 2 * h + 1, v);
                    }
                    store_terms(arow + s * SLOT_COLS + 16, v);
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                }
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
        int ucount = 0;
        for (int u = blockIdx.x; u < a.units; u += gridDim.x, ucount++) {
            const int tn = u % a.tiles_n, tm = u / a.tiles_n;
            const int b = ucount % NACC;
            if (*abort_flag || !mbar_wait_spin(bar_accf(b), (ucount / NACC) & 1)) { fail(); break; }
            tc_fence_after();
            const int n = tn * TM + quarter * 32 + lane;     // weight row = output column
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + b * ACC_COLS;
#pragma unroll 1
            for (int c0 = 0; c0 < TN; c0 += 32) {
                float v[32];
                tmem_ld32(taddr + c0, v);
#pragma unroll
                for (int i = 0; i < 32; i++) a.Y[(int64_t)(tm * TN + c0 + i) * a.N + n] = v[i];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acce(b));
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

// M % 128 == 0, N % 128 == 0, K % 64 == 0 (checked by the caller); wf: BQG_Q4_0 or BQG_Q8_0
int gemm_bf16(int wf, const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K, cudaStream_t stream,
              int sms)
{
    static std::mutex mu;
    auto enc = tensor_map_encoder();
    if (!enc) return BQG_ERR_CUDA;
    CUtensorMap map;
    const cuuint64_t gdim[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t gstride[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {XATOM, TN};
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
    a.W = static_cast<const uint8_t *>(Wp);
    a.Y = Y;
    a.row_bytes = row_bytes;
    a.M = M;
    a.N = (int)N;
    a.K = (int)K;
    a.tiles_n = (int)(N / TM);
    a.units = a.tiles_n * (M / TN);
    // Below K = 1024 a product of few terms can be dominated by one weight,
    // and the one bf16 rounding of (q - 8) d (relative error up to 2^-9) can
    // then exceed the parity bound 1e-3 sum |w x|; those calls split each
    // weight exactly into bf16 terms (two for q4_0, three for q8_0).  From
    // K = 1024 on, one rounding per weight (the config's bf16 dequantization).
    const bool exact = K < kGemmExactBelowK;
    {
        std::lock_guard<std::mutex> lk(mu);
        static bool attr = false;
        if (!attr) {
            if (cudaFuncSetAttribute(gemm_bf16_kernel<BQG_Q4_0, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     GemmSmem<BQG_Q4_0, Pipe<1>::NSTAGE>::SMEM_BYTES) != cudaSuccess ||
                cudaFuncSetAttribute(gemm_bf16_kernel<BQG_Q4_0, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     GemmSmem<BQG_Q4_0, Pipe<2>::NSTAGE>::SMEM_BYTES) != cudaSuccess ||
                cudaFuncSetAttribute(gemm_bf16_kernel<BQG_Q8_0, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     GemmSmem<BQG_Q8_0, Pipe<1>::NSTAGE>::SMEM_BYTES) != cudaSuccess ||
                cudaFuncSetAttribute(gemm_bf16_kernel<BQG_Q8_0, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     GemmSmem<BQG_Q8_0, Pipe<3>::NSTAGE>::SMEM_BYTES) != cudaSuccess)
                return BQG_ERR_CUDA;
            attr = true;
        }
    }
    const int grid = std::min(a.units, sms);
    if (wf == BQG_Q8_0 && exact)
        gemm_bf16_kernel<BQG_Q8_0, 3><<<grid, NUM_THREADS, GemmSmem<BQG_Q8_0, Pipe<3>::NSTAGE>::SMEM_BYTES, stream>>>(
            map, cmap, smap, a);
    else if (wf == BQG_Q8_0)
        gemm_bf16_kernel<BQG_Q8_0, 1><<<grid, NUM_THREADS, GemmSmem<BQG_Q8_0, Pipe<1>::NSTAGE>::SMEM_BYTES, stream>>>(
            map, cmap, smap, a);
    else if (exact)
        gemm_bf16_kernel<BQG_Q4_0, 2><<<grid, NUM_THREADS, GemmSmem<BQG_Q4_0, Pipe<2>::NSTAGE>::SMEM_BYTES, stream>>>(
            map, cmap, smap, a);
    else
        gemm_bf16_kernel<BQG_Q4_0, 1><<<grid, NUM_THREADS, GemmSmem<BQG_Q4_0, Pipe<1>::NSTAGE>::SMEM_BYTES, stream>>>(
            map, cmap, smap, a);
    return cudaGetLastError() == cudaSuccess ? BQG_OK : BQG_ERR_CUDA;
}

}  // namespace bqg
