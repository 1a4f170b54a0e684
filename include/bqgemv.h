/*
 * bqgemv.h -- block-quantized skinny GEMV / prefill GEMM for GB300 (sm_103a).
 *
 * What it computes (all entry points):
 *     Y[m, n] = sum_k  W[n, k] * X[m, k]          m < M, n < N, k < K
 * with W stored as N rows of K weights and X as M rows of K activations:
 * the memory-bound decode shape (M = 1..8) of "The Shape That Actually
 * Matters" (amarbaro.com), and the M = 512 prefill GEMM over dequantized
 * weight tiles of "llama-3x-prompt-speed" ("the tile").  Outputs are fp32.
 *
 * Block formats (32 elements per block, little-endian fp16 scales):
 *   BQG_Q8_0  34 B = fp16 d | int8 q[32]                  w = q * d
 *   BQG_Q4_0  18 B = fp16 d | 16 bytes of 4-bit codes      w = (q - 8) * d
 *             (the 18-byte block of "MI50 megakernel", hypothesis ledger;
 *              byte j holds element j in its low nibble, j+16 in its high)
 *   BQG_Q8_1  36 B = fp16 d | fp16 s | int8 q[32]          x = q * d,
 *             s = fp16(d * sum q)   (the activation side of the "Q4_0 x Q8_1"
 *             matvec of "rx-6700xt-llama2-decode", Approach & Methodology)
 *   BQG_BF16  2 B per element, no blocks.
 * A "canonical" weight matrix is N rows, each K/32 consecutive blocks.
 *
 * Repacked weights (the layout every GEMV/GEMM entry point reads), produced
 * once at load time by bqg_repack_weights.  nb = K/32 blocks per row,
 * T = ceil(nb/32) tiles per row, a tile = 32 consecutive blocks of one row:
 *   bf16 : row-major N x K, identical to canonical.
 *   q4_0 : tile of 576 B: block 32t+s has its 16 code bytes at 16*s and its
 *          fp16 scale at 512 + 2*s.
 *   q8_0 : tile of 1088 B: block 32t+s has codes 0..15 at 16*s, codes 16..31
 *          at 512 + 16*s, and its fp16 scale at 1024 + 2*s.
 * Rows follow each other with a stride of T tiles; unused slots of a row's
 * last tile are zero.  Every 32 lanes of a warp then read 512 contiguous
 * bytes per 128-bit load, and scales sit beside their codes.
 *
 * Rounding rules of the encoders (the pages name the formats only):
 *   the scale is computed in fp32 and rounded once to fp16 (nearest-even);
 *   codes divide by the STORED fp16 scale in IEEE fp32 and round half away
 *   from zero; q8: d = amax/127, q clamped to [-127, 127], d = 0 gives q = 0;
 *   q4_0: m = first element of largest |x|, d = m / -8,
 *         q = clamp(round(x/d) + 8, 0, 15), d = 0 gives q = 8.
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers on the current CUDA device unless stated.
 *     The caller owns every buffer; the library never allocates, frees or
 *     keeps a pointer after the call returns.
 *   - Every call is asynchronous on `stream` (0 = legacy default stream) and
 *     returns a bqg_status.  Arguments are validated on the host before any
 *     launch; an invalid call launches nothing.
 *   - Device pointers must be 16-byte aligned (BQG_ERR_MISALIGNED otherwise).
 *   - K must be a positive multiple of 32 (BQG_ERR_UNSUPPORTED_SHAPE).
 *   - Only sm_103 devices are accepted (BQG_ERR_UNSUPPORTED_DEVICE).
 *   - There is no CPU fallback and no silent change of route.
 */
#ifndef BQGEMV_H
#define BQGEMV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* formats */
enum { BQG_BF16 = 0, BQG_Q8_0 = 1, BQG_Q4_0 = 2, BQG_Q8_1 = 3, BQG_F32 = 4 };

/* status codes */
enum {
    BQG_OK = 0,
    BQG_ERR_INVALID_ARG = 1,        /* null pointer, bad enum, M not allowed, N < 0 */
    BQG_ERR_UNSUPPORTED_SHAPE = 2,  /* K % 32 != 0, K or M beyond the kernel limits */
    BQG_ERR_MISALIGNED = 3,         /* a device pointer is not 16-byte aligned      */
    BQG_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not sm_103                 */
    BQG_ERR_CUDA = 5,               /* a CUDA runtime call or launch failed         */
    BQG_ERR_TIMEOUT = 6,            /* a bounded device-side wait gave up           */
    BQG_ERR_WORKSPACE = 7           /* the call needs a workspace that is missing   */
};

/* operation ids for bqg_workspace_size */
enum {
    BQG_OP_GEMV_BF16 = 0,
    BQG_OP_GEMV_Q8_0 = 1,
    BQG_OP_GEMV_Q4_0 = 2,
    BQG_OP_GEMV_Q4_0_Q8_1 = 3,
    BQG_OP_QKV_Q4_0_Q8_1 = 4,       /* N = Nq + 2*Nkv */
    BQG_OP_GATE_UP_Q4_0_Q8_1 = 5,   /* N = rows of each of gate and up */
    BQG_OP_GEMM_Q4_0_BF16 = 6,
    BQG_OP_GATE_UP_Q8_1_Q4_0_Q8_1 = 7, /* gate+up SwiGLU with q8_1 output; N = rows of each */
    BQG_OP_GEMM_Q8_0_BF16 = 8,
    BQG_OP_DECODE_LAYER_Q4_0_Q8_1 = 9  /* M = 1; N = Nff (rows of each of gate and up), K = model width */
};

/* ---- load time ------------------------------------------------------- */

/* Bytes of the repacked layout of an N x K matrix of `fmt` (BQG_BF16,
 * BQG_Q8_0 or BQG_Q4_0); 0 for an invalid format or K % 32 != 0. */
size_t bqg_repacked_size(int fmt, int64_t N, int64_t K);

/* Encode fp32 weights (N x K, row-major, device) into canonical q8_0 or
 * q4_0 blocks (N x K/32 blocks, device) with the rounding rules above.
 * fmt: BQG_Q8_0 or BQG_Q4_0.  `dst` needs N*(K/32)*(34 or 18) bytes and
 * may be 2-byte aligned (block rows are not 16-byte multiples). */
int bqg_quantize_weights(int fmt, const float *W, void *dst, int64_t N, int64_t K,
                         cudaStream_t stream);

/* Canonical -> repacked layout (above).  `src` canonical (2-byte aligned is
 * enough), `dst` bqg_repacked_size(fmt, N, K) bytes, 16-byte aligned; the
 * two must not overlap.  Pure byte permutation (bit-exact). */
int bqg_repack_weights(int fmt, const void *src, void *dst, int64_t N, int64_t K,
                       cudaStream_t stream);

/* ---- per token -------------------------------------------------------- */

/* Quantize activations to q8_1 blocks ("Q8_1" of rx-6700xt-llama2-decode).
 * x: M x K, x_dtype BQG_BF16 or BQG_F32, row-major.  xq: M x K/32 blocks of
 * 36 B, row-major.  1 <= M <= 65535.  Bit-exact with the rules above. */
int bqg_quantize_q8_1(const void *x, int x_dtype, void *xq, int M, int64_t K,
                      cudaStream_t stream);

/* Fused RMSNorm + q8_1 quantization: the normalisation that precedes each
 * projection folded into the activation encoder, one launch instead of two
 * ("MI50 megakernel", hypothesis ledger: neighbouring steps fused into one
 * dispatch).  The pages name the fusion, not its arithmetic; per row m
 * the definition is
 *     s   = sum_k x[m,k]^2                 (exact for bf16 inputs)
 *     r   = fp32( 1 / sqrt(s / K + eps) )  (one rounding to fp32)
 *     y_k = fp32( fp32(x[m,k] * r) * gamma[k] )   (gamma NULL: no gain)
 * then y is encoded like bqg_quantize_q8_1.  x: M x K, x_dtype BQG_BF16 or
 * BQG_F32 (2- or 4-byte aligned); gamma: K fp32 or NULL (4-byte aligned);
 * eps >= 0 and finite; xq: M x K/32 blocks of 36 B (4-byte aligned);
 * 1 <= M <= 65535.  The kernel sums the squares as error-free fp32 pairs and
 * refines rsqrtf by one Newton step; before its final rounding r is within
 * about 2^-44 (relative) of the exact value, so r, and with it every byte,
 * matches the definition evaluated in fp64 unless the exact value lies that
 * close to an fp32 rounding boundary (about one row in 2^20). */
int bqg_rmsnorm_quantize_q8_1(const void *x, int x_dtype, const float *gamma, float eps, void *xq, int M,
                              int64_t K, cudaStream_t stream);

/* Skinny GEMV, M in {1, 2, 4, 8}.  Wp: repacked weights of the named format.
 * X: M x K bf16 (row-major).  Y: M x N fp32 (row-major).
 * ws/ws_bytes: workspace for split-K; bqg_workspace_size(op, M, N, K) bytes
 * are required when that size is non-zero (BQG_ERR_WORKSPACE otherwise); it
 * needs no initialisation and must not be shared by calls that overlap.
 * fp32 accumulation.  At M = 1 and 2 (and where the route below does not
 * apply) bqg_gemv_q8_0/q4_0 dequantize (q*d, (q-8)*d) exactly and add the
 * products in fp32.  At M = 4 and 8 (and for q4_0 at M = 2; staged
 * activations M*K*2 bytes within 80 KiB; bf16 weights with N >= 16 * 76)
 * the products go to the tensor
 * cores (mma.sync, bf16 operands: q8_0 codes, q4_0 values q-8 and bf16
 * weights are exact in bf16, each product exact in fp32); each block's sum
 * over its 32 values is then scaled by its d in fp32, and bf16 weights
 * accumulate in the MMA's fp32 fragment.  Either way the result lies
 * within 1e-3 * sum_k |w x| + 1e-6 of the exact sum (the bound the tests
 * hold every route to).
 * Y may also be page-locked host memory given by its bqg_host_alias address
 * (the outputs are written there with plain stores over the CPU-GPU link);
 * this holds for the four bqg_gemv_* entries of a single matrix and
 * bqg_gemv_q4_0_q8_1_noalloc.  X and Wp must be device memory. */
int bqg_gemv_bf16(const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K,
                  void *ws, size_t ws_bytes, cudaStream_t stream);
int bqg_gemv_q8_0(const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K,
                  void *ws, size_t ws_bytes, cudaStream_t stream);
int bqg_gemv_q4_0(const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K,
                  void *ws, size_t ws_bytes, cudaStream_t stream);

/* q4_0 weights x q8_1 activations (M in {1, 2, 4, 8}).  Per block the
 * integer dot sumi = sum_i (qw_i - 8) * qx_i is exact (int32 by dp4a; at
 * M = 8 on the tensor cores, from exact bf16 operands, an fp32 sum of
 * integers below 2^15 in magnitude, so exact as well), and
 * Y += (d_w * d_x) * sumi in fp32.  Xq: M x K/32 q8_1 blocks. */
int bqg_gemv_q4_0_q8_1(const void *Wp, const void *Xq, float *Y, int M, int64_t N, int64_t K,
                       void *ws, size_t ws_bytes, cudaStream_t stream);

/* No counterpart on the pages.  An allocation-free variant of
 * bqg_gemv_q4_0_q8_1 for callers that cannot hand the library a workspace
 * from cudaMalloc: a runtime whose device memory plan is fixed when the
 * model loads, a decode loop in which an allocation may block or
 * synchronize the device, or C code with no allocator of its own.  Same
 * arguments and arithmetic as bqg_gemv_q4_0_q8_1 without the workspace:
 * split-K partial sums go to a fixed array of bqg_noalloc_scratch_bytes()
 * (32 KiB) inside the library, which every device that loads the library
 * holds until the process exits.
 *  - The first call on each device looks up the array's device address (a
 *    synchronous runtime call); make that first call before any stream
 *    capture.  The address is kept for the life of the process: a
 *    cudaDeviceReset of that device afterwards (which reloads the library's
 *    device image, perhaps elsewhere) leaves it stale, so this entry point
 *    must not be called on a device after that device has been reset.
 *  - A shape whose split-K partials would not fit the array returns
 *    BQG_ERR_WORKSPACE and launches nothing.
 *  - Every call shares the array.  Nothing in it has to start at zero (a
 *    call writes every partial sum it reads), but calls that overlap on the
 *    GPU, on one stream or several, race on it.
 *  - It calls no cudaMalloc, cudaFree or allocating library routine. */
int bqg_gemv_q4_0_q8_1_noalloc(const void *Wp, const void *Xq, float *Y, int M, int64_t N, int64_t K,
                               cudaStream_t stream);
size_t bqg_noalloc_scratch_bytes(void);

/* Q, K and V projections of one shared activation in a single launch
 * (the grouped QKV launch of "rx-6700xt-llama2-decode", Approach &
 * Methodology).  Wq: Nq x K, Wk/Wv: Nkv x K repacked q4_0;
 * Yq: M x Nq, Yk/Yv: M x Nkv fp32.  Same arithmetic as bqg_gemv_q4_0_q8_1. */
int bqg_gemv_q4_0_q8_1_qkv(const void *Wq, const void *Wk, const void *Wv, const void *Xq,
                           float *Yq, float *Yk, float *Yv, int M, int64_t Nq, int64_t Nkv,
                           int64_t K, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Feed-forward gate and up projections in one launch with the SwiGLU
 * epilogue applied before the store (the grouped feed-forward launch of
 * "rx-6700xt-llama2-decode", Approach & Methodology):
 * H[m, n] = silu(g) * u with g = (Wg Xq)[m, n], u = (Wu Xq)[m, n],
 * silu(g) = g / (1 + exp(-g)).
 * Wg, Wu: N x K repacked q4_0; H: M x N fp32. */
int bqg_gemv_q4_0_q8_1_gate_up_swiglu(const void *Wg, const void *Wu, const void *Xq, float *H,
                                      int M, int64_t N, int64_t K, void *ws, size_t ws_bytes,
                                      cudaStream_t stream);

/* The same gate+up+SwiGLU whose epilogue writes h as q8_1 blocks, ready for
 * the down projection (bqg_gemv_q4_0_q8_1 at K = N), instead of fp32: the
 * standalone encoder between the two launches goes away ("rx-6700xt-
 * llama2-decode", Approach & Methodology: the fused gate+up writes the
 * SwiGLU result directly).  Hq: M x N/32 blocks of 36 B (4-byte aligned);
 * N must be a multiple of 32.  Each block is encoded, with the rules of
 * bqg_quantize_q8_1, from the fp32 values h = silu(g) * u that
 * bqg_gemv_q4_0_q8_1_gate_up_swiglu would write, so the two agree byte for
 * byte with bqg_quantize_q8_1 applied to the latter.
 * ws: bqg_workspace_size(BQG_OP_GATE_UP_Q8_1_Q4_0_Q8_1, M, N, K) bytes,
 * 16-byte aligned.  Without split-K it holds an fp32 staging copy of h and
 * one counter per block, which must be ZERO before the first call on that
 * workspace (every successful call leaves them zero; after a
 * BQG_ERR_TIMEOUT report, zero them again).  Calls that share a workspace
 * must not overlap. */
int bqg_gemv_q4_0_q8_1_gate_up_swiglu_q8_1(const void *Wg, const void *Wu, const void *Xq, void *Hq, int M,
                                           int64_t N, int64_t K, void *ws, size_t ws_bytes,
                                           cudaStream_t stream);

/* One decode layer's three projection groups in one persistent launch
 * ("MI50 megakernel", hypothesis ledger: neighbouring steps fused into one
 * dispatch with a grid-wide barrier between dependent steps; "rx-6700xt-
 * llama2-decode", Approach & Methodology: the q4_0 x q8_1 matvec and its fused
 * QKV and gate+up/SwiGLU dispatches).  M = 1.  Computes, as the separate
 * entry points would:
 *   xqa = q8_1(xa), xqb = q8_1(xb)              (the rules of bqg_quantize_q8_1)
 *   Yq, Yk, Yv = Wq . xqa, Wk . xqa, Wv . xqa   (bqg_gemv_q4_0_q8_1_qkv)
 *   hq = q8_1(silu(Wg . xqb) * (Wu . xqb))      (..._gate_up_swiglu_q8_1)
 *   Y  = Wd . hq                                (bqg_gemv_q4_0_q8_1)
 * xa, xb: K values each, x_dtype BQG_BF16 or BQG_F32 (2- or 4-byte aligned).
 * Wq: Nq x K, Wk and Wv: Nkv x K, Wg and Wu: Nff x K, Wd: K x Nff, all
 * repacked q4_0 (16-byte aligned).  Yq: Nq, Yk and Yv: Nkv, Y: K fp32.
 * K and Nff multiples of 32.  The launch is cooperative (every CTA resident
 * at once, as the grid barrier needs; the runtime refuses it otherwise,
 * reported as BQG_ERR_CUDA).  ws: bqg_workspace_size(
 * BQG_OP_DECODE_LAYER_Q4_0_Q8_1, 1, Nff, K) bytes, 16-byte aligned, ZERO
 * before the first call on it (every successful call leaves its counters
 * zero; after a BQG_ERR_TIMEOUT report zero it again); it holds h (fp32),
 * the q8_1 blocks of h, their arrival counters and the grid barrier.  Calls
 * sharing a workspace must not overlap.  Errors: INVALID_ARG (null pointer,
 * non-positive size, other x_dtype), UNSUPPORTED_SHAPE (M != 1, K or Nff not
 * a multiple of 32 or above 65536, stages that do not fit in shared memory),
 * MISALIGNED, WORKSPACE (ws too small); a bounded device wait that gives up
 * (one stage, or the grid barrier after about a second) is reported by
 * bqg_last_device_error. */
int bqg_decode_layer_q4_0_q8_1(const void *xa, const void *xb, int x_dtype, const void *Wq, const void *Wk,
                               const void *Wv, const void *Wg, const void *Wu, const void *Wd, float *Yq, float *Yk,
                               float *Yv, float *Y, int M, int64_t Nq, int64_t Nkv, int64_t Nff, int64_t K, void *ws,
                               size_t ws_bytes, cudaStream_t stream);

/* Prefill GEMM ("llama-3x-prompt-speed", "the tile"): each weight tile is
 * dequantized once to bf16 into the tensor memory the MMA reads and fed to
 * the tensor cores with fp32 accumulation.  For K >= 1024 each weight
 * (q-8)*d is rounded once to nearest-even bf16 (relative error <= 2^-9 per
 * weight); for K < 1024, where one large term can dominate a short sum and
 * that rounding could exceed the library's parity bound 1e-3 * sum|w x|,
 * each weight is written exactly as a sum of two bf16 terms, one MMA each.
 * Wp: repacked q4_0 N x K; X: M x K bf16; Y: M x N fp32.
 * M a positive multiple of 128, N a multiple of 128, K a multiple of 64.
 * The kernel's shared-memory limit is raised once per process, on the
 * device current at the first call of each weight format and K range: a
 * process that calls the GEMM on a second device gets BQG_ERR_CUDA there
 * (nothing is launched). */
int bqg_gemm_q4_0_bf16(const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K,
                       void *ws, size_t ws_bytes, cudaStream_t stream);

/* The same prefill GEMM with q8_0 weights (the q8_0 tile of
 * "llama-3x-prompt-speed", "the free 2x"): q * d rounded to nearest-even
 * bf16 for K >= 1024, and for K < 1024 written exactly as three bf16 terms
 * (an 8-bit code times an fp16 scale has up to 19 significant bits).
 * Wp: repacked q8_0 N x K; other arguments as bqg_gemm_q4_0_bf16. */
int bqg_gemm_q8_0_bf16(const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K,
                       void *ws, size_t ws_bytes, cudaStream_t stream);

/* Check export: the exact per-block integer dots
 *     dots[n, b] = sum_{i<32} (qw[n, 32b+i] - 8) * qx[32b+i]
 * of q4_0 x q8_1 for one activation row (the integer-dot Q4_0 x Q8_1
 * matvec of "rx-6700xt-llama2-decode", Approach & Methodology), exactly as
 * bqg_gemv_q4_0_q8_1 computes them at M = 1 on this device: a check
 * instantiation of the GEMV's own kernel for the plan that call would use
 * (same staging of the activation row, same weight stream and dot routine;
 * it writes the dots instead of the outputs), or, for the shapes that call
 * serves with the K-slice kernel, that kernel's routine.
 * Wp: repacked q4_0 N x K; Xq: K/32 q8_1 blocks (4-byte alignment is
 * enough); dots: N x K/32 int32, row-major (4-byte alignment).  |dot| <=
 * 32 * 8 * 127.  Errors as bqg_gemv_q4_0_q8_1. */
int bqg_debug_q4_0_q8_1_block_dots(const void *Wp, const void *Xq, int32_t *dots, int64_t N,
                                   int64_t K, cudaStream_t stream);

/* The same dots from the K-slice kernel's routine (q4_0_q8_1_sumi on the
 * operands as that kernel loads them), whatever the shape: the routine the
 * GEMV entry points use where the lanes-per-row kernel's staged
 * activations do not fit (for example M = 8 at K = 11008).  Arguments and
 * errors as bqg_debug_q4_0_q8_1_block_dots. */
int bqg_debug_q4_0_q8_1_block_dots_kslice(const void *Wp, const void *Xq, int32_t *dots, int64_t N,
                                          int64_t K, cudaStream_t stream);

/* ---- utilities -------------------------------------------------------- */

/* Workspace bytes that op needs for this shape on the current device
 * (0 = none).  For BQG_OP_QKV_Q4_0_Q8_1 pass N = Nq + 2*Nkv. */
size_t bqg_workspace_size(int op, int M, int64_t N, int64_t K);

/* Which kernel serves a GEMV call of this shape on the current device
 * (op: BQG_OP_GEMV_BF16, _Q8_0, _Q4_0 or _Q4_0_Q8_1): *route receives one
 * of the BQG_ROUTE_* values below.  No launch; the choice depends only on
 * the shape, the device and the BQG_* tuning variables.  Errors as the
 * GEMV entry points' shape checks. */
enum {
    BQG_ROUTE_K_SLICE = 0,                /* K-slice kernel (staged activations too large) */
    BQG_ROUTE_LANES_PER_ROW = 1,          /* lanes-per-row kernel, general form (split K) */
    BQG_ROUTE_LANES_PER_ROW_ROWS = 2,     /* lanes-per-row kernel, whole rows per stage */
    BQG_ROUTE_TENSOR_CORE = 3             /* tensor-core kernel (M = 4, 8 with bf16 activations, q4_0 x bf16 at M = 2,
                                             q4_0 x q8_1 at M = 8) */
};
int bqg_gemv_route(int op, int M, int64_t N, int64_t K, int *route);

/* Reads and clears this device's error word, which a bounded device-side
 * wait sets when it gives up (0 = none).  Synchronizes `stream` first.
 * Returns BQG_OK or BQG_ERR_CUDA; *out receives the word. */
int bqg_last_device_error(cudaStream_t stream, int *out);

/* ---- host memory on the coherent CPU-GPU link ------------------------- */

/* Device-side address of page-locked host memory (cudaHostAlloc,
 * cudaMallocHost, or cudaHostRegister with mapping); under unified
 * addressing it equals `host`.  Kernels that read or write it cross the
 * CPU-GPU link (NVLink-C2C on a Grace node) with no copy-engine transfer.
 * *dev receives the address.  BQG_ERR_INVALID_ARG for null arguments;
 * BQG_ERR_CUDA when the memory is not page-locked and mapped (nothing is
 * left pending on the CUDA runtime). */
int bqg_host_alias(const void *host, void **dev);

/* Copy `bytes` from src to dst with a kernel (the SMs) instead of a copy
 * engine: for moving an activation row in from, or a result out to, memory
 * named by bqg_host_alias, where a copy-engine transfer of a few KB costs
 * more in latency than the bytes.  Either pointer may be device memory or a
 * host alias.  Ordered on `stream` like any launch; with programmatic
 * dependent launch on (bqg_set_pdl) it waits for the previous kernel before
 * it reads or writes anything.  Both pointers 16-byte aligned and bytes a
 * multiple of 16 (BQG_ERR_MISALIGNED); the ranges must not overlap
 * (BQG_ERR_INVALID_ARG).  bytes = 0 launches nothing and accepts any
 * pointers (null included). */
int bqg_copy_sm(void *dst, const void *src, size_t bytes, cudaStream_t stream);

/* Programmatic dependent launch for the GEMV kernels (default off).
 * When on, a GEMV may start and begin streaming its weights while the
 * previous kernel on the stream finishes; it waits for that kernel before
 * reading X or writing Y.  Weights must not be written by a kernel that is
 * still running when the GEMV is enqueued.  Returns the previous setting. */
int bqg_set_pdl(int enable);

/* Name of the CUDA error behind the calling thread's last BQG_ERR_CUDA
 * ("no error" if there was none). */
const char *bqg_last_cuda_error(void);

/* Static description of a status code. */
const char *bqg_status_string(int status);

/* Library version, e.g. "bqgemv 0.1 sm_103a". */
const char *bqg_version(void);

#ifdef __cplusplus
}
#endif
#endif /* BQGEMV_H */
