// bqg_layer.cu -- one decode layer's three projection groups in one persistent launch.
//
// "MI50 megakernel" (the hypothesis ledger: fusing neighbouring steps into
// one dispatch, a grid-wide barrier between dependent steps) and "rx-6700xt-
// llama2-decode" (the q4_0 x q8_1 matvec, the fused QKV and gate+up/SwiGLU
// dispatches), for M = 1:
//
//   phase 1 (no dependency between its parts):
//     CTAs [0, cq)     : qkv = W_{q,k,v} . q8_1(xa)              (three outputs)
//     CTAs [cq, grid)  : h   = silu(Wg . q8_1(xb)) * (Wu . q8_1(xb)),
//                        written as q8_1 blocks hq (the SwiGLU -> q8_1 epilogue)
//   grid barrier (bounded wait)
//   phase 2          : y   = Wd . hq                              (every CTA)
//
// Each CTA encodes its own activation row into q8_1 in shared memory with
// the encoder of bqg_quantize_q8_1 (the same bytes), so the layer is one
// launch.  The CTA is the lanes-per-row GEMV of bqg_gemv.cuh with one slot
// per warp: each warp streams groups of RL rows (group g of the CTA to warp
// g mod NW).  A warp requests its first down-projection stage as soon as its
// last phase-1 stage is consumed, before the grid barrier (the weights do
// not depend on h), so most of phase 2's weights are in shared memory when
// the barrier opens.  Every wait is bounded; on a timeout the kernel sets
// its error word, stops issuing copies and waits (bounded) for the ones in
// flight before it exits.
#include "bqg_gemv.cuh"

namespace bqg {

static __device__ int g_layer_error;

constexpr int kLayerRL1 = 2;   // phase 1: a gate/up group is one (gate, up) pair; qkv pairs of rows
constexpr int kLayerRL2 = 1;   // phase 2: long rows (K = Nff), one per group

__device__ __forceinline__ float layer_load_act(const void *x, int x_f32, int64_t i)
{
    if (x_f32) return reinterpret_cast<const float *>(x)[i];
    const uint16_t b = reinterpret_cast<const uint16_t *>(x)[i];
    return __uint_as_float((uint32_t)b << 16);
}

// Virtual rows [v0, v1) of part `cta` of `ncta` (in pairs when gate and up
// rows alternate).
__device__ __forceinline__ void layer_rows(const GemvParams &p, int cta, int ncta, int64_t &v0, int64_t &v1)
{
    const int64_t unit = (p.nmat == 2) ? 2 : 1;
    const int64_t units = p.Nv / unit;
    v0 = (int64_t)cta * units / ncta * unit;
    v1 = (int64_t)(cta + 1) * units / ncta * unit;
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier of the cooperative launch on one 64-bit word in the
// workspace: generation in the high half, arrivals in the low half.  A CTA
// arrives with one atomic add, which also returns the generation it arrived
// in; the last arrival resets the count and advances the generation with
// one more add; the others wait (bounded) for the generation to change.
// The CTA's earlier global writes are ordered before its arrival by the CTA
// barrier and a fence of the arriving thread.  False on a timeout.
__device__ bool layer_grid_barrier(unsigned long long *gbar, unsigned nctas, int *s_flag)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        bool ok = true;
        __threadfence();
        const unsigned long long old = atomicAdd(gbar, 1ull);
        const unsigned g0 = (unsigned)(old >> 32);
        if ((unsigned)old + 1u == nctas) {
            __threadfence();
            atomicAdd(gbar, (1ull << 32) - nctas);
        } else {
            const long long t0 = clock64();
            while ((unsigned)(ld_acquire_gpu_u64(gbar) >> 32) == g0) {
                __nanosleep(32);
                if (clock64() - t0 > kWaitTimeoutCycles) { ok = false; break; }
            }
        }
        __threadfence();
        *s_flag = ok ? 1 : 0;
    }
    __syncthreads();
    return *reinterpret_cast<volatile int *>(s_flag) != 0;
}

// q8_1 blocks of the XB values each lane holds (block j is this warp's
// j-th block), with the steps of q8_1_encode_warp taken for all blocks at
// once so that their reductions and divisions overlap; the same bytes.
template <int XB>
__device__ __forceinline__ void q8_1_encode_warp_batch(const float (&v)[XB], int lane, int warp, int nwarps, int nb,
                                                       uint8_t *out)
{
    float a[XB];
#pragma unroll
    for (int j = 0; j < XB; j++) a[j] = fabsf(v[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int j = 0; j < XB; j++) a[j] = fmaxf(a[j], __shfl_xor_sync(0xffffffffu, a[j], o));
    uint32_t dbits[XB];
    int q[XB], sm[XB];
#pragma unroll
    for (int j = 0; j < XB; j++) {
        const __half dh = __float2half_rn(__fdiv_rn(a[j], 127.0f));
        dbits[j] = __half_as_ushort(dh);
        q[j] = q8_code(v[j], __half2float(dh));
        sm[j] = q[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int j = 0; j < XB; j++) sm[j] += __shfl_xor_sync(0xffffffffu, sm[j], o);
#pragma unroll
    for (int j = 0; j < XB; j++) {
        const int b = warp + j * nwarps;
        if (b >= nb) continue;
        uint8_t *blk = out + (size_t)b * Q8_1_BYTES;
        blk[4 + lane] = (uint8_t)(int8_t)q[j];
        if (lane == 0) {
            const float d = __half2float(__ushort_as_half((unsigned short)dbits[j]));
            const __half sh = __float2half_rn(d * (float)sm[j]);   // exact product, one rounding
            *reinterpret_cast<uint32_t *>(blk) = dbits[j] | ((uint32_t)__half_as_ushort(sh) << 16);
        }
    }
}

// One stage of a phase: the RL virtual rows from vs (those below v1), whole
// rows, one bulk copy per run of consecutive rows of one matrix.
template <int RL>
__device__ __forceinline__ void layer_issue(const GemvParams &p, uint32_t slot, uint32_t bar, int64_t vs, int64_t v1)
{
    issue_stage<W_Q4_0>(p, slot, bar, vs, RL, v1, 0, p.row_bytes);
}

// This warp's groups of RL rows of [v0, v1) (group g to warp g mod NW),
// streamed through its one slot.  The warp's first group was requested
// before the call (pending); each later one is requested as soon as the
// previous one has been read.  SWIGLU: a group is one (gate, up) pair and the
// output h = silu(g) * u goes to the fp32 staging row p.Y[0]; else every row
// goes to its matrix's output.  ok turns false (warp-uniform) when a wait
// gives up; the warp then does no more work.
template <int RL, bool SWIGLU>
__device__ __forceinline__ void layer_phase(const GemvParams &p, int64_t v0, int64_t v1, int warp, int NW, int lane,
                                            const uint8_t *slot_ptr, uint32_t slot, uint32_t bar, uint32_t &ph,
                                            bool &pending, const uint8_t *xs, bool &ok)
{
    constexpr int CPT = TileTraits<W_Q4_0>::CPT;
    const int nt = (p.nc + CPT - 1) / CPT;
    const int tail = min(32, p.nb - 32 * (nt - 1));
    const int ds_off = ((p.nc + 31) / 32) * XPieces<W_Q4_0, X_Q8_1>::P * 512;
    const int ng = (int)((v1 - v0 + RL - 1) / RL);
    for (int g = warp; g < ng; g += NW) {
        const int64_t vs = v0 + (int64_t)g * RL;
        if (ok) {
            const bool w = mbar_wait_bounded(bar, ph);
            ok = __all_sync(0xffffffffu, w);
            if (ok) {
                pending = false;
                ph ^= 1;
            } else if (lane == 0) {
                atomicExch(&g_layer_error, 1);
            }
        }
        if (!ok) continue;
        float acc[RL][1][2];
#pragma unroll
        for (int i = 0; i < RL; i++) acc[i][0][0] = acc[i][0][1] = 0.f;
        lpr_tiles<W_Q4_0, X_Q8_1, 1, RL>(acc, slot_ptr, p.row_stride, xs, p.x_row_bytes, ds_off, 0, nt, tail, lane);
        // the warp is done with its slot: request its next group
        __syncwarp();
        if (lane == 0 && g + NW < ng) {
            fence_proxy_async_smem();
            layer_issue<RL>(p, slot, bar, vs + (int64_t)NW * RL, v1);
            pending = true;
        }
        float tot[RL];
#pragma unroll
        for (int i = 0; i < RL; i++) {
            float a = acc[i][0][0] + acc[i][0][1];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
            tot[i] = a;
        }
        if (lane != 0) continue;
        if constexpr (SWIGLU) {
            p.Y[0][staged_vrow(p, vs, RL, 0) >> 1] = silu(tot[0]) * tot[RL - 1];
        } else {
#pragma unroll
            for (int i = 0; i < RL; i++) {
                const int64_t v = staged_vrow(p, vs, RL, i);
                if (v >= v1) continue;
                int mat; int64_t rr;
                map_row(p, v, mat, rr);
                p.Y[mat][rr] = tot[i];
            }
        }
    }
}

__global__ void __launch_bounds__(384, 2) decode_layer_kernel(const LayerParams lp)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_flag;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int NW = blockDim.x >> 5;
    const bool is_qkv = (int)blockIdx.x < lp.cq;
    const int cta1 = is_qkv ? (int)blockIdx.x : (int)blockIdx.x - lp.cq;
    const int n1 = is_qkv ? lp.cq : (int)gridDim.x - lp.cq;
    const uint8_t *slot_ptr = smem + (size_t)warp * lp.slot_bytes;
    const uint32_t slot = smem_u32(slot_ptr);
    const uint32_t bar = smem_u32(smem + lp.bar_off) + 8 * warp;
    uint8_t *xs = smem + lp.x_off;
    uint8_t *xraw = smem + lp.xraw_off;
    const uint32_t xbar = smem_u32(smem + lp.bar_off) + 8 * NW;   // phase 2's activation copy

    // this CTA's activation row, loaded before any weight copy is requested
    // (lane l of warp w holds element l of blocks w, w + NW, ...) so that the
    // loads do not wait behind the weight stream
    constexpr int XB = 12;                         // blocks per lane held at once
    const void *x = is_qkv ? lp.xa : lp.xb;
    const int nb1 = lp.qkv.nb;
    float xv[XB];
#pragma unroll
    for (int j = 0; j < XB; j++) {
        const int b = warp + j * NW;
        xv[j] = (b < nb1) ? layer_load_act(x, lp.x_f32, (int64_t)b * QK + lane) : 0.f;
    }

    if (lane == 0) {
        mbar_init(bar, 1);                         // lane 0's arrive + bytes
        if (warp == 0) mbar_init(xbar, 1);
        mbar_fence_init();
    }
    __syncthreads();

    int64_t a0, a1, d0, d1;
    if (is_qkv) layer_rows(lp.qkv, cta1, n1, a0, a1);
    else layer_rows(lp.gu, cta1, n1, a0, a1);
    layer_rows(lp.dn, blockIdx.x, gridDim.x, d0, d1);
    uint32_t ph = 0;
    bool pending = false, ok = true;

    // the warp's first phase-1 stage: weights depend on nothing
    if (lane == 0 && (int64_t)warp * kLayerRL1 < a1 - a0) {
        if (is_qkv) layer_issue<kLayerRL1>(lp.qkv, slot, bar, a0 + (int64_t)warp * kLayerRL1, a1);
        else layer_issue<kLayerRL1>(lp.gu, slot, bar, a0 + (int64_t)warp * kLayerRL1, a1);
        pending = true;
    }

    // the activation row as q8_1 blocks (the encoder of bqg_quantize_q8_1),
    // then in the staged layout (qkv and gate/up share K)
    q8_1_encode_warp_batch<XB>(xv, lane, warp, NW, nb1, xraw);
    for (int b = warp + XB * NW; b < nb1; b += NW)     // rows longer than XB * NW blocks
        q8_1_encode_warp(layer_load_act(x, lp.x_f32, (int64_t)b * QK + lane), lane, xraw + (size_t)b * Q8_1_BYTES);
    __syncthreads();
    expand_x<W_Q4_0, X_Q8_1>(lp.qkv, xraw, xs, 1, tid, blockDim.x);
    __syncthreads();

    if (is_qkv)
        layer_phase<kLayerRL1, false>(lp.qkv, a0, a1, warp, NW, lane, slot_ptr, slot, bar, ph, pending, xs, ok);
    else
        layer_phase<kLayerRL1, true>(lp.gu, a0, a1, warp, NW, lane, slot_ptr, slot, bar, ph, pending, xs, ok);

    // the warp's first down-projection stage, into its now free slot
    __syncwarp();
    if (lane == 0 && ok && (int64_t)warp * kLayerRL2 < d1 - d0) {
        fence_proxy_async_smem();
        layer_issue<kLayerRL2>(lp.dn, slot, bar, d0 + (int64_t)warp * kLayerRL2, d1);
        pending = true;
    }

    // h of this CTA's outputs as q8_1 blocks (counted arrivals per block)
    if (!is_qkv) swiglu_q8_1_finish(lp.gu, 1, a0 >> 1, a1 >> 1, 1, warp, NW, lane);

    const bool gok = layer_grid_barrier(lp.gbar, gridDim.x, &s_flag);
    if (!gok) {
        if (tid == 0) atomicExch(&g_layer_error, 1);
        ok = false;
    }
    // h's q8_1 blocks in one bulk copy (written by other CTAs through the
    // generic proxy; the barrier's acquire, then a proxy fence, order them
    // before this async-proxy read), then in the staged layout
    bool xok = gok;
    if (gok) {
        // rounded up to 16 bytes: the workspace pads h's blocks to 16, and
        // the raw area holds that much
        const uint32_t bytes = ((uint32_t)lp.dn.nb * Q8_1_BYTES + 15u) & ~15u;
        if (tid == 0) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            mbar_arrive_expect_tx(xbar, bytes);
            bulk_g2s(smem_u32(xraw), lp.dn.X, bytes, xbar);
        }
        xok = mbar_wait_bounded(xbar, 0);
        if (!xok) {
            if (lane == 0) atomicExch(&g_layer_error, 1);
            ok = false;
        }
        if (xok) expand_x<W_Q4_0, X_Q8_1>(lp.dn, xraw, xs, 1, tid, blockDim.x);
    }
    __syncthreads();
    ok = ok && xok;
    layer_phase<kLayerRL2, false>(lp.dn, d0, d1, warp, NW, lane, slot_ptr, slot, bar, ph, pending, xs, ok);

    // after a timeout: do not leave while this warp's copy is in flight
    if (lane == 0 && pending) mbar_wait_bounded(bar, ph);
    if (tid == 0 && gok && !xok) mbar_wait_bounded(xbar, 0);
}

cudaError_t layer_occupancy(int threads, size_t smem, int *bpsm)
{
    int dev = 0, optin = 0;
    cudaFuncAttributes fa;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, decode_layer_kernel);
    if (e == cudaSuccess && smem + fa.sharedSizeBytes > (size_t)optin) return cudaErrorInvalidValue;
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(bpsm, decode_layer_kernel, threads, smem);
}

// A cooperative launch: the runtime refuses it unless every CTA can be
// resident at once, which the grid barrier needs.
cudaError_t layer_launch(const LayerParams &lp, int grid, int threads, size_t smem, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_layer_kernel, lp);
}

// Reads and clears this translation unit's error words.
cudaError_t layer_take_error(int *out)
{
    int a = 0, b = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&a, g_layer_error, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&b, g_gemv_error, sizeof(int));
    if (e != cudaSuccess) return e;
    *out = a | b;
    if (a) e = cudaMemcpyToSymbol(g_layer_error, &zero, sizeof(int));
    if (e == cudaSuccess && b) e = cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(int));
    return e;
}

}  // namespace bqg
