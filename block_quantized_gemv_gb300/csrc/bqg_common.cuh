// bqg_common.cuh -- device helpers shared by the sm_103a kernels of libbqgemv.
//
// Block formats (32 elements per block) and the repacked weight layout are
// described in include/bqgemv.h.  Nothing here is shared with the CPU oracle.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "../../include/bqgemv.h"

namespace bqg {

constexpr int QK = 32;              // elements per block
constexpr int Q8_0_BYTES = 34;
constexpr int Q4_0_BYTES = 18;
constexpr int Q8_1_BYTES = 36;
constexpr int Q4_0_TILE = 576;      // 32 blocks: 512 B codes + 64 B scales
constexpr int Q8_0_TILE = 1088;     // 32 blocks: 1024 B codes + 64 B scales

// ---------------------------------------------------------------------------
// loads
// ---------------------------------------------------------------------------
// Weights are read exactly once per call: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ldg_stream_v4(const void *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_stream_u16(const void *p)
{
    unsigned short v;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg_v4(const void *p)
{
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// Warm L2 with a contiguous byte range (no data is consumed, so it is safe
// to issue before the previous grid on the stream has finished).
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Programmatic dependent launch: no-ops when the kernel was launched
// without the programmatic-serialization attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// mbarriers and bulk copies (shared memory staging)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Test the phase; if it is not complete the thread is suspended (not
// spinning) until it completes or about `suspend_ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t suspend_ns = 1000000u)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity), "r"(suspend_ns)
                 : "memory");
    return ok != 0;
}
// ~1 s at 2 GHz: no correct launch waits this long on one phase.
constexpr long long kWaitTimeoutCycles = 1ll << 31;
// Wait for the phase with the given parity; false if it did not complete in
// time.  Between failed tests the warp sleeps (backing off to ~0.5 us) so
// that waiting warps leave the issue slots to the warps doing work.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    unsigned ns = 32;
    while (!mbar_try_wait(bar, parity)) {
        __nanosleep(ns);
        ns = min(ns * 2, 512u);
        if (clock64() - t0 > kWaitTimeoutCycles) return false;
    }
    return true;
}
// Tight variant for short pipeline waits (a few hundred cycles): plain
// try_wait (hardware time limit), no sleep between tests; still bounded.
__device__ __forceinline__ bool mbar_try_wait_nohint(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait_nohint(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; i++)
            if (mbar_try_wait_nohint(bar, parity)) return true;
        if (clock64() - t0 > kWaitTimeoutCycles) return false;
    }
}

// Order this thread's generic-proxy shared-memory accesses before its later
// async-proxy ones (bulk copies, tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---------------------------------------------------------------------------
// q8 block encoding (one warp per 32-element block, lane i = element i):
// d = fp16_rn(amax / 127), q = round_half_away(x / d) in IEEE fp32, clamped
// to [-127, 127]; d == 0 gives q = 0.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ int warp_sum_int(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// q8 code of v given the stored scale d (as float)
__device__ __forceinline__ int q8_code(float v, float d)
{
    if (d == 0.0f) return 0;
    const float q = fminf(fmaxf(roundf(__fdiv_rn(v, d)), -127.0f), 127.0f);
    return (int)q;
}

// One q8_1 block (36 bytes at `out`, 4-byte aligned): fp16 d, fp16 s =
// fp16_rn(d * sum q), 32 int8 codes; `v` is this lane's element.
__device__ __forceinline__ void q8_1_encode_warp(float v, int lane, uint8_t *out)
{
    const float amax = warp_max(fabsf(v));
    const __half dh = __float2half_rn(__fdiv_rn(amax, 127.0f));
    const float d = __half2float(dh);
    const int q = q8_code(v, d);
    const int sum = warp_sum_int(q);
    out[4 + lane] = (uint8_t)(int8_t)q;
    if (lane == 0) {
        // d | s as one little-endian word
        const __half sh = __float2half_rn(d * (float)sum);   // exact product, one rounding
        const uint32_t db = __half_as_ushort(dh), sb = __half_as_ushort(sh);
        *reinterpret_cast<uint32_t *>(out) = db | (sb << 16);
    }
}

// Bulk copy global -> this CTA's shared memory, completing `bytes` on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// ---------------------------------------------------------------------------
// scalar conversions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// eight bf16 (16 bytes, element k in bits 16 (k & 1) of word k / 2) -> fp32
__device__ __forceinline__ void bf16x8_to_f32(const uint4 &v, float (&x)[8])
{
    x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xffff0000u);
    x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xffff0000u);
    x[4] = __uint_as_float(v.z << 16); x[5] = __uint_as_float(v.z & 0xffff0000u);
    x[6] = __uint_as_float(v.w << 16); x[7] = __uint_as_float(v.w & 0xffff0000u);
}

__device__ __forceinline__ float half_bits_to_float(uint32_t h)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// Byte j of `w` (an unsigned code u) as the exact float u + 2^23, built by
// placing u in the mantissa of 2^23 (one byte permute, no int->float unit).
template <int J>
__device__ __forceinline__ float byte_plus_2p23(uint32_t w)
{
    return __uint_as_float(__byte_perm(w, 0x4b000000u, J | (4 << 4) | (4 << 8) | (7 << 12)));
}

// ---------------------------------------------------------------------------
// packed fp32 pairs (sm_100+): one instruction for two lanes of work
// ---------------------------------------------------------------------------
// (d0, d1) += (a0, a1) * (b0, b1), each with one rounding
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rd, {%0, %1};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rd;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// (a0 + c, a1 + c) with one rounding each
// (a0, a1) *= (c, c), one packed instruction
__device__ __forceinline__ void fmul2(float &a0, float &a1, float c)
{
    asm("{\n\t.reg .b64 ra, rc;\n\t"
        "mov.b64 ra, {%0, %1};\n\t"
        "mov.b64 rc, {%2, %2};\n\t"
        "mul.rn.f32x2 ra, ra, rc;\n\t"
        "mov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(c));
}
__device__ __forceinline__ void fadd2(float &a0, float &a1, float c)
{
    asm("{\n\t.reg .b64 ra, rc;\n\t"
        "mov.b64 ra, {%0, %1};\n\t"
        "mov.b64 rc, {%2, %2};\n\t"
        "add.rn.f32x2 ra, ra, rc;\n\t"
        "mov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(c));
}

// ---------------------------------------------------------------------------
// warp reductions
// ---------------------------------------------------------------------------
// Reduce V values per lane over the 32 lanes of a warp by recursive halving:
// after log2(V) exchange steps each lane keeps one partial of index
// (lane >> (5 - log2 V)) & (V - 1), then a butterfly over the remaining lane
// bits completes it.  The full sum of value i ends in lane i << (5 - log2 V).
// V must be a power of two <= 32.  Cost: V - 1 + (5 - log2 V) shuffles.
template <int V>
struct WarpReduce {
    static constexpr int L = (V >= 32) ? 5 : (V >= 16) ? 4 : (V >= 8) ? 3 : (V >= 4) ? 2 : (V >= 2) ? 1 : 0;
    static_assert((1 << L) == V, "V must be a power of two <= 32");

    __device__ __forceinline__ static float run(float (&v)[V], int lane)
    {
#pragma unroll
        for (int step = 0; step < L; step++) {
            const int off = 16 >> step;
            const int half = V >> (step + 1);
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int j = 0; j < half; j++) {
                float send = upper ? v[j] : v[j + half];
                float keep = upper ? v[j + half] : v[j];
                v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
        }
        float s = v[0];
#pragma unroll
        for (int off = 16 >> L; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        return s;
    }
    __device__ __forceinline__ static int index_of_lane(int lane) { return (lane >> (5 - L)) & (V - 1); }
    __device__ __forceinline__ static int lane_of_index(int i) { return i << (5 - L); }
    __device__ __forceinline__ static bool is_holder(int lane) { return (lane & ((32 >> L) - 1)) == 0; }
};

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

}  // namespace bqg
