// bqg_noalloc.cu -- a q4_0 x q8_1 GEMV entry point that allocates nothing.
//
// Some callers cannot hand the library a workspace from cudaMalloc: a
// runtime whose memory plan is fixed when the model loads (an inference
// server that reserves the whole device for weights and KV cache up front),
// a latency-critical decode loop where an allocation may block or
// synchronize the device, or plain C code with no allocator of its own.
// For them this entry point takes its split-K scratch from a fixed array
// that lives in the library's device image instead.
#include <mutex>

#include "bqg_common.cuh"

namespace bqg {

// Scratch for the split-K partial sums: bqg_noalloc_scratch_bytes() bytes.
// Every device that loads the library holds this array until the process
// exits; every call shares it.
constexpr size_t kNoAllocScratchBytes = 32 * 1024;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64] = {};
bool g_noalloc_ready[64] = {};

// Device address of the scratch array on the current device.  The host-side
// name of the array is only a stand-in, so the address is looked up once per
// device with that device current.
int noalloc_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BQG_ERR_CUDA;
    if (dev < 0 || dev >= 64) return BQG_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ready[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return BQG_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
        g_noalloc_ready[dev] = true;
    }
    *out = g_noalloc_ptr[dev];
    return BQG_OK;
}
}  // namespace

}  // namespace bqg

extern "C" {

size_t bqg_noalloc_scratch_bytes(void) { return bqg::kNoAllocScratchBytes; }

int bqg_gemv_q4_0_q8_1_noalloc(const void *Wp, const void *Xq, float *Y, int M, int64_t N, int64_t K,
                               cudaStream_t stream)
{
    if (!Wp || !Xq || !Y || N < 0) return BQG_ERR_INVALID_ARG;
    if (M != 1 && M != 2 && M != 4 && M != 8) return BQG_ERR_INVALID_ARG;
    if (K <= 0 || K % 32) return BQG_ERR_UNSUPPORTED_SHAPE;
    void *scratch = nullptr;
    if (int st = bqg::noalloc_scratch(&scratch)) return st;
    // the shape's split-K partials must fit the fixed array
    const size_t need = bqg_workspace_size(BQG_OP_GEMV_Q4_0_Q8_1, M, N, K);
    if (need > bqg::kNoAllocScratchBytes) return BQG_ERR_WORKSPACE;
    return bqg_gemv_q4_0_q8_1(Wp, Xq, Y, M, N, K, scratch, bqg::kNoAllocScratchBytes, stream);
}

}  // extern "C"
