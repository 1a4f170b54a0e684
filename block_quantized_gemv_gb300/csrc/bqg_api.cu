// bqg_api.cu -- the C ABI of libbqgemv: argument validation, launch planning
// and dispatch.  Declarations and contracts: include/bqgemv.h.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <cmath>
#include <mutex>
#include <tuple>

#include <cudaTypedefs.h>

#include "bqg_gemv.cuh"
#include "bqg_gemv_mma.cuh"

namespace bqg {
cudaError_t gemv_run_bf16(const GemvParams &, int, int, dim3, int, size_t, cudaStream_t, bool, int *);
cudaError_t gemv_run_q8_0(const GemvParams &, int, int, dim3, int, size_t, cudaStream_t, bool, int *);
cudaError_t gemv_run_q4_0(const GemvParams &, int, int, dim3, int, size_t, cudaStream_t, bool, int *);
cudaError_t gemv_run_q4_0_q8_1(const GemvParams &, int, int, dim3, int, size_t, cudaStream_t, bool, int *);
cudaError_t gemv_error_bf16(int *);
cudaError_t gemv_error_q8_0(int *);
cudaError_t gemv_error_q4_0(int *);
cudaError_t gemv_error_q4_0_q8_1(int *);
cudaError_t gemv_lpr_run_bf16(const GemvParams &, int, dim3, int, size_t, cudaStream_t, bool, int *);
cudaError_t gemv_lpr_run_q8_0(const GemvParams &, int, dim3, int, size_t, cudaStream_t, bool, int *);
cudaError_t gemv_lpr_run_q4_0(const GemvParams &, int, dim3, int, size_t, cudaStream_t, bool, int *);
cudaError_t gemv_lpr_run_q4_0_q8_1(const GemvParams &, int, dim3, int, size_t, cudaStream_t, bool, int *);
cudaError_t gemv_lpr_dots_run_q4_0_q8_1(const GemvParams &, dim3, int, size_t, cudaStream_t, int *);
using MmaFn = cudaError_t (*)(const CUtensorMap &, const CUtensorMap &, const MmaParams &, int, dim3, int, size_t, cudaStream_t, bool, int *);
cudaError_t gemv_mma_run_bf16(const CUtensorMap &, const CUtensorMap &, const MmaParams &, int, dim3, int, size_t, cudaStream_t, bool, int *);
cudaError_t gemv_mma_run_q8_0(const CUtensorMap &, const CUtensorMap &, const MmaParams &, int, dim3, int, size_t, cudaStream_t, bool, int *);
cudaError_t gemv_mma_run_q4_0(const CUtensorMap &, const CUtensorMap &, const MmaParams &, int, dim3, int, size_t, cudaStream_t, bool, int *);
cudaError_t gemv_mma_run_q4_0_q8_1(const CUtensorMap &, const CUtensorMap &, const MmaParams &, int, dim3, int, size_t, cudaStream_t, bool, int *);
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
int gemv_x_stage_bytes_bf16(int, int, int);
int gemv_x_stage_bytes_q8_0(int, int, int);
int gemv_x_stage_bytes_q4_0(int, int, int);
int gemv_x_stage_bytes_q4_0_q8_1(int, int, int);
cudaError_t layer_occupancy(int threads, size_t smem, int *bpsm);
cudaError_t layer_launch(const LayerParams &lp, int grid, int threads, size_t smem, cudaStream_t stream);
cudaError_t layer_take_error(int *out);
cudaError_t launch_quantize_q8_1(const void *, int, void *, int, int64_t, cudaStream_t, bool);
cudaError_t launch_rmsnorm_q8_1(const void *, int, const float *, float, void *, int, int64_t, cudaStream_t, bool);
cudaError_t launch_quantize_weights(int, const float *, void *, int64_t, int64_t, cudaStream_t);
cudaError_t launch_repack(int, const void *, void *, int64_t, int64_t, cudaStream_t);
cudaError_t launch_block_dots(const void *, const void *, int32_t *, int64_t, int64_t, int64_t, cudaStream_t);
cudaError_t launch_copy_sm(void *, const void *, int64_t, int, cudaStream_t, bool);
cudaError_t launch_splitk_reduce(const GemvParams &, int, int, int, cudaStream_t, bool);
int gemm_bf16(int, const void *, const void *, float *, int, int64_t, int64_t, cudaStream_t, int);
size_t gemm_workspace(int, int64_t, int64_t);
int gemm_read_error(cudaStream_t, int *);
}  // namespace bqg

using namespace bqg;

namespace {

std::atomic<int> g_pdl{0};
thread_local cudaError_t t_last_cuda = cudaSuccess;

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return BQG_OK;
    t_last_cuda = e;
    return BQG_ERR_CUDA;
}


struct DevInfo {
    bool init = false;
    bool ok = false;
    int sms = 0;
};
std::mutex g_mu;
DevInfo g_dev[64];
std::map<std::tuple<int, int, int, int, int, int, int, size_t>, int> g_occ;

// Current device, checked to be sm_103.
int current_device(DevInfo *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BQG_ERR_CUDA;
    if (dev < 0 || dev >= 64) return BQG_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo &d = g_dev[dev];
    if (!d.init) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return BQG_ERR_CUDA;
        d.ok = (major == 10 && minor == 3);
        d.sms = sms;
        d.init = true;
    }
    *out = d;
    return d.ok ? BQG_OK : BQG_ERR_UNSUPPORTED_DEVICE;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool valid_m(int M) { return M == 1 || M == 2 || M == 4 || M == 8; }

int64_t repacked_row_bytes(int fmt, int64_t K)
{
    const int64_t nb = K / QK, T = (nb + 31) / 32;
    if (fmt == BQG_BF16) return 2 * K;
    if (fmt == BQG_Q4_0) return T * Q4_0_TILE;
    if (fmt == BQG_Q8_0) return T * Q8_0_TILE;
    return 0;
}

// chunk index space of one row (include/bqgemv.h layout, one 16-byte code load per chunk)
int chunk_space(int wf, int64_t K)
{
    const int64_t nb = K / QK, T = (nb + 31) / 32;
    if (wf == W_BF16) return (int)(K / 8);
    if (wf == W_Q8_0) return (int)(64 * T);
    return (int)nb;
}

using RunFn = cudaError_t (*)(const GemvParams &, int, int, dim3, int, size_t, cudaStream_t, bool, int *);
RunFn runner(int wf, int xf)
{
    if (xf == X_Q8_1) return gemv_run_q4_0_q8_1;
    if (wf == W_BF16) return gemv_run_bf16;
    if (wf == W_Q8_0) return gemv_run_q8_0;
    return gemv_run_q4_0;
}

using LprFn = cudaError_t (*)(const GemvParams &, int, dim3, int, size_t, cudaStream_t, bool, int *);
LprFn lpr_runner(int wf, int xf)
{
    if (xf == X_Q8_1) return gemv_lpr_run_q4_0_q8_1;
    if (wf == W_BF16) return gemv_lpr_run_bf16;
    if (wf == W_Q8_0) return gemv_lpr_run_q8_0;
    return gemv_lpr_run_q4_0;
}
// staged bytes of one activation row (bf16 rows staged as bf16 when bf16 != 0, else fp32)
int x_stage_bytes(int wf, int xf, int nc, int nb, int bf16)
{
    if (xf == X_Q8_1) return gemv_x_stage_bytes_q4_0_q8_1(nc, nb, 0);
    if (wf == W_BF16) return gemv_x_stage_bytes_bf16(nc, nb, bf16);
    if (wf == W_Q8_0) return gemv_x_stage_bytes_q8_0(nc, nb, bf16);
    return gemv_x_stage_bytes_q4_0(nc, nb, bf16);
}

struct GemvPlan {
    bool lpr;               // lanes-per-row kernel
    bool x_bf16s;           // bf16 activations staged as bf16 (M = 1 as well)
    int L, x_off, x_row_bytes, xraw_off, early, rl, piece_chunks, wg, ng;
    int C, TPR, RG, RPS, nc, cps, splits, threads, ncons, S, NS, stride, win_stages, part_off, bar_off, ctas;
    dim3 grid;
    size_t smem, ws_bytes;
};

constexpr int kMaxK = 65536;
constexpr int kLprMaxWarps = 12;       // the lanes-per-row kernel's launch bound: 384 threads
// Staged weights per CTA.  Two CTAs per SM stream a GEMV; when one of them
// finishes, the next GEMV's CTA takes its place and starts its own weight
// stream while the other drains (programmatic dependent launch).
constexpr int kStageBudget = 100 * 1024;

// Tuning knobs read once from the environment (unset = defaults above):
//   BQG_STAGE_KB     staged-weight budget per CTA in KiB
//   BQG_CTAS_PER_SM  cap on resident GEMV CTAs per SM (1 or 2)
//   BQG_LPR_KB, BQG_LPR_OVERLAP_KB, BQG_OVERLAP_SHARE_KB, BQG_LPR_L, BQG_LPR_D,
//   BQG_LPR_EARLY, BQG_LPR_RL, BQG_LPR_PIECE, BQG_LPR_STAGE_KB
//                    lanes-per-row geometry (see plan_lpr)
//   BQG_NO_LPR       1: serve every M with the K-slice kernel
int env_int(const char *name, int dflt)
{
    const char *v = getenv(name);
    return (v && *v) ? atoi(v) : dflt;
}
int stage_budget()
{
    static const int b = std::max(16, std::min(200, env_int("BQG_STAGE_KB", kStageBudget / 1024))) * 1024;
    return b;
}
int ctas_per_sm_cap()
{
    static const int c = std::max(1, std::min(2, env_int("BQG_CTAS_PER_SM", 2)));
    return c;
}

// Bytes of a row holding chunks [0, cps) in the repacked layout.
int64_t range_bytes(int wf, int cps)
{
    if (wf == W_BF16) return 16ll * cps;
    const int per_tile = (wf == W_Q8_0) ? 64 : 32;
    const int64_t tb = (wf == W_Q8_0) ? Q8_0_TILE : Q4_0_TILE;
    return (int64_t)((cps + per_tile - 1) / per_tile) * tb;
}

// Launch geometry for Nv virtual rows.  `unit` = 2 keeps (gate, up) pairs
// in one CTA.  Returns a status.
int plan_gemv(int wf, int xf, int M, int64_t Nv, int64_t K, int unit, const DevInfo &dev, int device,
              GemvPlan *pl)
{
    GemvPlan g{};
    g.nc = chunk_space(wf, K);
    g.RPS = (M == 8) ? 1 : 4 / M;
    const int align = (wf == W_Q8_0) ? 64 : 32;        // splits start on whole tiles
    const int maxs = std::max(1, std::min(16, g.nc / std::max(align, 64)));
    // Split K when there are too few rows to give every SM a few stages of
    // work, or when a staged row would not leave room for two stages.
    g.splits = 1;
    if (Nv < (int64_t)dev.sms * 4)
        g.splits = (int)std::min<int64_t>(maxs, ((int64_t)dev.sms * 4 + Nv - 1) / std::max<int64_t>(Nv, 1));
    for (;;) {
        g.cps = g.nc;
        if (g.splits > 1) {
            g.cps = ((g.nc + g.splits - 1) / g.splits + align - 1) / align * align;
            g.splits = (g.nc + g.cps - 1) / g.cps;
        }
        g.C = 1;
        while ((g.cps + g.C - 1) / g.C > 512 && g.C < 4) g.C *= 2;
        g.TPR = ((g.cps + g.C - 1) / g.C + 31) / 32 * 32;
        // row groups per CTA: at most 512 consumer threads, and few enough rows
        // per stage that at least four stages fit the budget
        g.RG = std::max(1, std::min(std::min(8, 512 / g.TPR),
                                    (int)(stage_budget() / (4ll * g.RPS * range_bytes(wf, g.cps)))));
        // a stage is SUB passes of RG x RPS rows; gate/up stages need an even row count
        g.S = g.RG * g.RPS * ((unit == 2 && (g.RG * g.RPS) % 2) ? 2 : 1);
        g.stride = (int)range_bytes(wf, g.cps);
        const bool fits = (g.cps + g.C - 1) / g.C <= 512 && 2ll * g.S * g.stride <= 2 * stage_budget();
        if (fits) break;
        if (g.splits >= maxs) return BQG_ERR_UNSUPPORTED_SHAPE;
        g.splits++;
    }
    g.ncons = g.RG * g.TPR;
    g.threads = g.ncons + 32;
    g.NS = (int)std::max<int64_t>(2, std::min<int64_t>(8, stage_budget() / ((int64_t)g.S * g.stride)));
    const int WPG = g.TPR / 32;
    g.win_stages = std::max(1, (64 + g.S - 1) / g.S);
    g.part_off = g.NS * g.S * g.stride;
    const int part_bytes = g.win_stages * g.S * WPG * M * (int)sizeof(float);
    g.bar_off = (g.part_off + part_bytes + 15) / 16 * 16;
    g.smem = (size_t)g.bar_off + 16 * g.NS;
    if (g.smem > 232448) return BQG_ERR_UNSUPPORTED_SHAPE;

    int bpsm = 0;
    {
        auto key = std::make_tuple(device, wf, xf, M, g.C, g.threads, 0, g.smem);
        std::unique_lock<std::mutex> lk(g_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) {
            bpsm = it->second;
        } else {
            lk.unlock();
            GemvParams dummy{};
            const cudaError_t e = runner(wf, xf)(dummy, M, g.C, dim3(1), g.threads, g.smem, 0, false, &bpsm);
            if (e != cudaSuccess) return cuda_status(e);
            lk.lock();
            g_occ[key] = bpsm;
        }
    }
    if (bpsm < 1) return BQG_ERR_UNSUPPORTED_SHAPE;
    bpsm = std::min(bpsm, ctas_per_sm_cap());
    const int64_t units = Nv / unit;
    const int64_t want = ((int64_t)dev.sms * bpsm + g.splits - 1) / g.splits;
    g.ctas = (int)std::max<int64_t>(1, std::min(units, want));
    g.grid = dim3((unsigned)g.ctas, (unsigned)g.splits);
    g.ws_bytes = (g.splits > 1) ? (size_t)g.splits * M * Nv * sizeof(float) : 0;
    *pl = g;
    return BQG_OK;
}


// Launch geometry of the lanes-per-row kernel (M = 1, 2, 4, 8).  Returns
// BQG_ERR_UNSUPPORTED_SHAPE when the staged activations would not fit, in
// which case the K-slice kernel (plan_gemv) serves the call.
//
// Two CTAs per SM stream the call, each with about half of the SM's shared
// memory.  An optional "overlap" geometry (BQG_OVERLAP_SHARE_KB > 0: SMs
// whose weight share is at most that many KiB) keeps each CTA to a quarter
// of the SM so that the next call's CTAs can be resident while this call
// drains; measured on the decode shapes it loses more to the smaller
// per-CTA ring and warp count than it gains, so it is off by default.
int plan_lpr(int wf, int xf, int M, int64_t Nv, int64_t K, int unit, const DevInfo &dev, int device,
             GemvPlan *pl)
{
    if (M != 1 && M != 2 && M != 4 && M != 8) return BQG_ERR_UNSUPPORTED_SHAPE;
    static const bool off = env_int("BQG_NO_LPR", 0) != 0;
    if (off) return BQG_ERR_UNSUPPORTED_SHAPE;
    static const int big_kb = std::max(16, std::min(220, env_int("BQG_LPR_KB", 113)));
    static const int small_kb = std::max(16, std::min(110, env_int("BQG_LPR_OVERLAP_KB", 54)));
    static const int share_kb = env_int("BQG_OVERLAP_SHARE_KB", 0);       // measured: off
    static const int force_L = env_int("BQG_LPR_L", 0);
    static const int force_D = env_int("BQG_LPR_D", 0);
    static const int early = std::max(0, env_int("BQG_LPR_EARLY", 1));
    static const int force_rl = env_int("BQG_LPR_RL", 0);
    static const int force_pg = env_int("BQG_LPR_PIECE", 0);
    static const int max_stage_kb = std::max(1, env_int("BQG_LPR_STAGE_KB", 16));
    GemvPlan g{};
    g.lpr = true;
    g.nc = chunk_space(wf, K);
    const int nb = (int)(K / QK);
    const int align = (wf == W_Q8_0) ? 64 : 32;
    const int maxs = std::max(1, std::min(16, g.nc / std::max(align, 64)));
    g.splits = 1;
    if (Nv < (int64_t)dev.sms * 4)
        g.splits = (int)std::min<int64_t>(maxs, ((int64_t)dev.sms * 4 + Nv - 1) / std::max<int64_t>(Nv, 1));
    // bf16 activations at M = 4, 8 (fp32 rows would not fit) and, measured
    // faster for every weight format, at M = 1, 2 (half the shared-memory
    // reads per weight): rows staged as bf16, copied in place (no raw copy);
    // else staged rows plus their raw copy (the 16-byte-aligned span around
    // X: up to 15 bytes of slack on either side)
    static const int bf16x_m1 = env_int("BQG_LPR_BF16X", 1);
    const bool bf16s = xf == X_BF16 && (M >= 4 || bf16x_m1);
    g.x_bf16s = bf16s;
    g.x_row_bytes = (x_stage_bytes(wf, xf, g.nc, nb, bf16s ? 1 : 0) + 15) / 16 * 16;
    const int xraw = bf16s ? 0 : (int)((M * ((xf == X_Q8_1) ? (int64_t)nb * Q8_1_BYTES : K * 2) + 30) / 16 * 16);
    const int xbytes = M * g.x_row_bytes + xraw + 16;
    if (xbytes > 80 * 1024) return BQG_ERR_UNSUPPORTED_SHAPE;
    g.cps = g.nc;
    if (g.splits > 1) {
        g.cps = ((g.nc + g.splits - 1) / g.splits + align - 1) / align * align;
        g.splits = (g.nc + g.cps - 1) / g.cps;
    }
    g.stride = (int)range_bytes(wf, g.cps);          // bytes of a row's split range
    // A warp works on RL rows at a time with all 32 lanes (gate/up blocks
    // need an even RL); every activation load serves the RL rows.  The rows
    // stream in K-pieces of whole tiles: the whole split range when RL rows
    // of it fit in `max_stage` bytes, so that each stage is one bulk copy of
    // consecutive rows (the copy engine costs about as much per copy as per
    // few KiB moved).
    g.L = 32;
    // measured on the decode and sweep shapes: two rows per lane for q4_0
    // (q8_1 or bf16 activations) at M = 1 and for every format at M = 2, one
    // otherwise (q8_0 at M = 1 below)
    int rl = ((M == 1 && wf == W_Q4_0) || M == 2) ? 2 : 1;
    // q8_0 x bf16 at M = 1 (bf16-staged): two rows per lane (each activation
    // piece converted once for both rows), with one slot per warp when each
    // CTA has few rows (N = 4096: 13 per CTA) and two otherwise (measured at
    // N = 12288 / 14336 / 24576: 10.85 -> 10.51, 12.12 -> 11.29, 18.11 -> 17.03 us
    // against one row and two slots)
    const bool q8_m1 = bf16x_m1 && M == 1 && wf == W_Q8_0 && xf == X_BF16;
    const bool q8_m1_few = q8_m1 && Nv < (int64_t)dev.sms * 2 * 24;
    if (q8_m1) rl = 2;
    // (four rows per lane: instantiated for fp32- or q8_1-staged M = 1 only)
    if (force_rl == 1 || force_rl == 2 || (force_rl == 4 && M == 1 && !bf16s)) rl = force_rl;
    // M = 4, 8 (measured on the sweep shapes): two rows per lane, but one
    // for q8_0 at M = 8, whose dequant registers then spill
    if (force_rl == 0 && M >= 4) rl = (wf == W_Q8_0 && M == 8) ? 1 : 2;
    if (unit == 2 && (rl & 1)) rl = 2;
    g.rl = rl;
    g.wg = 1;
    g.S = rl;
    const int cpt = (wf == W_Q8_0) ? 64 : 32;                        // chunks per tile
    const int64_t tile_bytes = (wf == W_Q8_0) ? Q8_0_TILE : (wf == W_Q4_0) ? Q4_0_TILE : 512;
    const int64_t per_sm = Nv * (int64_t)g.stride * g.splits / std::max(1, dev.sms);
    const bool overlap = per_sm <= (int64_t)share_kb * 1024;
    const int64_t budget = (int64_t)(overlap ? small_kb : big_kb) * 1024 - xbytes - 1024;
    const int max_tiles = (g.cps + cpt - 1) / cpt;
    int ntile = (int)std::max<int64_t>(1, (int64_t)max_stage_kb * 1024 / ((int64_t)g.S * tile_bytes));
    ntile = std::min(ntile, max_tiles);
    if (force_pg > 0) ntile = std::min(force_pg, max_tiles);
    g.piece_chunks = ntile * cpt;
    g.stride = (int)range_bytes(wf, std::min(g.piece_chunks, g.cps));
    const int64_t stage = (int64_t)g.S * g.stride;
    if (budget < stage) return BQG_ERR_UNSUPPORTED_SHAPE;
    static const int force_warps = env_int("BQG_LPR_WARPS", 0);
    int max_warps = (overlap || M >= 4) ? 8 : kLprMaxWarps;         // M >= 4: the kernel's 256-thread bound
    if (force_warps >= 1) max_warps = std::min(max_warps, force_warps);
    const int slots = (int)std::min<int64_t>(64, budget / stage);
    int ng = std::max(1, std::min(max_warps, slots / 2));
    int D = std::max(1, slots / ng);
    // measured: at M = 1 q8_1 activations and q4_0 weights gain more from more
    // warps with one slot each than from double slots, bf16 and q8_0 weights
    // keep two; at M = 2 and 4 two slots per warp win by 1-4 % on the sweep
    // shape (q4_0 x bf16 at M = 2 excepted), at M = 8 one slot
    const bool two_slots_m24 = (M == 2 || M == 4) && !(M == 2 && wf == W_Q4_0 && xf == X_BF16);
    const bool one_slot = !two_slots_m24 && (xf == X_Q8_1 || M >= 2 || wf == W_Q4_0 || q8_m1_few);
    const int want_D = (force_D > 0) ? force_D : one_slot ? 1 : two_slots_m24 ? 2 : 0;
    if (want_D > 0) { D = want_D; ng = std::max(1, std::min(max_warps, slots / D)); }
    g.ng = ng;
    g.NS = D;
    g.TPR = 32 * g.ng;
    g.RG = 1;
    g.C = 1;
    g.ncons = g.TPR;
    g.threads = g.TPR;
    g.x_off = (int)(g.ng * (int64_t)D * stage);
    g.xraw_off = (g.x_off + M * g.x_row_bytes + 15) / 16 * 16;
    g.bar_off = (int)(g.xraw_off + xraw);
    g.smem = (size_t)g.bar_off + 8 * (g.ng * D + 1);
    g.early = std::min(D, early);
    if (g.smem > 232448) return BQG_ERR_UNSUPPORTED_SHAPE;

    int bpsm = 0;
    {
        auto key = std::make_tuple(device, wf, xf, M, g.rl, g.threads, 1, g.smem);
        std::unique_lock<std::mutex> lk(g_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) {
            bpsm = it->second;
        } else {
            lk.unlock();
            GemvParams dummy{};
            dummy.rl = g.rl;
            dummy.x_bf16s = g.x_bf16s ? 1 : 0;
            const cudaError_t e = lpr_runner(wf, xf)(dummy, M, dim3(1), g.threads, g.smem, 0, false, &bpsm);
            if (e != cudaSuccess) return cuda_status(e);
            lk.lock();
            g_occ[key] = bpsm;
        }
    }
    if (bpsm < 1) return BQG_ERR_UNSUPPORTED_SHAPE;
    bpsm = std::min(bpsm, ctas_per_sm_cap());
    const int64_t units = Nv / unit;
    const int64_t want = ((int64_t)dev.sms * bpsm + g.splits - 1) / g.splits;
    g.ctas = (int)std::max<int64_t>(1, std::min(units, want));
    g.grid = dim3((unsigned)g.ctas, (unsigned)g.splits);
    g.ws_bytes = (g.splits > 1) ? (size_t)g.splits * M * Nv * sizeof(float) : 0;
    *pl = g;
    return BQG_OK;
}

// The plan a GEMV call uses: lanes-per-row when it applies, else K-slice.
int plan_any(int wf, int xf, int M, int64_t Nv, int64_t K, int unit, const DevInfo &dev, int device, GemvPlan *g)
{
    int st = plan_lpr(wf, xf, M, Nv, K, unit, dev, device, g);
    if (st == BQG_OK) return st;
    if (st != BQG_ERR_UNSUPPORTED_SHAPE) return st;
    return plan_gemv(wf, xf, M, Nv, K, unit, dev, device, g);
}

// Common path of every GEMV entry point.
// Workspace of a SwiGLU call with a q8_1 output and no split-K: fp32 staging
// of the M x N outputs, then one int32 arrival counter per q8_1 block.
size_t swiglu_q8_1_staging(int M, int64_t N)
{
    return ((size_t)M * N * 4 + 15) / 16 * 16 + (size_t)M * (N / 32) * 4;
}

// Does the lanes-per-row plan fit gemv_lpr_rows_kernel: one matrix, no
// split of K, each stage whole rows, outputs stored as they are?
bool rows_kernel_applies(const GemvPlan &g, const GemvParams &p)
{
    static const bool off = env_int("BQG_NO_ROWS_KERNEL", 0) != 0;
    return !off && g.lpr && g.splits == 1 && p.nmat == 1 && p.epi == EPI_STORE && !p.hq &&
           g.piece_chunks >= g.nc;
}

// The plan's geometry in the kernel parameters.
void apply_plan(GemvParams &p, const GemvPlan &g, int64_t K)
{
    p.K = (int)K;
    p.nb = (int)(K / QK);
    p.nc = g.nc;
    p.TPR = g.TPR;
    p.RG = g.RG;
    p.chunks_per_split = g.cps;
    p.nstages = g.NS;
    p.stage_rows = g.S;
    p.row_stride = g.stride;
    p.win_stages = g.win_stages;
    p.part_off = g.part_off;
    p.bar_off = g.bar_off;
    p.ctas = g.ctas;
    p.L = g.L;
    p.wg = g.wg;
    p.ng = g.ng;
    p.x_off = g.x_off;
    p.xraw_off = g.xraw_off;
    p.early = g.early;
    p.rl = g.rl;
    p.piece_chunks = g.piece_chunks;
    p.x_bf16s = g.x_bf16s ? 1 : 0;
    p.x_row_bytes = g.x_row_bytes;
}

int run_gemv(int wf, int xf, GemvParams p, int M, int64_t K, int final_epi, void *ws, size_t ws_bytes,
             cudaStream_t stream, uint8_t *hq = nullptr)
{
    DevInfo dev;
    int dv = 0;
    int st = current_device(&dev);
    if (st) return st;
    cudaGetDevice(&dv);
    if (p.Nv == 0) return BQG_OK;
    const int unit = (final_epi == EPI_SWIGLU) ? 2 : 1;
    GemvPlan g;
    st = plan_any(wf, xf, M, p.Nv, K, unit, dev, dv, &g);
    if (st) return st;
    const size_t need = (hq && g.splits == 1) ? swiglu_q8_1_staging(M, p.rows[0]) : g.ws_bytes;
    if (need > 0) {
        if (!ws || ws_bytes < need) return BQG_ERR_WORKSPACE;
        if (!aligned16(ws)) return BQG_ERR_MISALIGNED;
    }
    if (hq) {
        p.hq = hq;
        if (g.splits == 1) {
            p.Y[0] = static_cast<float *>(ws);
            p.cnt = reinterpret_cast<int *>(static_cast<uint8_t *>(ws) + ((size_t)M * p.rows[0] * 4 + 15) / 16 * 16);
        }
    }
    apply_plan(p, g, K);
    p.ws = (g.splits > 1) ? (float *)ws : nullptr;
    p.epi = (g.splits > 1) ? EPI_PARTIAL : final_epi;
    p.rows_kernel = rows_kernel_applies(g, p) ? 1 : 0;
    const bool pdl = g_pdl.load() != 0;
    cudaError_t e = g.lpr ? lpr_runner(wf, xf)(p, M, g.grid, g.threads, g.smem, stream, pdl, nullptr)
                          : runner(wf, xf)(p, M, g.C, g.grid, g.threads, g.smem, stream, pdl, nullptr);
    if (e != cudaSuccess) return cuda_status(e);
    if (g.splits > 1) {
        e = launch_splitk_reduce(p, M, g.splits, final_epi, stream, pdl);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return BQG_OK;
}

// Workspace of the persistent decode layer (Nff = rows of gate and of up):
// fp32 h staging, one arrival counter per q8_1 block of h, the q8_1 blocks
// of h, then the two grid-barrier words (16-byte aligned parts).
struct LayerWs {
    size_t h, cnt, hq, gbar, total;
};
LayerWs layer_ws(int64_t Nff)
{
    auto up16 = [](size_t b) { return (b + 15) / 16 * 16; };
    LayerWs w;
    w.h = 0;
    w.cnt = up16((size_t)Nff * 4);
    w.hq = w.cnt + up16((size_t)(Nff / QK) * 4);
    w.gbar = w.hq + up16((size_t)(Nff / QK) * Q8_1_BYTES);
    w.total = w.gbar + 16;
    return w;
}

int check_k(int64_t K)
{
    if (K <= 0 || K % QK) return BQG_ERR_UNSUPPORTED_SHAPE;
    if (K > kMaxK) return BQG_ERR_UNSUPPORTED_SHAPE;
    return BQG_OK;
}

// The tensor-core route (bqg_gemv_mma.cuh): M = 4 or 8, bf16 activations
// (and q4_0 x bf16 at M = 2, q4_0 x q8_1 at M = 8), one matrix, outputs stored as they are, staged activations within 80 KiB
// (M K <= about 40960).  One CTA per SM, eight warps; as many slots per warp
// (at most four) as the shared memory left by the staged activation rows
// and the partial records holds.  Measured on the sweep shape (K = 4096,
// N = 14336) against the lanes-per-row kernel: M = 8 bf16 41.7 -> 21.7 us,
// q8_0 43.0 -> 17.5, q4_0 34.5 -> 13.5; M = 4 q8_0 20.9 -> 16.7, q4_0
// 19.9 -> 12.5, bf16 23.3 -> 21.2.  Eight warps with two slots each beat
// sixteen warps in pairs sharing slots, and four.  Returns
// BQG_ERR_UNSUPPORTED_SHAPE when it does not apply (the lanes-per-row plan
// then serves the call).
struct MmaPlan {
    MmaParams p;
    dim3 grid;
    int threads;
    size_t smem;
};

MmaFn mma_runner(int wf, int xf)
{
    if (xf == X_Q8_1) return gemv_mma_run_q4_0_q8_1;
    return (wf == W_BF16) ? gemv_mma_run_bf16 : (wf == W_Q8_0) ? gemv_mma_run_q8_0 : gemv_mma_run_q4_0;
}

int plan_mma(int wf, int xf, int M, int64_t N, int64_t K, const DevInfo &dev, int device, MmaPlan *pl)
{
    static const bool off = env_int("BQG_NO_MMA", 0) != 0;
    static const int force_D = env_int("BQG_MMA_D", 0);
    static const int force_nw = env_int("BQG_MMA_WARPS", 0);
    static const int force_gw = env_int("BQG_MMA_GROUP", 0);
    if (off || N <= 0) return BQG_ERR_UNSUPPORTED_SHAPE;
    // M = 2: q4_0 x bf16 only (its lanes-per-row dot is bound by the
    // conversion; measured 13.70 -> 12.28 us at N = 14336, 6.18 -> 5.83 at 4096)
    if (M != 4 && M != 8 && !(M == 2 && wf == W_Q4_0 && xf == X_BF16)) return BQG_ERR_UNSUPPORTED_SHAPE;
    // q8_1 activations (q4_0 weights): at M = 8, where the integer-dot
    // lanes-per-row kernel is bound by its dots (at M = 4 it is faster)
    if (xf == X_Q8_1 && (wf != W_Q4_0 || M != 8)) return BQG_ERR_UNSUPPORTED_SHAPE;
    MmaParams p{};
    p.N = N;
    p.K = (int)K;
    p.nb = (int)(K / QK);
    const int slot = (wf == W_Q8_0) ? MmaGeom<W_Q8_0>::SLOT : (wf == W_Q4_0) ? MmaGeom<W_Q4_0>::SLOT
                                                                              : MmaGeom<W_BF16>::SLOT;
    p.T = (wf == W_BF16) ? (int)((K + 255) / 256) : (wf == W_Q4_0) ? (p.nb + 31) / 32 : (p.nb + 15) / 16;
    p.units = (N + 15) / 16;
    // bf16 weights over fewer units than half the SMs: the lanes-per-row
    // kernel (split K) is faster (measured at N = 1024, M = 4 and 8)
    if (wf == W_BF16 && p.units < dev.sms / 2) return BQG_ERR_UNSUPPORTED_SHAPE;
    p.x_pitch = (int)((2 * K + 127) / 128 * 128 + 64);
    const int xdbytes = (xf == X_Q8_1) ? p.nb * 8 * 4 : 0;              // q8_1: the scale table
    const int xbytes = M * p.x_pitch + xdbytes;
    if (M * p.x_pitch > 80 * 1024) return BQG_ERR_UNSUPPORTED_SHAPE;
    p.gw = (force_gw == 1 || force_gw == 2) ? force_gw : 1;
    p.nw = (force_nw >= 1 && force_nw <= 16) ? force_nw : 8;
    p.nw = std::max(p.gw, p.nw / p.gw * p.gw);
    const int ng = p.nw / p.gw;
    const int ctas = (int)std::min<int64_t>(p.units, dev.sms);
    const int64_t upc = (p.units + ctas - 1) / ctas;                 // units of the largest CTA
    const int64_t maxS = upc * p.T;
    if (maxS * ng >= ((int64_t)1 << 30) || upc * 16 * M >= ((int64_t)1 << 30)) return BQG_ERR_UNSUPPORTED_SHAPE;
    const int64_t spg = (maxS + ng - 1) / ng;                        // stages of the busiest group
    p.rmax = (int)std::max<int64_t>(1, std::min<int64_t>(upc, (spg + p.T - 2) / p.T + 1));
    const int rec = p.nw * p.rmax * 512;
    const int64_t xarea = std::max<int64_t>(xbytes, (int64_t)M * (16 * upc + 1) * 4 + 15) / 16 * 16;
    if (xarea > 120 * 1024) return BQG_ERR_UNSUPPORTED_SHAPE;
    const int budget = 232448 - 512 - 128 - (int)xarea - rec - 8 * ng * 4;
    int D = std::min(4, budget / (ng * slot));
    if (force_D > 0) D = std::min(D, force_D);
    if (D < 1) return BQG_ERR_UNSUPPORTED_SHAPE;
    p.D = D;
    static const int force_early = env_int("BQG_MMA_EARLY", -1);
    p.early = (force_early >= 0) ? std::min(force_early, D) : D;   // weights do not wait for the previous grid
    p.x_off = ng * D * slot;
    p.xd_off = p.x_off + M * p.x_pitch;
    // the activation area also holds the CTA's sums before they go out
    p.rec_off = p.x_off + (int)xarea;
    p.bar_off = p.rec_off + rec;
    MmaPlan g{};
    g.smem = (size_t)p.bar_off + 8 * ng * D + 128;      // + alignment slack
    g.threads = 32 * p.nw;
    g.grid = dim3((unsigned)ctas);
    MmaFn fn = mma_runner(wf, xf);
    int bpsm = 0;
    {
        auto key = std::make_tuple(device, wf, xf, M, 0, g.threads, 2, g.smem);
        std::unique_lock<std::mutex> lk(g_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) {
            bpsm = it->second;
        } else {
            lk.unlock();
            CUtensorMap dummy_map{};
            const cudaError_t e = fn(dummy_map, dummy_map, p, M, dim3(1), g.threads, g.smem, 0, false, &bpsm);
            if (e != cudaSuccess) return cuda_status(e);
            lk.lock();
            g_occ[key] = bpsm;
        }
    }
    if (bpsm < 1) return BQG_ERR_UNSUPPORTED_SHAPE;
    g.p = p;
    *pl = g;
    return BQG_OK;
}

int run_mma(int wf, int xf, int fmt, const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K,
            cudaStream_t stream)
{
    DevInfo dev;
    int dv = 0;
    int st = current_device(&dev);
    if (st) return st;
    cudaGetDevice(&dv);
    MmaPlan g;
    st = plan_mma(wf, xf, M, N, K, dev, dv, &g);
    if (st) return st;
    auto enc = tensor_map_encoder();
    if (!enc) return BQG_ERR_UNSUPPORTED_SHAPE;
    // the repacked rows as 8-byte units; boxes of 16 rows: the stage's data
    // plus the pitch pad (q8_0: a low or high code half; the scales)
    const int64_t row_bytes = repacked_row_bytes(fmt, K);
    const int box = (wf == W_Q8_0) ? MmaGeom<W_Q8_0>::BOX : (wf == W_Q4_0) ? MmaGeom<W_Q4_0>::BOX
                                                                          : MmaGeom<W_BF16>::BOX;
    cuuint64_t gdim[2] = {(cuuint64_t)(row_bytes / 8), (cuuint64_t)N};
    cuuint64_t gstride[1] = {(cuuint64_t)row_bytes};
    cuuint32_t wbox[2] = {(cuuint32_t)box, 16u};
    cuuint32_t sbox[2] = {(cuuint32_t)MmaGeom<W_Q8_0>::SC_BOX, 16u};
    cuuint32_t estride[2] = {1u, 1u};
    CUtensorMap wmap, smap;
    if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(Wp), gdim, gstride, wbox, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return BQG_ERR_UNSUPPORTED_SHAPE;
    smap = wmap;
    if (wf == W_Q8_0 &&
        enc(&smap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(Wp), gdim, gstride, sbox, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return BQG_ERR_UNSUPPORTED_SHAPE;
    g.p.X = static_cast<const uint8_t *>(X);
    g.p.Y = Y;
    return cuda_status(mma_runner(wf, xf)(wmap, smap, g.p, M, g.grid, g.threads, g.smem, stream, g_pdl.load() != 0,
                                          nullptr));
}

int gemv_plain(int wf, int xf, int fmt, const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K,
               void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!Wp || !X || !Y || N < 0 || !valid_m(M)) return BQG_ERR_INVALID_ARG;
    if (int st = check_k(K)) return st;
    if (wf == W_BF16 && K > 16384) return BQG_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(Wp) || !aligned16(Y) || !aligned(X, xf == X_Q8_1 ? 4 : 16)) return BQG_ERR_MISALIGNED;
    if ((M == 2 || M == 4 || M == 8) && N > 0) {
        const int st = run_mma(wf, xf, fmt, Wp, X, Y, M, N, K, stream);
        if (st != BQG_ERR_UNSUPPORTED_SHAPE) return st;
    }
    GemvParams p{};
    p.W[0] = (const uint8_t *)Wp;
    p.Y[0] = Y;
    p.rows[0] = N;
    p.nmat = 1;
    p.X = (const uint8_t *)X;
    p.Nv = N;
    p.row_bytes = repacked_row_bytes(fmt, K);
    return run_gemv(wf, xf, p, M, K, EPI_STORE, ws, ws_bytes, stream);
}

}  // namespace

extern "C" {

const char *bqg_status_string(int s)
{
    switch (s) {
    case BQG_OK: return "ok";
    case BQG_ERR_INVALID_ARG: return "invalid argument";
    case BQG_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case BQG_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case BQG_ERR_UNSUPPORTED_DEVICE: return "unsupported device (sm_103 required)";
    case BQG_ERR_CUDA: return "CUDA error";
    case BQG_ERR_TIMEOUT: return "bounded device wait timed out";
    case BQG_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

const char *bqg_version(void) { return "bqgemv 0.1 sm_103a"; }

const char *bqg_last_cuda_error(void) { return cudaGetErrorString(t_last_cuda); }

int bqg_set_pdl(int enable) { return g_pdl.exchange(enable ? 1 : 0); }

int bqg_host_alias(const void *host, void **dev)
{
    if (!host || !dev) return BQG_ERR_INVALID_ARG;
    DevInfo di;
    if (int st = current_device(&di)) return st;
    void *d = nullptr;
    const cudaError_t e = cudaHostGetDevicePointer(&d, const_cast<void *>(host), 0);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();   // not page-locked and mapped: report it, leave no error pending
        return cuda_status(e);
    }
    *dev = d;
    return BQG_OK;
}

int bqg_copy_sm(void *dst, const void *src, size_t bytes, cudaStream_t stream)
{
    DevInfo dev;
    if (bytes == 0) return current_device(&dev);   // nothing to copy: any pointers, no launch
    if (!dst || !src) return BQG_ERR_INVALID_ARG;
    if (!aligned16(dst) || !aligned16(src) || bytes % 16) return BQG_ERR_MISALIGNED;
    const uintptr_t a = reinterpret_cast<uintptr_t>(dst), b = reinterpret_cast<uintptr_t>(src);
    if (a < b + bytes && b < a + bytes) return BQG_ERR_INVALID_ARG;   // overlapping ranges
    if (int st = current_device(&dev)) return st;
    return cuda_status(launch_copy_sm(dst, src, (int64_t)bytes, dev.sms, stream, g_pdl.load() != 0));
}

size_t bqg_repacked_size(int fmt, int64_t N, int64_t K)
{
    if (N < 0 || K <= 0 || K % QK) return 0;
    if (fmt != BQG_BF16 && fmt != BQG_Q8_0 && fmt != BQG_Q4_0) return 0;
    return (size_t)(N * repacked_row_bytes(fmt, K));
}

int bqg_quantize_weights(int fmt, const float *W, void *dst, int64_t N, int64_t K, cudaStream_t stream)
{
    if (!W || !dst || N < 0 || (fmt != BQG_Q8_0 && fmt != BQG_Q4_0)) return BQG_ERR_INVALID_ARG;
    if (int st = check_k(K)) return st;
    if (!aligned(W, 4) || !aligned(dst, 2)) return BQG_ERR_MISALIGNED;
    DevInfo dev;
    if (int st = current_device(&dev)) return st;
    if (N == 0) return BQG_OK;
    return cuda_status(launch_quantize_weights(fmt, W, dst, N, K, stream));
}

int bqg_repack_weights(int fmt, const void *src, void *dst, int64_t N, int64_t K, cudaStream_t stream)
{
    if (!src || !dst || N < 0 || (fmt != BQG_BF16 && fmt != BQG_Q8_0 && fmt != BQG_Q4_0)) return BQG_ERR_INVALID_ARG;
    if (int st = check_k(K)) return st;
    if (!aligned(src, 2) || !aligned16(dst)) return BQG_ERR_MISALIGNED;
    DevInfo dev;
    if (int st = current_device(&dev)) return st;
    if (N == 0) return BQG_OK;
    return cuda_status(launch_repack(fmt, src, dst, N, K, stream));
}

int bqg_quantize_q8_1(const void *x, int x_dtype, void *xq, int M, int64_t K, cudaStream_t stream)
{
    if (!x || !xq || M < 1 || M > 65535 || (x_dtype != BQG_BF16 && x_dtype != BQG_F32)) return BQG_ERR_INVALID_ARG;
    if (int st = check_k(K)) return st;
    if (!aligned(x, x_dtype == BQG_F32 ? 4 : 2) || !aligned(xq, 4)) return BQG_ERR_MISALIGNED;
    DevInfo dev;
    if (int st = current_device(&dev)) return st;
    return cuda_status(launch_quantize_q8_1(x, x_dtype == BQG_F32, xq, M, K, stream, g_pdl.load() != 0));
}

int bqg_rmsnorm_quantize_q8_1(const void *x, int x_dtype, const float *gamma, float eps, void *xq, int M, int64_t K,
                              cudaStream_t stream)
{
    if (!x || !xq || M < 1 || M > 65535 || (x_dtype != BQG_BF16 && x_dtype != BQG_F32)) return BQG_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return BQG_ERR_INVALID_ARG;
    if (int st = check_k(K)) return st;
    if (!aligned(x, x_dtype == BQG_F32 ? 4 : 2) || !aligned(xq, 4) || (gamma && !aligned(gamma, 4)))
        return BQG_ERR_MISALIGNED;
    DevInfo dev;
    if (int st = current_device(&dev)) return st;
    return cuda_status(launch_rmsnorm_q8_1(x, x_dtype == BQG_F32, gamma, eps, xq, M, K, stream, g_pdl.load() != 0));
}

int bqg_gemv_bf16(const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K, void *ws, size_t ws_bytes,
                  cudaStream_t stream)
{
    return gemv_plain(W_BF16, X_BF16, BQG_BF16, Wp, X, Y, M, N, K, ws, ws_bytes, stream);
}

int bqg_gemv_q8_0(const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K, void *ws, size_t ws_bytes,
                  cudaStream_t stream)
{
    return gemv_plain(W_Q8_0, X_BF16, BQG_Q8_0, Wp, X, Y, M, N, K, ws, ws_bytes, stream);
}

int bqg_gemv_q4_0(const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K, void *ws, size_t ws_bytes,
                  cudaStream_t stream)
{
    return gemv_plain(W_Q4_0, X_BF16, BQG_Q4_0, Wp, X, Y, M, N, K, ws, ws_bytes, stream);
}

int bqg_gemv_q4_0_q8_1(const void *Wp, const void *Xq, float *Y, int M, int64_t N, int64_t K, void *ws,
                       size_t ws_bytes, cudaStream_t stream)
{
    return gemv_plain(W_Q4_0, X_Q8_1, BQG_Q4_0, Wp, Xq, Y, M, N, K, ws, ws_bytes, stream);
}

int bqg_gemv_q4_0_q8_1_qkv(const void *Wq, const void *Wk, const void *Wv, const void *Xq, float *Yq, float *Yk,
                           float *Yv, int M, int64_t Nq, int64_t Nkv, int64_t K, void *ws, size_t ws_bytes,
                           cudaStream_t stream)
{
    if (!Wq || !Wk || !Wv || !Xq || !Yq || !Yk || !Yv || Nq < 0 || Nkv < 0 || !valid_m(M)) return BQG_ERR_INVALID_ARG;
    if (int st = check_k(K)) return st;
    if (!aligned16(Wq) || !aligned16(Wk) || !aligned16(Wv) || !aligned(Xq, 4) || !aligned16(Yq) || !aligned16(Yk) ||
        !aligned16(Yv))
        return BQG_ERR_MISALIGNED;
    GemvParams p{};
    p.W[0] = (const uint8_t *)Wq; p.W[1] = (const uint8_t *)Wk; p.W[2] = (const uint8_t *)Wv;
    p.Y[0] = Yq; p.Y[1] = Yk; p.Y[2] = Yv;
    p.rows[0] = Nq; p.rows[1] = Nkv; p.rows[2] = Nkv;
    p.nmat = 3;
    p.X = (const uint8_t *)Xq;
    p.Nv = Nq + 2 * Nkv;
    p.row_bytes = repacked_row_bytes(BQG_Q4_0, K);
    return run_gemv(W_Q4_0, X_Q8_1, p, M, K, EPI_STORE, ws, ws_bytes, stream);
}

int bqg_gemv_q4_0_q8_1_gate_up_swiglu(const void *Wg, const void *Wu, const void *Xq, float *H, int M, int64_t N,
                                      int64_t K, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!Wg || !Wu || !Xq || !H || N < 0 || !valid_m(M)) return BQG_ERR_INVALID_ARG;
    if (int st = check_k(K)) return st;
    if (!aligned16(Wg) || !aligned16(Wu) || !aligned(Xq, 4) || !aligned16(H)) return BQG_ERR_MISALIGNED;
    GemvParams p{};
    p.W[0] = (const uint8_t *)Wg; p.W[1] = (const uint8_t *)Wu;
    p.Y[0] = H;
    p.rows[0] = N; p.rows[1] = N;
    p.nmat = 2;
    p.X = (const uint8_t *)Xq;
    p.Nv = 2 * N;
    p.row_bytes = repacked_row_bytes(BQG_Q4_0, K);
    return run_gemv(W_Q4_0, X_Q8_1, p, M, K, EPI_SWIGLU, ws, ws_bytes, stream);
}

int bqg_gemv_q4_0_q8_1_gate_up_swiglu_q8_1(const void *Wg, const void *Wu, const void *Xq, void *Hq, int M,
                                           int64_t N, int64_t K, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!Wg || !Wu || !Xq || !Hq || N < 0 || !valid_m(M)) return BQG_ERR_INVALID_ARG;
    if (int st = check_k(K)) return st;
    if (N % QK) return BQG_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(Wg) || !aligned16(Wu) || !aligned(Xq, 4) || !aligned(Hq, 4)) return BQG_ERR_MISALIGNED;
    GemvParams p{};
    p.W[0] = (const uint8_t *)Wg; p.W[1] = (const uint8_t *)Wu;
    p.rows[0] = N; p.rows[1] = N;
    p.nmat = 2;
    p.X = (const uint8_t *)Xq;
    p.Nv = 2 * N;
    p.row_bytes = repacked_row_bytes(BQG_Q4_0, K);
    return run_gemv(W_Q4_0, X_Q8_1, p, M, K, EPI_SWIGLU, ws, ws_bytes, stream, (uint8_t *)Hq);
}

int bqg_decode_layer_q4_0_q8_1(const void *xa, const void *xb, int x_dtype, const void *Wq, const void *Wk,
                               const void *Wv, const void *Wg, const void *Wu, const void *Wd, float *Yq, float *Yk,
                               float *Yv, float *Y, int M, int64_t Nq, int64_t Nkv, int64_t Nff, int64_t K, void *ws,
                               size_t ws_bytes, cudaStream_t stream)
{
    if (!xa || !xb || !Wq || !Wk || !Wv || !Wg || !Wu || !Wd || !Yq || !Yk || !Yv || !Y || !ws)
        return BQG_ERR_INVALID_ARG;
    if (Nq <= 0 || Nkv <= 0 || Nff <= 0 || (x_dtype != BQG_BF16 && x_dtype != BQG_F32)) return BQG_ERR_INVALID_ARG;
    if (M != 1) return BQG_ERR_UNSUPPORTED_SHAPE;
    if (int st = check_k(K)) return st;
    if (int st = check_k(Nff)) return st;
    const bool f32 = (x_dtype == BQG_F32);
    if (!aligned16(Wq) || !aligned16(Wk) || !aligned16(Wv) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd) ||
        !aligned16(ws) || !aligned(xa, f32 ? 4 : 2) || !aligned(xb, f32 ? 4 : 2) || !aligned(Yq, 4) ||
        !aligned(Yk, 4) || !aligned(Yv, 4) || !aligned(Y, 4))
        return BQG_ERR_MISALIGNED;
    const LayerWs w = layer_ws(Nff);
    if (ws_bytes < w.total) return BQG_ERR_WORKSPACE;
    DevInfo dev;
    if (int st = current_device(&dev)) return st;

    // shared memory: one slot per warp (the larger stage of the two phases),
    // staged activations (the larger phase), phase 1's q8_1 blocks, barriers
    constexpr int NW = 12, RL1 = 2, RL2 = 1;
    const int64_t rb1 = repacked_row_bytes(BQG_Q4_0, K), rb2 = repacked_row_bytes(BQG_Q4_0, Nff);
    const int nb1 = (int)(K / QK), nb2 = (int)(Nff / QK);
    const int nc1 = chunk_space(W_Q4_0, K), nc2 = chunk_space(W_Q4_0, Nff);
    const int xrb1 = (x_stage_bytes(W_Q4_0, X_Q8_1, nc1, nb1, 0) + 15) / 16 * 16;
    const int xrb2 = (x_stage_bytes(W_Q4_0, X_Q8_1, nc2, nb2, 0) + 15) / 16 * 16;
    LayerParams lp{};
    lp.slot_bytes = (int)std::max<int64_t>(RL1 * rb1, RL2 * rb2);
    lp.x_off = NW * lp.slot_bytes;
    lp.xraw_off = lp.x_off + std::max(xrb1, xrb2);
    lp.bar_off = lp.xraw_off + (std::max(nb1, nb2) * Q8_1_BYTES + 15) / 16 * 16;
    const size_t smem = (size_t)lp.bar_off + 8 * (NW + 1);
    if (smem > 232448) return BQG_ERR_UNSUPPORTED_SHAPE;
    int bpsm = 0;
    if (cudaError_t e = layer_occupancy(32 * NW, smem, &bpsm)) return cuda_status(e);
    bpsm = std::min(bpsm, 2);
    if (bpsm < 1) return BQG_ERR_UNSUPPORTED_SHAPE;
    const int grid = dev.sms * bpsm;
    // phase 1's CTAs split between qkv and gate/up in proportion to their bytes
    const double qb = (double)(Nq + 2 * Nkv), gb = (double)(2 * Nff);
    lp.cq = (int)std::min<int64_t>(grid - 1, std::max<int64_t>(1, (int64_t)(grid * qb / (qb + gb) + 0.5)));

    uint8_t *wsb = static_cast<uint8_t *>(ws);
    GemvParams &a = lp.qkv;
    a.W[0] = (const uint8_t *)Wq; a.W[1] = (const uint8_t *)Wk; a.W[2] = (const uint8_t *)Wv;
    a.Y[0] = Yq; a.Y[1] = Yk; a.Y[2] = Yv;
    a.rows[0] = Nq; a.rows[1] = Nkv; a.rows[2] = Nkv;
    a.nmat = 3;
    a.Nv = Nq + 2 * Nkv;
    GemvParams &g = lp.gu;
    g.W[0] = (const uint8_t *)Wg; g.W[1] = (const uint8_t *)Wu;
    g.Y[0] = reinterpret_cast<float *>(wsb + w.h);
    g.rows[0] = Nff; g.rows[1] = Nff;
    g.nmat = 2;
    g.Nv = 2 * Nff;
    g.hq = wsb + w.hq;
    g.cnt = reinterpret_cast<int *>(wsb + w.cnt);
    for (GemvParams *q : {&a, &g}) {
        q->epi = (q == &g) ? EPI_SWIGLU : EPI_STORE;
        q->row_bytes = rb1;
        q->row_stride = (int)rb1;
        q->K = (int)K;
        q->nb = nb1;
        q->nc = nc1;
        q->x_row_bytes = xrb1;
    }
    GemvParams &d = lp.dn;
    d.W[0] = (const uint8_t *)Wd;
    d.Y[0] = Y;
    d.rows[0] = K;
    d.nmat = 1;
    d.Nv = K;
    d.epi = EPI_STORE;
    d.X = wsb + w.hq;
    d.row_bytes = rb2;
    d.row_stride = (int)rb2;
    d.K = (int)Nff;
    d.nb = nb2;
    d.nc = nc2;
    d.x_row_bytes = xrb2;
    lp.xa = xa;
    lp.xb = xb;
    lp.x_f32 = f32 ? 1 : 0;
    lp.gbar = reinterpret_cast<unsigned long long *>(wsb + w.gbar);
    if (cudaError_t e = layer_launch(lp, grid, 32 * NW, smem, stream)) return cuda_status(e);
    return BQG_OK;
}

static int gemm_entry(int fmt, const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K, void *ws,
                      size_t ws_bytes, cudaStream_t stream)
{
    (void)ws; (void)ws_bytes;
    if (!Wp || !X || !Y || M <= 0 || N < 0) return BQG_ERR_INVALID_ARG;
    if (M % 128 || N % 128 || K <= 0 || K % 64 || K > kMaxK) return BQG_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(Wp) || !aligned16(X) || !aligned16(Y)) return BQG_ERR_MISALIGNED;
    DevInfo dev;
    if (int st = current_device(&dev)) return st;
    if (N == 0) return BQG_OK;
    return gemm_bf16(fmt, Wp, X, Y, M, N, K, stream, dev.sms);
}

int bqg_gemm_q4_0_bf16(const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K, void *ws,
                       size_t ws_bytes, cudaStream_t stream)
{
    return gemm_entry(BQG_Q4_0, Wp, X, Y, M, N, K, ws, ws_bytes, stream);
}

int bqg_gemm_q8_0_bf16(const void *Wp, const void *X, float *Y, int M, int64_t N, int64_t K, void *ws,
                       size_t ws_bytes, cudaStream_t stream)
{
    return gemm_entry(BQG_Q8_0, Wp, X, Y, M, N, K, ws, ws_bytes, stream);
}

int bqg_debug_q4_0_q8_1_block_dots(const void *Wp, const void *Xq, int32_t *dots, int64_t N, int64_t K,
                                   cudaStream_t stream)
{
    if (!Wp || !Xq || !dots || N < 0) return BQG_ERR_INVALID_ARG;
    if (int st = check_k(K)) return st;
    if (!aligned16(Wp) || !aligned(Xq, 4) || !aligned(dots, 4)) return BQG_ERR_MISALIGNED;
    DevInfo dev;
    if (int st = current_device(&dev)) return st;
    if (N == 0) return BQG_OK;
    int dv = 0;
    cudaGetDevice(&dv);
    // the route bqg_gemv_q4_0_q8_1 takes at M = 1: the lanes-per-row kernel,
    // else (staged activations too large) the K-slice kernel
    GemvPlan g;
    int st = plan_lpr(W_Q4_0, X_Q8_1, 1, N, K, 1, dev, dv, &g);
    if (st == BQG_ERR_UNSUPPORTED_SHAPE)
        return cuda_status(launch_block_dots(Wp, Xq, dots, N, K, repacked_row_bytes(BQG_Q4_0, K), stream));
    if (st) return st;
    GemvParams p{};
    p.W[0] = (const uint8_t *)Wp;
    p.rows[0] = N;
    p.nmat = 1;
    p.X = (const uint8_t *)Xq;
    p.Nv = N;
    p.row_bytes = repacked_row_bytes(BQG_Q4_0, K);
    apply_plan(p, g, K);
    p.epi = (g.splits > 1) ? EPI_PARTIAL : EPI_STORE;     // no output is written either way
    p.dots = dots;
    p.rows_kernel = rows_kernel_applies(g, p) ? 1 : 0;    // the kernel bqg_gemv_q4_0_q8_1 would run
    int occ = 0;
    if (cudaError_t e = gemv_lpr_dots_run_q4_0_q8_1(p, g.grid, g.threads, g.smem, stream, &occ)) return cuda_status(e);
    if (occ < 1) return BQG_ERR_UNSUPPORTED_SHAPE;
    return cuda_status(gemv_lpr_dots_run_q4_0_q8_1(p, g.grid, g.threads, g.smem, stream, nullptr));
}

int bqg_debug_q4_0_q8_1_block_dots_kslice(const void *Wp, const void *Xq, int32_t *dots, int64_t N, int64_t K,
                                          cudaStream_t stream)
{
    if (!Wp || !Xq || !dots || N < 0) return BQG_ERR_INVALID_ARG;
    if (int st = check_k(K)) return st;
    if (!aligned16(Wp) || !aligned(Xq, 4) || !aligned(dots, 4)) return BQG_ERR_MISALIGNED;
    DevInfo dev;
    if (int st = current_device(&dev)) return st;
    if (N == 0) return BQG_OK;
    return cuda_status(launch_block_dots(Wp, Xq, dots, N, K, repacked_row_bytes(BQG_Q4_0, K), stream));
}

size_t bqg_workspace_size(int op, int M, int64_t N, int64_t K)
{
    if (N <= 0 || K <= 0 || K % QK || K > kMaxK) return 0;
    if (op == BQG_OP_GEMM_Q4_0_BF16 || op == BQG_OP_GEMM_Q8_0_BF16) return gemm_workspace(M, N, K);
    if (op == BQG_OP_DECODE_LAYER_Q4_0_Q8_1) return (M == 1 && N % QK == 0 && N <= kMaxK) ? layer_ws(N).total : 0;
    if (!valid_m(M)) return 0;
    DevInfo dev;
    int dv = 0;
    if (current_device(&dev) != BQG_OK) return 0;
    cudaGetDevice(&dv);
    int wf = W_Q4_0, xf = X_Q8_1, unit = 1;
    int64_t Nv = N;
    switch (op) {
    case BQG_OP_GEMV_BF16: wf = W_BF16; xf = X_BF16; break;
    case BQG_OP_GEMV_Q8_0: wf = W_Q8_0; xf = X_BF16; break;
    case BQG_OP_GEMV_Q4_0: wf = W_Q4_0; xf = X_BF16; break;
    case BQG_OP_GEMV_Q4_0_Q8_1: break;
    case BQG_OP_QKV_Q4_0_Q8_1: break;
    case BQG_OP_GATE_UP_Q4_0_Q8_1: Nv = 2 * N; unit = 2; break;
    case BQG_OP_GATE_UP_Q8_1_Q4_0_Q8_1: Nv = 2 * N; unit = 2; break;
    default: return 0;
    }
    if (op == BQG_OP_GEMV_BF16 || op == BQG_OP_GEMV_Q8_0 || op == BQG_OP_GEMV_Q4_0 || op == BQG_OP_GEMV_Q4_0_Q8_1) {
        MmaPlan mp;
        if (plan_mma(wf, xf, M, N, K, dev, dv, &mp) == BQG_OK) return 0;   // the tensor-core route
    }
    GemvPlan g;
    if (plan_any(wf, xf, M, Nv, K, unit, dev, dv, &g) != BQG_OK) return 0;
    if (op == BQG_OP_GATE_UP_Q8_1_Q4_0_Q8_1 && g.splits == 1) return N % QK ? 0 : swiglu_q8_1_staging(M, N);
    return g.ws_bytes;
}

int bqg_gemv_route(int op, int M, int64_t N, int64_t K, int *route)
{
    if (!route || N <= 0 || !valid_m(M)) return BQG_ERR_INVALID_ARG;
    if (int st = check_k(K)) return st;
    int wf = W_Q4_0, xf = X_Q8_1;
    switch (op) {
    case BQG_OP_GEMV_BF16: wf = W_BF16; xf = X_BF16; break;
    case BQG_OP_GEMV_Q8_0: wf = W_Q8_0; xf = X_BF16; break;
    case BQG_OP_GEMV_Q4_0: wf = W_Q4_0; xf = X_BF16; break;
    case BQG_OP_GEMV_Q4_0_Q8_1: break;
    default: return BQG_ERR_INVALID_ARG;
    }
    if (wf == W_BF16 && K > 16384) return BQG_ERR_UNSUPPORTED_SHAPE;
    DevInfo dev;
    int dv = 0;
    int st = current_device(&dev);
    if (st) return st;
    cudaGetDevice(&dv);
    if (M == 2 || M == 4 || M == 8) {
        MmaPlan mp;
        st = plan_mma(wf, xf, M, N, K, dev, dv, &mp);
        if (st == BQG_OK) {
            *route = BQG_ROUTE_TENSOR_CORE;
            return BQG_OK;
        }
        if (st != BQG_ERR_UNSUPPORTED_SHAPE) return st;
    }
    GemvPlan g;
    st = plan_any(wf, xf, M, N, K, 1, dev, dv, &g);
    if (st) return st;
    GemvParams p{};
    p.nmat = 1;
    p.epi = (g.splits > 1) ? EPI_PARTIAL : EPI_STORE;
    *route = !g.lpr ? BQG_ROUTE_K_SLICE : rows_kernel_applies(g, p) ? BQG_ROUTE_LANES_PER_ROW_ROWS
                                                                      : BQG_ROUTE_LANES_PER_ROW;
    return BQG_OK;
}

int bqg_last_device_error(cudaStream_t stream, int *out)
{
    if (!out) return BQG_ERR_INVALID_ARG;
    int word = 0;
    if (int st = gemm_read_error(stream, &word)) return st;
    int w = 0;
    for (auto fn : {gemv_error_bf16, gemv_error_q8_0, gemv_error_q4_0, gemv_error_q4_0_q8_1, layer_take_error}) {
        if (fn(&w) != cudaSuccess) return BQG_ERR_CUDA;
        word |= w;
    }
    *out = word;
    return BQG_OK;
}

}  // extern "C"
