"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars (the oracle is the reference in every case):
  * encoders, repack and the q4_0 x q8_1 block dots: bit-exact;
  * every float output: |y_gpu - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-6;
  * SwiGLU output h = silu(g) u: the bound of g and u carried through silu
    (|silu'| <= 1.1) plus 1e-6 |h| + 1e-6.
Outputs are pre-filled with NaN so that an element the kernel never writes
fails the test ("llama-3x-prompt-speed", the negative: unwritten memory read
back as -inf).
"""
import numpy as np
import pytest
import torch

import block_quantized_gemv_gb300 as bqg
from block_quantized_gemv_gb300 import build as bqg_build
from block_quantized_gemv_gb300 import synth
from oracle import BF16, F32, Q4_0, Q8_0, Q8_1

pytestmark = pytest.mark.gpu

FMT_FN = {BF16: "gemv_bf16", Q8_0: "gemv_q8_0", Q4_0: "gemv_q4_0"}


@pytest.fixture(scope="module", autouse=True)
def lib():
    bqg_build.build()
    return bqg.load()


def nan_like(shape):
    return torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")


def check_close(y_gpu, Y, A, what):
    y = y_gpu.detach().cpu().double().numpy() if isinstance(y_gpu, torch.Tensor) else y_gpu
    assert np.all(np.isfinite(y)), f"{what}: unwritten or non-finite outputs"
    err = np.abs(y - Y)
    bound = 1e-3 * A + 1e-6
    worst = np.max(err / bound)
    assert np.all(err <= bound), f"{what}: max err/bound = {worst:.3g}"
    return worst


def make_weights(ora, fmt, N, K, seed):
    """canonical weights from the oracle encoders (bf16: bits) + the GPU repack"""
    Wf = synth.weights_f32(N, K, seed)
    if fmt == BF16:
        canon = synth.bf16_bits(Wf)
    else:
        canon = ora.quantize(fmt, Wf)
    return Wf, canon


def gpu_repacked(fmt, canon, N, K):
    return bqg.repack_weights(fmt, synth.u8_tensor(canon), N, K)


# ---------------------------------------------------------------------------
# encoders and layout: bit-exact
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("src", ["bf16", "f32"])
@pytest.mark.parametrize("M,K", [(1, 32), (1, 4096), (3, 1056), (8, 4096), (1, 11008), (2, 65536)])
def test_quantize_q8_1_bitexact(ora, src, M, K):
    x = synth.activations_f32(M, K, seed=100 + M + K) * 3
    x[0, :32] = 0.0                                    # an all-zero block
    x[0, 32:64] = np.arange(32) - 16.0 if K >= 64 else x[0, 32:64]   # ties at .5 after scaling
    if src == "bf16":
        bits = synth.bf16_bits(x)
        xt = synth.bf16_tensor(bits)
        xref = np.array(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float())
    else:
        xt = torch.from_numpy(x).cuda()
        xref = x
    got = bqg.quantize_q8_1(xt).cpu().numpy()
    want = ora.quantize(Q8_1, xref)
    assert np.array_equal(got.reshape(-1), want.reshape(-1))


@pytest.mark.parametrize("src", ["bf16", "f32"])
@pytest.mark.parametrize("gain", [False, True])
@pytest.mark.parametrize("M,K,eps", [(1, 32, 1e-5), (1, 4096, 1e-5), (3, 1056, 1e-6), (8, 4096, 0.0),
                                     (1, 11008, 1e-5), (2, 65536, 1e-5)])
def test_rmsnorm_quantize_q8_1_bitexact(ora, src, gain, M, K, eps):
    """Fused RMSNorm -> q8_1 against the oracle's definition, byte for byte."""
    x = synth.activations_f32(M, K, seed=300 + M + K) * 2
    if M > 1:
        x[1] = 0.0 if eps > 0 else 1.0                  # a zero row (eps > 0) or a constant row
    if src == "bf16":
        bits = synth.bf16_bits(x)
        xt = synth.bf16_tensor(bits)
        xref = np.array(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float())
    else:
        xt = torch.from_numpy(x).cuda()
        xref = x
    g = np.random.default_rng(K).uniform(0.25, 2.0, K).astype(np.float32) if gain else None
    gt = torch.from_numpy(g).cuda() if gain else None
    got = bqg.rmsnorm_quantize_q8_1(xt, gt, eps).cpu().numpy()
    want = ora.rmsnorm_q8_1(xref, g, eps)
    assert np.array_equal(got.reshape(-1), want.reshape(-1))


@pytest.mark.parametrize("fmt", [Q8_0, Q4_0])
@pytest.mark.parametrize("N,K", [(1, 32), (5, 1056), (64, 4096), (3, 11008)])
def test_quantize_weights_bitexact(ora, fmt, N, K):
    W = synth.weights_f32(N, K, seed=7 + N)
    W[0, :32] = 0.0
    if K >= 64:
        W[0, 32:64] = 0.0
        W[0, 35], W[0, 40] = -2.0, 2.0                 # equal magnitude, opposite sign
    if K >= 96:
        W[0, 64:96] = (np.arange(32) - 16) * 0.25      # the hand-worked q4_0 block
    got = bqg.quantize_weights(fmt, torch.from_numpy(W).cuda()).cpu().numpy()
    want = ora.quantize(fmt, W)
    assert np.array_equal(got.reshape(-1), want.reshape(-1))


@pytest.mark.parametrize("fmt", [BF16, Q8_0, Q4_0])
@pytest.mark.parametrize("N,K", [(1, 32), (3, 1056), (17, 4096), (2, 11008)])
def test_repack_bitexact_and_roundtrip(ora, fmt, N, K):
    _, canon = make_weights(ora, fmt, N, K, seed=N * K)
    packed = gpu_repacked(fmt, canon, N, K).cpu().numpy()
    assert packed.size == ora.repacked_size(fmt, N, K)
    assert np.array_equal(packed, ora.repack(fmt, canon, N, K))
    assert np.array_equal(ora.unrepack(fmt, packed, N, K), np.ascontiguousarray(canon).reshape(-1).view(np.uint8))


def plant_extreme_blocks(canon, xq, N, K):
    """Blocks at the ends of the integer range, written as bytes: weight codes
    all 0 (q - 8 = -8), all 15 (+7), and the two nibble halves apart (0x0f,
    0xf0), against activation codes all +127, all -127 and alternating +-127
    (|sum| up to 32 * 8 * 127).  Scales 1.0 (fp16 0x3c00); the q8_1 s field
    is fp16(d * sum q)."""
    nb = K // 32
    W = canon.reshape(N, nb, 18)
    X = xq.reshape(nb, 36)
    patterns = [0x00, 0xFF, 0x0F, 0xF0]
    for r in range(min(N, 4)):
        for b in range(min(nb, 4)):
            W[r, b, 0:2] = (0x00, 0x3C)
            W[r, b, 2:] = patterns[(r + b) % 4]
    xcodes = [np.full(32, 127), np.full(32, -127), np.where(np.arange(32) % 2, 127, -127), np.full(32, 127)]
    for b in range(min(nb, 4)):
        q = xcodes[b].astype(np.int8)
        X[b, 0:2] = (0x00, 0x3C)
        X[b, 2:4] = np.array([q.astype(np.int64).sum()], dtype=np.float16).view(np.uint8)   # exact: |s| <= 4064
        X[b, 4:] = q.view(np.uint8)
    return canon, xq


@pytest.mark.parametrize("route", ["gemv", "kslice"])
@pytest.mark.parametrize("N,K", [(8, 64), (33, 1056), (256, 4096), (16, 11008), (4096, 11008), (5, 65536)])
def test_block_dots_bitexact(ora, route, N, K):
    """The int32 block dots sum (qw - 8) qx, bit-exact with the oracle, from
    the GEMV's own lanes-per-row kernel (route "gemv": the plan
    bqg_gemv_q4_0_q8_1 uses at M = 1) and from the K-slice kernel's routine."""
    _, canon = make_weights(ora, Q4_0, N, K, seed=3)
    xq = ora.quantize(Q8_1, synth.rms_normalised_f32(1, K, seed=4))
    canon, xq = plant_extreme_blocks(canon, xq, N, K)
    fn = bqg.debug_q4_0_q8_1_block_dots if route == "gemv" else bqg.debug_q4_0_q8_1_block_dots_kslice
    out = torch.full((N, K // 32), -(2 ** 31), dtype=torch.int32, device="cuda")   # unwritten dots fail
    dots = fn(gpu_repacked(Q4_0, canon, N, K), synth.u8_tensor(xq), N, K, out=out).cpu().numpy()
    want = ora.block_dots_q4_0_q8_1(canon, xq, N, K)
    if min(N, K // 32) >= 2:
        assert want[0, 0] == -32 * 8 * 127 and want[1, 0] == 32 * 7 * 127     # the planted extremes arrived
    assert np.array_equal(dots, want)


# ---------------------------------------------------------------------------
# GEMV parity
# ---------------------------------------------------------------------------
SHAPES = [(1, 32), (7, 1056), (300, 1024), (1000, 4096), (130, 11008)]


def run_gemv(ora, fmt, xf, M, N, K, seed=0, rows=None):
    _, canon = make_weights(ora, fmt, N, K, seed=seed)
    Wp = gpu_repacked(fmt, canon, N, K)
    if xf == BF16:
        xbits = synth.bf16_bits(synth.activations_f32(M, K, seed=seed + 1))
        X = synth.bf16_tensor(xbits)
        xref = xbits
        fn = FMT_FN[fmt]
    else:
        xref = ora.quantize(Q8_1, synth.rms_normalised_f32(M, K, seed=seed + 1))
        X = synth.u8_tensor(xref).view(M, -1)
        fn = "gemv_q4_0_q8_1"
    op = {"gemv_bf16": bqg.OP_GEMV_BF16, "gemv_q8_0": bqg.OP_GEMV_Q8_0, "gemv_q4_0": bqg.OP_GEMV_Q4_0,
          "gemv_q4_0_q8_1": bqg.OP_GEMV_Q4_0_Q8_1}[fn]
    ws = bqg.workspace(op, M, N, K)
    Y = nan_like((M, N))
    getattr(bqg, fn)(Wp, X, N, K, out=Y, ws=ws)
    torch.cuda.synchronize()
    Yr, Ar = ora.gemv(fmt, canon, xf, xref, M, N, K, rows=rows, nthreads=8)
    y = Y.cpu().double().numpy()
    if rows is not None:
        assert np.all(np.isfinite(y)), "unwritten outputs"
        y = y[:, rows]
    return check_close(y, Yr, Ar, f"{fn} M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 2, 4, 8])
@pytest.mark.parametrize("fmt", [BF16, Q8_0, Q4_0])
@pytest.mark.parametrize("N,K", SHAPES)
def test_gemv_bf16_activations(ora, fmt, M, N, K):
    run_gemv(ora, fmt, BF16, M, N, K, seed=N + K + M)


@pytest.mark.parametrize("M", [1, 2, 4, 8])
@pytest.mark.parametrize("N,K", SHAPES)
def test_gemv_q4_0_q8_1(ora, M, N, K):
    run_gemv(ora, Q4_0, Q8_1, M, N, K, seed=N + K + M)


OPS = {BF16: bqg.OP_GEMV_BF16, Q8_0: bqg.OP_GEMV_Q8_0, Q4_0: bqg.OP_GEMV_Q4_0}
# Shapes the tensor-core kernel serves at M = 4 and 8: N not a multiple of
# its 16-row units (17, 1300, 2437) and K whose last stage is partial (K =
# 1056: one block past a q4_0 tile, one past a q8_0 half tile, 32 values
# past a bf16 tile; K = 4128 likewise after four tiles).  bf16 weights take
# the route from N = 16 * 76 rows on.
TC_SHAPES = [(17, 1056), (1300, 4128), (2437, 1056), (2437, 4096)]


@pytest.mark.parametrize("M", [4, 8])
@pytest.mark.parametrize("fmt", [BF16, Q8_0, Q4_0])
@pytest.mark.parametrize("N,K", TC_SHAPES)
def test_gemv_tensor_core_route(ora, fmt, M, N, K):
    route = bqg.gemv_route(OPS[fmt], M, N, K)
    want_tc = not (fmt == BF16 and N < 16 * 76)
    assert (route == bqg.ROUTE_TENSOR_CORE) == want_tc, bqg.ROUTE_NAMES[route]
    run_gemv(ora, fmt, BF16, M, N, K, seed=3 * N + K + M)


@pytest.mark.parametrize("N,K", TC_SHAPES)
def test_gemv_q4_0_q8_1_tensor_core_route(ora, N, K):
    """q4_0 x q8_1 at M = 8 on the tensor cores: each block's MMA sum is the
    exact integer dot, scaled by d_w d_x."""
    assert bqg.gemv_route(bqg.OP_GEMV_Q4_0_Q8_1, 8, N, K) == bqg.ROUTE_TENSOR_CORE
    run_gemv(ora, Q4_0, Q8_1, 8, N, K, seed=5 * N + K)


def test_gemv_routes():
    """The route each shape class takes (no launch)."""
    tc, rows = bqg.ROUTE_TENSOR_CORE, bqg.ROUTE_LANES_PER_ROW_ROWS
    assert bqg.gemv_route(bqg.OP_GEMV_Q8_0, 8, 14336, 4096) == tc
    assert bqg.gemv_route(bqg.OP_GEMV_BF16, 4, 14336, 4096) == tc
    assert bqg.gemv_route(bqg.OP_GEMV_Q4_0, 4, 14336, 4096) == tc
    # M = 2: q4_0 x bf16 on the tensor cores, the other formats on the lanes-per-row kernel
    assert bqg.gemv_route(bqg.OP_GEMV_Q4_0, 2, 14336, 4096) == tc
    assert bqg.gemv_route(bqg.OP_GEMV_Q8_0, 2, 14336, 4096) == rows
    # M = 1: the whole-row lanes-per-row kernel on the headline shape
    assert bqg.gemv_route(bqg.OP_GEMV_BF16, 1, 12288, 4096) == rows
    assert bqg.gemv_route(bqg.OP_GEMV_Q4_0_Q8_1, 1, 12288, 4096) == rows
    # q8_1 activations: the tensor-core route at M = 8, the integer-dot kernel at M = 4
    assert bqg.gemv_route(bqg.OP_GEMV_Q4_0_Q8_1, 8, 14336, 4096) == tc
    assert bqg.gemv_route(bqg.OP_GEMV_Q4_0_Q8_1, 4, 14336, 4096) == rows
    # staged activations above 80 KiB (M = 8, K = 11008): not the tensor-core route
    assert bqg.gemv_route(bqg.OP_GEMV_Q8_0, 8, 4096, 11008) != tc


@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("N,K", [(64, 1024), (1000, 4096), (130, 11008)])
def test_gemv_q4_0_q8_1_float_is_the_exact_integer_dots_scaled(ora, M, N, K):
    """Each output is sum_b fp32(d_w d_x) * sumi_b with sumi_b the exact
    integer dot: against that sum (fp64, from the oracle's dots and scales)
    the GPU may differ only by fp32 accumulation, |err| <= (nb + 2) 2^-24
    sum_b |fp32(d_w d_x) sumi_b| -- far inside the benchmark spec's bound, so a
    wrong integer would show.  At M = 1 the integer-dot kernels compute the
    dots; at M = 8 with K <= 5056 the tensor-core kernel does (exact bf16
    operands, integer sums below 2^15)."""
    _, canon = make_weights(ora, Q4_0, N, K, seed=5)
    xq = ora.quantize(Q8_1, synth.rms_normalised_f32(M, K, seed=6))
    Wp = gpu_repacked(Q4_0, canon, N, K)
    Y = nan_like((M, N))
    bqg.gemv_q4_0_q8_1(Wp, synth.u8_tensor(xq).view(M, -1), N, K, out=Y,
                       ws=bqg.workspace(bqg.OP_GEMV_Q4_0_Q8_1, M, N, K))
    torch.cuda.synchronize()
    if M == 8 and K <= 5056:
        assert bqg.gemv_route(bqg.OP_GEMV_Q4_0_Q8_1, M, N, K) == bqg.ROUTE_TENSOR_CORE
    nb = K // 32
    dw = canon.reshape(N, nb, 18)[:, :, 0:2].copy().view(np.float16).reshape(N, nb).astype(np.float32)
    y = Y.cpu().double().numpy()
    assert np.all(np.isfinite(y))
    xrows = np.asarray(xq).reshape(M, nb * 36)
    for m in range(M):
        xm = np.ascontiguousarray(xrows[m])
        dots = ora.block_dots_q4_0_q8_1(canon, xm, N, K).astype(np.float64)
        dx = xm.reshape(nb, 36)[:, 0:2].copy().view(np.float16).reshape(nb).astype(np.float32)
        scale = (dw * dx[None, :]).astype(np.float64)       # the fp32 product, rounded as the kernel rounds it
        terms = scale * dots
        want = terms.sum(axis=1)
        bound = (nb + 2) * 2.0 ** -24 * np.abs(terms).sum(axis=1) + 1e-30
        assert np.all(np.abs(y[m] - want) <= bound), f"row {m}: max err/bound {np.max(np.abs(y[m] - want) / bound):.3g}"


@pytest.mark.parametrize("fmt,xf", [(BF16, BF16), (Q8_0, BF16), (Q4_0, Q8_1), (Q4_0, BF16)])
def test_gemv_splitk_small_n(ora, fmt, xf):
    # few rows, long K: the plan splits K across CTAs and needs a workspace
    M, N, K = 1, 24, 16384
    op = {BF16: bqg.OP_GEMV_BF16, Q8_0: bqg.OP_GEMV_Q8_0}.get(fmt, bqg.OP_GEMV_Q4_0_Q8_1 if xf == Q8_1 else bqg.OP_GEMV_Q4_0)
    assert bqg.workspace_size(op, M, N, K) > 0
    run_gemv(ora, fmt, xf, M, N, K, seed=11)


def test_splitk_requires_workspace_and_is_deterministic(ora):
    M, N, K = 2, 16, 8192
    _, canon = make_weights(ora, Q8_0, N, K, seed=1)
    Wp = gpu_repacked(Q8_0, canon, N, K)
    X = synth.bf16_tensor(synth.bf16_bits(synth.activations_f32(M, K, seed=2)))
    with pytest.raises(bqg.BqgError) as e:
        bqg.gemv_q8_0(Wp, X, N, K)
    assert e.value.status == 7
    ws = bqg.workspace(bqg.OP_GEMV_Q8_0, M, N, K)
    a = bqg.gemv_q8_0(Wp, X, N, K, ws=ws).clone()
    b = bqg.gemv_q8_0(Wp, X, N, K, ws=ws)
    assert torch.equal(a, b)


def test_gemv_bitwise_deterministic(ora):
    M, N, K = 1, 4096, 4096
    _, canon = make_weights(ora, BF16, N, K, seed=9)
    Wp = gpu_repacked(BF16, canon, N, K)
    X = synth.bf16_tensor(synth.bf16_bits(synth.activations_f32(M, K, seed=10)))
    a = bqg.gemv_bf16(Wp, X, N, K).clone()
    for _ in range(3):
        assert torch.equal(a, bqg.gemv_bf16(Wp, X, N, K))


# ---------------------------------------------------------------------------
# fused entries
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M", [1, 2, 8])
@pytest.mark.parametrize("Nq,Nkv,K", [(256, 64, 1024), (4096, 4096, 4096), (96, 32, 11008)])
def test_qkv(ora, M, Nq, Nkv, K):
    mats = [make_weights(ora, Q4_0, n, K, seed=21 + i)[1] for i, n in enumerate((Nq, Nkv, Nkv))]
    packed = [gpu_repacked(Q4_0, c, n, K) for c, n in zip(mats, (Nq, Nkv, Nkv))]
    xq = ora.quantize(Q8_1, synth.rms_normalised_f32(M, K, seed=20))
    out = (nan_like((M, Nq)), nan_like((M, Nkv)), nan_like((M, Nkv)))
    N = Nq + 2 * Nkv
    ws = bqg.workspace(bqg.OP_QKV_Q4_0_Q8_1, M, N, K)
    bqg.gemv_q4_0_q8_1_qkv(*packed, synth.u8_tensor(xq).view(M, -1), Nq, Nkv, K, out=out, ws=ws)
    torch.cuda.synchronize()
    for c, n, y, name in zip(mats, (Nq, Nkv, Nkv), out, "qkv"):
        # large matrices: every 7th row against the oracle (all rows must still be written)
        rows = None if n * K <= 4096 * 4096 else np.arange(0, n, 7)
        Yr, Ar = ora.gemv(Q4_0, c, Q8_1, xq, M, n, K, rows=rows, nthreads=8)
        yv = y.cpu().double().numpy()
        assert np.all(np.isfinite(yv)), f"qkv[{name}]: unwritten outputs"
        check_close(yv if rows is None else yv[:, rows], Yr, Ar, f"qkv[{name}]")


def swiglu_bound(ora, Yg, Ag, Yu, Au):
    tg, tu = 1e-3 * Ag + 1e-6, 1e-3 * Au + 1e-6
    silu = ora.swiglu(Yg.reshape(-1), np.ones(Yg.size)).reshape(Yg.shape)
    h = silu * Yu
    return h, 1.1 * tg * (np.abs(Yu) + tu) + np.abs(silu) * tu + 1e-6 * np.abs(h) + 1e-6


@pytest.mark.parametrize("M", [1, 2, 8])
@pytest.mark.parametrize("N,K", [(64, 1024), (11008, 4096), (40, 11008)])
def test_gate_up_swiglu(ora, M, N, K):
    _, cg = make_weights(ora, Q4_0, N, K, seed=31)
    _, cu = make_weights(ora, Q4_0, N, K, seed=32)
    xq = ora.quantize(Q8_1, synth.rms_normalised_f32(M, K, seed=33))
    H = nan_like((M, N))
    ws = bqg.workspace(bqg.OP_GATE_UP_Q4_0_Q8_1, M, N, K)
    bqg.gemv_q4_0_q8_1_gate_up_swiglu(gpu_repacked(Q4_0, cg, N, K), gpu_repacked(Q4_0, cu, N, K),
                                      synth.u8_tensor(xq).view(M, -1), N, K, out=H, ws=ws)
    torch.cuda.synchronize()
    Yg, Ag = ora.gemv(Q4_0, cg, Q8_1, xq, M, N, K, nthreads=8)
    Yu, Au = ora.gemv(Q4_0, cu, Q8_1, xq, M, N, K, nthreads=8)
    h_ref, bound = swiglu_bound(ora, Yg, Ag, Yu, Au)
    h = H.cpu().double().numpy()
    assert np.all(np.isfinite(h))
    assert np.all(np.abs(h - h_ref) <= bound), float(np.max(np.abs(h - h_ref) / bound))


@pytest.mark.parametrize("M", [1, 2, 4, 8])
@pytest.mark.parametrize("N,K", [(64, 1024), (11008, 4096), (32, 11008), (4096, 4096)])
def test_gate_up_swiglu_q8_1(ora, M, N, K):
    """SwiGLU epilogue writing q8_1: (1) byte for byte the q8_1 encoding of the
    fp32 h the plain entry point writes; (2) within the SwiGLU bound plus half
    a quantization step of the oracle's h; (3) the workspace's block counters
    are re-armed, so a second call gives the same bytes."""
    _, cg = make_weights(ora, Q4_0, N, K, seed=41)
    _, cu = make_weights(ora, Q4_0, N, K, seed=42)
    xq = ora.quantize(Q8_1, synth.rms_normalised_f32(M, K, seed=43))
    Wg, Wu = gpu_repacked(Q4_0, cg, N, K), gpu_repacked(Q4_0, cu, N, K)
    xt = synth.u8_tensor(xq).view(M, -1)
    ws = bqg.workspace(bqg.OP_GATE_UP_Q8_1_Q4_0_Q8_1, M, N, K)
    Hq = bqg.gemv_q4_0_q8_1_gate_up_swiglu_q8_1(Wg, Wu, xt, N, K, ws=ws)
    Hq2 = bqg.gemv_q4_0_q8_1_gate_up_swiglu_q8_1(Wg, Wu, xt, N, K, ws=ws)
    H = bqg.gemv_q4_0_q8_1_gate_up_swiglu(Wg, Wu, xt, N, K, ws=bqg.workspace(bqg.OP_GATE_UP_Q4_0_Q8_1, M, N, K))
    torch.cuda.synchronize()
    got = Hq.cpu().numpy().reshape(-1)
    assert np.array_equal(ora.quantize(Q8_1, H.cpu().numpy()).reshape(-1), got)
    assert np.array_equal(Hq2.cpu().numpy().reshape(-1), got)
    Yg, Ag = ora.gemv(Q4_0, cg, Q8_1, xq, M, N, K, nthreads=8)
    Yu, Au = ora.gemv(Q4_0, cu, Q8_1, xq, M, N, K, nthreads=8)
    h_ref, bound = swiglu_bound(ora, Yg, Ag, Yu, Au)
    deq = ora.dequantize(Q8_1, got, M, N)
    blocks = got.reshape(M, N // 32, 36)
    d = np.frombuffer(blocks[:, :, 0:2].copy().tobytes(), dtype=np.float16).astype(np.float64).reshape(M, N // 32)
    half_step = np.repeat(d / 2, 32, axis=1)
    assert np.all(np.abs(deq - h_ref) <= bound + half_step * (1 + 2.0 ** -10)), \
        float(np.max(np.abs(deq - h_ref) - bound - half_step))


# ---------------------------------------------------------------------------
# error paths on a real device (nothing is launched)
# ---------------------------------------------------------------------------
def test_device_is_accepted_and_errors_are_reported():
    L = bqg.load()
    W = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    X = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(16, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert L.bqg_gemv_bf16(W.data_ptr(), X.data_ptr(), Y.data_ptr(), 3, 8, 64, None, 0, s) == 1
    assert L.bqg_gemv_bf16(W.data_ptr(), X.data_ptr(), Y.data_ptr(), 1, 8, 48, None, 0, s) == 2
    assert L.bqg_gemv_bf16(W.data_ptr() + 2, X.data_ptr(), Y.data_ptr(), 1, 8, 64, None, 0, s) == 3
    assert L.bqg_gemv_bf16(W.data_ptr(), X.data_ptr(), Y.data_ptr(), 1, 0, 64, None, 0, s) == 0
    assert bqg.last_device_error() == 0
