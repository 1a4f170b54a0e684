"""Parity at the full sizes of the five benchmark configurations, through the
same entry points and launch geometry the benchmark times.

  C1 q8_0 GEMV M=1 K=4096 N=4096                       all outputs
  C2 bf16 GEMV M=1 K=4096 N=12288                      all outputs
  C3 q4_0 x q8_1 decode layer (QKV, gate+up+SwiGLU, down) every stage
  C4 skinny-M sweep M in {1,2,4,8}, K=4096, N=14336    sampled rows
  C5 prefill GEMM M=512 K=4096 N=14336 (q4_0)          sampled outputs
Bars as in test_gpu_parity.
"""
import numpy as np
import pytest
import torch

import block_quantized_gemv_gb300 as bqg
from block_quantized_gemv_gb300 import build as bqg_build
from block_quantized_gemv_gb300 import synth
from oracle import BF16, Q4_0, Q8_0, Q8_1

from test_gpu_parity import check_close, gpu_repacked, make_weights, nan_like, swiglu_bound

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def lib():
    bqg_build.build()
    return bqg.load()


def gemv_call(fmt, xf, Wp, X, N, K, M):
    fn = {BF16: bqg.gemv_bf16, Q8_0: bqg.gemv_q8_0, Q4_0: bqg.gemv_q4_0}[fmt] if xf == BF16 else bqg.gemv_q4_0_q8_1
    op = {BF16: bqg.OP_GEMV_BF16, Q8_0: bqg.OP_GEMV_Q8_0, Q4_0: bqg.OP_GEMV_Q4_0}[fmt] if xf == BF16 \
        else bqg.OP_GEMV_Q4_0_Q8_1
    Y = nan_like((M, N))
    fn(Wp, X, N, K, out=Y, ws=bqg.workspace(op, M, N, K))
    torch.cuda.synchronize()
    return Y


def test_c1_q8_0_m1_k4096_n4096(ora):
    N, K = 4096, 4096
    # the weights come from the GPU encoder, which must equal the oracle's
    Wf = synth.weights_f32(N, K, seed=1)
    canon_gpu = bqg.quantize_weights(Q8_0, torch.from_numpy(Wf).cuda())
    canon = ora.quantize(Q8_0, Wf)
    assert np.array_equal(canon_gpu.cpu().numpy().reshape(-1), canon.reshape(-1))
    xb = synth.bf16_bits(synth.activations_f32(1, K, seed=2))
    Y = gemv_call(Q8_0, BF16, bqg.repack_weights(Q8_0, canon_gpu, N, K), synth.bf16_tensor(xb), N, K, 1)
    Yr, Ar = ora.gemv(Q8_0, canon, BF16, xb, 1, N, K, nthreads=16)
    check_close(Y, Yr, Ar, "C1")


def test_c2_bf16_m1_k4096_n12288(ora):
    N, K = 12288, 4096
    wb = synth.bf16_bits(synth.weights_f32(N, K, seed=1))
    xb = synth.bf16_bits(synth.activations_f32(1, K, seed=2))
    Wp = bqg.repack_weights(BF16, synth.u8_tensor(wb), N, K)
    Y = gemv_call(BF16, BF16, Wp, synth.bf16_tensor(xb), N, K, 1)
    Yr, Ar = ora.gemv(BF16, wb, BF16, xb, 1, N, K, nthreads=16)
    check_close(Y, Yr, Ar, "C2")


def test_c3_decode_layer(ora):
    K, Nq, Nff = 4096, 4096, 11008
    canon = {k: make_weights(ora, Q4_0, n, kk, seed=40 + i)[1]
             for i, (k, n, kk) in enumerate([("q", Nq, K), ("k", Nq, K), ("v", Nq, K),
                                             ("g", Nff, K), ("u", Nff, K), ("d", K, Nff)])}
    shapes = {"q": (Nq, K), "k": (Nq, K), "v": (Nq, K), "g": (Nff, K), "u": (Nff, K), "d": (K, Nff)}
    Wp = {k: gpu_repacked(Q4_0, canon[k], *shapes[k]) for k in canon}
    x = synth.rms_normalised_f32(1, K, seed=50)
    xq = bqg.quantize_q8_1(torch.from_numpy(x).cuda())
    xq_ref = ora.quantize(Q8_1, x)
    assert np.array_equal(xq.cpu().numpy().reshape(-1), xq_ref.reshape(-1))
    out = (nan_like((1, Nq)), nan_like((1, Nq)), nan_like((1, Nq)))
    bqg.gemv_q4_0_q8_1_qkv(Wp["q"], Wp["k"], Wp["v"], xq, Nq, Nq, K, out=out,
                           ws=bqg.workspace(bqg.OP_QKV_Q4_0_Q8_1, 1, 3 * Nq, K))
    H = nan_like((1, Nff))
    bqg.gemv_q4_0_q8_1_gate_up_swiglu(Wp["g"], Wp["u"], xq, Nff, K, out=H,
                                      ws=bqg.workspace(bqg.OP_GATE_UP_Q4_0_Q8_1, 1, Nff, K))
    hq = bqg.quantize_q8_1(H)
    Y = nan_like((1, K))
    bqg.gemv_q4_0_q8_1(Wp["d"], hq, K, Nff, out=Y, ws=bqg.workspace(bqg.OP_GEMV_Q4_0_Q8_1, 1, K, Nff))
    torch.cuda.synchronize()
    for name, y in zip("qkv", out):
        Yr, Ar = ora.gemv(Q4_0, canon[name], Q8_1, xq_ref, 1, Nq, K, nthreads=16)
        check_close(y, Yr, Ar, f"C3 {name}")
    Yg, Ag = ora.gemv(Q4_0, canon["g"], Q8_1, xq_ref, 1, Nff, K, nthreads=16)
    Yu, Au = ora.gemv(Q4_0, canon["u"], Q8_1, xq_ref, 1, Nff, K, nthreads=16)
    h_ref, bound = swiglu_bound(ora, Yg, Ag, Yu, Au)
    h = H.cpu().double().numpy()
    assert np.all(np.isfinite(h)) and np.all(np.abs(h - h_ref) <= bound)
    # the down projection consumes the GPU's own q8_1(h); its bytes must be the oracle's
    hq_ref = ora.quantize(Q8_1, H.cpu().numpy())
    assert np.array_equal(hq.cpu().numpy().reshape(-1), hq_ref.reshape(-1))
    Yr, Ar = ora.gemv(Q4_0, canon["d"], Q8_1, hq_ref, 1, K, Nff, nthreads=16)
    check_close(Y, Yr, Ar, "C3 down")
    # per-block integer dots of the down projection, bit-exact, from the
    # GEMV's own kernel and plan and from the K-slice routine
    rows = np.arange(0, K, 97)
    want = ora.block_dots_q4_0_q8_1(canon["d"].reshape(K, -1)[rows], hq_ref, rows.size, Nff)
    for fn in (bqg.debug_q4_0_q8_1_block_dots, bqg.debug_q4_0_q8_1_block_dots_kslice):
        dots = fn(Wp["d"], hq, K, Nff)
        assert np.array_equal(dots.cpu().numpy()[rows], want), fn.__name__


@pytest.mark.parametrize("M", [1, 2, 4, 8])
@pytest.mark.parametrize("fmt,xf", [(BF16, BF16), (Q8_0, BF16), (Q4_0, BF16), (Q4_0, Q8_1)])
def test_c4_skinny_sweep(ora, M, fmt, xf):
    N, K = 14336, 4096
    _, canon = make_weights(ora, fmt, N, K, seed=60)
    Wp = gpu_repacked(fmt, canon, N, K)
    if xf == BF16:
        xref = synth.bf16_bits(synth.activations_f32(M, K, seed=61))
        X = synth.bf16_tensor(xref)
    else:
        xref = ora.quantize(Q8_1, synth.rms_normalised_f32(M, K, seed=61))
        X = synth.u8_tensor(xref).view(M, -1)
    Y = gemv_call(fmt, xf, Wp, X, N, K, M)
    rows = np.unique(np.concatenate([np.arange(0, N, 29), [N - 1]]))
    Yr, Ar = ora.gemv(fmt, canon, xf, xref, M, N, K, rows=rows, nthreads=16)
    y = Y.cpu().double().numpy()
    assert np.all(np.isfinite(y))
    check_close(y[:, rows], Yr, Ar, f"C4 M={M}")
