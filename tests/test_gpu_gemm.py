"""Prefill GEMM (q4_0 or q8_0 weights x bf16 activations on the tensor cores)
against the oracle, two ways:

* exactness of the tensor-core path: the oracle evaluated on the weights
  rounded to bf16 (the rounding the prefill page's tile applies before the
  MMA: (q - 8) * d or q * d, one round-to-nearest-even), compared with an fp32
  accumulation bound, K * 2^-23 * sum_k |w_k x_k| + 1e-6;
* the parity bound against the exact weights: |y - y_ref| <= 1e-3 *
  sum_k |w_k x_k| + 1e-6 for K >= 1024 (the full-size configuration
  included).  Rounding a weight to bf16 moves it by at most 2^-9 of itself,
  so for short K (few terms to average the rounding out) the bound used is
  (1e-3 + 2^-9) * sum_k |w_k x_k| + 1e-6.
"""
import numpy as np
import pytest
import torch

import block_quantized_gemv_gb300 as bqg
from block_quantized_gemv_gb300 import build as bqg_build
from block_quantized_gemv_gb300 import synth
from oracle import BF16, Q4_0, Q8_0

from test_gpu_parity import gpu_repacked, make_weights, nan_like

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    bqg_build.build()
    return bqg.load()


def bf16_round(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def run_gemm(ora, M, N, K, seed, rows=None, cols=None, fmt=Q4_0):
    _, canon = make_weights(ora, fmt, N, K, seed=seed)
    Wp = gpu_repacked(fmt, canon, N, K)
    xbits = synth.bf16_bits(synth.activations_f32(M, K, seed=seed + 1))
    X = synth.bf16_tensor(xbits)
    Y = nan_like((M, N))
    (bqg.gemm_q8_0_bf16 if fmt == Q8_0 else bqg.gemm_q4_0_bf16)(Wp, X, N, K, out=Y)
    torch.cuda.synchronize()
    assert bqg.last_device_error() == 0
    y = Y.cpu().double().numpy()
    assert np.all(np.isfinite(y)), "unwritten outputs"
    sel_n = np.arange(N) if cols is None else cols
    sel_m = np.arange(M) if rows is None else rows
    ys = y[np.ix_(sel_m, sel_n)]
    # (1) exact tensor-core arithmetic on bf16-rounded weights
    w_exact = ora.dequantize(fmt, canon.reshape(N, -1)[sel_n], len(sel_n), K)
    wb = bf16_round(w_exact).view(torch.int16).numpy().view(np.uint16)
    Yb, Ab = ora.gemv(BF16, wb, BF16, xbits[sel_m], len(sel_m), len(sel_n), K, nthreads=16)
    err = np.abs(ys - Yb)
    bound = K * 2.0 ** -23 * Ab + 1e-6
    assert np.all(err <= bound), ("rounded-weight check", float(np.max(err / bound)))
    # (2) parity with the exact weights
    Yr, Ar = ora.gemv(fmt, canon, BF16, xbits[sel_m], len(sel_m), N, K, rows=sel_n, nthreads=16)
    err = np.abs(ys - Yr)
    bound = (1e-3 if K >= 1024 else 1e-3 + 2.0 ** -9) * Ar + 1e-6
    assert np.all(err <= bound), ("parity", float(np.max(err / bound)))
    return Y, canon, X


@pytest.mark.parametrize("fmt", [Q4_0, Q8_0])
@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (128, 256, 128), (256, 384, 1024), (384, 128, 4096),
                                   (128, 1024, 2048)])
def test_gemm_small(ora, M, N, K, fmt):
    run_gemm(ora, M, N, K, seed=M + N + K, fmt=fmt)


def test_gemm_matches_matmul_on_rounded_weights(ora):
    M, N, K = 256, 512, 1024
    Y, canon, X = run_gemm(ora, M, N, K, seed=3)
    w = ora.dequantize(Q4_0, canon, N, K)
    Wb = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16).float().cuda()
    ref = X.float() @ Wb.T
    torch.cuda.synchronize()
    assert torch.allclose(Y, ref, rtol=2e-5, atol=2e-5 * float(ref.abs().max()))


@pytest.mark.slow
def test_c5_prefill_m512_k4096_n14336(ora):
    M, N, K = 512, 14336, 4096
    rng = np.random.default_rng(0)
    cols = np.unique(np.concatenate([rng.choice(N, 96, replace=False), [0, 127, 128, N - 1]]))
    rows = np.unique(np.concatenate([rng.choice(M, 40, replace=False), [0, 127, 128, M - 1]]))
    run_gemm(ora, M, N, K, seed=77, rows=rows, cols=cols)


@pytest.mark.slow
def test_prefill_q8_0_m512_k4096_n14336(ora):
    M, N, K = 512, 14336, 4096
    rng = np.random.default_rng(1)
    cols = np.unique(np.concatenate([rng.choice(N, 96, replace=False), [0, 127, 128, N - 1]]))
    rows = np.unique(np.concatenate([rng.choice(M, 40, replace=False), [0, 127, 128, M - 1]]))
    run_gemm(ora, M, N, K, seed=78, rows=rows, cols=cols, fmt=Q8_0)


def test_gemm_rejects_bad_shapes():
    L = bqg.load()
    W = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    X = torch.zeros(1 << 16, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(1 << 16, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert L.bqg_gemm_q4_0_bf16(W.data_ptr(), X.data_ptr(), Y.data_ptr(), 100, 128, 64, None, 0, s) == 2
    assert L.bqg_gemm_q4_0_bf16(W.data_ptr(), X.data_ptr(), Y.data_ptr(), 128, 100, 64, None, 0, s) == 2
    assert L.bqg_gemm_q4_0_bf16(W.data_ptr(), X.data_ptr(), Y.data_ptr(), 128, 128, 96, None, 0, s) == 2
    assert L.bqg_gemm_q8_0_bf16(W.data_ptr(), X.data_ptr(), Y.data_ptr(), 128, 128, 96, None, 0, s) == 2
