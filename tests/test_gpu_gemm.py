"""Prefill GEMM (q4_0 or q8_0 weights x bf16 activations on the tensor cores)
against the oracle:

* the parity bound against the exact weights at every K:
  |y - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-6;
* exactness of the tensor-core path, within an fp32 accumulation bound
  K * 2^-23 * sum_k |w_k x_k| + 1e-6.  From K = 1024 on each weight is
  rounded once to bf16 (the prefill page's tile: (q - 8) * d or q * d,
  round-to-nearest-even), so the reference is the oracle evaluated on those
  rounded weights; below K = 1024 the kernel splits each weight exactly into
  bf16 terms, so the reference is the oracle on the exact weights.
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


EXACT_BELOW_K = 1024     # the kernel's split into exact bf16 terms applies below this K


def run_gemm(ora, M, N, K, seed, rows=None, cols=None, fmt=Q4_0, canon=None, x=None):
    if canon is None:
        _, canon = make_weights(ora, fmt, N, K, seed=seed)
    Wp = gpu_repacked(fmt, canon, N, K)
    xbits = synth.bf16_bits(synth.activations_f32(M, K, seed=seed + 1) if x is None else x)
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
    Yr, Ar = ora.gemv(fmt, canon, BF16, xbits[sel_m], len(sel_m), N, K, rows=sel_n, nthreads=16)
    # (1) the tensor-core arithmetic: fp32 accumulation of exactly the weights it was given
    if K < EXACT_BELOW_K:
        Yb, Ab = Yr, Ar
    else:
        w_exact = ora.dequantize(fmt, canon.reshape(N, -1)[sel_n], len(sel_n), K)
        wb = bf16_round(w_exact).view(torch.int16).numpy().view(np.uint16)
        Yb, Ab = ora.gemv(BF16, wb, BF16, xbits[sel_m], len(sel_m), len(sel_n), K, nthreads=16)
    err = np.abs(ys - Yb)
    bound = K * 2.0 ** -23 * Ab + 1e-6
    assert np.all(err <= bound), ("tensor-core arithmetic", float(np.max(err / bound)))
    # (2) parity with the exact weights, the stated bound at every K
    err = np.abs(ys - Yr)
    bound = 1e-3 * Ar + 1e-6
    assert np.all(err <= bound), ("parity", float(np.max(err / bound)))
    return Y, canon, X


@pytest.mark.parametrize("fmt", [Q4_0, Q8_0])
@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (128, 256, 128), (128, 128, 960), (256, 384, 1024),
                                   (384, 128, 4096), (128, 1024, 2048)])
def test_gemm_small(ora, M, N, K, fmt):
    run_gemm(ora, M, N, K, seed=M + N + K, fmt=fmt)


@pytest.mark.parametrize("fmt", [Q4_0, Q8_0])
@pytest.mark.parametrize("M,N,K", [(256, 10240, 1024), (640, 5120, 2048)])
def test_gemm_big_units(ora, M, N, K, fmt):
    """Shapes whose order keeps units of 256 activation rows whole on a
    152-SM part (more than half the CTAs take one): every unit big (M = 256),
    and big units followed by single-tile units (M / 128 odd).  Sampled rows
    cover both 128-row halves of every big unit and the single tile."""
    rng = np.random.default_rng(M + N)
    cols = np.unique(np.concatenate([rng.choice(N, 64, replace=False), [0, 127, 128, N - 1]]))
    rows = np.unique(np.concatenate([rng.choice(M, 48, replace=False), [0, 127, 128, 255, M - 128, M - 1]]))
    run_gemm(ora, M, N, K, seed=M + K, rows=rows, cols=cols, fmt=fmt)


@pytest.mark.parametrize("fmt", [Q4_0, Q8_0])
def test_gemm_one_dominant_term(ora, fmt):
    """Short K with one activation per row far larger than the rest: the sum is
    one product, so a single bf16 rounding of that weight (up to 2^-9 of it)
    would break the 1e-3 bound; the exact split must not."""
    M, N, K = 128, 256, 64
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((M, K)) * 1e-3).astype(np.float32)
    x[np.arange(M), rng.integers(0, K, M)] = 100.0
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    # scales with a full 11-bit significand, so (q - 8) d needs more than bf16's 8 bits
    W[:, :32] *= 1.0 + 1023.0 / 1024.0
    run_gemm(ora, M, N, K, seed=5, fmt=fmt, canon=ora.quantize(fmt, W), x=x)


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
