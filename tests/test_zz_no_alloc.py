"""The allocation-free q4_0 x q8_1 GEMV entry point (bqg_gemv_q4_0_q8_1_noalloc).

It serves callers that cannot give the library a cudaMalloc'd workspace (a
fixed device-memory plan, a decode loop where allocating may block, C code
without an allocator): its split-K scratch is a fixed array inside the
library.  Here it is called through the C ABI on shapes that split K, twice
in a row (the array keeps the previous call's contents), and each result
must match the CPU oracle and the existing entry point (given a workspace
of its own), both within the parity bound of the other tests,
|y - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-6.  This file is collected last
on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_quantized_gemv_gb300 as bqg
from block_quantized_gemv_gb300 import build as bqg_build
from block_quantized_gemv_gb300 import synth
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    bqg_build.build()
    return bqg.load()


def _case(N, K, M, seed):
    ora = oracle.default()
    canon = ora.quantize(oracle.Q4_0, synth.weights_f32(N, K, seed))
    Wp = bqg.repack_weights(bqg.Q4_0, synth.u8_tensor(canon), N, K)
    xq_host = ora.quantize(oracle.Q8_1, synth.rms_normalised_f32(M, K, seed + 1))
    Xq = synth.u8_tensor(xq_host).view(M, -1)
    Y, A = ora.gemv(oracle.Q4_0, canon, oracle.Q8_1, xq_host, M, N, K, nthreads=8)
    return Wp, Xq, Y, A


@pytest.mark.parametrize("N,K,M", [(24, 16384, 1), (200, 8192, 2), (40, 11008, 8)])
def test_noalloc_matches_the_workspace_entry_point(L, N, K, M):
    Wp, Xq, Y_ref, A = _case(N, K, M, seed=N + K + M)
    need = bqg.workspace_size(bqg.OP_GEMV_Q4_0_Q8_1, M, N, K)
    assert 0 < need <= L.bqg_noalloc_scratch_bytes()      # the shape really splits K
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ref = torch.full((M, N), float("nan"), device="cuda")
    bqg.gemv_q4_0_q8_1(Wp, Xq, N, K, out=ref, ws=ws)
    stream = torch.cuda.current_stream().cuda_stream
    bound = 1e-3 * A + 1e-6
    for _ in range(2):
        y = torch.full((M, N), float("nan"), device="cuda")
        st = L.bqg_gemv_q4_0_q8_1_noalloc(Wp.data_ptr(), Xq.data_ptr(), y.data_ptr(), M, N, K, stream)
        assert st == 0, bqg.status_string(st)
        torch.cuda.synchronize()
        yh = y.cpu().double().numpy()
        assert np.all(np.isfinite(yh)), "unwritten outputs"
        assert np.all(np.abs(yh - Y_ref) <= bound), "differs from the oracle"
        assert np.all(np.abs(yh - ref.cpu().double().numpy()) <= bound), "differs from the workspace entry point"


def test_noalloc_rejects_a_shape_beyond_its_scratch(L):
    # M = 8 rows of 600 outputs split 2 ways need 2 * 8 * 600 * 4 = 38400 bytes > 32 KiB
    M, N, K = 8, 600, 32768
    assert bqg.workspace_size(bqg.OP_GEMV_Q4_0_Q8_1, M, N, K) > L.bqg_noalloc_scratch_bytes()
    W = torch.zeros(bqg.repacked_size(bqg.Q4_0, N, K), dtype=torch.uint8, device="cuda")
    X = torch.zeros(M * (K // 32) * 36, dtype=torch.uint8, device="cuda")
    Y = torch.zeros((M, N), device="cuda")
    st = L.bqg_gemv_q4_0_q8_1_noalloc(W.data_ptr(), X.data_ptr(), Y.data_ptr(), M, N, K,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == 7        # BQG_ERR_WORKSPACE, nothing launched
