"""Edge cases of the GEMV entries against the oracle.

  * the largest K each entry accepts (65536 for the block formats, 16384 for
    bf16 weights), at M = 1 and M = 8 (the latter through the K-slice kernel,
    whose activations do not fit the lanes-per-row staging), and the first K
    each refuses;
  * degenerate canonical blocks that the encoders never write but the
    format allows: scale 0, -0, the smallest fp16 subnormal (2^-24) and the
    largest finite fp16 (65504), and q8_0 codes of -128;
  * an all-zero activation row (every output exactly zero).
"""
import numpy as np
import pytest
import torch

import block_quantized_gemv_gb300 as bqg
from block_quantized_gemv_gb300 import build as bqg_build
from block_quantized_gemv_gb300 import synth
from oracle import BF16, Q4_0, Q8_0, Q8_1

from test_gpu_parity import check_close, gpu_repacked, nan_like, run_gemv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    bqg_build.build()
    return bqg.load()


@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("fmt,xf,K", [(Q8_0, BF16, 65536), (Q4_0, BF16, 65536), (Q4_0, Q8_1, 65536),
                                      (BF16, BF16, 16384)])
def test_gemv_at_the_largest_k(ora, fmt, xf, K, M):
    run_gemv(ora, fmt, xf, M, 40, K, seed=K + M)


@pytest.mark.parametrize("fn,fmt,K", [("gemv_q8_0", Q8_0, 65536 + 32), ("gemv_q4_0", Q4_0, 65536 + 32),
                                      ("gemv_bf16", BF16, 16384 + 32)])
def test_gemv_refuses_k_beyond_the_largest(fn, fmt, K):
    # weights of the full repacked size, so that the binding's size check
    # passes and the library's own shape check is what refuses
    Wp = torch.zeros(bqg.repacked_size(fmt, 8, K), dtype=torch.uint8, device="cuda")
    X = torch.zeros((1, K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bqg.BqgError) as e:
        getattr(bqg, fn)(Wp, X, 8, K, out=torch.zeros((1, 8), device="cuda"))
    assert e.value.status == 2


def degenerate_canonical(fmt, N, K, seed):
    """Random codes; per-row scale patterns: 0 everywhere, -0 everywhere,
    the smallest subnormal, the largest finite fp16, scattered zero blocks,
    then ordinary scales."""
    rng = np.random.default_rng(seed)
    nb, bb = K // 32, (34 if fmt == Q8_0 else 18)
    canon = rng.integers(0, 256, size=(N, nb, bb), dtype=np.uint8)
    if fmt == Q8_0:
        canon[5, :, 2:] = 0x80                                   # every code -128
    d = (rng.standard_normal((N, nb)) * 2e-4).astype(np.float16)
    bits = d.view(np.uint16)
    bits[0, :] = 0x0000                                          # +0
    bits[1, :] = 0x8000                                          # -0
    bits[2, :] = 0x0001                                          # 2^-24, subnormal
    bits[3, :] = 0x7BFF                                          # 65504
    bits[4, ::3] = 0x0000                                        # scattered zero blocks
    canon[:, :, 0:2] = bits.view(np.uint8).reshape(N, nb, 2)
    return canon.reshape(N, nb * bb)


@pytest.mark.parametrize("M", [2, 4, 8])
@pytest.mark.parametrize("fmt,xf", [(Q8_0, BF16), (Q4_0, BF16), (Q4_0, Q8_1)])
def test_gemv_degenerate_blocks_and_a_zero_row(ora, fmt, xf, M):
    N, K = 64, 4096
    if xf == BF16 and M >= 4:      # these calls take the tensor-core route
        op = bqg.OP_GEMV_Q8_0 if fmt == Q8_0 else bqg.OP_GEMV_Q4_0
        assert bqg.gemv_route(op, M, N, K) == bqg.ROUTE_TENSOR_CORE
    canon = degenerate_canonical(fmt, N, K, seed=M + fmt)
    Wp = gpu_repacked(fmt, canon, N, K)
    x = synth.activations_f32(M, K, seed=77)
    x[1, :] = 0.0                                                # an all-zero row
    if xf == BF16:
        xref = synth.bf16_bits(x)
        X = synth.bf16_tensor(xref)
        fn, op = ("gemv_q8_0", bqg.OP_GEMV_Q8_0) if fmt == Q8_0 else ("gemv_q4_0", bqg.OP_GEMV_Q4_0)
    else:
        xref = ora.quantize(Q8_1, x)
        X = synth.u8_tensor(xref).view(M, -1)
        fn, op = "gemv_q4_0_q8_1", bqg.OP_GEMV_Q4_0_Q8_1
    Y = nan_like((M, N))
    getattr(bqg, fn)(Wp, X, N, K, out=Y, ws=bqg.workspace(op, M, N, K))
    torch.cuda.synchronize()
    Yr, Ar = ora.gemv(fmt, canon, xf, xref, M, N, K, nthreads=8)
    check_close(Y, Yr, Ar, f"{fn} degenerate blocks M={M}")
    y = Y.cpu()
    assert not y[1].any(), "an all-zero activation row must give exact zeros"
    assert not y[:, 0].any() and not y[:, 1].any(), "rows with zero scales must give exact zeros"


def test_weights_smaller_than_their_layout_are_refused_before_launch():
    """The C boundary takes the weights as a bare pointer; the binding checks
    them against the repacked size of the call's shape and refuses a tensor
    that is too small (ValueError) before anything is enqueued."""
    N, K = 64, 256
    W = torch.zeros(bqg.repacked_size(bqg.Q4_0, N, K) - 16, dtype=torch.uint8, device="cuda")
    X = torch.zeros((1, K), dtype=torch.bfloat16, device="cuda")
    Y = torch.full((1, N), 7.0, device="cuda")
    torch.cuda.synchronize()
    with pytest.raises(ValueError, match="Wp holds"):
        bqg.gemv_q4_0(W, X, N, K, out=Y)
    torch.cuda.synchronize()
    assert torch.all(Y == 7.0)          # nothing ran


def test_tensor_on_another_device_is_refused_before_launch(monkeypatch):
    """The binding launches on the current device: a tensor that lives on
    another one is refused (ValueError) before anything is enqueued.  With
    one GPU the mismatch is made by pretending the current device is 1."""
    N, K = 64, 256
    W = torch.zeros(bqg.repacked_size(bqg.BF16, N, K), dtype=torch.uint8, device="cuda")
    X = torch.zeros((1, K), dtype=torch.bfloat16, device="cuda")
    Y = torch.full((1, N), 7.0, device="cuda")
    torch.cuda.synchronize()
    monkeypatch.setattr(bqg, "_current_device", lambda: 1)
    with pytest.raises(ValueError, match="current device is cuda:1"):
        bqg.gemv_bf16(W, X, N, K, out=Y)
    monkeypatch.undo()
    torch.cuda.synchronize()
    assert torch.all(Y == 7.0)          # nothing ran


@pytest.mark.parametrize("fmt", [BF16, Q8_0, Q4_0])
@pytest.mark.parametrize("K,tensor_core", [(5056, True), (5088, False)])
def test_tensor_core_route_at_its_largest_k(ora, fmt, K, tensor_core):
    """At M = 8 the tensor-core route stages the activation rows at a pitch of
    round_up(2K, 128) + 64 bytes within 80 KiB: K = 5056 is the largest that
    fits, K = 5088 goes to the lanes-per-row kernel.  Both match the oracle."""
    M, N = 8, 2437
    op = {BF16: bqg.OP_GEMV_BF16, Q8_0: bqg.OP_GEMV_Q8_0, Q4_0: bqg.OP_GEMV_Q4_0}[fmt]
    assert (bqg.gemv_route(op, M, N, K) == bqg.ROUTE_TENSOR_CORE) == tensor_core
    Wf = synth.weights_f32(N, K, seed=K + fmt)
    canon = synth.bf16_bits(Wf) if fmt == BF16 else ora.quantize(fmt, Wf)
    Wp = gpu_repacked(fmt, canon, N, K)
    xref = synth.bf16_bits(synth.activations_f32(M, K, seed=K + 1))
    Y = nan_like((M, N))
    fn = {BF16: bqg.gemv_bf16, Q8_0: bqg.gemv_q8_0, Q4_0: bqg.gemv_q4_0}[fmt]
    fn(Wp, synth.bf16_tensor(xref), N, K, out=Y, ws=bqg.workspace(op, M, N, K))
    torch.cuda.synchronize()
    Yr, Ar = ora.gemv(fmt, canon, BF16, xref, M, N, K, nthreads=8)
    check_close(Y, Yr, Ar, f"fmt {fmt} M=8 K={K}")

