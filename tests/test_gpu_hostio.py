"""Host memory on the CPU-GPU link: bqg_host_alias, bqg_copy_sm, and GEMV
outputs written straight into page-locked host memory.

  * bqg_copy_sm moves every byte (device to device, host to device, device
    to host) at sizes from one 16-byte piece to several MB with ragged
    tails, and writes nothing past the end;
  * a GEMV given a pinned host Y writes the same bits as the same call with a
    device Y (same kernel, same order), on the single-pass and the split-K
    paths, and those bits are within |dy| <= 1e-3 * sum|w x| + 1e-6 of the oracle;
  * a chain of steps (copy in, GEMV out) enqueued back to back with
    programmatic dependent launch on keeps stream order: every step sees its
    own activation and leaves its own output.
"""
import numpy as np
import pytest
import torch

import block_quantized_gemv_gb300 as bqg
from block_quantized_gemv_gb300 import build as bqg_build
from block_quantized_gemv_gb300 import synth
from oracle import BF16, Q4_0, Q8_0, Q8_1

from test_gpu_parity import check_close, gpu_repacked, make_weights, nan_like

pytestmark = pytest.mark.gpu

FN = {BF16: "gemv_bf16", Q8_0: "gemv_q8_0", Q4_0: "gemv_q4_0"}
OP = {"gemv_bf16": bqg.OP_GEMV_BF16, "gemv_q8_0": bqg.OP_GEMV_Q8_0, "gemv_q4_0": bqg.OP_GEMV_Q4_0,
      "gemv_q4_0_q8_1": bqg.OP_GEMV_Q4_0_Q8_1}


@pytest.fixture(scope="module", autouse=True)
def lib():
    bqg_build.build()
    return bqg.load()


def pinned(shape, dtype):
    return torch.empty(shape, dtype=dtype).pin_memory()


@pytest.mark.parametrize("where", ["d2d", "h2d", "d2h"])
@pytest.mark.parametrize("nbytes", [16, 8192, 8192 + 48, 4 << 20, (4 << 20) + 16 * 257])
def test_copy_sm_moves_every_byte(where, nbytes):
    g = torch.Generator().manual_seed(nbytes)
    ref = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g)
    src = ref.pin_memory() if where == "h2d" else ref.cuda()
    if where == "d2h":
        dst = pinned((nbytes + 64,), torch.uint8)
        dst.zero_()
    else:
        dst = torch.zeros(nbytes + 64, dtype=torch.uint8, device="cuda")
    bqg.copy_sm(dst, src)
    torch.cuda.synchronize()
    got = dst.cpu()
    assert torch.equal(got[:nbytes], ref)
    assert not got[nbytes:].any(), "bytes written past the end"
    assert bqg.last_device_error() == 0


def test_copy_sm_empty_launches_nothing():
    dst = torch.full((32,), 7, dtype=torch.uint8, device="cuda")
    bqg.copy_sm(dst, torch.empty(0, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert bool((dst == 7).all())


def test_host_alias_of_pinned_memory_and_of_pageable_memory():
    t = pinned((1024,), torch.float32)
    assert bqg.host_alias(t) != 0
    # pageable memory: an error status (nothing left pending), or on a node
    # whose driver maps all host memory, a usable address
    try:
        a = bqg.host_alias(torch.zeros(1024))
        assert a != 0
    except bqg.BqgError as e:
        assert e.status == 5
    x = torch.ones(64, device="cuda")
    assert float((x * 2).sum().item()) == 128.0      # the context is healthy
    with pytest.raises(TypeError):
        bqg.gemv_bf16(torch.zeros(64, dtype=torch.uint8, device="cuda"),
                      torch.zeros((1, 32), dtype=torch.bfloat16, device="cuda"), 1, 32,
                      out=torch.zeros((1, 1)))       # pageable CPU output: refused by the binding


def weights_and_x(ora, fmt, xf, M, N, K, seed):
    _, canon = make_weights(ora, fmt, N, K, seed=seed)
    Wp = gpu_repacked(fmt, canon, N, K)
    if xf == BF16:
        xref = synth.bf16_bits(synth.activations_f32(M, K, seed=seed + 1))
        X = synth.bf16_tensor(xref)
        fn = FN[fmt]
    else:
        xref = ora.quantize(Q8_1, synth.rms_normalised_f32(M, K, seed=seed + 1))
        X = synth.u8_tensor(xref).view(M, -1)
        fn = "gemv_q4_0_q8_1"
    return canon, Wp, X, xref, fn


@pytest.mark.parametrize("fmt,xf", [(BF16, BF16), (Q8_0, BF16), (Q4_0, BF16), (Q4_0, Q8_1)])
@pytest.mark.parametrize("M,N,K", [(1, 1000, 4096), (2, 392, 1056), (1, 24, 16384), (1, 12288, 4096)])
def test_gemv_output_in_pinned_host_memory(ora, fmt, xf, M, N, K):
    canon, Wp, X, xref, fn = weights_and_x(ora, fmt, xf, M, N, K, seed=N + K + M)
    ws = bqg.workspace(OP[fn], M, N, K)
    Yd = nan_like((M, N))
    getattr(bqg, fn)(Wp, X, N, K, out=Yd, ws=ws)
    Yh = pinned((M, N), torch.float32)
    Yh.fill_(float("nan"))
    getattr(bqg, fn)(Wp, X, N, K, out=Yh, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(Yh, Yd.cpu()), "host output differs from the device output"
    if N * K <= 1 << 22:
        Yr, Ar = ora.gemv(fmt, canon, xf, xref, M, N, K, nthreads=8)
        check_close(Yh, Yr, Ar, f"{fn} host Y M={M} N={N} K={K}")


def test_noalloc_gemv_output_in_pinned_host_memory(ora):
    M, N, K = 1, 40, 8192
    canon, Wp, X, xref, fn = weights_and_x(ora, Q4_0, Q8_1, M, N, K, seed=3)
    Yh = pinned((M, N), torch.float32)
    Yh.fill_(float("nan"))
    bqg.gemv_q4_0_q8_1_noalloc(Wp, X, N, K, out=Yh)
    torch.cuda.synchronize()
    Yr, Ar = ora.gemv(Q4_0, canon, Q8_1, xref, M, N, K, nthreads=8)
    check_close(Yh, Yr, Ar, "noalloc host Y")


@pytest.mark.parametrize("pdl", [True, False])
def test_chained_steps_copy_in_and_write_out_keep_stream_order(ora, pdl):
    """Eight steps enqueued without a host sync: step i copies its own pinned
    activation row into ONE device buffer and writes its own pinned output.
    A step that read the buffer before its copy landed, or a copy that
    overwrote it while the previous GEMV still read it, changes the bits."""
    M, N, K, S = 1, 4096, 4096, 8
    _, canon = make_weights(ora, BF16, N, K, seed=21)
    Wp = gpu_repacked(BF16, canon, N, K)
    xs = [synth.bf16_tensor(synth.bf16_bits(synth.activations_f32(M, K, seed=300 + i))) for i in range(S)]
    ref = []
    for x in xs:
        y = nan_like((M, N))
        bqg.gemv_bf16(Wp, x, N, K, out=y)
        ref.append(y)
    torch.cuda.synchronize()
    xh = [x.cpu().pin_memory() for x in xs]
    yh = [pinned((M, N), torch.float32) for _ in range(S)]
    for y in yh:
        y.fill_(float("nan"))
    Xd = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    prev = bqg.set_pdl(pdl)
    try:
        for i in range(S):
            bqg.copy_sm(Xd, xh[i])
            bqg.gemv_bf16(Wp, Xd, N, K, out=yh[i])
        torch.cuda.synchronize()
    finally:
        bqg.set_pdl(prev)
    for i in range(S):
        assert torch.equal(yh[i], ref[i].cpu()), f"step {i}"
    assert bqg.last_device_error() == 0
