"""The persistent decode layer (one launch: q8_1 of both activation rows,
QKV, gate+up+SwiGLU written as q8_1, grid barrier, down projection) against
the oracle, stage by stage, through the entry point the benchmark times.

  * QKV outputs: within |dy| <= 1e-3 * sum|w x| + 1e-6 of the oracle on q8_1(xa);
  * h: its q8_1 blocks (read from the workspace) dequantize to within the
    SwiGLU bound plus half a quantization step of the oracle's h, and at the
    decode shape they are byte for byte those of the separate entry points
    (same arithmetic, same order);
  * down output: within the same bound of the oracle on those blocks;
  * the workspace's counters and barrier are re-armed: a second call gives
    the same bytes and leaves them zero.
"""
import numpy as np
import pytest
import torch

import block_quantized_gemv_gb300 as bqg
from block_quantized_gemv_gb300 import build as bqg_build
from block_quantized_gemv_gb300 import synth
from oracle import Q4_0, Q8_1

from test_gpu_parity import check_close, gpu_repacked, make_weights, nan_like, swiglu_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    bqg_build.build()
    return bqg.load()


def run_layer(ora, K, Nq, Nkv, Nff, dtype, seed):
    shapes = {"q": (Nq, K), "k": (Nkv, K), "v": (Nkv, K), "g": (Nff, K), "u": (Nff, K), "d": (K, Nff)}
    canon = {k: make_weights(ora, Q4_0, n, kk, seed=seed + i)[1] for i, (k, (n, kk)) in enumerate(shapes.items())}
    Wp = {k: gpu_repacked(Q4_0, canon[k], *shapes[k]) for k in canon}
    xs = [synth.rms_normalised_f32(1, K, seed=seed + 10 + j) for j in range(2)]
    if dtype == "bf16":
        bits = [synth.bf16_bits(x) for x in xs]
        xt = [synth.bf16_tensor(b) for b in bits]
        xval = [t.float().cpu().numpy() for t in xt]
    else:
        xt = [torch.from_numpy(x).cuda() for x in xs]
        xval = xs
    ws = bqg.workspace(bqg.OP_DECODE_LAYER_Q4_0_Q8_1, 1, Nff, K)
    out = tuple(nan_like((1, n)) for n in (Nq, Nkv, Nkv, K))
    bqg.decode_layer_q4_0_q8_1(xt[0], xt[1], Wp["q"], Wp["k"], Wp["v"], Wp["g"], Wp["u"], Wp["d"], Nq, Nkv, Nff, K,
                               out=out, ws=ws)
    torch.cuda.synchronize()
    xqa, xqb = ora.quantize(Q8_1, xval[0]), ora.quantize(Q8_1, xval[1])
    for name, y, n in zip("qkv", out[:3], (Nq, Nkv, Nkv)):
        Yr, Ar = ora.gemv(Q4_0, canon[name], Q8_1, xqa, 1, n, K, nthreads=16)
        check_close(y, Yr, Ar, f"layer {name} K={K}")
    hq = bqg.layer_hq(ws, Nff).cpu().numpy().copy()
    Yg, Ag = ora.gemv(Q4_0, canon["g"], Q8_1, xqb, 1, Nff, K, nthreads=16)
    Yu, Au = ora.gemv(Q4_0, canon["u"], Q8_1, xqb, 1, Nff, K, nthreads=16)
    h_ref, bound = swiglu_bound(ora, Yg, Ag, Yu, Au)
    deq = ora.dequantize(Q8_1, hq, 1, Nff)
    d = np.frombuffer(hq.reshape(Nff // 32, 36)[:, 0:2].copy().tobytes(), dtype=np.float16).astype(np.float64)
    half_step = np.repeat(d / 2, 32).reshape(1, Nff)
    assert np.all(np.abs(deq - h_ref) <= bound + half_step * (1 + 2.0 ** -10)), \
        float(np.max(np.abs(deq - h_ref) - bound - half_step))
    Yr, Ar = ora.gemv(Q4_0, canon["d"], Q8_1, hq, 1, K, Nff, nthreads=16)
    check_close(out[3], Yr, Ar, f"layer down K={K} Nff={Nff}")
    # re-armed: counters and barrier arrivals back at zero, same bytes again
    up16 = lambda b: (b + 15) // 16 * 16
    wsn = ws.cpu().numpy()
    c0 = up16(Nff * 4)
    assert not wsn[c0:c0 + Nff // 32 * 4].any(), "block counters not re-armed"
    g0 = up16(c0 + Nff // 32 * 4) + up16(Nff // 32 * 36)
    assert not wsn[g0:g0 + 4].any(), "barrier arrivals not re-armed"
    out2 = tuple(nan_like((1, n)) for n in (Nq, Nkv, Nkv, K))
    bqg.decode_layer_q4_0_q8_1(xt[0], xt[1], Wp["q"], Wp["k"], Wp["v"], Wp["g"], Wp["u"], Wp["d"], Nq, Nkv, Nff, K,
                               out=out2, ws=ws)
    torch.cuda.synchronize()
    for a, b in zip(out, out2):
        assert torch.equal(a, b)
    assert np.array_equal(bqg.layer_hq(ws, Nff).cpu().numpy(), hq)
    assert bqg.last_device_error() == 0
    return Wp, xt, hq


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("K,Nq,Nkv,Nff", [(1024, 256, 64, 512), (1056, 101, 37, 1056), (4096, 512, 128, 2048)])
def test_decode_layer_small(ora, K, Nq, Nkv, Nff, dtype):
    run_layer(ora, K, Nq, Nkv, Nff, dtype, seed=K + Nq + Nff)


def test_decode_layer_c3_shape_matches_the_separate_entries(ora):
    """C3: K=4096, QKV 3 x 4096, gate/up 2 x 11008, down 4096 x 11008."""
    K, Nq, Nff = 4096, 4096, 11008
    Wp, xt, hq = run_layer(ora, K, Nq, Nq, Nff, "bf16", seed=70)
    xqb = bqg.quantize_q8_1(xt[1])
    hq2 = bqg.gemv_q4_0_q8_1_gate_up_swiglu_q8_1(Wp["g"], Wp["u"], xqb, Nff, K,
                                                 ws=bqg.workspace(bqg.OP_GATE_UP_Q8_1_Q4_0_Q8_1, 1, Nff, K))
    torch.cuda.synchronize()
    assert np.array_equal(hq2.cpu().numpy().reshape(-1), hq.reshape(-1))


def test_decode_layer_rejects_small_workspace():
    K, Nq, Nff = 1024, 256, 512
    z = torch.zeros(1, dtype=torch.uint8, device="cuda")

    def w(n, k):           # zero weights of the repacked size (the binding checks it)
        return torch.zeros(bqg.repacked_size(bqg.Q4_0, n, k), dtype=torch.uint8, device="cuda")

    with pytest.raises(bqg.BqgError) as e:
        bqg.decode_layer_q4_0_q8_1(torch.zeros((1, K), dtype=torch.bfloat16, device="cuda"),
                                   torch.zeros((1, K), dtype=torch.bfloat16, device="cuda"),
                                   w(Nq, K), w(Nq, K), w(Nq, K), w(Nff, K), w(Nff, K), w(K, Nff),
                                   Nq, Nq, Nff, K, ws=z)
    assert e.value.status == 7


def test_decode_layer_barrier_timeout_is_reported_and_recoverable(ora):
    """The grid barrier's bounded wait, made to run out without any fault: the
    workspace's arrival count is preset (against the zero-workspace contract)
    so that no arrival can ever complete the barrier.  Every CTA gives up
    after about a second, sets the error word, drains its copies and exits;
    the host reads the error, and after the workspace is zeroed again the
    same context computes the layer correctly."""
    K, Nq, Nkv, Nff = 1024, 256, 64, 512
    up16 = lambda b: (b + 15) // 16 * 16
    gbar = up16(Nff * 4) + up16(Nff // 32 * 4) + up16(Nff // 32 * 36)
    shapes = {"q": (Nq, K), "k": (Nkv, K), "v": (Nkv, K), "g": (Nff, K), "u": (Nff, K), "d": (K, Nff)}
    canon = {k: make_weights(ora, Q4_0, n, kk, seed=90 + i)[1] for i, (k, (n, kk)) in enumerate(shapes.items())}
    Wp = {k: gpu_repacked(Q4_0, canon[k], *shapes[k]) for k in canon}
    x = synth.bf16_tensor(synth.bf16_bits(synth.rms_normalised_f32(1, K, seed=99)))
    ws = bqg.workspace(bqg.OP_DECODE_LAYER_Q4_0_Q8_1, 1, Nff, K)
    assert bqg.last_device_error() == 0
    ws[gbar:gbar + 4] = torch.tensor([0xff, 0xff, 0xff, 0x7f], dtype=torch.uint8, device="cuda")
    args = (x, x, Wp["q"], Wp["k"], Wp["v"], Wp["g"], Wp["u"], Wp["d"], Nq, Nkv, Nff, K)
    bqg.decode_layer_q4_0_q8_1(*args, ws=ws)
    torch.cuda.synchronize()
    assert bqg.last_device_error() != 0
    assert bqg.last_device_error() == 0            # read and cleared
    ws.zero_()
    Yq, Yk, Yv, Y = bqg.decode_layer_q4_0_q8_1(*args, ws=ws)
    torch.cuda.synchronize()
    assert bqg.last_device_error() == 0
    xq = ora.quantize(Q8_1, x.float().cpu().numpy())
    Yr, Ar = ora.gemv(Q4_0, canon["q"], Q8_1, xq, 1, Nq, K, nthreads=16)
    check_close(Yq.view(1, -1), Yr, Ar, "layer q after a barrier timeout")
    hq = bqg.layer_hq(ws, Nff).cpu().numpy().copy()
    Yr, Ar = ora.gemv(Q4_0, canon["d"], Q8_1, hq, 1, K, Nff, nthreads=16)
    check_close(Y.view(1, -1), Yr, Ar, "layer down after a barrier timeout")
