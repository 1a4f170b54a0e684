"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every symbol include/bqgemv.h declares, and validates arguments on the host
before touching the device.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

import block_quantized_gemv_gb300 as bqg
from block_quantized_gemv_gb300 import build as bqg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bqgemv.h")


@pytest.fixture(scope="module")
def L():
    bqg_build.build()
    return bqg.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bqg_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("bqg_gemv_bf16", "bqg_gemv_q8_0", "bqg_gemv_q4_0_q8_1", "bqg_quantize_q8_1",
                 "bqg_repack_weights", "bqg_gemv_q4_0_q8_1_qkv", "bqg_gemv_q4_0_q8_1_gate_up_swiglu",
                 "bqg_gemm_q4_0_bf16", "bqg_debug_q4_0_q8_1_block_dots", "bqg_workspace_size",
                 "bqg_last_device_error", "bqg_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    # and the binding knows every one of them
    assert set(declared_functions()) <= set(bqg.EXPORTS)


def test_status_strings_and_version(L):
    assert bqg.version().startswith("bqgemv")
    for s in range(8):
        assert bqg.status_string(s) and "unknown" not in bqg.status_string(s)
    assert "unknown" in bqg.status_string(99)


def test_repacked_size_matches_the_oracle(L, ora):
    import oracle
    for fmt in (bqg.BF16, bqg.Q8_0, bqg.Q4_0):
        for N, K in ((1, 32), (7, 1056), (4096, 4096), (4096, 11008), (3, 65536)):
            assert bqg.repacked_size(fmt, N, K) == ora.repacked_size(fmt, N, K)
    assert bqg.repacked_size(bqg.Q4_0, 4, 48) == 0
    assert bqg.repacked_size(7, 4, 64) == 0


FAKE = 0x10000  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("call,status", [
    (lambda L: L.bqg_gemv_bf16(None, FAKE, FAKE, 1, 8, 64, None, 0, None), 1),
    (lambda L: L.bqg_gemv_bf16(FAKE, FAKE, FAKE, 3, 8, 64, None, 0, None), 1),     # M = 3
    (lambda L: L.bqg_gemv_bf16(FAKE, FAKE, FAKE, 1, -1, 64, None, 0, None), 1),    # N < 0
    (lambda L: L.bqg_gemv_q8_0(FAKE, FAKE, FAKE, 1, 8, 48, None, 0, None), 2),     # K % 32
    (lambda L: L.bqg_gemv_q4_0(FAKE, FAKE, FAKE, 1, 8, 0, None, 0, None), 2),      # K = 0
    (lambda L: L.bqg_gemv_bf16(FAKE, FAKE, FAKE, 1, 8, 32768, None, 0, None), 2),  # bf16 K limit
    (lambda L: L.bqg_gemv_q4_0_q8_1(FAKE + 8, FAKE, FAKE, 1, 8, 64, None, 0, None), 3),
    (lambda L: L.bqg_gemv_q4_0_q8_1(FAKE, FAKE + 2, FAKE, 1, 8, 64, None, 0, None), 3),
    (lambda L: L.bqg_quantize_q8_1(FAKE, 9, FAKE, 1, 64, None), 1),                # dtype
    (lambda L: L.bqg_quantize_q8_1(FAKE, 0, FAKE, 0, 64, None), 1),                # M = 0
    (lambda L: L.bqg_repack_weights(5, FAKE, FAKE, 4, 64, None), 1),
    (lambda L: L.bqg_repack_weights(2, FAKE, FAKE + 4, 4, 64, None), 3),
    (lambda L: L.bqg_gemm_q4_0_bf16(FAKE, FAKE, FAKE, 100, 128, 64, None, 0, None), 2),  # M % 128
    (lambda L: L.bqg_gemm_q4_0_bf16(FAKE, FAKE, FAKE, 128, 128, 96, None, 0, None), 2),  # K % 64
    (lambda L: L.bqg_gemv_q4_0_q8_1_qkv(FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 1, 8, 8, 64, None, 0, None), 1),
    (lambda L: L.bqg_gemv_q4_0_q8_1_gate_up_swiglu(FAKE, FAKE, FAKE, FAKE, 2, 8, 40, None, 0, None), 2),
    (lambda L: L.bqg_debug_q4_0_q8_1_block_dots(FAKE, FAKE, None, 8, 64, None), 1),
    (lambda L: L.bqg_rmsnorm_quantize_q8_1(FAKE, 0, None, -1.0, FAKE, 1, 64, None), 1),          # eps < 0
    (lambda L: L.bqg_rmsnorm_quantize_q8_1(FAKE, 0, None, float("nan"), FAKE, 1, 64, None), 1),  # eps NaN
    (lambda L: L.bqg_rmsnorm_quantize_q8_1(FAKE, 0, FAKE + 2, 1e-5, FAKE, 1, 64, None), 3),     # gamma
    (lambda L: L.bqg_rmsnorm_quantize_q8_1(FAKE, 0, None, 1e-5, FAKE, 1, 40, None), 2),         # K % 32
    (lambda L: L.bqg_gemv_q4_0_q8_1_gate_up_swiglu_q8_1(FAKE, FAKE, FAKE, FAKE, 1, 40, 64, None, 0, None), 2),  # N % 32
    (lambda L: L.bqg_gemv_q4_0_q8_1_gate_up_swiglu_q8_1(FAKE, FAKE, FAKE, FAKE + 2, 1, 64, 64, None, 0, None), 3),
    # persistent decode layer: (xa, xb, dtype, Wq, Wk, Wv, Wg, Wu, Wd, Yq, Yk, Yv, Y, M, Nq, Nkv, Nff, K, ws, bytes, s)
    (lambda L: L.bqg_decode_layer_q4_0_q8_1(FAKE, FAKE, 0, *[FAKE] * 10, 1, 64, 64, 128, 64, None, 0, None), 1),   # ws
    (lambda L: L.bqg_decode_layer_q4_0_q8_1(FAKE, FAKE, 7, *[FAKE] * 10, 1, 64, 64, 128, 64, FAKE, 1 << 20, None), 1),
    (lambda L: L.bqg_decode_layer_q4_0_q8_1(FAKE, FAKE, 0, *[FAKE] * 10, 2, 64, 64, 128, 64, FAKE, 1 << 20, None), 2),
    (lambda L: L.bqg_decode_layer_q4_0_q8_1(FAKE, FAKE, 0, *[FAKE] * 10, 1, 64, 64, 120, 64, FAKE, 1 << 20, None), 2),
    (lambda L: L.bqg_decode_layer_q4_0_q8_1(FAKE, FAKE, 0, *[FAKE] * 10, 1, 64, 0, 128, 64, FAKE, 1 << 20, None), 1),
    (lambda L: L.bqg_decode_layer_q4_0_q8_1(FAKE, FAKE, 0, FAKE + 8, *[FAKE] * 9, 1, 64, 64, 128, 64, FAKE, 1 << 20,
                                            None), 3),
    (lambda L: L.bqg_decode_layer_q4_0_q8_1(FAKE, FAKE, 0, *[FAKE] * 10, 1, 64, 64, 128, 64, FAKE, 64, None), 7),
    # SM copy and host alias: (dst, src, bytes, stream), (host, &dev)
    (lambda L: L.bqg_copy_sm(None, FAKE, 16, None), 1),
    (lambda L: L.bqg_copy_sm(FAKE, FAKE + 0x1008, 16, None), 3),       # src not 16-byte aligned
    (lambda L: L.bqg_copy_sm(FAKE, FAKE + 0x1000, 24, None), 3),       # bytes % 16
    (lambda L: L.bqg_copy_sm(FAKE + 16, FAKE, 64, None), 1),           # overlapping ranges
    (lambda L: L.bqg_copy_sm(FAKE, FAKE + 48, 64, None), 1),
    (lambda L: L.bqg_host_alias(None, FAKE), 1),
    (lambda L: L.bqg_host_alias(FAKE, None), 1),
])
def test_host_validation_rejects_before_launch(L, call, status):
    assert call(L) == status


def test_no_device_is_an_error_not_a_fallback(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid-looking arguments reach the device check, which must fail loudly
    st = L.bqg_gemv_bf16(FAKE, FAKE, FAKE, 1, 8, 64, None, 0, None)
    assert st in (4, 5)
    assert L.bqg_workspace_size(0, 1, 8, 64) == 0
    out = ctypes.c_int(0)
    assert L.bqg_last_device_error(None, None) == 1
    assert L.bqg_copy_sm(FAKE, FAKE + 0x1000, 16, None) in (4, 5)
    dev = ctypes.c_void_p(0)
    assert L.bqg_host_alias(FAKE, ctypes.addressof(dev)) in (4, 5)
    assert L.bqg_copy_sm(FAKE, FAKE + 0x1000, 0, None) in (4, 5)    # even an empty copy checks the device


def test_pdl_switch_roundtrip(L):
    prev = bqg.set_pdl(True)
    assert bqg.set_pdl(prev) is True


def test_tensor_on_another_device_is_refused():
    # the binding launches on the current device; a tensor elsewhere is an error, not a launch
    bqg.check_device(0, 0, "X")
    with pytest.raises(ValueError, match="cuda:1"):
        bqg.check_device(1, 0, "X")
