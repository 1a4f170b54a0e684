"""The binding's host-side checks, on the CPU.

The C boundary takes weights as bare pointers, so the binding checks each
weight tensor against the size of the repacked layout before calling the
library.  Here a stand-in library records the calls: every entry point
passes operands of exactly the required size through, and refuses a weight
tensor one byte short (ValueError naming it) before anything reaches the
library.  The binding's layout formula is checked against the library's
own bqg_repacked_size."""
import pytest
import torch

import block_quantized_gemv_gb300 as bqg
from block_quantized_gemv_gb300 import build as bqg_build
from block_quantized_gemv_gb300 import BF16, Q4_0, Q8_0, Q8_1


def test_weight_bytes_matches_the_library():
    bqg_build.build()
    L = bqg.load()
    for fmt in (BF16, Q8_0, Q4_0):
        for N in (1, 7, 128, 4096):
            for K in (32, 64, 992, 1024, 1056, 4096, 11008, 65536, 65568):
                assert bqg.weight_bytes(fmt, N, K) == L.bqg_repacked_size(fmt, N, K), (fmt, N, K)
        for N, K in ((4, 0), (4, 48), (4, -32), (0, 64)):
            assert bqg.weight_bytes(fmt, N, K) is None       # the library refuses these shapes itself


class StubLib:
    """Stands in for libbqgemv: records which entry point was called."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def entry(*args):
            self.calls.append(name)
            return 0
        return entry


@pytest.fixture
def stub(monkeypatch):
    lib = StubLib()

    def dev(t, name, dtype=None, numel=None):      # as _dev, for CPU tensors
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a tensor")
        bqg._check_tensor(t, name, dtype, numel)
        return 16

    monkeypatch.setattr(bqg, "load", lambda path=None: lib)
    monkeypatch.setattr(bqg, "_dev", dev)
    monkeypatch.setattr(bqg, "_dev_or_host", dev)
    monkeypatch.setattr(bqg, "_stream", lambda stream=None: 0)
    return lib


def u8(n):
    return torch.zeros(n, dtype=torch.uint8)


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def q8_1(M, K):
    return torch.zeros((M, bqg.row_bytes(Q8_1, K)), dtype=torch.uint8)


N, K, M = 100, 1056, 2          # K = 33 blocks: two tiles per repacked row
Nq, Nkv, Nff = 96, 64, 160


def cases():
    """(C entry point, {weight name: (format, rows, cols)}, call(weights))"""
    wb = bqg.weight_bytes
    yield ("bqg_gemv_bf16", {"Wp": (BF16, N, K)}, lambda w: bqg.gemv_bf16(w["Wp"], bf16(M, K), N, K))
    yield ("bqg_gemv_q8_0", {"Wp": (Q8_0, N, K)}, lambda w: bqg.gemv_q8_0(w["Wp"], bf16(M, K), N, K))
    yield ("bqg_gemv_q4_0", {"Wp": (Q4_0, N, K)}, lambda w: bqg.gemv_q4_0(w["Wp"], bf16(M, K), N, K))
    yield ("bqg_gemv_q4_0_q8_1", {"Wp": (Q4_0, N, K)}, lambda w: bqg.gemv_q4_0_q8_1(w["Wp"], q8_1(M, K), N, K))
    yield ("bqg_gemv_q4_0_q8_1_noalloc", {"Wp": (Q4_0, N, K)},
           lambda w: bqg.gemv_q4_0_q8_1_noalloc(w["Wp"], q8_1(M, K), N, K))
    yield ("bqg_gemv_q4_0_q8_1_qkv", {"Wq": (Q4_0, Nq, K), "Wk": (Q4_0, Nkv, K), "Wv": (Q4_0, Nkv, K)},
           lambda w: bqg.gemv_q4_0_q8_1_qkv(w["Wq"], w["Wk"], w["Wv"], q8_1(M, K), Nq, Nkv, K))
    yield ("bqg_gemv_q4_0_q8_1_gate_up_swiglu", {"Wg": (Q4_0, Nff, K), "Wu": (Q4_0, Nff, K)},
           lambda w: bqg.gemv_q4_0_q8_1_gate_up_swiglu(w["Wg"], w["Wu"], q8_1(M, K), Nff, K))
    yield ("bqg_gemv_q4_0_q8_1_gate_up_swiglu_q8_1", {"Wg": (Q4_0, Nff, K), "Wu": (Q4_0, Nff, K)},
           lambda w: bqg.gemv_q4_0_q8_1_gate_up_swiglu_q8_1(w["Wg"], w["Wu"], q8_1(M, K), Nff, K))
    layer = {"Wq": (Q4_0, Nq, K), "Wk": (Q4_0, Nkv, K), "Wv": (Q4_0, Nkv, K), "Wg": (Q4_0, Nff, K),
             "Wu": (Q4_0, Nff, K), "Wd": (Q4_0, K, Nff)}      # the down projection: K rows of Nff
    yield ("bqg_decode_layer_q4_0_q8_1", layer,
           lambda w: bqg.decode_layer_q4_0_q8_1(bf16(1, K), bf16(1, K), w["Wq"], w["Wk"], w["Wv"], w["Wg"],
                                                w["Wu"], w["Wd"], Nq, Nkv, Nff, K))
    yield ("bqg_gemm_q4_0_bf16", {"Wp": (Q4_0, 256, K)}, lambda w: bqg.gemm_q4_0_bf16(w["Wp"], bf16(128, K), 256, K))
    yield ("bqg_gemm_q8_0_bf16", {"Wp": (Q8_0, 256, K)}, lambda w: bqg.gemm_q8_0_bf16(w["Wp"], bf16(128, K), 256, K))
    yield ("bqg_debug_q4_0_q8_1_block_dots", {"Wp": (Q4_0, N, K)},
           lambda w: bqg.debug_q4_0_q8_1_block_dots(w["Wp"], q8_1(1, K), N, K))
    yield ("bqg_debug_q4_0_q8_1_block_dots_kslice", {"Wp": (Q4_0, N, K)},
           lambda w: bqg.debug_q4_0_q8_1_block_dots_kslice(w["Wp"], q8_1(1, K), N, K))
    assert wb(Q4_0, K, Nff) != wb(Q4_0, Nff, K)      # the down projection's shape matters


CASES = list(cases())


@pytest.mark.parametrize("entry,weights,call", CASES, ids=[c[0] for c in CASES])
def test_exactly_sized_weights_pass_through(stub, entry, weights, call):
    call({n: u8(bqg.weight_bytes(*s)) for n, s in weights.items()})
    assert stub.calls == [entry]


@pytest.mark.parametrize("entry,weights,call", CASES, ids=[c[0] for c in CASES])
def test_a_weight_one_byte_short_is_refused_before_the_library(stub, entry, weights, call):
    for short in weights:
        w = {n: u8(bqg.weight_bytes(*s) - (n == short)) for n, s in weights.items()}
        with pytest.raises(ValueError, match=f"{short} holds"):
            call(w)
    assert stub.calls == []
