"""The arithmetic behind the prefill GEMM's packed-bf16 q4_0 dequantization,
checked exhaustively on the CPU (every finite fp16 scale x every 4-bit code).

The kernel forms each weight (q - 8) * d rounded once to bf16 (the prefill
tile of "llama-3x-prompt-speed": the weight tile dequantized to bf16) without
fp32 arithmetic:
  * e = q - 8 from the bf16 bit pattern 0x43 n (= 128 + n) minus 136;
  * d = dh + dl with dh = bf16(d) (round to nearest even) and dl = d - dh;
  * one bf16 fused multiply-add r = RN(e * dh + RN(e * dl)).
That equals RN_bf16(e * d) for every input exactly when
  (1) 0x43 n is 128 + n and 128 + n - 136 is exact in bf16,
  (2) dl is a bf16 value (so it is passed without rounding),
  (3) e * dl is a bf16 value (so the product before the FMA is exact);
then e * dh + e * dl = e * d exactly and the FMA rounds it once.  (4) No
value leaves bf16's normal range.  The GPU tests check the kernel's outputs;
this test checks the identity they rest on for all 1 048 576 (d, q) pairs.
"""
import numpy as np
import torch


def bf16_rne(a64):
    """float64 values that are exact in float32 -> nearest-even bf16, as float64"""
    return torch.from_numpy(np.asarray(a64, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def is_bf16(a64):
    return np.array_equal(bf16_rne(a64), a64)


def bf16_bits_value(bits):
    return torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16) \
        .to(torch.float64).numpy()


def test_code_pattern_is_128_plus_n_and_the_shift_is_exact():
    n = np.arange(16)
    v = bf16_bits_value(0x4300 | n)
    assert np.array_equal(v, 128.0 + n)
    assert np.array_equal(bf16_rne(v - 136.0), n - 8.0)


def test_scale_split_and_products_are_exact_for_every_fp16_scale():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    d = bits.view(np.float16).astype(np.float64)
    d = d[np.isfinite(d)]                                  # 63 488 finite scales, both zeros included
    dh = bf16_rne(d)
    dl = d - dh                                            # exact in float64
    assert np.array_equal(np.asarray(dl, np.float32).astype(np.float64), dl), "d - dh not exact in fp32"
    assert is_bf16(dl), "the remainder of an fp16 scale is not a bf16 value"
    e = np.arange(-8, 8, dtype=np.float64)[:, None]
    prod_lo = e * dl                                       # exact in float64
    assert is_bf16(prod_lo), "(q - 8) * dl is not exact in bf16"
    exact = e * d                                          # at most 15 significant bits: exact in float64 and float32
    assert np.array_equal(e * dh + prod_lo, exact)
    # the FMA's single rounding of the exact sum is the bf16 rounding of the weight
    r = bf16_rne(exact)
    assert np.all(np.isfinite(r))
    nz = np.abs(exact[exact != 0])
    assert nz.min() >= 2.0 ** -24 and nz.max() <= 8 * 65504.0   # far inside bf16's normal range
    # and the rounding is what the config's one rounding of the fp32 product gives
    assert np.array_equal(r, bf16_rne(np.asarray(exact, np.float32).astype(np.float64)))


def test_q8_0_codes_do_not_admit_the_same_split():
    """Why q8_0 keeps its fp32 route: an 8-bit code times the remainder of
    the scale is not always a bf16 value."""
    d = np.array([1.0 + 3.0 / 1024.0])                     # remainder 3 / 1024 after bf16's 7 fraction bits
    dl = d - bf16_rne(d)
    assert dl[0] == 3.0 / 1024.0
    assert not is_bf16(np.array([127.0]) * dl)             # 127 * 3 = 381 needs 9 significant bits
