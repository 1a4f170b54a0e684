"""Pins that tie the CPU oracle to things other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with an independent fact:
  * values derived by hand for worked blocks (tests/golden/*.txt),
  * a library routine for special cases (numpy float16, torch bfloat16),
  * exact rational arithmetic on tiny inputs (Python fractions, decoding the
    raw bytes here with struct, independently of the C decoder),
  * closed forms and invariants of the block encodings.
They are plain functions so that ``test_oracle_pins`` can run them against the
real oracle and ``test_oracle_mutants`` against deliberately broken copies.
"""
from __future__ import annotations

import math
import os
import struct
from fractions import Fraction

import numpy as np

import oracle
from oracle import BF16, Q4_0, Q8_0, Q8_1

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            out[key.strip()] = val.split()
    return out


def _hexbytes(tokens):
    return np.array([int(t, 16) for t in tokens], dtype=np.uint8)


# ---------------------------------------------------------------------------
# independent decoders (struct's IEEE half, plain integer arithmetic)
# ---------------------------------------------------------------------------
def _half(b: bytes) -> Fraction:
    return Fraction(struct.unpack("<e", b)[0])


def _bf16(u: int) -> Fraction:
    return Fraction(struct.unpack("<f", struct.pack("<I", (u & 0xFFFF) << 16))[0])


def exact_row(fmt, row: bytes, K: int):
    """Exact rational values of one row of K elements, decoded in Python."""
    vals = []
    if fmt == BF16:
        for k in range(K):
            vals.append(_bf16(row[2 * k] | (row[2 * k + 1] << 8)))
        return vals
    nb = K // 32
    for b in range(nb):
        if fmt == Q8_0:
            blk = row[34 * b: 34 * b + 34]
            d = _half(blk[0:2])
            vals += [d * struct.unpack("<b", blk[2 + i: 3 + i])[0] for i in range(32)]
        elif fmt == Q8_1:
            blk = row[36 * b: 36 * b + 36]
            d = _half(blk[0:2])
            vals += [d * struct.unpack("<b", blk[4 + i: 5 + i])[0] for i in range(32)]
        elif fmt == Q4_0:
            blk = row[18 * b: 18 * b + 18]
            d = _half(blk[0:2])
            lo = [blk[2 + j] & 15 for j in range(16)]
            hi = [blk[2 + j] >> 4 for j in range(16)]
            vals += [d * (q - 8) for q in lo + hi]
    return vals


# ---------------------------------------------------------------------------
# scalar formats against library routines
# ---------------------------------------------------------------------------
def pin_fp16_decode_all_patterns(o):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    for b in range(0, 65536, 1):
        v = o.fp16_to_double(b)
        r = ref[b]
        if math.isnan(r):
            assert math.isnan(v), hex(b)
        else:
            assert v == r, (hex(b), v, r)


def pin_fp16_encode_vs_numpy(o):
    rng = np.random.default_rng(1234)
    xs = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6,
          2.0 ** -14, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -26, 1e-10,
          0.1, 1 / 3, 2049.0, 2051.0, 4097.0, 1 + 2 ** -11, 1 + 3 * 2 ** -11]
    # exact ties between binary16 neighbours in every binade (both parities)
    for e in range(-24, 16):
        for m in (1, 3, 1023, 1025, 2047):
            xs.append(float(np.float32(m * 2.0 ** (e - 11))))
    xs += list(rng.standard_normal(4000) * 10.0 ** rng.uniform(-9, 5, 4000))
    xs = np.array(xs, dtype=np.float32)
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    for x, r in zip(xs, ref):
        got = o.fp16_from_float(float(x))
        assert got == int(r), (float(x), hex(got), hex(int(r)))


def pin_bf16_decode_vs_torch(o):
    import torch
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    for b, r in zip(bits, ref):
        v = o.bf16_to_double(int(b))
        assert (math.isnan(v) and math.isnan(r)) or v == r, (hex(int(b)), v, r)


# ---------------------------------------------------------------------------
# hand-worked blocks
# ---------------------------------------------------------------------------
def pin_q4_0_hand_block(o):
    g = _read_golden("q4_0_hand_block.txt")
    x = np.array([float(t) for t in g["x"]], dtype=np.float32)
    got = o.quantize(Q4_0, x)[0]
    assert np.array_equal(got, _hexbytes(g["bytes"])), got
    vals = o.dequantize(Q4_0, got, 1, 32)[0]
    assert np.array_equal(vals, np.array([float(t) for t in g["values"]])), vals


def pin_q8_0_hand_block(o):
    g = _read_golden("q8_0_hand_block.txt")
    x = np.array([float(t) for t in g["x"]], dtype=np.float32)
    got = o.quantize(Q8_0, x)[0]
    assert np.array_equal(got, _hexbytes(g["bytes"])), got


def pin_q8_1_hand_blocks(o):
    g = _read_golden("q8_1_hand_blocks.txt")
    for tag in ("A", "B"):
        x = np.array([float(t) for t in g["x" + tag]], dtype=np.float32)
        got = o.quantize(Q8_1, x)[0]
        assert np.array_equal(got, _hexbytes(g["bytes" + tag])), (tag, got)


# ---------------------------------------------------------------------------
# brute force on tiny inputs, exact rational arithmetic
# ---------------------------------------------------------------------------
def _tiny_case(rng, wfmt, xfmt, M, N, K):
    Wf = rng.normal(0, 0.02, (N, K)).astype(np.float32)
    Xf = rng.normal(0, 1, (M, K)).astype(np.float32)
    if wfmt == BF16:
        W = _to_bf16_bits(Wf)
    else:
        W = o_quant(wfmt, Wf)
    if xfmt == BF16:
        X = _to_bf16_bits(Xf)
    else:
        X = o_quant(xfmt, Xf)
    return W, X


_Q = {}


def o_quant(fmt, x):
    # inputs for the brute-force pins come from the oracle under test
    return _Q["o"].quantize(fmt, x)


def _to_bf16_bits(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def pin_gemv_brute_force(o):
    _Q["o"] = o
    rng = np.random.default_rng(7)
    for wfmt in (BF16, Q8_0, Q4_0):
        for xfmt in (BF16, Q8_1):
            for (M, N, K) in ((1, 3, 32), (2, 5, 64), (1, 8, 64)):
                W, X = _tiny_case(rng, wfmt, xfmt, M, N, K)
                Y, A = o.gemv(wfmt, W, xfmt, X, M, N, K)
                wb = np.ascontiguousarray(W).view(np.uint8).reshape(N, -1)
                xb = np.ascontiguousarray(X).view(np.uint8).reshape(M, -1)
                for m in range(M):
                    xv = exact_row(xfmt, bytes(xb[m]), K)
                    for n in range(N):
                        wv = exact_row(wfmt, bytes(wb[n]), K)
                        exact = sum((a * b for a, b in zip(wv, xv)), Fraction(0))
                        absum = sum((abs(a * b) for a, b in zip(wv, xv)), Fraction(0))
                        # fp64 left-to-right sum: |err| <= K * 2^-53 * sum|wx| (products exact)
                        bound = K * 2.0 ** -52 * float(absum) + 1e-300
                        assert abs(Y[m, n] - float(exact)) <= bound, (wfmt, xfmt, m, n, Y[m, n], float(exact))
                        assert abs(A[m, n] - float(absum)) <= bound, (wfmt, xfmt, m, n)


def pin_block_dots_brute_force(o):
    _Q["o"] = o
    rng = np.random.default_rng(11)
    N, K = 6, 96
    W = o.quantize(Q4_0, rng.normal(0, 0.02, (N, K)).astype(np.float32))
    X = o.quantize(Q8_1, rng.normal(0, 1, (1, K)).astype(np.float32))
    dots = o.block_dots_q4_0_q8_1(W, X, N, K)
    xb = X.reshape(-1)
    for n in range(N):
        for b in range(K // 32):
            blk = W[n, 18 * b: 18 * b + 18]
            qw = [int(blk[2 + j]) & 15 for j in range(16)] + [int(blk[2 + j]) >> 4 for j in range(16)]
            qx = [int(np.int8(xb[36 * b + 4 + i])) for i in range(32)]
            assert dots[n, b] == sum((a - 8) * c for a, c in zip(qw, qx)), (n, b)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------
def _q8_0_row(codes, dbits):
    """Canonical q8_0 row built byte by byte from codes and a raw fp16 scale."""
    K = len(codes)
    out = bytearray()
    for b in range(K // 32):
        out += struct.pack("<H", dbits)
        out += bytes(int(c) & 0xFF for c in codes[32 * b: 32 * b + 32])
    return np.frombuffer(bytes(out), dtype=np.uint8)


def pin_closed_forms(o):
    K = 256
    c = 0.75  # exact in bf16
    xbits = np.full(K, 0x3F40, dtype=np.uint16)   # bf16 0.75
    ones = _q8_0_row([1] * K, 0x3C00)             # q = 1, d = 1.0 -> w = 1
    Y, _ = o.gemv(Q8_0, ones, BF16, xbits, 1, 1, K)
    assert Y[0, 0] == K * c
    # one-hot row selects x_j * 2^-5 exactly
    xr = _to_bf16_bits(np.random.default_rng(3).normal(0, 1, K).astype(np.float32))
    for j in (0, 17, 31, 32, 200, 255):
        codes = [0] * K
        codes[j] = 1
        row = _q8_0_row(codes, 0x2800)            # fp16 2^-5
        Y, _ = o.gemv(Q8_0, row, BF16, xr, 1, 1, K)
        assert Y[0, 0] == float(_bf16(int(xr[j]))) * 2.0 ** -5, j
    # alternating weights against a constant activation sum to zero
    alt = _q8_0_row([1 if k % 2 == 0 else -1 for k in range(K)], 0x3C00)
    Y, _ = o.gemv(Q8_0, alt, BF16, xbits, 1, 1, K)
    assert Y[0, 0] == 0.0
    # q4_0: codes 9 and 7 alternate (+d, -d) -> zero; code 8 everywhere -> zero
    row = bytearray()
    for b in range(K // 32):
        row += struct.pack("<H", 0x3C00) + bytes([0x79] * 16)  # low 9, high 7
    Y, _ = o.gemv(Q4_0, np.frombuffer(bytes(row), np.uint8), BF16, xbits, 1, 1, K)
    assert Y[0, 0] == 0.0
    # linearity: y(W, 2x) == 2 y(W, x) exactly (doubling is exact)
    rng = np.random.default_rng(5)
    W = _to_bf16_bits(rng.normal(0, 0.02, (4, K)).astype(np.float32))
    x = rng.normal(0, 1, (1, K)).astype(np.float32)
    y1, _ = o.gemv(BF16, W, BF16, _to_bf16_bits(x), 1, 4, K)
    y2, _ = o.gemv(BF16, W, BF16, _to_bf16_bits(2 * x), 1, 4, K)
    assert np.array_equal(y2, 2 * y1)


# ---------------------------------------------------------------------------
# invariants of the encodings
# ---------------------------------------------------------------------------
def pin_quantize_invariants(o):
    rng = np.random.default_rng(99)
    K = 32 * 64
    for scale in (0.02, 1.0, 300.0):
        x = (rng.standard_normal((4, K)) * scale).astype(np.float32)
        # adversarial: exact halves of the scale and a dominant element per block
        x[0, ::7] = np.round(x[0, ::7] * 4) / 4
        for fmt, off in ((Q8_0, 2), (Q8_1, 4)):
            q = o.quantize(fmt, x)
            bs = 34 if fmt == Q8_0 else 36
            blocks = q.reshape(-1, bs)
            d = blocks[:, 0:2].copy().view(np.float16).astype(np.float64).reshape(-1)
            codes = blocks[:, off:].view(np.int8).astype(np.int64)
            assert np.all(np.abs(codes) <= 127)
            xv = x.reshape(-1, 32).astype(np.float64)
            err = np.abs(codes * d[:, None] - xv)
            assert np.all(err <= d[:, None] / 2 * (1 + 2 ** -20)), (fmt, float((err - d[:, None] / 2).max()))
            # amax maps to +-127 or to the value nearest the fp16-rounded scale
            amax = np.abs(xv).max(axis=1)
            assert np.all(np.abs(np.abs(codes).max(axis=1) - 127) <= 1)
            assert np.all(np.abs(d - amax / 127) <= amax / 127 * 2 ** -11)
            if fmt == Q8_1:
                s = blocks[:, 2:4].copy().view(np.float16).astype(np.float64).reshape(-1)
                ref = (d * codes.sum(axis=1)).astype(np.float16).astype(np.float64)
                assert np.array_equal(s, ref)
        q = o.quantize(Q4_0, x).reshape(-1, 18)
        d = q[:, 0:2].copy().view(np.float16).astype(np.float64).reshape(-1)
        lo = (q[:, 2:] & 15).astype(np.int64)
        hi = (q[:, 2:] >> 4).astype(np.int64)
        codes = np.concatenate([lo, hi], axis=1)
        xv = x.reshape(-1, 32).astype(np.float64)
        imax = np.argmax(np.abs(xv), axis=1)       # first index of the max |x|
        assert np.all(codes[np.arange(len(imax)), imax] == 0)
        r = xv / d[:, None]
        clamped = r > 7.5
        err = np.abs((codes - 8) * d[:, None] - xv)
        ad = np.broadcast_to(np.abs(d)[:, None], err.shape)
        assert np.all(err[~clamped] <= ad[~clamped] / 2 * (1 + 2 ** -20))
        # clamped codes (x/d > 7.5) read back 7d; |x/d| <= 8 (1 + 2^-11) because
        # d is m/-8 rounded to fp16, so the error stays below |d| (1 + 2^-8)
        assert np.all(err[clamped] <= ad[clamped] * (1 + 2 ** -8))
        assert np.all(codes[clamped] == 15)
        assert np.all(codes[r < 6.5 - 1e-6] < 15)


def pin_degenerate_blocks(o):
    z = np.zeros(64, dtype=np.float32)
    q8 = o.quantize(Q8_0, z)[0]
    assert not q8.any()
    q1 = o.quantize(Q8_1, z)[0]
    assert not q1.any()
    q4 = o.quantize(Q4_0, z)[0].reshape(2, 18)
    # m = +0 gives d = 0 / -8 = -0.0 (fp16 0x8000); every code is 8 (value 0)
    assert np.all(q4[:, 0] == 0x00) and np.all(q4[:, 1] == 0x80) and np.all(q4[:, 2:] == 0x88)
    # a single non-zero element: it maps to the extreme code
    x = np.zeros(32, dtype=np.float32)
    x[5] = -3.0
    q4 = o.quantize(Q4_0, x)[0]
    assert struct.unpack("<e", bytes(q4[:2]))[0] == 0.375 and (q4[2 + 5] & 15) == 0
    q8 = o.quantize(Q8_0, x)[0]
    assert np.int8(q8[2 + 5]) == -127
    # equal magnitudes of opposite sign: the first one sets the sign of d
    x = np.zeros(32, dtype=np.float32)
    x[3], x[9] = -2.0, 2.0
    q4 = o.quantize(Q4_0, x)[0]
    assert struct.unpack("<e", bytes(q4[:2]))[0] == 0.25
    assert (q4[2 + 3] & 15) == 0 and (q4[2 + 9] & 15) == 15


def pin_swiglu(o):
    rng = np.random.default_rng(2)
    g = rng.normal(0, 3, 1000)
    u = rng.normal(0, 1, 1000)
    h = o.swiglu(g, u)
    ref = g * 0.5 * (1 + np.tanh(g / 2)) * u          # sigma(g) = (1 + tanh(g/2)) / 2
    assert np.allclose(h, ref, rtol=1e-13, atol=1e-300)
    ones = np.ones_like(g)
    hp, hn = o.swiglu(g, ones), o.swiglu(-g, ones)
    assert np.allclose(hn, hp - g, rtol=1e-12, atol=1e-14)   # silu(-g) = silu(g) - g
    assert o.swiglu(np.array([0.0]), np.array([5.0]))[0] == 0.0


def pin_second_reference(o):
    _Q["o"] = o
    rng = np.random.default_rng(4)
    M, N, K = 2, 16, 512
    for wfmt in (BF16, Q8_0, Q4_0):
        W, X = _tiny_case(rng, wfmt, BF16, M, N, K)
        Y, A = o.gemv(wfmt, W, BF16, X, M, N, K)
        Yf = o.gemv_f32acc(wfmt, W, BF16, X, M, N, K)
        assert np.all(np.abs(Yf - Y) <= 2 * K * 2.0 ** -24 * A)


def pin_rows_and_threads(o):
    _Q["o"] = o
    rng = np.random.default_rng(8)
    M, N, K = 2, 40, 320
    W, X = _tiny_case(rng, Q4_0, Q8_1, M, N, K)
    Y, A = o.gemv(Q4_0, W, Q8_1, X, M, N, K)
    rows = np.array([39, 0, 17, 17, 5])
    Ys, As = o.gemv(Q4_0, W, Q8_1, X, M, N, K, rows=rows)
    assert np.array_equal(Ys, Y[:, rows]) and np.array_equal(As, A[:, rows])
    Yt, At = o.gemv(Q4_0, W, Q8_1, X, M, N, K, nthreads=4)
    assert np.array_equal(Yt, Y) and np.array_equal(At, A)


def pin_repack_layout(o):
    cases = []
    with open(os.path.join(GOLDEN, "repack_layout.txt")) as f:
        for line in f:
            t = line.split()
            if not t or t[0].startswith("#"):
                continue
            if t[0] == "case":
                kv = dict(s.split("=") for s in t[2:5])
                cases.append({"fmt": t[1], "N": int(kv["N"]), "K": int(kv["K"]),
                              "size": int(kv["size"]), "full": t[5] == "full", "moves": []})
            else:
                cases[-1]["moves"].append(tuple(int(v) for v in t[1:4]))
    for c in cases:
        fmt = Q4_0 if c["fmt"] == "q4_0" else Q8_0
        N, K = c["N"], c["K"]
        nbytes = N * (K // 32) * (18 if fmt == Q4_0 else 34)
        canon = ((np.arange(nbytes) * 7 + 3) % 251 + 1).astype(np.uint8)   # no zero bytes
        assert o.repacked_size(fmt, N, K) == c["size"]
        packed = o.repack(fmt, canon, N, K)
        assert packed.size == c["size"]
        covered = np.zeros(packed.size, dtype=bool)
        for p, q, n in c["moves"]:
            assert np.array_equal(packed[p:p + n], canon[q:q + n]), (c["fmt"], p, q)
            covered[p:p + n] = True
        if c["full"]:
            assert not packed[~covered].any()
        assert np.array_equal(o.unrepack(fmt, packed, N, K), canon)
    rng = np.random.default_rng(0)
    bf = rng.integers(0, 65536, 64 * 8, dtype=np.uint16)
    assert np.array_equal(o.repack(BF16, bf, 8, 64), bf.view(np.uint8))


def _fp16(u: int) -> float:
    return float(_half(struct.pack("<H", u & 0xFFFF)))


def _bf16_values(x):
    """fp32 array rounded to bf16 (nearest even), returned as fp32."""
    bits = _to_bf16_bits(x).astype(np.uint32) << 16
    return bits.view(np.float32)


def pin_rmsnorm_q8_1_hand_block(o):
    """The hand-worked block: a constant row normalises to ones."""
    g = _read_golden("rmsnorm_q8_1_hand_block.txt")
    want = _hexbytes(g["bytes"])
    for key in ("x1", "xhalf"):
        x = np.array([float(v) for v in g[key]], dtype=np.float32)
        got = o.rmsnorm_q8_1(x, None, 0.0)[0]
        assert np.array_equal(got, want), (key, bytes(got).hex())


def pin_rmsnorm_q8_1_properties(o):
    """Against the definition, with the sum of squares taken exactly
    (fractions) and the square root from the math library:
      * every dequantized output is within half a step (d/2) of
        x_k / sqrt(mean(x^2) + eps) * gamma_k, up to the fp32 roundings of r
        and of the two products;
      * gamma of ones is no gamma; gamma of 2 doubles d and s and keeps the codes;
      * a zero row (eps > 0) gives all-zero blocks."""
    rng = np.random.default_rng(21)
    M, K = 3, 1024
    x = _bf16_values(rng.normal(0, 1, (M, K)).astype(np.float32))
    for eps, gamma in ((1e-5, None), (0.5, None), (1e-6, rng.uniform(0.5, 1.5, K).astype(np.float32))):
        out = o.rmsnorm_q8_1(x, gamma, eps)
        deq = o.dequantize(Q8_1, out.reshape(-1), M, K)
        for m in range(M):
            s = sum(Fraction(float(v)) ** 2 for v in x[m])
            inv = 1.0 / math.sqrt(float(s / K) + float(np.float32(eps)))
            ref = x[m].astype(np.float64) * inv * (1.0 if gamma is None else gamma.astype(np.float64))
            for b in range(K // 32):
                blk = out[m, b * 36:(b + 1) * 36]
                d = _fp16(int(blk[0]) | int(blk[1]) << 8)
                err = np.abs(deq[m, b * 32:(b + 1) * 32] - ref[b * 32:(b + 1) * 32])
                slack = 4 * 2.0 ** -24 * np.abs(ref[b * 32:(b + 1) * 32])
                assert np.all(err <= d / 2 + slack + 1e-12), (eps, m, b, float(err.max()), d)
    # gamma of ones == no gamma; gamma of 2 doubles the scales exactly
    a = o.rmsnorm_q8_1(x, None, 1e-5)
    assert np.array_equal(o.rmsnorm_q8_1(x, np.ones(K, np.float32), 1e-5), a)
    two = o.rmsnorm_q8_1(x, np.full(K, 2.0, np.float32), 1e-5)
    for m in range(M):
        for b in range(K // 32):
            ba, bt = a[m, b * 36:(b + 1) * 36], two[m, b * 36:(b + 1) * 36]
            assert np.array_equal(ba[4:], bt[4:])
            for off in (0, 2):
                ha, ht = int(ba[off]) | int(ba[off + 1]) << 8, int(bt[off]) | int(bt[off + 1]) << 8
                assert _fp16(ht) == 2 * _fp16(ha), (m, b, off)
    z = o.rmsnorm_q8_1(np.zeros((2, 64), np.float32), None, 1e-5)
    assert not z.any()


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
