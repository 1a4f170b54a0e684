"""CPU oracle for block-quantized skinny GEMV -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``block_quantized_gemv_gb300``) never imports, links or calls it, and this
package never imports the product.  The arithmetic lives in
``bqg_oracle.c`` (plain C, fp64 accumulation); this module only compiles it
with gcc and marshals numpy arrays through ctypes.

``Oracle(path)`` binds one compiled copy of the C file; the module-level
functions use the default build.  The pin tests also build deliberately
broken copies (mutants) and check that some pin rejects each of them.

Parity status: every function is pinned (brute force, hand-worked blocks,
closed forms, invariants or a library routine); see tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

BF16, Q8_0, Q4_0, Q8_1, F32 = 0, 1, 2, 3, 4
BLOCK_BYTES = {Q8_0: 34, Q4_0: 18, Q8_1: 36}
QK = 32

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "bqg_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lock = threading.Lock()
_default = None


def compile_source(src: str, out: str) -> str:
    """gcc, no fast-math and no FMA contraction (same results on x86 and Arm)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", src, "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(out + ".tmp", out)
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _LIB)
    return _LIB


def row_bytes(fmt: int, K: int) -> int:
    if fmt == BF16:
        return 2 * K
    if fmt == F32:
        return 4 * K
    return (K // QK) * BLOCK_BYTES[fmt]


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    return a.reshape(-1).view(np.uint8)


class Oracle:
    """ctypes binding of one compiled copy of bqg_oracle.c."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        sig = {
            "ref_fp16_to_double": ([ctypes.c_uint16], ctypes.c_double),
            "ref_fp16_from_float": ([ctypes.c_float], ctypes.c_uint16),
            "ref_bf16_to_double": ([ctypes.c_uint16], ctypes.c_double),
            "ref_quantize": ([I, P, I64, I64, P], I),
            "ref_dequantize": ([I, P, I64, I64, P], I),
            "ref_gemv": ([I, P, I, P, I64, I64, I64, P, I64, P, P, I], I),
            "ref_gemv_f32acc": ([I, P, I, P, I64, I64, I64, P], I),
            "ref_block_dots_q4_0_q8_1": ([P, P, I64, I64, P], I),
            "ref_swiglu": ([P, P, I64, P], None),
            "ref_rmsnorm_q8_1": ([P, P, ctypes.c_float, I64, I64, P], I),
            "ref_repacked_size": ([I, I64, I64], I64),
            "ref_repack": ([I, P, I64, I64, P], I),
            "ref_unrepack": ([I, P, I64, I64, P], I),
            "ref_openmp_max_threads": ([], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes, fn.restype = args, res
        self.L = L
        self.path = path

    # --- scalars -------------------------------------------------------------
    def fp16_to_double(self, h: int) -> float:
        return self.L.ref_fp16_to_double(int(h) & 0xFFFF)

    def fp16_from_float(self, f: float) -> int:
        return int(self.L.ref_fp16_from_float(float(np.float32(f))))

    def bf16_to_double(self, b: int) -> float:
        return self.L.ref_bf16_to_double(int(b) & 0xFFFF)

    # --- encoders / decoders ---------------------------------------------------
    def quantize(self, fmt: int, x: np.ndarray) -> np.ndarray:
        """fp32 rows x K -> canonical blocks (uint8, rows x row_bytes)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim == 1:
            x = x[None, :]
        rows, K = x.shape
        out = np.zeros((rows, row_bytes(fmt, K)), dtype=np.uint8)
        rc = self.L.ref_quantize(fmt, _ptr(x), rows, K, _ptr(out))
        if rc:
            raise ValueError(f"ref_quantize failed ({rc})")
        return out

    def rmsnorm_q8_1(self, x: np.ndarray, gamma=None, eps: float = 1e-5) -> np.ndarray:
        """fp32 rows x K (bf16 inputs given exactly as fp32) -> RMS-normalised,
        optionally scaled by gamma (K fp32), q8_1 blocks (uint8, rows x K/32*36)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim == 1:
            x = x[None, :]
        rows, K = x.shape
        g = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.float32)
        out = np.zeros((rows, row_bytes(Q8_1, K)), dtype=np.uint8)
        rc = self.L.ref_rmsnorm_q8_1(_ptr(x), None if g is None else _ptr(g), ctypes.c_float(eps), rows, K, _ptr(out))
        if rc:
            raise ValueError(f"ref_rmsnorm_q8_1 failed ({rc})")
        return out

    def dequantize(self, fmt: int, data, rows: int, K: int) -> np.ndarray:
        data = _u8(data)
        assert data.size >= rows * row_bytes(fmt, K)
        out = np.empty((rows, K), dtype=np.float64)
        rc = self.L.ref_dequantize(fmt, _ptr(data), rows, K, _ptr(out))
        if rc:
            raise ValueError(f"ref_dequantize failed ({rc})")
        return out

    def gemv(self, wfmt: int, W, xfmt: int, X, M: int, N: int, K: int, rows=None, nthreads: int = 1):
        """Y[m, j] = sum_k W[rows[j], k] X[m, k] in fp64; returns (Y, A = sum_k |W X|)."""
        W, X = _u8(W), _u8(X)
        assert W.size >= N * row_bytes(wfmt, K) and X.size >= M * row_bytes(xfmt, K)
        if rows is None:
            nsel, rp = N, None
        else:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            assert rows.size == 0 or (rows.min() >= 0 and rows.max() < N)
            nsel, rp = rows.size, _ptr(rows)
        Y = np.zeros((M, nsel), dtype=np.float64)
        A = np.zeros((M, nsel), dtype=np.float64)
        if nsel:
            rc = self.L.ref_gemv(wfmt, _ptr(W), xfmt, _ptr(X), M, N, K, rp, nsel,
                                 _ptr(Y), _ptr(A), nthreads)
            if rc:
                raise ValueError(f"ref_gemv failed ({rc})")
        return Y, A

    def gemv_f32acc(self, wfmt: int, W, xfmt: int, X, M: int, N: int, K: int) -> np.ndarray:
        W, X = _u8(W), _u8(X)
        Y = np.zeros((M, N), dtype=np.float32)
        rc = self.L.ref_gemv_f32acc(wfmt, _ptr(W), xfmt, _ptr(X), M, N, K, _ptr(Y))
        if rc:
            raise ValueError(f"ref_gemv_f32acc failed ({rc})")
        return Y

    def block_dots_q4_0_q8_1(self, W, Xq, N: int, K: int) -> np.ndarray:
        W, Xq = _u8(W), _u8(Xq)
        out = np.zeros((N, K // QK), dtype=np.int32)
        rc = self.L.ref_block_dots_q4_0_q8_1(_ptr(W), _ptr(Xq), N, K, _ptr(out))
        if rc:
            raise ValueError(f"ref_block_dots failed ({rc})")
        return out

    def swiglu(self, g, u) -> np.ndarray:
        g = np.ascontiguousarray(g, dtype=np.float64).reshape(-1)
        u = np.ascontiguousarray(u, dtype=np.float64).reshape(-1)
        h = np.empty_like(g)
        self.L.ref_swiglu(_ptr(g), _ptr(u), g.size, _ptr(h))
        return h

    def repacked_size(self, fmt: int, N: int, K: int) -> int:
        return int(self.L.ref_repacked_size(fmt, N, K))

    def repack(self, fmt: int, canon, N: int, K: int) -> np.ndarray:
        canon = _u8(canon)
        out = np.zeros(self.repacked_size(fmt, N, K), dtype=np.uint8)
        rc = self.L.ref_repack(fmt, _ptr(canon), N, K, _ptr(out))
        if rc:
            raise ValueError(f"ref_repack failed ({rc})")
        return out

    def unrepack(self, fmt: int, packed, N: int, K: int) -> np.ndarray:
        packed = _u8(packed)
        out = np.zeros(N * row_bytes(fmt, K), dtype=np.uint8)
        rc = self.L.ref_unrepack(fmt, _ptr(packed), N, K, _ptr(out))
        if rc:
            raise ValueError(f"ref_unrepack failed ({rc})")
        return out

    def openmp_threads(self) -> int:
        return int(self.L.ref_openmp_max_threads())


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def tolerance(A) -> np.ndarray:
    """Per-output parity bound: 1e-3 * sum_k |w_k x_k| + 1e-6."""
    return 1e-3 * np.asarray(A) + 1e-6


def __getattr__(name):
    # module-level convenience: oracle.gemv(...) == oracle.default().gemv(...)
    if name in ("fp16_to_double", "fp16_from_float", "bf16_to_double", "quantize",
                "dequantize", "gemv", "gemv_f32acc", "block_dots_q4_0_q8_1", "swiglu",
                "repacked_size", "repack", "unrepack", "openmp_threads"):
        return getattr(default(), name)
    raise AttributeError(name)
