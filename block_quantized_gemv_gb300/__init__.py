"""Python binding of libbqgemv (block-quantized skinny GEMV for sm_103a).

A thin ctypes layer over the C ABI in include/bqgemv.h: every function here
has the name of its C entry point without the ``bqg_`` prefix, checks that
the torch tensors it is given match the C contract, and passes raw device
pointers plus the current CUDA stream.  Where the C contract allows host
memory (the output of a single-matrix GEMV, either side of copy_sm), a pinned
CPU tensor is passed as its device-side alias (bqg_host_alias).  All
arithmetic runs in the library's CUDA kernels; PyTorch only provides memory
and streams.  There is no fallback: if the shared library is missing, every
call raises.  Every CUDA tensor must be on the current device (ValueError
otherwise, before anything is launched).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

BF16, Q8_0, Q4_0, Q8_1, F32 = 0, 1, 2, 3, 4
OP_GEMV_BF16, OP_GEMV_Q8_0, OP_GEMV_Q4_0, OP_GEMV_Q4_0_Q8_1 = 0, 1, 2, 3
OP_QKV_Q4_0_Q8_1, OP_GATE_UP_Q4_0_Q8_1, OP_GEMM_Q4_0_BF16 = 4, 5, 6
OP_GATE_UP_Q8_1_Q4_0_Q8_1, OP_GEMM_Q8_0_BF16, OP_DECODE_LAYER_Q4_0_Q8_1 = 7, 8, 9
BLOCK_BYTES = {Q8_0: 34, Q4_0: 18, Q8_1: 36}
QK = 32
TILE_BYTES = {Q8_0: 1088, Q4_0: 576}     # 32 blocks of one repacked row

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libbqgemv.so")

EXPORTS = {
    # name: (argtypes, restype)
    "bqg_repacked_size": (["i", "i64", "i64"], "size"),
    "bqg_quantize_weights": (["i", "p", "p", "i64", "i64", "p"], "i"),
    "bqg_repack_weights": (["i", "p", "p", "i64", "i64", "p"], "i"),
    "bqg_quantize_q8_1": (["p", "i", "p", "i", "i64", "p"], "i"),
    "bqg_rmsnorm_quantize_q8_1": (["p", "i", "p", "f", "p", "i", "i64", "p"], "i"),
    "bqg_gemv_bf16": (["p", "p", "p", "i", "i64", "i64", "p", "size", "p"], "i"),
    "bqg_gemv_q8_0": (["p", "p", "p", "i", "i64", "i64", "p", "size", "p"], "i"),
    "bqg_gemv_q4_0": (["p", "p", "p", "i", "i64", "i64", "p", "size", "p"], "i"),
    "bqg_gemv_q4_0_q8_1": (["p", "p", "p", "i", "i64", "i64", "p", "size", "p"], "i"),
    "bqg_gemv_q4_0_q8_1_qkv": (["p", "p", "p", "p", "p", "p", "p", "i", "i64", "i64", "i64", "p", "size", "p"], "i"),
    "bqg_gemv_q4_0_q8_1_gate_up_swiglu": (["p", "p", "p", "p", "i", "i64", "i64", "p", "size", "p"], "i"),
    "bqg_gemv_q4_0_q8_1_gate_up_swiglu_q8_1": (["p", "p", "p", "p", "i", "i64", "i64", "p", "size", "p"], "i"),
    "bqg_decode_layer_q4_0_q8_1": (["p", "p", "i", "p", "p", "p", "p", "p", "p", "p", "p", "p", "p", "i", "i64",
                                    "i64", "i64", "i64", "p", "size", "p"], "i"),
    "bqg_gemm_q4_0_bf16": (["p", "p", "p", "i", "i64", "i64", "p", "size", "p"], "i"),
    "bqg_gemm_q8_0_bf16": (["p", "p", "p", "i", "i64", "i64", "p", "size", "p"], "i"),
    "bqg_debug_q4_0_q8_1_block_dots": (["p", "p", "p", "i64", "i64", "p"], "i"),
    "bqg_debug_q4_0_q8_1_block_dots_kslice": (["p", "p", "p", "i64", "i64", "p"], "i"),
    "bqg_workspace_size": (["i", "i", "i64", "i64"], "size"),
    "bqg_gemv_route": (["i", "i", "i64", "i64", "p"], "i"),
    "bqg_last_device_error": (["p", "p"], "i"),
    "bqg_set_pdl": (["i"], "i"),
    "bqg_host_alias": (["p", "p"], "i"),
    "bqg_copy_sm": (["p", "p", "size", "p"], "i"),
    "bqg_status_string": (["i"], "str"),
    "bqg_version": ([], "str"),
    "bqg_last_cuda_error": ([], "str"),
    "bqg_gemv_q4_0_q8_1_noalloc": (["p", "p", "p", "i", "i64", "i64", "p"], "i"),
    "bqg_noalloc_scratch_bytes": ([], "size"),
}
_CT = {"i": ctypes.c_int, "i64": ctypes.c_int64, "p": ctypes.c_void_p, "size": ctypes.c_size_t,
       "str": ctypes.c_char_p, "f": ctypes.c_float}

_lock = threading.Lock()
_lib = None


class BqgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = f" [{load().bqg_last_cuda_error().decode()}]" if status == 5 else ""
        super().__init__(f"{where}: {status_string(status)} (status {status}){detail}")


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (once) and return the shared library; raises if it is not built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libbqgemv is not built ({p} missing); run "
                                   "block_quantized_gemv_gb300.build.build()")
            L = ctypes.CDLL(p)
            for name, (args, res) in EXPORTS.items():
                fn = getattr(L, name)
                fn.argtypes = [_CT[a] for a in args]
                fn.restype = _CT[res]
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return load().bqg_status_string(int(status)).decode()


def version() -> str:
    return load().bqg_version().decode()


def _check(status: int, where: str):
    if status != 0:
        raise BqgError(status, where)


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream=None) -> int:
    """The stream handle to enqueue on: `stream`, else torch's current stream
    of the current device (read without building a Stream object)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None and _cur_device is not None:
        return _raw_stream(_cur_device())
    return torch.cuda.current_stream().cuda_stream


def _current_device() -> int:
    return _cur_device() if _cur_device is not None else torch.cuda.current_device()


def check_device(index: int, current: int, name: str) -> None:
    """A CUDA tensor must live on the current device: the library launches
    on the current device and would otherwise dereference another GPU's
    memory."""
    if index != current:
        raise ValueError(f"{name} is on cuda:{index} but the current device is cuda:{current}; "
                         f"call under torch.cuda.device({index})")


def _check_tensor(t: torch.Tensor, name: str, dtype=None, numel=None) -> None:
    """Layout, dtype and size checks shared by device and host operands:
    `numel` is the byte count the call will touch."""
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.nbytes < numel:
        raise ValueError(f"{name} holds {t.nbytes} bytes, needs {numel}")


def _dev(t: torch.Tensor, name: str, dtype=None, numel=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    check_device(t.device.index, _current_device(), name)
    _check_tensor(t, name, dtype, numel)
    return t.data_ptr()


def weight_bytes(fmt: int, N: int, K: int):
    """Bytes of N repacked weight rows of K values (the layout of
    include/bqgemv.h: bf16 row-major; q4_0 / q8_0 rows of ceil(K/32/32)
    tiles of 576 / 1088 bytes), or None for a shape the library refuses by
    itself (K not a positive multiple of 32, N < 1).  The C boundary takes
    the weights as a bare pointer, so the binding checks their size."""
    if N < 1 or K < 1 or K % QK:
        return None
    if fmt == BF16:
        return N * K * 2
    return N * ((K // QK + 31) // 32) * TILE_BYTES[fmt]


def host_alias(t: torch.Tensor) -> int:
    """Device-side address of a page-locked (pinned) CPU tensor's memory:
    kernels given it read or write host memory over the CPU-GPU link."""
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError("host_alias wants a pinned CPU tensor")
    if not t.is_contiguous():
        raise ValueError("the tensor must be contiguous")
    out = ctypes.c_void_p(0)
    _check(load().bqg_host_alias(t.data_ptr(), ctypes.addressof(out)), "bqg_host_alias")
    return out.value


def _dev_or_host(t: torch.Tensor, name: str, dtype=None, numel=None):
    """_dev for a CUDA tensor; the host alias for a pinned CPU tensor."""
    if isinstance(t, torch.Tensor) and not t.is_cuda and t.is_pinned():
        _check_tensor(t, name, dtype, numel)
        return host_alias(t)
    return _dev(t, name, dtype, numel)


def copy_sm(dst: torch.Tensor, src: torch.Tensor, stream=None) -> torch.Tensor:
    """Copy src's bytes into dst with a kernel instead of a copy engine; each
    of the two may be a CUDA tensor or a pinned CPU tensor."""
    n = src.nbytes
    _check(load().bqg_copy_sm(_dev_or_host(dst, "dst", numel=n), _dev_or_host(src, "src"), n, _stream(stream)),
           "bqg_copy_sm")
    return dst


def _ws(ws):
    if ws is None:
        return None, 0
    return _dev(ws, "ws"), ws.nbytes


def row_bytes(fmt: int, K: int) -> int:
    """Bytes of one canonical row (bf16: 2K; block formats: K/32 blocks)."""
    return 2 * K if fmt == BF16 else (K // QK) * BLOCK_BYTES[fmt]


# --- load time -----------------------------------------------------------------
def repacked_size(fmt: int, N: int, K: int) -> int:
    return int(load().bqg_repacked_size(fmt, N, K))


def quantize_weights(fmt: int, W: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """fp32 N x K -> canonical q8_0/q4_0 blocks (uint8, N x row_bytes)."""
    N, K = W.shape
    if out is None:
        out = torch.empty((N, row_bytes(fmt, K)), dtype=torch.uint8, device=W.device)
    _check(load().bqg_quantize_weights(fmt, _dev(W, "W", torch.float32),
                                       _dev(out, "out", numel=N * row_bytes(fmt, K)), N, K, _stream(stream)),
           "bqg_quantize_weights")
    return out


def repack_weights(fmt: int, src: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    size = repacked_size(fmt, N, K)
    if out is None:
        out = torch.empty(size, dtype=torch.uint8, device=src.device)
    _check(load().bqg_repack_weights(fmt, _dev(src, "src", numel=N * row_bytes(fmt, K)),
                                     _dev(out, "out", numel=size), N, K, _stream(stream)),
           "bqg_repack_weights")
    return out


# --- per token -----------------------------------------------------------------
def quantize_q8_1(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """bf16 or fp32 M x K -> q8_1 blocks (uint8, M x K/32*36)."""
    M, K = x.shape
    dt = {torch.bfloat16: BF16, torch.float32: F32}.get(x.dtype)
    if dt is None:
        raise TypeError("x must be bf16 or fp32")
    if out is None:
        out = torch.empty((M, row_bytes(Q8_1, K)), dtype=torch.uint8, device=x.device)
    _check(load().bqg_quantize_q8_1(_dev(x, "x"), dt, _dev(out, "out", numel=M * row_bytes(Q8_1, K)), M, K,
                                    _stream(stream)), "bqg_quantize_q8_1")
    return out


def rmsnorm_quantize_q8_1(x: torch.Tensor, gamma: torch.Tensor | None = None, eps: float = 1e-5,
                          out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Fused RMSNorm (optional fp32 gain `gamma`) + q8_1 quantization:
    bf16 or fp32 M x K -> q8_1 blocks (uint8, M x K/32*36)."""
    M, K = x.shape
    dt = {torch.bfloat16: BF16, torch.float32: F32}.get(x.dtype)
    if dt is None:
        raise TypeError("x must be bf16 or fp32")
    if out is None:
        out = torch.empty((M, row_bytes(Q8_1, K)), dtype=torch.uint8, device=x.device)
    g = None if gamma is None else _dev(gamma, "gamma", torch.float32, K * 4)
    _check(load().bqg_rmsnorm_quantize_q8_1(_dev(x, "x"), dt, g, float(eps),
                                            _dev(out, "out", numel=M * row_bytes(Q8_1, K)), M, K, _stream(stream)),
           "bqg_rmsnorm_quantize_q8_1")
    return out


def _gemv(fn: str, wfmt: int, Wp, X, N: int, K: int, M: int, out, ws, stream, xbytes):
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=X.device)
    wsp, wsb = _ws(ws)
    _check(getattr(load(), fn)(_dev(Wp, "Wp", numel=weight_bytes(wfmt, N, K)), _dev(X, "X", numel=xbytes),
                               _dev_or_host(out, "Y", torch.float32, M * N * 4), M, N, K, wsp, wsb, _stream(stream)),
           fn)
    return out


def gemv_bf16(Wp, X, N, K, out=None, ws=None, stream=None):
    return _gemv("bqg_gemv_bf16", BF16, Wp, X, N, K, X.shape[0], out, ws, stream, X.shape[0] * K * 2)


def gemv_q8_0(Wp, X, N, K, out=None, ws=None, stream=None):
    return _gemv("bqg_gemv_q8_0", Q8_0, Wp, X, N, K, X.shape[0], out, ws, stream, X.shape[0] * K * 2)


def gemv_q4_0(Wp, X, N, K, out=None, ws=None, stream=None):
    return _gemv("bqg_gemv_q4_0", Q4_0, Wp, X, N, K, X.shape[0], out, ws, stream, X.shape[0] * K * 2)


def gemv_q4_0_q8_1(Wp, Xq, N, K, out=None, ws=None, stream=None):
    M = Xq.shape[0]
    return _gemv("bqg_gemv_q4_0_q8_1", Q4_0, Wp, Xq, N, K, M, out, ws, stream, M * row_bytes(Q8_1, K))


def gemv_q4_0_q8_1_noalloc(Wp, Xq, N, K, out=None, stream=None):
    """bqg_gemv_q4_0_q8_1 without a workspace argument: split-K scratch comes
    from a fixed array inside the library (for callers that cannot allocate)."""
    M = Xq.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=Xq.device)
    _check(load().bqg_gemv_q4_0_q8_1_noalloc(_dev(Wp, "Wp", numel=weight_bytes(Q4_0, N, K)), _dev(Xq, "Xq", numel=M * row_bytes(Q8_1, K)),
                                             _dev_or_host(out, "Y", torch.float32, M * N * 4), M, N, K,
                                             _stream(stream)), "bqg_gemv_q4_0_q8_1_noalloc")
    return out


def gemv_q4_0_q8_1_qkv(Wq, Wk, Wv, Xq, Nq, Nkv, K, out=None, ws=None, stream=None):
    M = Xq.shape[0]
    dev = Xq.device
    if out is None:
        out = (torch.empty((M, Nq), dtype=torch.float32, device=dev),
               torch.empty((M, Nkv), dtype=torch.float32, device=dev),
               torch.empty((M, Nkv), dtype=torch.float32, device=dev))
    Yq, Yk, Yv = out
    wsp, wsb = _ws(ws)
    _check(load().bqg_gemv_q4_0_q8_1_qkv(_dev(Wq, "Wq", numel=weight_bytes(Q4_0, Nq, K)),
                                         _dev(Wk, "Wk", numel=weight_bytes(Q4_0, Nkv, K)),
                                         _dev(Wv, "Wv", numel=weight_bytes(Q4_0, Nkv, K)),
                                         _dev(Xq, "Xq", numel=M * row_bytes(Q8_1, K)),
                                         _dev(Yq, "Yq", torch.float32, M * Nq * 4),
                                         _dev(Yk, "Yk", torch.float32, M * Nkv * 4),
                                         _dev(Yv, "Yv", torch.float32, M * Nkv * 4),
                                         M, Nq, Nkv, K, wsp, wsb, _stream(stream)), "bqg_gemv_q4_0_q8_1_qkv")
    return out


def gemv_q4_0_q8_1_gate_up_swiglu(Wg, Wu, Xq, N, K, out=None, ws=None, stream=None):
    M = Xq.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=Xq.device)
    wsp, wsb = _ws(ws)
    _check(load().bqg_gemv_q4_0_q8_1_gate_up_swiglu(_dev(Wg, "Wg", numel=weight_bytes(Q4_0, N, K)),
                                                    _dev(Wu, "Wu", numel=weight_bytes(Q4_0, N, K)),
                                                    _dev(Xq, "Xq", numel=M * row_bytes(Q8_1, K)),
                                                    _dev(out, "H", torch.float32, M * N * 4), M, N, K, wsp, wsb,
                                                    _stream(stream)), "bqg_gemv_q4_0_q8_1_gate_up_swiglu")
    return out


def gemv_q4_0_q8_1_gate_up_swiglu_q8_1(Wg, Wu, Xq, N, K, out=None, ws=None, stream=None):
    """gate+up+SwiGLU writing h as q8_1 blocks (uint8, M x N/32*36).  `ws`
    (workspace(OP_GATE_UP_Q8_1_Q4_0_Q8_1, ...)) must start zero-filled."""
    M = Xq.shape[0]
    if out is None:
        out = torch.empty((M, row_bytes(Q8_1, N)), dtype=torch.uint8, device=Xq.device)
    wsp, wsb = _ws(ws)
    _check(load().bqg_gemv_q4_0_q8_1_gate_up_swiglu_q8_1(_dev(Wg, "Wg", numel=weight_bytes(Q4_0, N, K)),
                                                         _dev(Wu, "Wu", numel=weight_bytes(Q4_0, N, K)),
                                                         _dev(Xq, "Xq", numel=M * row_bytes(Q8_1, K)),
                                                         _dev(out, "Hq", numel=M * row_bytes(Q8_1, N)), M, N, K,
                                                         wsp, wsb, _stream(stream)),
           "bqg_gemv_q4_0_q8_1_gate_up_swiglu_q8_1")
    return out


def decode_layer_q4_0_q8_1(xa, xb, Wq, Wk, Wv, Wg, Wu, Wd, Nq, Nkv, Nff, K, out=None, ws=None, stream=None):
    """One decode layer (M = 1) in one persistent launch: q8_1 of xa and xb,
    QKV from xa, gate+up+SwiGLU (h as q8_1) from xb, down projection of h.
    xa, xb: (1, K) bf16 or fp32.  Returns (Yq, Yk, Yv, Y).  `ws`
    (workspace(OP_DECODE_LAYER_Q4_0_Q8_1, 1, Nff, K)) must start zero-filled;
    it also holds h's q8_1 blocks (see `layer_hq`)."""
    if xa.dtype not in (torch.bfloat16, torch.float32) or xb.dtype != xa.dtype:
        raise TypeError("xa and xb must both be bfloat16 or both float32")
    dt = F32 if xa.dtype == torch.float32 else BF16
    nx = K * xa.element_size()
    if out is None:
        dev = xa.device
        out = tuple(torch.empty(n, dtype=torch.float32, device=dev) for n in (Nq, Nkv, Nkv, K))
    Yq, Yk, Yv, Y = out
    wsp, wsb = _ws(ws)
    _check(load().bqg_decode_layer_q4_0_q8_1(_dev(xa, "xa", numel=nx), _dev(xb, "xb", numel=nx), dt,
                                             _dev(Wq, "Wq", numel=weight_bytes(Q4_0, Nq, K)),
                                             _dev(Wk, "Wk", numel=weight_bytes(Q4_0, Nkv, K)),
                                             _dev(Wv, "Wv", numel=weight_bytes(Q4_0, Nkv, K)),
                                             _dev(Wg, "Wg", numel=weight_bytes(Q4_0, Nff, K)),
                                             _dev(Wu, "Wu", numel=weight_bytes(Q4_0, Nff, K)),
                                             _dev(Wd, "Wd", numel=weight_bytes(Q4_0, K, Nff)),
                                             _dev(Yq, "Yq", torch.float32, Nq * 4), _dev(Yk, "Yk", torch.float32, Nkv * 4),
                                             _dev(Yv, "Yv", torch.float32, Nkv * 4), _dev(Y, "Y", torch.float32, K * 4),
                                             1, Nq, Nkv, Nff, K, wsp, wsb, _stream(stream)),
           "bqg_decode_layer_q4_0_q8_1")
    return out


def layer_hq(ws, Nff):
    """The q8_1 blocks of h (uint8, Nff/32 * 36) inside a decode-layer workspace."""
    up16 = lambda b: (b + 15) // 16 * 16
    off = up16(Nff * 4) + up16(Nff // QK * 4)
    return ws[off:off + Nff // QK * BLOCK_BYTES[Q8_1]]


def gemm_q4_0_bf16(Wp, X, N, K, out=None, ws=None, stream=None):
    M = X.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=X.device)
    wsp, wsb = _ws(ws)
    _check(load().bqg_gemm_q4_0_bf16(_dev(Wp, "Wp", numel=weight_bytes(Q4_0, N, K)), _dev(X, "X", torch.bfloat16, M * K * 2),
                                     _dev(out, "Y", torch.float32, M * N * 4), M, N, K, wsp, wsb, _stream(stream)),
           "bqg_gemm_q4_0_bf16")
    return out


def gemm_q8_0_bf16(Wp, X, N, K, out=None, ws=None, stream=None):
    M = X.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=X.device)
    wsp, wsb = _ws(ws)
    _check(load().bqg_gemm_q8_0_bf16(_dev(Wp, "Wp", numel=weight_bytes(Q8_0, N, K)), _dev(X, "X", torch.bfloat16, M * K * 2),
                                     _dev(out, "Y", torch.float32, M * N * 4), M, N, K, wsp, wsb, _stream(stream)),
           "bqg_gemm_q8_0_bf16")
    return out


def _block_dots(fn, Wp, Xq, N, K, out, stream):
    if out is None:
        out = torch.empty((N, K // QK), dtype=torch.int32, device=Xq.device)
    _check(getattr(load(), fn)(_dev(Wp, "Wp", numel=weight_bytes(Q4_0, N, K)), _dev(Xq, "Xq", numel=row_bytes(Q8_1, K)),
                               _dev(out, "dots", torch.int32, N * (K // QK) * 4), N, K, _stream(stream)), fn)
    return out


def debug_q4_0_q8_1_block_dots(Wp, Xq, N, K, out=None, stream=None):
    """The integer block dots as gemv_q4_0_q8_1 computes them at M = 1 (its
    own kernel and plan), N x K/32 int32."""
    return _block_dots("bqg_debug_q4_0_q8_1_block_dots", Wp, Xq, N, K, out, stream)


def debug_q4_0_q8_1_block_dots_kslice(Wp, Xq, N, K, out=None, stream=None):
    """The same dots from the K-slice kernel's routine."""
    return _block_dots("bqg_debug_q4_0_q8_1_block_dots_kslice", Wp, Xq, N, K, out, stream)


# --- utilities -----------------------------------------------------------------
def workspace_size(op: int, M: int, N: int, K: int) -> int:
    return int(load().bqg_workspace_size(op, M, N, K))


def workspace(op: int, M: int, N: int, K: int, device="cuda") -> torch.Tensor | None:
    """A workspace for `op` (zero-filled, as the q8_1-output SwiGLU requires)."""
    n = workspace_size(op, M, N, K)
    return torch.zeros(n, dtype=torch.uint8, device=device) if n else None


ROUTE_K_SLICE, ROUTE_LANES_PER_ROW, ROUTE_LANES_PER_ROW_ROWS, ROUTE_TENSOR_CORE = 0, 1, 2, 3
ROUTE_NAMES = {0: "k_slice", 1: "lanes_per_row", 2: "lanes_per_row_rows", 3: "tensor_core"}


def gemv_route(op: int, M: int, N: int, K: int) -> int:
    """Which kernel serves a GEMV call of this shape on the current device
    (one of the ROUTE_* values)."""
    out = ctypes.c_int(-1)
    _check(load().bqg_gemv_route(op, M, N, K, ctypes.addressof(out)), "bqg_gemv_route")
    return out.value


def last_device_error(stream=None) -> int:
    out = ctypes.c_int(0)
    _check(load().bqg_last_device_error(_stream(stream), ctypes.addressof(out)), "bqg_last_device_error")
    return out.value


def set_pdl(enable: bool) -> bool:
    return bool(load().bqg_set_pdl(1 if enable else 0))
