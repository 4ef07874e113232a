"""ctypes binding of ``libhcread.so``: the C ABI of include/hc_read.h, same names.

Argument marshalling only. Tensors are passed by ``data_ptr()``; every step of the
read runs in the library's CUDA kernels. There is no other implementation to fall
back to: if the library is missing or a call fails, an exception says so.

``hc_read`` and ``hc_read_path`` go through a small CPython module (``_hcpycall``,
built with the library) that converts the arguments in C and calls the loaded
library's own entry points: ctypes' per-call conversion of 11 arguments cost more
host time than the read's two kernel launches. Where that module was not built, the
calls go through ctypes.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhcread.so")

HC_OK = 0
HC_ERR_ARG = -1
HC_ERR_NOT_INIT = -2
HC_ERR_ARCH = -3
HC_ERR_CUDA = -4
HC_ERR_TIMEOUT = -5
HC_ERR_CHECK = -6
HC_ERR_NOMEM = -7
HC_ERR_BOUNDS = -8

HC_PATH_AUTO = 0
HC_PATH_DECODE = 1
HC_PATH_PREFILL = 2
HC_PATH_PREFILL_UNFUSED = 3
HC_PATH_DECODE_ONE_KERNEL = 4
HC_PATH_PREFILL_BF16_LO = 5

STREAMS, WIDTH, RANK = 4, 2560, 320

# every symbol include/hc_read.h declares
EXPORTS = ("hc_read_init", "hc_read", "hc_read_path", "hc_read_check", "hc_read_status",
           "hc_read_strerror", "hc_read_shutdown", "hc_read_version", "hc_read_noalloc",
           "hc_read_upmix", "hc_read_lo_bf16", "hc_read_y", "hc_read_set_wait_limit",
           "hc_read_bounds_checked")


class HcReadError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {code} ({strerror(code)})")


class hc_check_report(ctypes.Structure):
    _fields_ = [
        ("device", ctypes.c_int),
        ("sm_count", ctypes.c_int),
        ("tokens_checked", ctypes.c_int),
        ("repeat_bitwise", ctypes.c_int),
        ("pending_write_bitwise", ctypes.c_int),
        ("images_bitwise", ctypes.c_int),
        ("paths_agree", ctypes.c_int),
        ("max_rel_diff", ctypes.c_double),
        ("max_rel_tol", ctypes.c_double),
        ("device_name", ctypes.c_char * 64),
    ]

    def as_dict(self) -> dict:
        d = {k: getattr(self, k) for k, _ in self._fields_}
        d["device_name"] = self.device_name.decode(errors="replace")
        return d


_lib = None
_call = None        # the _hcpycall module, bound to _lib's entry points


def _bind_call(lib: ctypes.CDLL) -> None:
    global _call
    try:
        from . import _hcpycall
    except ImportError:
        return
    addr = lambda f: ctypes.cast(f, ctypes.c_void_p).value  # noqa: E731
    _hcpycall.bind(addr(lib.hc_read), addr(lib.hc_read_path))
    _call = _hcpycall


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the library (once). Raises ImportError if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m hyper_connection_residual_read_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
    lib.hc_read_init.argtypes = [i32, i32, ctypes.c_float]
    lib.hc_read_init.restype = i32
    lib.hc_read.argtypes = [i32] + [vp] * 10
    lib.hc_read.restype = i32
    lib.hc_read_path.argtypes = [i32, i32] + [vp] * 10
    lib.hc_read_path.restype = i32
    lib.hc_read_check.argtypes = [i32, u64, ctypes.POINTER(hc_check_report)]
    lib.hc_read_check.restype = i32
    lib.hc_read_status.argtypes = [vp]
    lib.hc_read_status.restype = i32
    lib.hc_read_strerror.argtypes = [i32]
    lib.hc_read_strerror.restype = ctypes.c_char_p
    lib.hc_read_shutdown.argtypes = []
    lib.hc_read_shutdown.restype = None
    lib.hc_read_version.argtypes = []
    lib.hc_read_version.restype = i32
    lib.hc_read_noalloc.argtypes = [i32] + [vp] * 9 + [ctypes.c_float, vp]
    lib.hc_read_noalloc.restype = i32
    lib.hc_read_upmix.argtypes = [i32, i32] + [vp] * 8
    lib.hc_read_upmix.restype = i32
    lib.hc_read_y.argtypes = [i32] + [vp] * 9
    lib.hc_read_y.restype = i32
    lib.hc_read_lo_bf16.argtypes = [i32, vp, vp]
    lib.hc_read_lo_bf16.restype = i32
    lib.hc_read_set_wait_limit.argtypes = [u64]
    lib.hc_read_set_wait_limit.restype = i32
    lib.hc_read_bounds_checked.argtypes = []
    lib.hc_read_bounds_checked.restype = i32
    _lib = lib
    _bind_call(lib)
    return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    raise TypeError(f"expected a tensor, an int pointer or None, got {type(x)!r}")


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if type(stream) is int:
        return stream
    return stream.cuda_stream


def _check(fn: str, code: int) -> int:
    if code != HC_OK:
        raise HcReadError(fn, code)
    return code


def strerror(code: int) -> str:
    return load().hc_read_strerror(code).decode()


def hc_read_version() -> int:
    return load().hc_read_version()


def hc_read_bounds_checked() -> bool:
    """True if the loaded library is the bounds-checked build."""
    return bool(load().hc_read_bounds_checked())


def hc_read_init(device: int = 0, max_tokens: int = 8, eps: float = 1e-6) -> None:
    _check("hc_read_init", load().hc_read_init(device, max_tokens, eps))


def hc_read(tokens, R, P, w_norm, W_down, W_up, Rmix, out_f32, out_bf16, out_fp16,
            stream=None) -> None:
    """Enqueues one read on ``stream`` (default: torch's current stream)."""
    lib = _lib if _lib is not None else load()
    if _call is not None:
        code = _call.read(tokens, R, P, w_norm, W_down, W_up, Rmix, out_f32, out_bf16, out_fp16,
                          _stream(stream))
    else:
        code = lib.hc_read(tokens, _ptr(R), _ptr(P), _ptr(w_norm), _ptr(W_down), _ptr(W_up),
                           _ptr(Rmix), _ptr(out_f32), _ptr(out_bf16), _ptr(out_fp16),
                           _stream(stream))
    if code != HC_OK:
        raise HcReadError("hc_read", code)


def hc_read_path(path, tokens, R, P, w_norm, W_down, W_up, Rmix, out_f32, out_bf16,
                 out_fp16, stream=None) -> None:
    """``hc_read`` with an explicit kernel path (HC_PATH_*)."""
    lib = _lib if _lib is not None else load()
    if _call is not None:
        code = _call.read_path(path, tokens, R, P, w_norm, W_down, W_up, Rmix, out_f32,
                               out_bf16, out_fp16, _stream(stream))
    else:
        code = lib.hc_read_path(path, tokens, _ptr(R), _ptr(P), _ptr(w_norm), _ptr(W_down),
                                _ptr(W_up), _ptr(Rmix), _ptr(out_f32), _ptr(out_bf16),
                                _ptr(out_fp16), _stream(stream))
    if code != HC_OK:
        raise HcReadError("hc_read_path", code)


def hc_read_noalloc(tokens, R, P, w_norm, W_down, W_up, Rmix, out_f32, out_bf16, out_fp16,
                    eps: float = 1e-6, stream=None) -> None:
    """The decode read with no allocation by the library (at most 64 tokens; the
    scratch is a fixed device array shared by every call on the device)."""
    _check("hc_read_noalloc", load().hc_read_noalloc(
        tokens, _ptr(R), _ptr(P), _ptr(w_norm), _ptr(W_down), _ptr(W_up), _ptr(Rmix),
        _ptr(out_f32), _ptr(out_bf16), _ptr(out_fp16), eps, _stream(stream)))


def hc_read_upmix(path, tokens, R, P, W_up, Rmix, out_f32, out_bf16, out_fp16,
                  stream=None) -> None:
    """Re-runs the up projection + gate + mix stage of the last tile-path call
    (``path``: HC_PATH_PREFILL, HC_PATH_PREFILL_UNFUSED or HC_PATH_PREFILL_BF16_LO) on
    the lo that call left in the library's scratch."""
    _check("hc_read_upmix", load().hc_read_upmix(
        path, tokens, _ptr(R), _ptr(P), _ptr(W_up), _ptr(Rmix), _ptr(out_f32), _ptr(out_bf16),
        _ptr(out_fp16), _stream(stream)))


def hc_read_y(tokens, R, P, w_norm, W_down, W_up, out_f32, out_bf16, out_fp16,
              stream=None) -> None:
    """The read with the 2560-wide read-out y = sum of the gated streams ([T][2560]
    fp32 and its bf16 / fp16 images) instead of the 4x4 mix."""
    _check("hc_read_y", load().hc_read_y(
        tokens, _ptr(R), _ptr(P), _ptr(w_norm), _ptr(W_down), _ptr(W_up), _ptr(out_f32),
        _ptr(out_bf16), _ptr(out_fp16), _stream(stream)))


def hc_read_lo_bf16(tokens, lo_out, stream=None) -> None:
    """Copies lo of the last tile-path call, rounded once to bf16 (the A operand of the
    HC_PATH_PREFILL_BF16_LO up GEMM), into ``lo_out`` ([tokens][320] 16-bit device
    tensor)."""
    _check("hc_read_lo_bf16", load().hc_read_lo_bf16(tokens, _ptr(lo_out), _stream(stream)))


def hc_read_check(max_tokens: int = 8, seed: int = 0) -> tuple[int, dict]:
    rep = hc_check_report()
    code = load().hc_read_check(max_tokens, seed, ctypes.byref(rep))
    return code, rep.as_dict()


def hc_read_set_wait_limit(ns: int) -> None:
    """Bound of the one-kernel decode read's wait for the other CTAs' lo, in ns (0:
    the default, 2 s). Tests of failure detection shorten it."""
    _check("hc_read_set_wait_limit", load().hc_read_set_wait_limit(ns))


def hc_read_status(stream=None) -> int:
    return load().hc_read_status(_stream(stream))


def hc_read_shutdown() -> None:
    load().hc_read_shutdown()
