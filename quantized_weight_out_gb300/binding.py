"""ctypes binding of librg (include/rg.h).  Argument marshalling only.

Every function has the C name and returns the C status code.  Data arguments
accept an int device address, or any object with ``data_ptr()`` (a PyTorch
tensor); ``stream`` accepts None (the legacy default stream), an int handle,
or an object with a ``cuda_stream`` attribute (torch.cuda.Stream).

The library is loaded on first use.  If ``librg.so`` has not been built the
first call raises: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "librg.so")

RG_OK, RG_ERR_ARG, RG_ERR_TYPE, RG_ERR_SHAPE = 0, -1, -2, -3
RG_ERR_ALIGN, RG_ERR_CUDA, RG_ERR_TIMEOUT, RG_ERR_RANGE = -4, -5, -6, -7
RG_VARIANT_AUTO, RG_VARIANT_TC, RG_VARIANT_SMALLT, RG_VARIANT_SIMT32 = 0, 1, 2, 3
RG_VARIANT_TC_SINGLE, RG_VARIANT_TC_PAIR = 4, 5
VARIANTS = {"auto": 0, "tc": 1, "smallt": 2, "simt32": 3, "tc1": 4, "tc2": 5}

class rg_plan_info(ctypes.Structure):
    """include/rg.h rg_plan_info."""
    _fields_ = [("variant", ctypes.c_int32), ("cta_group", ctypes.c_int32),
                ("tile_k", ctypes.c_int32), ("tile_t", ctypes.c_int32),
                ("n_splits", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("launches", ctypes.c_int32), ("stream_k", ctypes.c_int32),
                ("decode_ops", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


# (name, restype, argtypes) of every exported function
_I64, _VP, _F, _I, _SZ = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int, ctypes.c_size_t
SIGNATURES = [
    ("rg_out_prod", _I, [_I, _VP, _I64, _I64, _VP, _I64, _VP, _F, _VP]),
    ("rg_out_prod_variant", _I, [_I, _I, _VP, _I64, _I64, _VP, _I64, _VP, _F, _VP]),
    ("rg_workspace_bytes", _SZ, [_I, _I, _I64, _I64, _I64]),
    ("rg_out_prod_ws", _I, [_I, _I, _VP, _I64, _I64, _VP, _I64, _VP, _F, _VP, _SZ, _VP]),
    ("rg_select_variant", _I, [_I, _I64, _I64, _I64]),
    ("rg_dequant", _I, [_I, _VP, _I64, _I64, _VP]),
    ("rg_dequant_async", _I, [_I, _VP, _I64, _I64, _VP, _VP]),
    ("rg_row_bytes", _SZ, [_I, _I64]),
    ("rg_strerror", ctypes.c_char_p, [_I]),
    ("rg_check", _I, [_VP]),
    ("rg_version", _I, []),
    ("rg_debug_wait_probe", _I, [_I, _VP]),
    ("rg_profile_next_gemm", _I, [_VP, _VP]),
    ("rg_out_prod_noalloc", _I, [_I, _VP, _I64, _I64, _VP, _I64, _VP, _F, _VP]),
    ("rg_plan", _I, [_I, _I, _I64, _I64, _I64, ctypes.POINTER(rg_plan_info)]),
    ("rg_mul_mat", _I, [_I, _VP, _I64, _I64, _VP, _I64, _VP, _F, _VP]),
    ("rg_mul_mat_variant", _I, [_I, _I, _VP, _I64, _I64, _VP, _I64, _VP, _F, _VP]),
    ("rg_out_prod_lora", _I, [_I, _I, _VP, _I64, _I64, _VP, _I64, _VP, _F, _VP, _VP, _I64, _F, _VP]),
    ("rg_out_prod_ex", _I, [_I, _I, _VP, _I64, _I64, _I64, _VP, _I64, _I64, _I64, _I64, _VP, _I64,
                            _I64, _I64, _F, _VP]),
    ("rg_launch_count", ctypes.c_uint64, []),
    ("rg_mul_mat_workspace_bytes", _SZ, [_I, _I64, _I64, _I64]),
    ("rg_out_prod_batched", _I, [_I, _I, _VP, _I64, _I64, _I64, _I64, _I64, _I64, _VP, _I64, _I64,
                                 _I64, _I64, _I64, _VP, _I64, _I64, _I64, _I64, _I64, _F, _VP]),
]

RG_NOALLOC_SCRATCH_BYTES = 32 << 20

_lib = None
_lock = threading.Lock()


class RgError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} ({status})" if what else f"{strerror(status)} ({status})")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load librg.so (once) and declare its signatures."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with quantized_weight_out_gb300.build.build() "
                    "(there is no CPU fallback)")
            lib = ctypes.CDLL(path)
            for name, res, args in SIGNATURES:
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def rg_out_prod(wtype, W, N, K, dY, T, dX, beta, stream=None) -> int:
    return load().rg_out_prod(wtype, _ptr(W), N, K, _ptr(dY), T, _ptr(dX), beta, _stream(stream))


def rg_out_prod_variant(variant, wtype, W, N, K, dY, T, dX, beta, stream=None) -> int:
    return load().rg_out_prod_variant(variant, wtype, _ptr(W), N, K, _ptr(dY), T, _ptr(dX), beta,
                                      _stream(stream))


def rg_out_prod_noalloc(wtype, W, N, K, dY, T, dX, beta, stream=None) -> int:
    return load().rg_out_prod_noalloc(wtype, _ptr(W), N, K, _ptr(dY), T, _ptr(dX), beta,
                                      _stream(stream))


def rg_out_prod_ex(variant, wtype, W, N, K, w_batch_bytes, dY, T, dy_t, dy_n, dy_batch, dX, dx_t,
                   dx_batch, batch, beta, stream=None) -> int:
    return load().rg_out_prod_ex(variant, wtype, _ptr(W), N, K, w_batch_bytes, _ptr(dY), T, dy_t,
                                 dy_n, dy_batch, _ptr(dX), dx_t, dx_batch, batch, beta,
                                 _stream(stream))


def rg_out_prod_batched(variant, wtype, W, N, K, w_n2, w_n3, w_s2, w_s3, dY, T, dy_t, dy_n, dy_s2,
                        dy_s3, dX, dx_t, dx_s2, dx_s3, n2, n3, beta, stream=None) -> int:
    return load().rg_out_prod_batched(variant, wtype, _ptr(W), N, K, w_n2, w_n3, w_s2, w_s3,
                                      _ptr(dY), T, dy_t, dy_n, dy_s2, dy_s3, _ptr(dX), dx_t, dx_s2,
                                      dx_s3, n2, n3, beta, _stream(stream))


def rg_mul_mat(wtype, W, N, K, X, T, Y, beta, stream=None) -> int:
    return load().rg_mul_mat(wtype, _ptr(W), N, K, _ptr(X), T, _ptr(Y), beta, _stream(stream))


def rg_mul_mat_variant(variant, wtype, W, N, K, X, T, Y, beta, stream=None) -> int:
    return load().rg_mul_mat_variant(variant, wtype, _ptr(W), N, K, _ptr(X), T, _ptr(Y), beta,
                                     _stream(stream))


def rg_mul_mat_workspace_bytes(wtype, N, K, T) -> int:
    return load().rg_mul_mat_workspace_bytes(wtype, N, K, T)


def rg_out_prod_lora(variant, wtype, W, N, K, dY, T, dX, beta, lora_a, lora_b, rank, scale,
                     stream=None) -> int:
    return load().rg_out_prod_lora(variant, wtype, _ptr(W), N, K, _ptr(dY), T, _ptr(dX), beta,
                                   _ptr(lora_a), _ptr(lora_b), rank, scale, _stream(stream))


def rg_workspace_bytes(variant, wtype, N, K, T) -> int:
    return load().rg_workspace_bytes(variant, wtype, N, K, T)


def rg_out_prod_ws(variant, wtype, W, N, K, dY, T, dX, beta, workspace, workspace_bytes,
                   stream=None) -> int:
    return load().rg_out_prod_ws(variant, wtype, _ptr(W), N, K, _ptr(dY), T, _ptr(dX), beta,
                                 _ptr(workspace), workspace_bytes, _stream(stream))


def rg_select_variant(wtype, N, K, T) -> int:
    return load().rg_select_variant(wtype, N, K, T)


def rg_plan(variant, wtype, N, K, T, out: rg_plan_info) -> int:
    return load().rg_plan(variant, wtype, N, K, T, ctypes.byref(out))


def rg_launch_count() -> int:
    return int(load().rg_launch_count())


def rg_dequant(wtype, W, N, K, out) -> int:
    return load().rg_dequant(wtype, _ptr(W), N, K, _ptr(out))


def rg_dequant_async(wtype, W, N, K, out, stream=None) -> int:
    return load().rg_dequant_async(wtype, _ptr(W), N, K, _ptr(out), _stream(stream))


def rg_row_bytes(wtype, K) -> int:
    return load().rg_row_bytes(wtype, K)


def strerror(status: int) -> str:
    return load().rg_strerror(status).decode()


rg_strerror = strerror


def rg_check(stream=None) -> int:
    return load().rg_check(_stream(stream))


def rg_version() -> int:
    return load().rg_version()


def rg_debug_wait_probe(timeout_ms, stream=None) -> int:
    return load().rg_debug_wait_probe(timeout_ms, _stream(stream))


def _event(e):
    if e is None:
        return None
    if isinstance(e, int):
        return e
    return int(e.cuda_event)


def rg_profile_next_gemm(before, after) -> int:
    return load().rg_profile_next_gemm(_event(before), _event(after))


def check(status: int, what: str = "") -> None:
    """Raise RgError unless status is RG_OK."""
    if status != RG_OK:
        raise RgError(status, what)
