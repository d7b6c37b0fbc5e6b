"""ctypes loader for liblora_punica.so (the C ABI of include/lora_punica.h).

No fallback exists: if the library is missing or a call fails, an exception
is raised.  Build it with ``python -m expand_gemm_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "liblora_punica.so")

# Public entry points of include/lora_punica.h (checked by the test suite).
EXPORTS = ("lora_meta_prepare", "lora_meta_read_no_lora", "lora_shrink", "lora_expand",
           "lora_expand_bf16", "lora_linear", "lora_linear_noalloc", "lora_reload_options",
           "lora_status_string", "lora_version")

LORA_MAX_SLICES = 8
LORA_MAX_LORAS = 1024
LORA_MAX_RANK = 128
LORA_NOALLOC_MAX_FLOATS = 1 << 20


class LoraMetaC(ctypes.Structure):
    """Mirror of ``lora_meta_t``."""
    _fields_ = [
        ("token_lora_mapping", ctypes.c_void_p),
        ("token_indices_sorted_by_lora_ids", ctypes.c_void_p),
        ("num_tokens_per_lora", ctypes.c_void_p),
        ("lora_token_start_loc", ctypes.c_void_p),
        ("active_lora_ids", ctypes.c_void_p),
        ("no_lora_flag", ctypes.c_void_p),
        ("error_word", ctypes.c_void_p),
        ("max_loras", ctypes.c_int32),
        ("max_num_tokens", ctypes.c_int32),
        ("grid_sync", ctypes.c_void_p),
    ]


class LoraError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__("%s failed with status %d: %s" % (fn, status, msg))
        self.status = status


_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64


def load(path: str | None = None):
    """Load (once) and return the CUDA library; raise if it is not built.
    ``LORA_PUNICA_LIBRARY`` in the environment names another build of it
    (the debug-checks build) to load instead."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or os.environ.get("LORA_PUNICA_LIBRARY") or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                "liblora_punica.so is not built (expected at %s); run "
                "`python -m expand_gemm_gb300.build` -- there is no CPU fallback" % p)
        lib = ctypes.CDLL(p)
        lib.lora_meta_prepare.argtypes = [_P, _I32, ctypes.POINTER(LoraMetaC), _P]
        lib.lora_meta_prepare.restype = ctypes.c_int
        lib.lora_meta_read_no_lora.argtypes = [ctypes.POINTER(LoraMetaC), _P,
                                               ctypes.POINTER(ctypes.c_int32)]
        lib.lora_meta_read_no_lora.restype = ctypes.c_int
        lib.lora_shrink.argtypes = [_P, _I32, _I32, _I64, _P, _I32, _I32, _P,
                                    ctypes.POINTER(LoraMetaC), ctypes.c_float, _P]
        lib.lora_shrink.restype = ctypes.c_int
        lib.lora_expand.argtypes = [_P, _P, _P, _P, _I32, _I32, _P, _I64, _I32,
                                    _I32, _I32, ctypes.POINTER(LoraMetaC), _P]
        lib.lora_expand.restype = ctypes.c_int
        lib.lora_expand_bf16.argtypes = lib.lora_expand.argtypes
        lib.lora_expand_bf16.restype = ctypes.c_int
        lib.lora_linear.argtypes = [_P, _I32, _P, _I32, _I64, _P, _P, _P, _P, _I32, _I32,
                                    ctypes.c_float, _P, _P, _I64, ctypes.POINTER(LoraMetaC), _P]
        lib.lora_linear.restype = ctypes.c_int
        lib.lora_linear_noalloc.argtypes = [_P, _I32, _P, _I32, _I64, _P, _P, _P, _P, _I32,
                                            _I32, ctypes.c_float, _P, _I64,
                                            ctypes.POINTER(LoraMetaC), _P]
        lib.lora_linear_noalloc.restype = ctypes.c_int
        lib.lora_reload_options.argtypes = []
        lib.lora_reload_options.restype = None
        lib.lora_status_string.argtypes = [ctypes.c_int]
        lib.lora_status_string.restype = ctypes.c_char_p
        lib.lora_version.argtypes = []
        lib.lora_version.restype = ctypes.c_int
        _lib = lib
        return lib


def check(fn: str, status: int) -> None:
    if status != 0:
        msg = load().lora_status_string(status).decode()
        raise LoraError(fn, status, msg)
