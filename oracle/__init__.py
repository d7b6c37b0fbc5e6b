"""fp64 CPU oracle for the multi-LoRA shrink/expand path (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (``expand_gemm_gb300``)
never does: it runs on the GPU or fails.

The arithmetic lives in ``lora_oracle.c`` (plain C, double precision, one
token at a time); this module only builds that file with gcc and marshals
numpy arrays into it.  bf16 values travel as their raw ``uint16`` bit
patterns so that neither side has to trust the other's conversion.

What each function follows (API pages of vLLM's LoRA package):

* :func:`meta_prepare` -- page ``vllm.lora.ops.triton_ops.lora_kernel_metadata``,
  ``LoRAKernelMeta._reset`` and ``LoRAKernelMeta.prepare_tensors``.
* :func:`shrink` -- page ``vllm.lora.punica_wrapper.punica_gpu``,
  ``PunicaWrapperGPU.add_shrink`` (its "Semantics" docstring).
* :func:`expand` -- same page, ``PunicaWrapperGPU.add_expand`` (its
  "Semantics" docstring), with the bias handling of page
  ``vllm.lora.punica_wrapper.punica_tpu``, ``PunicaWrapperTPU._apply_bias``.

Every function is pinned by ``tests/test_oracle_*.py`` against values the
pages print, closed forms, invariants and library routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liblora_oracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32


def compile_source(src: str, out: str) -> str:
    """Compile an oracle C source into a shared library with the flags
    :func:`build` uses (the mutation tests build altered copies this way)."""
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=gnu11", "-O2", "-fopenmp", "-ffp-contract=off",
           "-fPIC", "-shared", "-Wall", "-o", tmp, src]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``lora_oracle.c`` into ``liblora_oracle.so`` beside it."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    lib.oracle_bf16_to_f64.argtypes = [_P, _I64, _P]
    lib.oracle_bf16_to_f64.restype = None
    lib.oracle_meta_prepare.argtypes = [_P, _I64, _I32, _P, _P, _P, _P, _P, _P]
    lib.oracle_meta_prepare.restype = _I64
    lib.oracle_shrink.argtypes = [_P, _I64, _I64, _I64, _P, _I32, _I32, _I32, _P,
                                  ctypes.c_double, _P, _P]
    lib.oracle_shrink.restype = None
    lib.oracle_expand.argtypes = [_P, _I64, _I32, _P, _P, _P, _I32, _I32, _P, _P, _I64,
                                  _I64, _I32, _P]
    lib.oracle_expand.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def load_library(path: str) -> None:
    """Bind this module to another build of the oracle source, such as a
    copy with a planted mistake (the mutation tests do this in a child
    process, to check that the pins catch the mistake)."""
    global _lib
    with _lock:
        _lib = _bind(ctypes.CDLL(os.path.abspath(path)))


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous, "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _ptr_array(arrays):
    """Host array of pointers (entries may be None -> NULL)."""
    arr = (ctypes.c_void_p * len(arrays))()
    for i, a in enumerate(arrays):
        arr[i] = None if a is None else _ptr(a)
    return arr


def num_threads() -> int:
    """Threads the oracle's OpenMP loops run on (OMP_NUM_THREADS, else the
    cores this process may use)."""
    return int(_load().oracle_num_threads())


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    src = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(src.shape, dtype=np.float64)
    _load().oracle_bf16_to_f64(_ptr(src), src.size, _ptr(out))
    return out


class Meta:
    """Host copy of the six LoRAKernelMeta buffers plus the invalid-id count."""

    def __init__(self, max_loras: int, max_num_tokens: int, fill: int = 0x7EADBEEF):
        # Buffers start at a sentinel so that "not written" is observable.
        self.token_lora_mapping = np.full(max_num_tokens, fill, np.int32)
        self.token_indices_sorted_by_lora_ids = np.full(max_num_tokens, fill, np.int32)
        self.active_lora_ids = np.full(max_loras + 1, fill, np.int32)
        self.num_tokens_per_lora = np.full(max_loras + 1, fill, np.int32)
        self.lora_token_start_loc = np.full(max_loras + 2, fill, np.int32)
        self.no_lora_flag = np.full(1, fill, np.int32)
        self.max_loras = max_loras
        self.invalid_ids = 0


def meta_prepare(token_lora_mapping: np.ndarray, max_loras: int,
                 meta: Meta | None = None) -> Meta:
    """Oracle of LoRAKernelMeta.prepare_tensors (see lora_oracle.c)."""
    m = np.ascontiguousarray(token_lora_mapping, dtype=np.int32)
    T = m.shape[0]
    if meta is None:
        meta = Meta(max_loras, max(T, 1))
    assert meta.max_loras == max_loras and meta.token_lora_mapping.shape[0] >= T
    meta.invalid_ids = int(_load().oracle_meta_prepare(
        _ptr(m), T, max_loras,
        _ptr(meta.token_lora_mapping), _ptr(meta.token_indices_sorted_by_lora_ids),
        _ptr(meta.active_lora_ids), _ptr(meta.num_tokens_per_lora),
        _ptr(meta.lora_token_start_loc), _ptr(meta.no_lora_flag)))
    return meta


def shrink(x_bits: np.ndarray, lora_a: list, token_lora_mapping: np.ndarray,
           scale: float, buf_in: np.ndarray) -> np.ndarray:
    """Oracle of lora_shrink: returns buf_in + scale * x @ A[s][id]^T in float64.

    x_bits: uint16 [T, H] (row stride may exceed H: pass a 2-D view whose
    rows are contiguous); lora_a: S arrays uint16 [L, r, H] (a leading
    singleton layer dimension is accepted); buf_in: float32 [S, T, r].
    """
    x2 = np.asarray(x_bits, dtype=np.uint16)
    T, H = x2.shape
    if x2.flags.c_contiguous:
        x_ld = H
    else:
        assert x2.strides[1] == 2 and x2.strides[0] % 2 == 0 and x2.strides[0] >= 2 * H, \
            "x rows must be contiguous with a non-negative row stride"
        x_ld = x2.strides[0] // 2
    xptr = x2.ctypes.data
    A = [np.ascontiguousarray(a, dtype=np.uint16) for a in lora_a]
    S = len(A)
    A = [a.reshape(-1, a.shape[-2], a.shape[-1]) for a in A]
    L, r, Ha = A[0].shape
    assert Ha == H and all(a.shape == (L, r, H) for a in A)
    m = np.ascontiguousarray(token_lora_mapping, dtype=np.int32)
    assert m.shape == (T,)
    bi = np.ascontiguousarray(buf_in, dtype=np.float32)
    assert bi.shape == (S, T, r)
    out = np.empty((S, T, r), np.float64)
    _load().oracle_shrink(xptr, T, H, x_ld, _ptr_array(A), S, r, L, _ptr(m),
                          float(scale), _ptr(bi), _ptr(out))
    return out


def expand(xin: np.ndarray, lora_b: list, token_lora_mapping: np.ndarray,
           y_in_bits: np.ndarray, slice_sizes, offset_start: int = 0,
           add_inputs: bool = True, lora_bias: list | None = None) -> np.ndarray:
    """Oracle of lora_expand with fused bias: returns y as float64 [T, y_ld].

    xin: float32 [S, T, r]; lora_b: S arrays uint16 [L, n_s, r];
    lora_bias: None or S entries (None or uint16 [L, n_s]);
    y_in_bits: uint16 [T, y_ld].
    """
    xi = np.ascontiguousarray(xin, dtype=np.float32)
    S, T, r = xi.shape
    B = [np.ascontiguousarray(b, dtype=np.uint16) for b in lora_b]
    B = [b.reshape(-1, b.shape[-2], b.shape[-1]) for b in B]
    assert len(B) == S == len(slice_sizes)
    L = B[0].shape[0]
    sizes = np.ascontiguousarray(slice_sizes, dtype=np.int32)
    for b, n in zip(B, sizes):
        assert b.shape == (L, int(n), r)
    y = np.ascontiguousarray(y_in_bits, dtype=np.uint16)
    assert y.shape[0] == T
    y_ld = y.shape[1]
    assert offset_start + int(sizes.sum()) <= y_ld
    bias_ptrs = None
    keep = []
    if lora_bias is not None:
        assert len(lora_bias) == S
        bl = []
        for b, n in zip(lora_bias, sizes):
            if b is None:
                bl.append(None)
            else:
                bb = np.ascontiguousarray(b, dtype=np.uint16).reshape(L, int(n))
                bl.append(bb)
        keep = bl
        bias_ptrs = _ptr_array(bl)
    m = np.ascontiguousarray(token_lora_mapping, dtype=np.int32)
    assert m.shape == (T,)
    out = np.empty((T, y_ld), np.float64)
    _load().oracle_expand(_ptr(xi), T, r, _ptr_array(B), bias_ptrs, _ptr(sizes),
                          S, L, _ptr(m), _ptr(y), y_ld, int(offset_start),
                          int(bool(add_inputs)), _ptr(out))
    del keep
    return out
