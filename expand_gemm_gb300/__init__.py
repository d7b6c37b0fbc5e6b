"""GB300 (sm_103a) multi-LoRA shrink/expand: thin PyTorch binding.

Every step runs in the CUDA kernels of ``liblora_punica.so`` (C ABI in
``include/lora_punica.h``); this module only checks tensor dtypes and
layouts, collects device pointers and the current CUDA stream, and calls the
library.  PyTorch provides device memory and streams, nothing else.  There
is no CPU fallback: without the built library every call raises.

Names follow vLLM's API pages:

* :class:`LoRAKernelMeta` -- page ``vllm.lora.ops.triton_ops.lora_kernel_metadata``
  (``make``, ``prepare_tensors``, ``meta_args``; ``no_lora`` is the host copy of
  the flag, the page's ``no_lora_flag_cpu``).
* :func:`lora_shrink`, :func:`lora_expand`, :func:`add_lora_linear`,
  :func:`add_lora_embedding`, :func:`add_lora_logits` -- page
  ``vllm.lora.punica_wrapper.punica_gpu`` (``PunicaWrapperGPU.add_shrink``,
  ``add_expand``, ``add_lora_linear``, ``add_lora_embedding``,
  ``add_lora_logits``).
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _lib
from ._lib import (LoraError, LORA_MAX_LORAS, LORA_MAX_RANK, LORA_MAX_SLICES,  # noqa: F401
                   LORA_NOALLOC_MAX_FLOATS)

__all__ = ["LoRAKernelMeta", "lora_meta_prepare", "lora_shrink", "lora_expand",
           "lora_linear", "lora_linear_noalloc", "add_lora_linear", "add_lora_embedding",
           "add_lora_logits", "reload_options", "LoraError", "library", "build"]


def library():
    """The loaded ctypes library (raises if it is not built)."""
    return _lib.load()


def build(force: bool = False) -> str:
    from .build import build as _build
    return _build(force=force)


def reload_options() -> None:
    """Re-read the LORA_PUNICA_* tuning variables (the library reads them
    once, at its first call): ``lora_reload_options``."""
    _lib.load().lora_reload_options()


def _stream_handle(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _need(t: torch.Tensor, name: str, dtype: torch.dtype) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (no CPU path exists)" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))


def _same_device(meta: "LoRAKernelMeta", named) -> None:
    """Every tensor of ``named`` ((name, tensor or None) pairs) must be on
    the GPU that holds the metadata: the kernels take raw pointers, so a
    tensor on another device would be read through the wrong address space."""
    dev = meta.no_lora_flag.get_device()
    for name, t in named:
        if t is not None and t.get_device() != dev:
            raise ValueError("%s is on cuda:%d, the metadata on cuda:%d"
                             % (name, t.get_device(), dev))


def _call(fn: str, device: torch.device, *args) -> None:
    """Calls library entry point `fn` with `device` current (the library
    looks up per-device state for the current device), then raises on a
    non-zero status."""
    with torch.cuda.device(device):
        st = getattr(_lib.load(), fn)(*args)
    _lib.check(fn, st)


def _ptr_array(tensors) -> ctypes.Array:
    arr = (ctypes.c_void_p * len(tensors))()
    for i, t in enumerate(tensors):
        arr[i] = None if t is None else t.data_ptr()
    return arr


class LoRAKernelMeta:
    """Per-forward metadata buffers (LoRAKernelMeta of the metadata page).

    Buffers are int32 device tensors allocated once by :meth:`make`; the
    no-LoRA flag lives on the device (the kernels read it there, so no host
    sync is needed; :meth:`no_lora` copies it to the host on request);
    ``error_word`` counts ids outside ``[-1, max_loras)`` seen by the last
    :meth:`prepare_tensors`.
    """

    def __init__(self, max_loras: int, max_num_tokens: int, device):
        if not 1 <= max_loras <= LORA_MAX_LORAS:
            raise ValueError("max_loras must be in [1, %d]" % LORA_MAX_LORAS)
        if max_num_tokens < 0:
            raise ValueError("max_num_tokens must be >= 0")
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.max_loras = int(max_loras)
        self.max_num_tokens = int(max_num_tokens)
        self.token_lora_mapping = torch.empty(max(max_num_tokens, 1), **i32)
        self.token_indices_sorted_by_lora_ids = torch.empty(max(max_num_tokens, 1), **i32)
        self.active_lora_ids = torch.full((max_loras + 1,), -1, **i32)
        self.num_tokens_per_lora = torch.zeros(max_loras + 1, **i32)
        self.lora_token_start_loc = torch.zeros(max_loras + 2, **i32)
        self.no_lora_flag = torch.ones(1, **i32)
        self.error_word = torch.zeros(1, **i32)
        # grid barrier of lora_linear's single-kernel path (left zero by every call)
        self.grid_sync = torch.zeros(2, **i32)
        self.c = _lib.LoraMetaC(
            self.token_lora_mapping.data_ptr(),
            self.token_indices_sorted_by_lora_ids.data_ptr(),
            self.num_tokens_per_lora.data_ptr(),
            self.lora_token_start_loc.data_ptr(),
            self.active_lora_ids.data_ptr(),
            self.no_lora_flag.data_ptr(),
            self.error_word.data_ptr(),
            self.max_loras, self.max_num_tokens,
            self.grid_sync.data_ptr())
        self.device = dev

    @staticmethod
    def make(max_loras: int, max_num_tokens: int, device) -> "LoRAKernelMeta":
        return LoRAKernelMeta(max_loras, max_num_tokens, device)

    def prepare_tensors(self, token_lora_mapping: torch.Tensor) -> None:
        lora_meta_prepare(token_lora_mapping, self)

    def meta_args(self, token_nums: int):
        """The six metadata tensors in the order the kernels take them."""
        return (self.token_lora_mapping[:token_nums],
                self.token_indices_sorted_by_lora_ids[:token_nums],
                self.num_tokens_per_lora, self.lora_token_start_loc,
                self.active_lora_ids, self.no_lora_flag)

    def no_lora(self) -> bool:
        """Host read of the flag through ``lora_meta_read_no_lora``
        (synchronises the current stream; the kernels never need it)."""
        out = ctypes.c_int32(-1)
        _call("lora_meta_read_no_lora", self.device, ctypes.byref(self.c),
              _stream_handle(self.device), ctypes.byref(out))
        return bool(out.value)


def lora_meta_prepare(token_lora_mapping: torch.Tensor, meta: LoRAKernelMeta) -> None:
    m = token_lora_mapping
    _need(m, "token_lora_mapping", torch.int32)
    if m.dim() != 1 or not m.is_contiguous():
        raise ValueError("token_lora_mapping must be a contiguous 1-D tensor")
    _same_device(meta, [("token_lora_mapping", m)])
    _call("lora_meta_prepare", meta.device, m.data_ptr() if m.numel() else None, m.numel(),
          ctypes.byref(meta.c), _stream_handle(meta.device))


def _weights(ws: Sequence[torch.Tensor], name: str):
    if isinstance(ws, torch.Tensor):
        ws = (ws,)
    out = []
    for i, w in enumerate(ws):
        _need(w, "%s[%d]" % (name, i), torch.bfloat16)
        if not w.is_contiguous():
            raise ValueError("%s[%d] must be contiguous" % (name, i))
        if w.dim() == 4 and w.size(1) == 1:          # [L, 1, rows, cols] layer dim
            w = w.view(w.size(0), w.size(2), w.size(3))
        if w.dim() != 3:
            raise ValueError("%s[%d] must be [max_loras, rows, cols]" % (name, i))
        out.append(w)
    return out


def lora_shrink(x: torch.Tensor, lora_a_stacked, y: torch.Tensor,
                meta: LoRAKernelMeta, scale: float) -> None:
    """y[s] += scale * x @ lora_a_stacked[s][id]^T for tokens with a LoRA."""
    _need(x, "x", torch.bfloat16)
    _need(y, "y", torch.float32)
    x2 = x.view(-1, x.shape[-1]) if x.dim() != 2 else x
    if x2.stride(1) != 1:
        raise ValueError("x rows must be contiguous")
    A = _weights(lora_a_stacked, "lora_a_stacked")
    T, H = x2.shape
    L, r, Ha = A[0].shape
    if Ha != H or any(a.shape != A[0].shape for a in A):
        raise ValueError("lora_a_stacked shapes must all be [L, r, %d]" % H)
    if L < meta.max_loras:
        raise ValueError("lora_a_stacked has %d LoRAs, metadata expects %d" % (L, meta.max_loras))
    if tuple(y.shape) != (len(A), T, r) or not y.is_contiguous():
        raise ValueError("y must be a contiguous fp32 [%d, %d, %d] tensor" % (len(A), T, r))
    _same_device(meta, [("x", x), ("y", y)] +
                 [("lora_a_stacked[%d]" % i, a) for i, a in enumerate(A)])
    _call("lora_shrink", x.device, x2.data_ptr(), T, H, x2.stride(0), _ptr_array(A), len(A), r,
          y.data_ptr(), ctypes.byref(meta.c), float(scale), _stream_handle(x.device))


def lora_expand(x: torch.Tensor, lora_b_stacked, y: torch.Tensor,
                meta: LoRAKernelMeta, offset_start: int = 0, add_inputs: bool = True,
                lora_bias_stacked: Optional[Sequence[Optional[torch.Tensor]]] = None) -> None:
    """y[:, off_s:off_s+n_s] (+)= x[s] @ lora_b_stacked[s][id]^T (+ bias).

    x is fp32 (the shrink's buffer; rounded to bf16 for the tensor cores) or
    bf16 (taken as it is: lora_expand_bf16)."""
    if not isinstance(x, torch.Tensor) or x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("x must be a float32 or bfloat16 torch.Tensor")
    _need(x, "x", x.dtype)
    _need(y, "y", torch.bfloat16)
    B = _weights(lora_b_stacked, "lora_b_stacked")
    if x.dim() != 3 or not x.is_contiguous() or x.size(0) != len(B):
        raise ValueError("x must be a contiguous [num_slices, T, r] tensor")
    S, T, r = x.shape
    L = B[0].size(0)
    if L < meta.max_loras:
        raise ValueError("lora_b_stacked has %d LoRAs, metadata expects %d" % (L, meta.max_loras))
    for i, b in enumerate(B):
        if b.size(0) != L or b.size(2) != r:
            raise ValueError("lora_b_stacked[%d] must be [%d, n, %d]" % (i, L, r))
    sizes = [b.size(1) for b in B]
    y2 = y.view(-1, y.shape[-1]) if y.dim() != 2 else y
    if y2.stride(1) != 1 or y2.size(0) != T:
        raise ValueError("y must be [T, width] with contiguous rows")
    bias_arr = None
    if lora_bias_stacked is not None:
        if len(lora_bias_stacked) != S:
            raise ValueError("lora_bias_stacked needs one entry per slice")
        bl = []
        for i, (bb, n) in enumerate(zip(lora_bias_stacked, sizes)):
            if bb is None:
                bl.append(None)
                continue
            _need(bb, "lora_bias_stacked[%d]" % i, torch.bfloat16)
            if not bb.is_contiguous() or bb.numel() != L * n:
                raise ValueError("lora_bias_stacked[%d] must be [%d, %d]" % (i, L, n))
            bl.append(bb)
        bias_arr = _ptr_array(bl)
    biases = () if lora_bias_stacked is None else lora_bias_stacked
    _same_device(meta, [("x", x), ("y", y)] +
                 [("lora_b_stacked[%d]" % i, b) for i, b in enumerate(B)] +
                 [("lora_bias_stacked[%d]" % i, b) for i, b in enumerate(biases)])
    size_arr = (ctypes.c_int32 * S)(*sizes)
    fn = "lora_expand_bf16" if x.dtype == torch.bfloat16 else "lora_expand"
    _call(fn, x.device, x.data_ptr(), _ptr_array(B), bias_arr, size_arr, S, r,
          y2.data_ptr(), y2.stride(0), T, int(offset_start), 1 if add_inputs else 0,
          ctypes.byref(meta.c), _stream_handle(x.device))


def add_lora_embedding(y: torch.Tensor, x: torch.Tensor, lora_b_stacked,
                       meta: LoRAKernelMeta, add_inputs: bool = True) -> None:
    """PunicaWrapperGPU.add_lora_embedding: y (+)= x @ lora_b_stacked[id]^T,
    where x is bf16 [T, r] (the embedding LoRA's A rows looked up per
    token) and add_inputs is passed through."""
    _need(x, "x", torch.bfloat16)
    x2 = x.view(-1, x.shape[-1])
    lora_expand(x2.unsqueeze(0), lora_b_stacked, y, meta, 0, add_inputs)


def add_lora_logits(y: torch.Tensor, x: torch.Tensor, lora_a_stacked, lora_b_stacked,
                    scale: float, meta: LoRAKernelMeta, *,
                    buffer: Optional[torch.Tensor] = None) -> None:
    """PunicaWrapperGPU.add_lora_logits: buffer = scale * x @ A[id]^T, then
    y += buffer @ B[id]^T, both driven by ``meta`` (the prompt/sampler
    metadata instance, one id per logits row)."""
    y2 = y.view(-1, y.shape[-1])
    x2 = x.view(-1, x.shape[-1])
    B = _weights(lora_b_stacked, "lora_b_stacked")
    if len(B) != 1:
        raise ValueError("add_lora_logits takes one lora_b tensor")
    r = B[0].size(-1)
    if buffer is None:
        buffer = torch.zeros((x2.size(0), r), dtype=torch.float32, device=x.device)
    lora_shrink(x2, lora_a_stacked, buffer.unsqueeze(0), meta, scale)
    lora_expand(buffer.unsqueeze(0), B, y2, meta, 0, True)


def add_lora_linear(y: torch.Tensor, x: torch.Tensor, lora_a_stacked, lora_b_stacked,
                    lora_bias_stacked, scale: float, output_slices, meta: LoRAKernelMeta,
                    *, buffer: Optional[torch.Tensor] = None) -> None:
    """PunicaWrapperGPU.add_lora_linear: shrink into an fp32 buffer, then
    expand into y with the bias fused into the expand kernel."""
    A = _weights(lora_a_stacked, "lora_a_stacked")
    B = _weights(lora_b_stacked, "lora_b_stacked")
    if not len(A) == len(B) == len(output_slices):
        raise ValueError("lora_a_stacked, lora_b_stacked and output_slices differ in length")
    if lora_bias_stacked is not None and len(lora_bias_stacked) != len(output_slices):
        raise ValueError("lora_bias_stacked needs one entry per slice")
    for b, n in zip(B, output_slices):
        if b.size(1) != n:
            raise ValueError("lora_b_stacked widths must match output_slices")
    x2 = x.view(-1, x.shape[-1])
    r = B[0].size(-1)
    if buffer is None:
        buffer = torch.zeros((len(output_slices), x2.size(0), r), dtype=torch.float32,
                             device=x.device)
    lora_shrink(x2, A, buffer, meta, scale)
    lora_expand(buffer, B, y, meta, 0, True, lora_bias_stacked)


def _linear_args(token_lora_mapping, x, lora_a_stacked, lora_b_stacked, lora_bias_stacked,
                 buffer, y):
    """Checks shared by lora_linear and lora_linear_noalloc; returns the
    marshalled C arguments in lora_linear's order (buffer pointer None when
    no buffer is given)."""
    m = token_lora_mapping
    _need(m, "token_lora_mapping", torch.int32)
    _need(x, "x", torch.bfloat16)
    _need(y, "y", torch.bfloat16)
    x2 = x.view(-1, x.shape[-1]) if x.dim() != 2 else x
    y2 = y.view(-1, y.shape[-1]) if y.dim() != 2 else y
    A = _weights(lora_a_stacked, "lora_a_stacked")
    B = _weights(lora_b_stacked, "lora_b_stacked")
    T, H = x2.shape
    if m.dim() != 1 or m.numel() != T or not m.is_contiguous():
        raise ValueError("token_lora_mapping must be a contiguous [T] tensor")
    if x2.stride(1) != 1 or y2.stride(1) != 1 or y2.size(0) != T:
        raise ValueError("x and y need contiguous rows and T rows")
    if len(A) != len(B):
        raise ValueError("lora_a_stacked and lora_b_stacked differ in length")
    L, r, Ha = A[0].shape
    if Ha != H or any(a.shape != A[0].shape for a in A):
        raise ValueError("lora_a_stacked shapes must all be [L, r, %d]" % H)
    for i, b in enumerate(B):
        if b.size(0) != B[0].size(0) or b.size(2) != r:
            raise ValueError("lora_b_stacked[%d] must be [%d, n, %d]" % (i, B[0].size(0), r))
    if buffer is not None:
        _need(buffer, "buffer", torch.float32)
        if tuple(buffer.shape) != (len(A), T, r) or not buffer.is_contiguous():
            raise ValueError("buffer must be a contiguous fp32 [%d, %d, %d] tensor"
                             % (len(A), T, r))
    sizes = [b.size(1) for b in B]
    bias_arr = None
    if lora_bias_stacked is not None:
        if len(lora_bias_stacked) != len(B):
            raise ValueError("lora_bias_stacked needs one entry per slice")
        for i, (bb, n) in enumerate(zip(lora_bias_stacked, sizes)):
            if bb is not None:
                _need(bb, "lora_bias_stacked[%d]" % i, torch.bfloat16)
                if not bb.is_contiguous() or bb.numel() != B[0].size(0) * n:
                    raise ValueError("lora_bias_stacked[%d] must be [L, %d]" % (i, n))
        bias_arr = _ptr_array(list(lora_bias_stacked))
    size_arr = (ctypes.c_int32 * len(B))(*sizes)
    named = ([("token_lora_mapping", m), ("x", x), ("y", y), ("buffer", buffer)] +
             [("lora_a_stacked[%d]" % i, a) for i, a in enumerate(A)] +
             [("lora_b_stacked[%d]" % i, b) for i, b in enumerate(B)] +
             [("lora_bias_stacked[%d]" % i, b)
              for i, b in enumerate(() if lora_bias_stacked is None else lora_bias_stacked)])
    return dict(L=L, nb=B[0].size(0), named=named,
                head=(m.data_ptr(), T, x2.data_ptr(), H, x2.stride(0), _ptr_array(A),
                      _ptr_array(B), bias_arr, size_arr, len(B), r),
                buf=None if buffer is None else buffer.data_ptr(),
                tail=(y2.data_ptr(), y2.stride(0)))


def lora_linear(token_lora_mapping: torch.Tensor, x: torch.Tensor, lora_a_stacked,
                lora_b_stacked, lora_bias_stacked, scale: float, buffer: torch.Tensor,
                y: torch.Tensor, meta: LoRAKernelMeta) -> None:
    """Metadata + shrink + expand of one LoRA layer in one library call
    (PunicaWrapperGPU.update_metadata followed by add_lora_linear).  Small
    batches run as one kernel, larger ones as three overlapping launches;
    see include/lora_punica.h."""
    if not isinstance(buffer, torch.Tensor):
        raise TypeError("buffer must be a torch.Tensor (lora_linear_noalloc needs none)")
    a = _linear_args(token_lora_mapping, x, lora_a_stacked, lora_b_stacked, lora_bias_stacked,
                     buffer, y)
    if a["L"] < meta.max_loras or a["nb"] < meta.max_loras:
        raise ValueError("weights hold fewer LoRAs than the metadata expects")
    _same_device(meta, a["named"])
    _call("lora_linear", x.device, *a["head"], float(scale), a["buf"], *a["tail"],
          ctypes.byref(meta.c), _stream_handle(x.device))


def lora_linear_noalloc(token_lora_mapping: torch.Tensor, x: torch.Tensor, lora_a_stacked,
                        lora_b_stacked, lora_bias_stacked, scale: float, y: torch.Tensor,
                        meta: LoRAKernelMeta) -> None:
    """lora_linear without a caller buffer: the fp32 intermediate lives in a
    fixed array the library owns on each device (at most
    LORA_NOALLOC_MAX_FLOATS = slices x tokens x rank floats), cleared by each
    call, so no device memory is allocated.  Calls on one device share that
    array and must not overlap; see include/lora_punica.h."""
    a = _linear_args(token_lora_mapping, x, lora_a_stacked, lora_b_stacked, lora_bias_stacked,
                     None, y)
    if a["L"] < meta.max_loras or a["nb"] < meta.max_loras:
        raise ValueError("weights hold fewer LoRAs than the metadata expects")
    _same_device(meta, a["named"])
    _call("lora_linear_noalloc", x.device, *a["head"], float(scale), *a["tail"],
          ctypes.byref(meta.c), _stream_handle(x.device))
