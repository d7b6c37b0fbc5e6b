"""lora_linear_noalloc: the library's fixed device buffer in place of the
caller's fp32 buffer.  Checked against lora_linear with a zeroed buffer (the
buffer add_lora_linear creates) and against the oracle, on two calls in a
row, so the second call shows that the fixed buffer is cleared between
calls.  Collected last: its buffer stays resident once loaded."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import (EXPAND_ATOL, EXPAND_RTOL, assert_close, bits_to_f64, dev_bf16,
                         dev_i32, host_bits)

pytestmark = pytest.mark.gpu


def _assert_same_up_to_atomic_order(got_bits, want_bits, d_abs, flip_abs, what):
    """Both runs compute y = bf16(y_in + d) from the same y_in and a zeroed
    buffer; the shrink's split-K fp32 atomic adds may sum the buffer in
    another order.  That moves the buffer by at most (terms) x 2^-24 x
    sum|x||A| per entry (2^-16 covers up to 256 partial sums; d_abs carries
    it through B), and can flip the bf16 rounding of a buffer entry fed to
    the tensor cores, moving its term by at most 2^-8 |buf| |B| (flip_abs =
    sum |buf| |B|).  On top comes one bf16 rounding step of each result
    (2^-8 relative, twice)."""
    got, want = bits_to_f64(got_bits), bits_to_f64(want_bits)
    tol = (2.0 ** -7 * np.maximum(np.abs(got), np.abs(want)) + 2.0 ** -16 * d_abs
           + 2.0 ** -8 * flip_abs + 1e-30)
    bad = np.abs(got - want) > tol
    assert not bad.any(), "%s: %d of %d elements differ beyond the bound" % (
        what, int(bad.sum()), bad.size)


@pytest.mark.parametrize("name,T", [("tiny", None), ("decode", None), ("mlp", 300)])
def test_noalloc_matches_lora_linear_on_two_calls(oracle_mod, name, T):
    import expand_gemm_gb300 as eg
    inp = W.generate(name, num_tokens=T)
    w = inp.workload
    T = inp.ids.shape[0]
    ids = dev_i32(inp.ids)
    x = dev_bf16(inp.x)
    A = [dev_bf16(a) for a in inp.lora_a]
    B = [dev_bf16(b) for b in inp.lora_b]
    bias = None if inp.lora_bias is None else [dev_bf16(b) for b in inp.lora_bias]
    y_na = dev_bf16(inp.y)
    y_ll = dev_bf16(inp.y)
    meta_na = eg.LoRAKernelMeta.make(w.max_loras, T, "cuda")
    meta_ll = eg.LoRAKernelMeta.make(w.max_loras, T, "cuda")
    r = inp.lora_a[0].shape[1]
    zero = np.zeros((len(A), T, r), np.float32)
    # sum over h and k of |x[t,h]| |A[k,h]| |B[n,k]| per output element
    absb = lambda bits: bits & np.uint16(0x7FFF)
    b_abs = oracle_mod.shrink(absb(inp.x), [absb(a) for a in inp.lora_a], inp.ids,
                              abs(w.scale), zero)
    d_abs = oracle_mod.expand(b_abs.astype(np.float32), [absb(b) for b in inp.lora_b], inp.ids,
                              np.zeros_like(inp.y), w.slices, 0, False, None)
    # sum over k of |buf[t,k]| |B[n,k]| with the exact buffer
    b_ref = oracle_mod.shrink(inp.x, inp.lora_a, inp.ids, w.scale, zero)
    flip_abs = oracle_mod.expand(np.abs(b_ref).astype(np.float32), [absb(b) for b in inp.lora_b],
                                 inp.ids, np.zeros_like(inp.y), w.slices, 0, False, None)
    y_ref = inp.y
    for call in range(2):
        y_ll.copy_(y_na)     # both calls start from the same y
        eg.lora_linear_noalloc(ids, x, A, B, bias, w.scale, y_na, meta_na)
        buf = torch.zeros((len(A), T, r), dtype=torch.float32, device="cuda")
        eg.lora_linear(ids, x, A, B, bias, w.scale, buf, y_ll, meta_ll)
        torch.cuda.synchronize()
        got, want = host_bits(y_na), host_bits(y_ll)
        b = oracle_mod.shrink(inp.x, inp.lora_a, inp.ids, w.scale, zero)
        ref = oracle_mod.expand(b.astype(np.float32), inp.lora_b, inp.ids, y_ref, w.slices, 0,
                                True, inp.lora_bias)
        assert_close(bits_to_f64(got), ref, EXPAND_ATOL, EXPAND_RTOL, "noalloc y, call %d" % call)
        _assert_same_up_to_atomic_order(got, want, d_abs, flip_abs, "noalloc vs lora_linear, call %d" % call)
        y_ref = got          # the next call adds onto what this one wrote
        np.testing.assert_array_equal(meta_na.active_lora_ids.cpu().numpy(),
                                      meta_ll.active_lora_ids.cpu().numpy())


def test_noalloc_rejects_a_batch_above_its_buffer():
    import expand_gemm_gb300 as eg
    S, r, H = 2, 128, 64
    T = eg.LORA_NOALLOC_MAX_FLOATS // (S * r) + 1
    ids = torch.zeros(T, dtype=torch.int32, device="cuda")
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    A = [torch.zeros((1, r, H), dtype=torch.bfloat16, device="cuda") for _ in range(S)]
    B = [torch.zeros((1, 64, r), dtype=torch.bfloat16, device="cuda") for _ in range(S)]
    y = torch.zeros((T, 128), dtype=torch.bfloat16, device="cuda")
    meta = eg.LoRAKernelMeta.make(1, T, "cuda")
    with pytest.raises(eg.LoraError, match="-9|fixed buffer"):
        eg.lora_linear_noalloc(ids, x, A, B, None, 1.0, y, meta)
    torch.cuda.synchronize()
    assert float(y.abs().sum()) == 0.0
