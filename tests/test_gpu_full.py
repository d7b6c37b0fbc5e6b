"""Full-size parity: every workload at its stated size, every token.

Three routes are checked against the oracle: ``lora_linear`` (the metadata
kernel, the shrink and the expand of one layer in one call: the step the
benchmark times, in the same launch configuration; on rank 128 one
tensor-core kernel after the metadata kernel), the same call with the shrink
and expand kernels apart (LORA_PUNICA_LINEAR_TC=0), and the separate
``lora_meta_prepare`` / ``lora_shrink`` / ``lora_expand`` calls.  For each:

* the metadata, bit-exact, in full;
* every entry of the fp32 shrink buffer of tokens with a LoRA, within the
  shrink tolerance;
* every element of every y row of tokens with a LoRA, within the expand
  tolerance;
* rows of tokens without a LoRA, bit-identical to the input (y) or still
  zero (buffer);
* no bounded pipeline wait gave up (bit 30 of the error word).

The oracle computes the large workload (16384 tokens, hidden 8192, rank 128,
three slices) in seconds on the host cores, so nothing is sampled.  Inputs
and oracle results are computed once per workload and shared by the routes.
"""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import (EXPAND_ATOL, EXPAND_RTOL, SHRINK_ATOL, SHRINK_RTOL, assert_close,
                         bits_to_f64, dev_bf16, dev_i32, host_bits)

pytestmark = pytest.mark.gpu

NAMES = ["tiny", "decode", "prefill", "mlp", "large", "none"]
_cache = {}


def _reference(oracle_mod, name):
    """Inputs and the oracle's results for workload `name` (computed once)."""
    if name not in _cache:
        _cache.clear()                       # one workload's arrays at a time
        inp = W.generate(name)
        w = inp.workload
        o = oracle_mod.meta_prepare(inp.ids, w.max_loras)
        ref_buf = oracle_mod.shrink(inp.x, inp.lora_a, inp.ids, w.scale, inp.buf)
        ref_y = oracle_mod.expand(ref_buf.astype(np.float32), inp.lora_b, inp.ids, inp.y,
                                  w.slices, w.offset_start, w.add_inputs, inp.lora_bias)
        _cache[name] = (inp, o, ref_buf, ref_y)
    return _cache[name]


def _device_inputs(inp):
    x = dev_bf16(inp.x)
    A = [dev_bf16(a) for a in inp.lora_a]
    B = [dev_bf16(b) for b in inp.lora_b]
    bias = None if inp.lora_bias is None else [dev_bf16(b) for b in inp.lora_bias]
    return x, A, B, bias


def _check(name, inp, o, ref_buf, ref_y, meta, buf, y):
    w = inp.workload
    T = w.num_tokens
    assert int(meta.no_lora_flag.item()) == int(o.no_lora_flag[0])
    np.testing.assert_array_equal(meta.active_lora_ids.cpu().numpy(), o.active_lora_ids)
    np.testing.assert_array_equal(meta.num_tokens_per_lora.cpu().numpy(), o.num_tokens_per_lora)
    np.testing.assert_array_equal(meta.lora_token_start_loc.cpu().numpy(), o.lora_token_start_loc)
    if not o.no_lora_flag[0]:
        np.testing.assert_array_equal(meta.token_indices_sorted_by_lora_ids[:T].cpu().numpy(),
                                      o.token_indices_sorted_by_lora_ids[:T])
        np.testing.assert_array_equal(meta.token_lora_mapping[:T].cpu().numpy(), inp.ids)
    err = int(meta.error_word.item())
    assert err & (1 << 30) == 0, "a bounded pipeline wait gave up"
    assert err & ~(1 << 30) == o.invalid_ids

    buf_h = buf.cpu().numpy()
    y_h = host_bits(y)
    act = inp.ids >= 0
    none = ~act
    # rows of tokens without a LoRA: untouched
    np.testing.assert_array_equal(y_h[none], inp.y[none])
    assert (buf_h[:, none] == 0).all()
    if not act.any():
        return
    assert_close(buf_h[:, act], ref_buf[:, act], SHRINK_ATOL, SHRINK_RTOL, "shrink[%s]" % name)
    assert_close(bits_to_f64(y_h[act]), ref_y[act], EXPAND_ATOL, EXPAND_RTOL,
                 "expand[%s]" % name)


def _run_lora_linear(eg, inp, x, A, B, bias, y, buf, meta):
    w = inp.workload
    eg.lora_linear(dev_i32(inp.ids), x, A, B, bias, w.scale, buf, y, meta)


def _run_lora_linear_three_kernels(eg, inp, x, A, B, bias, y, buf, meta):
    """lora_linear with its one-kernel tensor-core path turned off
    (LORA_PUNICA_LINEAR_TC=0): the rank-128 workloads, which take that path
    by default, run the metadata, shrink and expand kernels instead."""
    import os
    w = inp.workload
    old = os.environ.get("LORA_PUNICA_LINEAR_TC")
    os.environ["LORA_PUNICA_LINEAR_TC"] = "0"
    eg.reload_options()
    try:
        eg.lora_linear(dev_i32(inp.ids), x, A, B, bias, w.scale, buf, y, meta)
        torch.cuda.synchronize()
    finally:
        if old is None:
            del os.environ["LORA_PUNICA_LINEAR_TC"]
        else:
            os.environ["LORA_PUNICA_LINEAR_TC"] = old
        eg.reload_options()


def _run_separate(eg, inp, x, A, B, bias, y, buf, meta):
    w = inp.workload
    meta.prepare_tensors(dev_i32(inp.ids))
    eg.lora_shrink(x, A, buf, meta, w.scale)
    eg.lora_expand(buf, B, y, meta, w.offset_start, w.add_inputs, bias)


# lora_linear is the benchmark's step (on rank 128 the one tensor-core
# kernel after the metadata kernel); the same call with the separate kernels;
# the separate calls are the three entry points one by one.
ROUTES = [pytest.param(_run_lora_linear, id="lora_linear"),
          pytest.param(_run_lora_linear_three_kernels, id="lora_linear_three_kernels"),
          pytest.param(_run_separate, id="separate_calls")]


@pytest.mark.parametrize("route", ROUTES)
@pytest.mark.parametrize("name", NAMES)
def test_full_size_every_token(oracle_mod, name, route):
    import expand_gemm_gb300 as eg
    inp, o, ref_buf, ref_y = _reference(oracle_mod, name)
    w = inp.workload
    x, A, B, bias = _device_inputs(inp)
    y = dev_bf16(inp.y)
    buf = torch.zeros(inp.buf.shape, dtype=torch.float32, device="cuda")
    meta = eg.LoRAKernelMeta.make(w.max_loras, w.num_tokens, "cuda")
    route(eg, inp, x, A, B, bias, y, buf, meta)
    torch.cuda.synchronize()
    _check(name, inp, o, ref_buf, ref_y, meta, buf, y)
