"""GPU parity of lora_linear (metadata + shrink + expand in one call) against
the oracle composition, on each of its launch paths."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import (EXPAND_ATOL, EXPAND_RTOL, SHRINK_ATOL, SHRINK_RTOL, assert_close,
                         bits_to_f64, dev_bf16, dev_f32, dev_i32, host_bits)

pytestmark = pytest.mark.gpu

# (LORA_PUNICA_COOP, LORA_PUNICA_FUSED, LORA_PUNICA_SELF_META): one
# cooperative kernel (metadata, shrink, grid barrier, expand); one cluster
# kernel; the metadata kernel, then shrink and expand each loading before
# their grid-dependency wait; the shrink sorting the ids itself and writing
# the metadata, then the expand; the plain metadata kernel + shrink +
# expand.  Batches a path does not take fall through to the next.
PATHS = [pytest.param(("1", "0", None), id="coop"),
         pytest.param(("0", "1", None), id="fused"),
         pytest.param(("0", "0", None), id="early"),
         pytest.param(("0", "0", "1"), id="two_kernels"),
         pytest.param(("0", "0", "0"), id="three_kernels")]


def _set_path(knob, path):
    knob(LORA_PUNICA_COOP=path[0], LORA_PUNICA_FUSED=path[1], LORA_PUNICA_SELF_META=path[2])


def _check_linear(oracle_mod, inp, ids=None, buf0=None, L=None):
    import expand_gemm_gb300 as eg
    w = inp.workload
    ids = inp.ids if ids is None else ids
    L = w.max_loras if L is None else L
    T = ids.shape[0]
    b0 = inp.buf if buf0 is None else buf0
    x = dev_bf16(inp.x)
    A = [dev_bf16(a) for a in inp.lora_a]
    B = [dev_bf16(b) for b in inp.lora_b]
    bias = None if inp.lora_bias is None else [dev_bf16(b) for b in inp.lora_bias]
    y = dev_bf16(inp.y)
    buf = dev_f32(b0)
    meta = eg.LoRAKernelMeta.make(L, T, "cuda")
    eg.lora_linear(dev_i32(ids), x, A, B, bias, w.scale, buf, y, meta)
    torch.cuda.synchronize()

    o = oracle_mod.meta_prepare(ids, L)
    assert int(meta.no_lora_flag.item()) == int(o.no_lora_flag[0])
    np.testing.assert_array_equal(meta.active_lora_ids.cpu().numpy(), o.active_lora_ids)
    np.testing.assert_array_equal(meta.num_tokens_per_lora.cpu().numpy(), o.num_tokens_per_lora)
    np.testing.assert_array_equal(meta.lora_token_start_loc.cpu().numpy(), o.lora_token_start_loc)
    assert int(meta.error_word.item()) & ~(1 << 30) == o.invalid_ids
    assert int(meta.error_word.item()) & (1 << 30) == 0
    assert meta.grid_sync.cpu().tolist() == [0, 0]      # barrier words left clean
    if not o.no_lora_flag[0]:
        np.testing.assert_array_equal(meta.token_indices_sorted_by_lora_ids[:T].cpu().numpy(),
                                      o.token_indices_sorted_by_lora_ids[:T])
        np.testing.assert_array_equal(meta.token_lora_mapping[:T].cpu().numpy(), ids)

    ref_buf = oracle_mod.shrink(inp.x, inp.lora_a, ids, w.scale, b0)
    got_buf = buf.cpu().numpy()
    assert_close(got_buf, ref_buf, SHRINK_ATOL, SHRINK_RTOL, "lora_linear buffer")
    ref_y = oracle_mod.expand(ref_buf.astype(np.float32), inp.lora_b, ids, inp.y, w.slices,
                              0, True, inp.lora_bias)
    got_y = host_bits(y)
    assert_close(bits_to_f64(got_y), ref_y, EXPAND_ATOL, EXPAND_RTOL, "lora_linear y")
    none = (ids < 0) | (ids >= L)
    np.testing.assert_array_equal(got_y[none], inp.y[none])
    np.testing.assert_array_equal(got_buf[:, none], b0[:, none])


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name,T", [("tiny", None), ("decode", None), ("mlp", 200)])
def test_linear_workloads(oracle_mod, knob, path, name, T):
    _set_path(knob, path)
    _check_linear(oracle_mod, W.generate(name, num_tokens=T))


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T,H,r,L,slices,bias,ids", [
    (1, 64, 16, 1, (128,), False, "uniform"),              # single token
    (37, 320, 8, 3, (64, 200, 8), True, "uniform"),        # rank 8, ragged hidden blocks
    (130, 512, 24, 5, (256, 136), True, "uniform"),        # padded rank, two tiles per LoRA
    (300, 1024, 32, 4, (128, 128, 128, 128), False, "zipf_seq"),   # four slices, S*rp = 128
    (512, 2048, 64, 2, (512, 256), True, "zipf_seq"),      # the largest fused batch
    (513, 256, 16, 3, (128,), False, "uniform"),           # one past it: three kernels
    (200, 256, 16, 300, (64,), False, "uniform"),          # many LoRAs: three kernels
])
def test_linear_shapes(oracle_mod, knob, path, T, H, r, L, slices, bias, ids):
    _set_path(knob, path)
    w = W.Workload("lin", T + H + r, T, H, r, L, slices, ids, p_none=0.2, seq_len=(20, 90),
                   bias=bias, scale=0.8)
    inp = W.generate(w)
    b0 = np.random.default_rng(T).standard_normal(inp.buf.shape).astype(np.float32)
    _check_linear(oracle_mod, inp, buf0=b0)


@pytest.mark.parametrize("T,H,slices,L,bias,ids", [
    (300, 512, (128,), 4, False, "zipf_seq"),          # one slice
    (700, 200, (256, 64), 6, True, "uniform_p"),       # ragged hidden, per-token ids, bias
    (1100, 1024, (1024, 128, 192), 3, False, "zipf_seq"),   # three slices, a 64-column chunk
    (129, 128, (64, 64, 64), 2, True, "uniform"),      # a one-row tile, 64-column slices
    (2000, 2048, (512, 128, 128), 64, True, "mixed"),  # the large workload's id mix
])
def test_linear_one_kernel_tensor_core(oracle_mod, knob, T, H, slices, L, bias, ids):
    """lora_linear's one-kernel tensor-core path (rank 128, up to three
    slices: every tile's shrink, buffer update and expand on one SM) gives
    the oracle's metadata, buffer and y, with a non-zero starting buffer."""
    knob(LORA_PUNICA_LINEAR_TC="2")                 # required: no fallback
    w = W.Workload("lintc", T + H, T, H, 128, L, slices, ids, p_none=0.15, seq_len=(40, 400),
                   bias=bias, scale=0.7)
    inp = W.generate(w)
    b0 = np.random.default_rng(T + 1).standard_normal(inp.buf.shape).astype(np.float32)
    _check_linear(oracle_mod, inp, buf0=b0)


@pytest.mark.parametrize("T,H,slices,L,bias,ids", [
    (24000, 128, (64, 128, 192), 40, False, "uniform"),   # ~200 tiles of 128 runs each
    (30000, 256, (128,), 8, True, "zipf_seq"),             # ~235 tiles, bias
])
def test_linear_one_kernel_several_tiles_per_cta(oracle_mod, knob, T, H, slices, L, bias, ids):
    """More tiles than SMs: CTAs take a second tile, whose barrier phases,
    ring slots and TMEM buffers follow on from the first's."""
    knob(LORA_PUNICA_LINEAR_TC="2")                 # required: no fallback
    w = W.Workload("lintc_multi", T + H, T, H, 128, L, slices, ids, p_none=0.1,
                   seq_len=(100, 900), bias=bias, scale=0.25)
    inp = W.generate(w)
    b0 = np.random.default_rng(T).standard_normal(inp.buf.shape).astype(np.float32)
    _check_linear(oracle_mod, inp, buf0=b0)


@pytest.mark.parametrize("T,slices,min_tokens", [
    (1500, (200, 64), 1000),       # a slice width that is not a multiple of 64: separate kernels
    (600, (128, 128), None),       # below the default threshold (72 tokens per SM): separate
    (1024, (256, 64, 128), 1024),  # at a set threshold: the one kernel
    (12000, (128, 64), None),      # above the default threshold: the one kernel
])
def test_linear_rank128_default_rule(oracle_mod, knob, T, slices, min_tokens):
    """With the default rule (LORA_PUNICA_LINEAR_TC unset) rank-128 calls
    take the one kernel or the separate ones; both give the oracle's
    results."""
    knob(LORA_PUNICA_LINEAR_TC=None, LORA_PUNICA_LINEAR_TC_MIN_TOKENS=min_tokens)
    w = W.Workload("lintc_default", T, T, 512, 128, 5, slices, "zipf_seq", p_none=0.1,
                   seq_len=(40, 300), bias=True, scale=0.5)
    _check_linear(oracle_mod, W.generate(w))


def test_linear_one_kernel_required_refuses_what_it_does_not_take(knob):
    """LORA_PUNICA_LINEAR_TC=2 makes a call the kernel does not take fail
    (rank 64; a slice width that is not a multiple of 64) instead of
    running the separate kernels; y is left untouched."""
    import expand_gemm_gb300 as eg
    from expand_gemm_gb300._lib import LoraError
    knob(LORA_PUNICA_LINEAR_TC="2")
    for r, slices in ((64, (128,)), (128, (96,))):
        w = W.Workload("lintc_refuse", 5, 300, 256, r, 2, slices, "zipf_seq", p_none=0.1,
                       seq_len=(40, 200))
        inp = W.generate(w)
        y = dev_bf16(inp.y)
        meta = eg.LoRAKernelMeta.make(w.max_loras, w.num_tokens, "cuda")
        with pytest.raises(LoraError):
            eg.lora_linear(dev_i32(inp.ids), dev_bf16(inp.x), [dev_bf16(a) for a in inp.lora_a],
                           [dev_bf16(b) for b in inp.lora_b], None, w.scale,
                           dev_f32(inp.buf), y, meta)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host_bits(y), inp.y)


def test_linear_one_kernel_tensor_core_no_lora(oracle_mod, knob):
    """The one-kernel path on the all -1 batch and on invalid ids."""
    knob(LORA_PUNICA_LINEAR_TC="2")                 # required: no fallback
    inp = W.generate("large", num_tokens=640)
    _check_linear(oracle_mod, inp, ids=np.full(640, -1, np.int32))
    ids = inp.ids.copy()
    ids[::7] = 64
    ids[::11] = -5
    _check_linear(oracle_mod, inp, ids=ids)


@pytest.mark.parametrize("path", PATHS)
def test_linear_no_lora_and_invalid_ids(oracle_mod, knob, path):
    _set_path(knob, path)
    inp = W.generate("decode")
    _check_linear(oracle_mod, inp, ids=np.full(256, -1, np.int32))
    ids = inp.ids.copy()
    ids[::9] = 8
    ids[::13] = -3
    _check_linear(oracle_mod, inp, ids=ids)


def test_linear_repeated_calls_accumulate(oracle_mod):
    """Two calls in a row on the same buffers (the buffer accumulates)."""
    import expand_gemm_gb300 as eg
    inp = W.generate("tiny")
    w = inp.workload
    x, y = dev_bf16(inp.x), dev_bf16(inp.y)
    A = [dev_bf16(a) for a in inp.lora_a]
    B = [dev_bf16(b) for b in inp.lora_b]
    bias = [dev_bf16(b) for b in inp.lora_bias]
    buf = dev_f32(inp.buf)
    meta = eg.LoRAKernelMeta.make(w.max_loras, w.num_tokens, "cuda")
    ids = dev_i32(inp.ids)
    for _ in range(2):
        eg.lora_linear(ids, x, A, B, bias, w.scale, buf, y, meta)
    torch.cuda.synchronize()
    b1 = oracle_mod.shrink(inp.x, inp.lora_a, inp.ids, w.scale, inp.buf)
    y1 = oracle_mod.expand(b1.astype(np.float32), inp.lora_b, inp.ids, inp.y, w.slices, 0, True,
                           inp.lora_bias)
    y1_bits = W.bf16_bits(y1.astype(np.float32))
    b2 = oracle_mod.shrink(inp.x, inp.lora_a, inp.ids, w.scale, b1.astype(np.float32))
    y2 = oracle_mod.expand(b2.astype(np.float32), inp.lora_b, inp.ids, y1_bits, w.slices, 0,
                           True, inp.lora_bias)
    assert_close(buf.cpu().numpy(), b2, SHRINK_ATOL, SHRINK_RTOL, "buffer after two calls")
    assert_close(bits_to_f64(host_bits(y)), y2, 2 * EXPAND_ATOL, 2 * EXPAND_RTOL, "y after two calls")


def test_coop_barrier_timeout_reports_and_recovers(oracle_mod, knob):
    """The cooperative kernel's grid barrier is made to wait for one arrival
    that never comes (a test knob raises the expected count), with a short
    poll limit: every CTA gives up, bit 30 of the error word is set, the
    expand is skipped (y untouched), the shrink result is complete and the
    barrier words are back to zero.  The next call on the same metadata
    succeeds."""
    import expand_gemm_gb300 as eg
    inp = W.generate("decode")
    w = inp.workload
    T = w.num_tokens
    x = dev_bf16(inp.x)
    A = [dev_bf16(a) for a in inp.lora_a]
    B = [dev_bf16(b) for b in inp.lora_b]
    ids = dev_i32(inp.ids)
    meta = eg.LoRAKernelMeta.make(w.max_loras, T, "cuda")
    knob(LORA_PUNICA_COOP=1, LORA_PUNICA_COOP_TEST_EXTRA_ARRIVALS=1,
         LORA_PUNICA_COOP_TEST_TIMEOUT_CYCLES=20000000)   # ~10 ms
    y = dev_bf16(inp.y)
    buf = dev_f32(inp.buf)
    eg.lora_linear(ids, x, A, B, None, w.scale, buf, y, meta)
    torch.cuda.synchronize()
    assert int(meta.error_word.item()) & (1 << 30)
    assert meta.grid_sync.cpu().tolist() == [0, 0]
    np.testing.assert_array_equal(host_bits(y), inp.y)
    ref_buf = oracle_mod.shrink(inp.x, inp.lora_a, inp.ids, w.scale, inp.buf)
    assert_close(buf.cpu().numpy(), ref_buf, SHRINK_ATOL, SHRINK_RTOL, "buffer after timeout")

    knob(LORA_PUNICA_COOP_TEST_EXTRA_ARRIVALS=None, LORA_PUNICA_COOP_TEST_TIMEOUT_CYCLES=None)
    y = dev_bf16(inp.y)
    buf = dev_f32(inp.buf)
    eg.lora_linear(ids, x, A, B, None, w.scale, buf, y, meta)
    torch.cuda.synchronize()
    assert int(meta.error_word.item()) & (1 << 30) == 0
    assert meta.grid_sync.cpu().tolist() == [0, 0]
    assert_close(buf.cpu().numpy(), ref_buf, SHRINK_ATOL, SHRINK_RTOL, "buffer after recovery")
    ref_y = oracle_mod.expand(ref_buf.astype(np.float32), inp.lora_b, inp.ids, inp.y, w.slices,
                              0, True)
    assert_close(bits_to_f64(host_bits(y)), ref_y, EXPAND_ATOL, EXPAND_RTOL, "y after recovery")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name,T", [("decode", None), ("mlp", 512), ("prefill", 2048)])
def test_linear_alternating_no_lora_batches(oracle_mod, knob, path, name, T):
    """Calls with a mixed id map (with bias) and all -1 calls alternate on one
    metadata struct, back to back in one stream.  After every all -1 call, y
    and the buffer are bit-identical to what they were before it: no kernel
    of that call may act on the metadata of the mixed call before it (early
    mode fetches the metadata before its grid-dependency wait, so every
    kernel of the chain must pass its wait before it exits).  Every mixed
    call is checked against the oracle."""
    import expand_gemm_gb300 as eg
    _set_path(knob, path)
    w0 = W.generate(name, num_tokens=T).workload
    from dataclasses import replace
    w = replace(w0, bias=True, scale=0.9)
    inp = W.generate(w)
    T = w.num_tokens
    x = dev_bf16(inp.x)
    A = [dev_bf16(a) for a in inp.lora_a]
    B = [dev_bf16(b) for b in inp.lora_b]
    bias = [dev_bf16(b) for b in inp.lora_bias]
    ids_mixed = dev_i32(inp.ids)
    ids_none = dev_i32(np.full(T, -1, np.int32))
    meta = eg.LoRAKernelMeta.make(w.max_loras, T, "cuda")
    y = dev_bf16(inp.y)
    buf = torch.zeros(inp.buf.shape, dtype=torch.float32, device="cuda")
    ref_buf = oracle_mod.shrink(inp.x, inp.lora_a, inp.ids, w.scale, inp.buf)
    for it in range(3):
        y_before = host_bits(y)
        buf.zero_()
        eg.lora_linear(ids_mixed, x, A, B, bias, w.scale, buf, y, meta)
        eg.lora_linear(ids_none, x, A, B, bias, w.scale, buf, y, meta)
        y_after_none = host_bits(y)
        buf_after_none = buf.cpu().numpy()
        assert int(meta.no_lora_flag.item()) == 1
        assert int(meta.error_word.item()) == 0
        ref_y = oracle_mod.expand(ref_buf.astype(np.float32), inp.lora_b, inp.ids, y_before,
                                  w.slices, 0, True, inp.lora_bias)
        assert_close(buf_after_none, ref_buf, SHRINK_ATOL, SHRINK_RTOL, "buffer, round %d" % it)
        assert_close(bits_to_f64(y_after_none), ref_y, EXPAND_ATOL, EXPAND_RTOL,
                     "y, round %d" % it)
        # the all -1 call itself changed nothing: run it twice more and compare bits
        eg.lora_linear(ids_none, x, A, B, bias, w.scale, buf, y, meta)
        eg.lora_linear(ids_none, x, A, B, bias, w.scale, buf, y, meta)
        np.testing.assert_array_equal(host_bits(y), y_after_none)
        np.testing.assert_array_equal(buf.cpu().numpy(), buf_after_none)
