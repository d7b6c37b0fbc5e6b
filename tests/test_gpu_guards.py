"""Stray-write checks (the tools that would find them on the GPU are not
available): every tensor a call writes sits inside guard bands of a known
bit pattern, which must be bit-identical afterwards, on every launch path
of lora_linear and on the separate calls; and the debug-checks build
(LORA_PUNICA_DEBUG_CHECKS) reports metadata that points outside the batch
in bit 29 of the error word instead of using it.

The corrupted-metadata cases run only on the debug build, in a child
process, and every corrupted index is chosen to land inside the guard
bands that the buffers really have (rows past T, a LoRA past L, buffer
floats past the end), so that even an access the checks missed would stay
inside allocated memory and show up as a changed guard byte."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import (EXPAND_ATOL, EXPAND_RTOL, SHRINK_ATOL, SHRINK_RTOL, assert_close,
                         bits_to_f64, dev_i32, host_bits)

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GUARD_ROWS = 64          # rows before and after x and y
GUARD_COLS = 16          # columns left and right of x and y (keeps 32-byte alignment)
GUARD_BITS = 0x7FA5      # a bf16 NaN pattern no kernel writes
GUARD_F32 = -7.0e30      # fp32 guard value
GUARD_LORAS = 1          # LoRAs past max_loras in A, B and bias


def _guarded_bf16(bits: np.ndarray):
    """(full, view): `bits` placed inside guard rows and columns."""
    rows, cols = bits.shape
    full = np.full((rows + 2 * GUARD_ROWS, cols + 2 * GUARD_COLS), GUARD_BITS, np.uint16)
    full[GUARD_ROWS:GUARD_ROWS + rows, GUARD_COLS:GUARD_COLS + cols] = bits
    t = torch.from_numpy(full.view(np.int16)).view(torch.bfloat16).cuda()
    return t, t[GUARD_ROWS:GUARD_ROWS + rows, GUARD_COLS:GUARD_COLS + cols]


def _guarded_buf(shape, rank):
    n = int(np.prod(shape))
    g = GUARD_ROWS * rank * 2
    full = torch.full((n + 2 * g,), GUARD_F32, dtype=torch.float32, device="cuda")
    view = full[g:g + n].view(*shape)
    view.zero_()
    return full, view, g


def _weights_with_spare(arrs):
    """bf16 weights with GUARD_LORAS extra LoRAs after max_loras; returns
    the [max_loras, ...] views the calls take."""
    out = []
    for a in arrs:
        spare = np.full((GUARD_LORAS,) + a.shape[1:], 0x3C00, np.uint16)   # bf16 1/128
        full = np.concatenate([a, spare])
        t = torch.from_numpy(full.view(np.int16)).view(torch.bfloat16).cuda()
        out.append(t[:a.shape[0]])
    return out


def _check_guards(x_full, y_full, buf_full, buf_guard, T, what):
    for name, full in (("x", x_full), ("y", y_full)):
        h = host_bits(full)
        r0, c0 = GUARD_ROWS, GUARD_COLS
        band = np.ones(h.shape, bool)
        band[r0:h.shape[0] - r0, c0:h.shape[1] - c0] = False
        assert (h[band] == GUARD_BITS).all(), "%s: guard band of %s changed" % (what, name)
    b = buf_full.cpu().numpy()
    assert (b[:buf_guard] == np.float32(GUARD_F32)).all(), "%s: guard before the buffer" % what
    assert (b[-buf_guard:] == np.float32(GUARD_F32)).all(), "%s: guard after the buffer" % what


PATHS = [pytest.param(dict(LORA_PUNICA_COOP=1, LORA_PUNICA_FUSED=0), id="coop"),
         pytest.param(dict(LORA_PUNICA_COOP=0, LORA_PUNICA_FUSED=1), id="fused"),
         pytest.param(dict(LORA_PUNICA_COOP=0, LORA_PUNICA_FUSED=0), id="early"),
         pytest.param(dict(LORA_PUNICA_COOP=0, LORA_PUNICA_FUSED=0, LORA_PUNICA_SELF_META=1),
                      id="two_kernels"),
         pytest.param(dict(LORA_PUNICA_COOP=0, LORA_PUNICA_FUSED=0, LORA_PUNICA_SELF_META=0),
                      id="three_kernels"),
         pytest.param(dict(LORA_PUNICA_COOP=0, LORA_PUNICA_FUSED=0, LORA_PUNICA_UMMA_MIN_TOKENS=0,
                           LORA_PUNICA_UMMA_MIN_COLS=0, LORA_PUNICA_EXPAND_TC=2),
                      id="tensor_core_kernels"),
         pytest.param(dict(LORA_PUNICA_COOP=0, LORA_PUNICA_FUSED=0, LORA_PUNICA_UMMA_MIN_TOKENS=0,
                           LORA_PUNICA_UMMA_MIN_COLS=0, LORA_PUNICA_UMMA_PAIR=1),
                      id="cta_pair_shrink")]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name,T", [("tiny", None), ("decode", None), ("mlp", 384),
                                    ("prefill", 1536)])
def test_guard_bands_on_every_path(oracle_mod, knob, path, name, T):
    """lora_linear with x, y and the buffer inside guard bands: results
    within tolerance, rows without a LoRA and every guard byte untouched."""
    import expand_gemm_gb300 as eg
    knob(**path)
    inp = W.generate(name, num_tokens=T)
    w = inp.workload
    T = w.num_tokens
    x_full, x = _guarded_bf16(inp.x)
    y_full, y = _guarded_bf16(inp.y)
    buf_full, buf, g = _guarded_buf(inp.buf.shape, w.rank)
    A = _weights_with_spare(inp.lora_a)
    B = _weights_with_spare(inp.lora_b)
    bias = None if inp.lora_bias is None else _weights_with_spare(inp.lora_bias)
    meta = eg.LoRAKernelMeta.make(w.max_loras, T, "cuda")
    eg.lora_linear(dev_i32(inp.ids), x, A, B, bias, w.scale, buf, y, meta)
    torch.cuda.synchronize()
    _check_guards(x_full, y_full, buf_full, g, T, "lora_linear")
    assert int(meta.error_word.item()) == 0
    ref_buf = oracle_mod.shrink(inp.x, inp.lora_a, inp.ids, w.scale, inp.buf)
    assert_close(buf.cpu().numpy(), ref_buf, SHRINK_ATOL, SHRINK_RTOL, "buffer")
    ref_y = oracle_mod.expand(ref_buf.astype(np.float32), inp.lora_b, inp.ids, inp.y, w.slices,
                              0, True, inp.lora_bias)
    got_y = host_bits(y)
    assert_close(bits_to_f64(got_y), ref_y, EXPAND_ATOL, EXPAND_RTOL, "y")
    none = inp.ids < 0
    np.testing.assert_array_equal(got_y[none], inp.y[none])


def test_guard_bands_one_kernel_tensor_core(oracle_mod, knob):
    """lora_linear's rank-128 tensor-core kernel with x, y and the buffer
    inside guard bands (the large workload's shapes and id mix at 1536
    tokens: partial and fragmented tiles, halves on idle SMs)."""
    import expand_gemm_gb300 as eg
    knob(LORA_PUNICA_LINEAR_TC=2)                   # required: no fallback
    inp = W.generate("large", num_tokens=1536)
    w = inp.workload
    T = w.num_tokens
    x_full, x = _guarded_bf16(inp.x)
    y_full, y = _guarded_bf16(inp.y)
    buf_full, buf, g = _guarded_buf(inp.buf.shape, w.rank)
    A = _weights_with_spare(inp.lora_a)
    B = _weights_with_spare(inp.lora_b)
    meta = eg.LoRAKernelMeta.make(w.max_loras, T, "cuda")
    eg.lora_linear(dev_i32(inp.ids), x, A, B, None, w.scale, buf, y, meta)
    torch.cuda.synchronize()
    _check_guards(x_full, y_full, buf_full, g, T, "lora_linear (one tensor-core kernel)")
    assert int(meta.error_word.item()) == 0
    ref_buf = oracle_mod.shrink(inp.x, inp.lora_a, inp.ids, w.scale, inp.buf)
    assert_close(buf.cpu().numpy(), ref_buf, SHRINK_ATOL, SHRINK_RTOL, "buffer")
    ref_y = oracle_mod.expand(ref_buf.astype(np.float32), inp.lora_b, inp.ids, inp.y, w.slices,
                              0, True, None)
    got_y = host_bits(y)
    assert_close(bits_to_f64(got_y), ref_y, EXPAND_ATOL, EXPAND_RTOL, "y")
    none = inp.ids < 0
    np.testing.assert_array_equal(got_y[none], inp.y[none])


@pytest.mark.parametrize("tc", ["0", "2"])
def test_guard_bands_separate_calls_with_offset(oracle_mod, knob, tc):
    """lora_shrink and lora_expand (offset_start, add_inputs=False) with
    guard bands; the columns outside the slices stay untouched too."""
    import expand_gemm_gb300 as eg
    knob(LORA_PUNICA_EXPAND_TC=tc, LORA_PUNICA_UMMA_MIN_TOKENS=0, LORA_PUNICA_UMMA_MIN_COLS=0)
    w = W.Workload("guards", 41, 1300, 256, 64, 5, (192, 64), "zipf_seq", p_none=0.2,
                   seq_len=(100, 400), bias=True, offset_start=16)
    inp = W.generate(w)
    T = w.num_tokens
    x_full, x = _guarded_bf16(inp.x)
    y_full, y = _guarded_bf16(inp.y)
    buf_full, buf, g = _guarded_buf(inp.buf.shape, w.rank)
    A = _weights_with_spare(inp.lora_a)
    B = _weights_with_spare(inp.lora_b)
    bias = _weights_with_spare(inp.lora_bias)
    meta = eg.LoRAKernelMeta.make(w.max_loras, T, "cuda")
    meta.prepare_tensors(dev_i32(inp.ids))
    eg.lora_shrink(x, A, buf, meta, w.scale)
    eg.lora_expand(buf, B, y, meta, w.offset_start, False, bias)
    torch.cuda.synchronize()
    _check_guards(x_full, y_full, buf_full, g, T, "separate calls")
    assert int(meta.error_word.item()) == 0
    ref_buf = oracle_mod.shrink(inp.x, inp.lora_a, inp.ids, w.scale, inp.buf)
    ref_y = oracle_mod.expand(ref_buf.astype(np.float32), inp.lora_b, inp.ids, inp.y, w.slices,
                              w.offset_start, False, inp.lora_bias)
    got = host_bits(y)
    assert_close(bits_to_f64(got), ref_y, EXPAND_ATOL, EXPAND_RTOL, "y")
    np.testing.assert_array_equal(got[:, :w.offset_start], inp.y[:, :w.offset_start])


# The child process: runs on the debug-checks build (LORA_PUNICA_LIBRARY).
_CHILD = r'''
import json, os, sys
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, os.path.join(sys.argv[1], "tests"))
import numpy as np, torch
import test_gpu_guards as G
import workloads as W
import expand_gemm_gb300 as eg
from gpu_helpers import dev_i32
out = {"library": os.path.basename(eg.library()._name)}
w = W.Workload("dbg", 43, 700, 256, 32, 6, (128, 64), "zipf_seq", p_none=0.2,
               seq_len=(60, 200), bias=True)
inp = W.generate(w)
T = w.num_tokens

def run(corrupt, umma):
    os.environ["LORA_PUNICA_UMMA_MIN_TOKENS"] = "0" if umma else "1024"
    os.environ["LORA_PUNICA_UMMA_MIN_COLS"] = "0" if umma else "256"
    os.environ["LORA_PUNICA_EXPAND_TC"] = "2" if umma else "0"
    eg.reload_options()
    x_full, x = G._guarded_bf16(inp.x)
    y_full, y = G._guarded_bf16(inp.y)
    buf_full, buf, g = G._guarded_buf(inp.buf.shape, w.rank)
    A = G._weights_with_spare(inp.lora_a)
    B = G._weights_with_spare(inp.lora_b)
    bias = G._weights_with_spare(inp.lora_bias)
    # room for sorted-list entries past T
    meta = eg.LoRAKernelMeta.make(w.max_loras, T + G.GUARD_ROWS, "cuda")
    meta.prepare_tensors(dev_i32(inp.ids))
    # entries past the batch (reached only by the corrupted segment) point
    # into the guard rows
    meta.token_indices_sorted_by_lora_ids[T:] = T + 5
    torch.cuda.synchronize()
    if corrupt == "token":      # one sorted entry points 3 rows past the batch
        k = int(meta.lora_token_start_loc[1].item())
        meta.token_indices_sorted_by_lora_ids[k + 1] = T + 3
    elif corrupt == "lora":     # an active id equal to max_loras
        meta.active_lora_ids[1] = w.max_loras
    elif corrupt == "segment":  # the last segment runs 8 rows past T
        n = int((meta.num_tokens_per_lora > 0).sum().item())
        meta.num_tokens_per_lora[n - 1] += 8
        meta.lora_token_start_loc[n] += 8
    torch.cuda.synchronize()
    meta.error_word.zero_()
    eg.lora_shrink(x, A, buf, meta, w.scale)
    eg.lora_expand(buf, B, y, meta, 0, True, bias)
    torch.cuda.synchronize()
    guards = True
    try:
        G._check_guards(x_full, y_full, buf_full, g, T, corrupt)
    except AssertionError:
        guards = False
    return {"error_word": int(meta.error_word.item()), "guards_intact": guards}

for umma in (False, True):
    for corrupt in ("none", "token", "lora", "segment"):
        out["%s/%s" % ("tcgen05" if umma else "mma_sync", corrupt)] = run(corrupt, umma)
print(json.dumps(out))
'''


def test_debug_build_reports_metadata_outside_the_batch():
    """On the debug-checks build: a valid batch leaves bit 29 clear; a
    sorted entry past T, an active id equal to max_loras, or a segment
    running past T each set bit 29, and no guard byte changes (the checked
    accesses are skipped), on the mma.sync and the tcgen05 kernels."""
    from expand_gemm_gb300.build import build
    lib = build(debug=True)
    env = dict(os.environ, LORA_PUNICA_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["library"] == "liblora_punica_debug.so"
    for key, v in res.items():
        if key == "library":
            continue
        assert v["guards_intact"], key
        if key.endswith("/none"):
            assert v["error_word"] & (1 << 29) == 0, key
        else:
            assert v["error_word"] & (1 << 29), key
