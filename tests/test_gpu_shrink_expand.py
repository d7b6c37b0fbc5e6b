"""GPU parity of lora_shrink / lora_expand against the fp64 oracle.

Sizes are ones the oracle finishes in seconds but that still span several
token tiles, hidden chunks and column chunks, with ragged tails; the edge
cases cover empty and all-no-LoRA batches, a single token, padded ranks,
ragged hidden sizes, strided x, eight slices, unaligned outputs (scalar
epilogue), overwrite mode and offsets.
"""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import (EXPAND_ATOL, EXPAND_RTOL, SHRINK_ATOL, SHRINK_RTOL, assert_close,
                         bits_to_f64, dev_bf16, dev_f32, dev_i32, host_bits)

pytestmark = pytest.mark.gpu


def _eg():
    import expand_gemm_gb300 as eg
    return eg


def _meta(ids, L):
    eg = _eg()
    meta = eg.LoRAKernelMeta.make(L, max(ids.shape[0], 1), "cuda")
    meta.prepare_tensors(dev_i32(ids))
    return meta


def _run_shrink(inp, ids, scale, buf0=None, x_pad=0):
    eg = _eg()
    T, H = inp.x.shape
    if x_pad:
        xw = torch.zeros((T, H + x_pad), dtype=torch.bfloat16, device="cuda")
        xw[:, :H] = dev_bf16(inp.x)
        x = xw[:, :H]
    else:
        x = dev_bf16(inp.x)
    A = [dev_bf16(a) for a in inp.lora_a]
    buf = dev_f32(inp.buf if buf0 is None else buf0)
    meta = _meta(ids, inp.lora_a[0].shape[0])
    eg.lora_shrink(x, A, buf, meta, scale)
    torch.cuda.synchronize()
    assert int(meta.error_word.item()) & (1 << 30) == 0, "a pipeline wait timed out"
    return buf.cpu().numpy()


def _shrink_case(oracle_mod, inp, ids=None, scale=None, buf0=None, x_pad=0):
    ids = inp.ids if ids is None else ids
    scale = inp.workload.scale if scale is None else scale
    b0 = inp.buf if buf0 is None else buf0
    got = _run_shrink(inp, ids, scale, b0, x_pad)
    ref = oracle_mod.shrink(inp.x, inp.lora_a, ids, scale, b0)
    assert_close(got, ref, SHRINK_ATOL, SHRINK_RTOL, "shrink")
    none = (ids < 0) | (ids >= inp.lora_a[0].shape[0])
    np.testing.assert_array_equal(got[:, none], b0[:, none])     # bit-untouched
    return got


def _custom(T, H, r, L, slices, seed, ids="uniform", p_none=0.0, bias=False, scale=1.0):
    w = W.Workload("custom", seed, T, H, r, L, tuple(slices), ids, p_none=p_none,
                   seq_len=(3, 40), bias=bias, scale=scale)
    return W.generate(w)


# ------------------------------------------------------------------ shrink

@pytest.mark.parametrize("name,T", [("tiny", None), ("decode", None), ("prefill", 1536),
                                    ("mlp", 512), ("large", 384)])
def test_shrink_workloads_reduced(oracle_mod, name, T):
    inp = W.generate(name, num_tokens=T)
    _shrink_case(oracle_mod, inp)


@pytest.mark.parametrize("T,H,r,L,S", [
    (1, 64, 16, 1, 1),          # single token
    (7, 200, 8, 3, 2),          # ragged hidden (not a multiple of 64), rank 8
    (130, 512, 24, 5, 3),       # padded rank 24 -> 32, ragged token tile
    (257, 1024, 128, 4, 1),     # rank 128
    (96, 136, 40, 6, 8),        # eight slices, rank 40 -> 64
    (3000, 256, 16, 2, 1),      # many tiles, no split
])
def test_shrink_shapes(oracle_mod, T, H, r, L, S):
    inp = _custom(T, H, r, L, [16] * S, seed=T + H + r)
    _shrink_case(oracle_mod, inp, scale=0.37)


@pytest.mark.parametrize("T,H,r,L,S", [
    (1024, 256, 16, 2, 1),      # exactly whole 128-token tiles
    (1300, 320, 32, 3, 2),      # ragged hidden (5 blocks of 64), remainders
    (2100, 512, 64, 4, 1),
    (1500, 192, 128, 3, 3),     # rank 128, three slices: 384 TMEM columns
    (1100, 128, 24, 2, 2),      # padded rank 24 -> 32
])
@pytest.mark.parametrize("umma,partial,pair", [("0", "1", "0"), ("1", "1", "0"), ("1", "0", "0"),
                                               ("1", "1", "1")])
def test_shrink_long_segments(oracle_mod, knob, umma, partial, pair, T, H, r, L, S):
    """Long sequences per LoRA: with the tensor-core path forced on it takes
    every tile, the partial last tile of each segment included (partial=1),
    or the whole 128-token tiles with the remainders on mma.sync
    (partial=0); with it off, mma.sync covers everything.  pair=1 runs the
    CTA-pair kernel (256-token tiles, M = 256) where the padded rank is 64
    or 128, the single-CTA kernel elsewhere."""
    knob(LORA_PUNICA_UMMA=umma, LORA_PUNICA_UMMA_PARTIAL=partial, LORA_PUNICA_UMMA_MIN_COLS=0,
         LORA_PUNICA_UMMA_MIN_TOKENS=0, LORA_PUNICA_UMMA_PAIR=pair)
    w = W.Workload("long", T + r, T, H, r, L, tuple([16] * S), "zipf_seq", p_none=0.1,
                   seq_len=(200, 900), scale=0.75)
    inp = W.generate(w)
    rng = np.random.default_rng(3)
    b0 = rng.standard_normal(inp.buf.shape).astype(np.float32)
    _shrink_case(oracle_mod, inp, buf0=b0)


@pytest.mark.parametrize("ids", ["uniform", "uniform_p", "mixed"])
def test_shrink_tensor_core_fragmented_tiles(oracle_mod, knob, ids):
    """The tensor-core shrink on tiles whose tokens break into many runs
    (per-token ids: up to 128 one-row TMA boxes a stage; the decode-token
    prefix of a mixed batch): the pieces the producer warp builds cover
    every row of every tile exactly once."""
    knob(LORA_PUNICA_UMMA="1", LORA_PUNICA_UMMA_PARTIAL="1", LORA_PUNICA_UMMA_MIN_COLS=0,
         LORA_PUNICA_UMMA_MIN_TOKENS=0, LORA_PUNICA_UMMA_PAIR="0")
    w = W.Workload("frag", 1777, 1777, 256, 128, 3, (128, 128, 128), ids, p_none=0.1,
                   seq_len=(30, 300), n_decode=40, scale=0.5)
    inp = W.generate(w)
    b0 = np.random.default_rng(5).standard_normal(inp.buf.shape).astype(np.float32)
    _shrink_case(oracle_mod, inp, buf0=b0)


def test_shrink_accumulates_and_scales(oracle_mod):
    inp = _custom(300, 512, 32, 4, [8, 8], seed=9)
    rng = np.random.default_rng(0)
    b0 = rng.standard_normal(inp.buf.shape).astype(np.float32)
    _shrink_case(oracle_mod, inp, scale=-1.5, buf0=b0)
    got = _run_shrink(inp, inp.ids, 0.0, b0)
    np.testing.assert_array_equal(got, b0)


def test_shrink_strided_x(oracle_mod):
    inp = _custom(200, 264, 16, 3, [8], seed=11)
    _shrink_case(oracle_mod, inp, x_pad=24)


def test_shrink_zipf_segments_and_no_lora(oracle_mod):
    inp = _custom(2000, 256, 16, 9, [8, 8, 8], seed=12, ids="zipf_seq", p_none=0.3)
    _shrink_case(oracle_mod, inp)
    none = np.full(2000, -1, np.int32)
    b0 = np.random.default_rng(1).standard_normal(inp.buf.shape).astype(np.float32)
    got = _run_shrink(inp, none, 1.0, b0)
    np.testing.assert_array_equal(got, b0)


def test_shrink_invalid_ids_skipped(oracle_mod):
    inp = _custom(100, 128, 16, 3, [8], seed=13)
    ids = inp.ids.copy()
    ids[::7] = 5
    ids[::11] = -4
    _shrink_case(oracle_mod, inp, ids=ids)


# ------------------------------------------------------------------ expand

def _run_expand(inp, ids, xin, y_bits, slices, offset, add_inputs, bias, y_col_pad=0):
    eg = _eg()
    B = [dev_bf16(b) for b in inp.lora_b]
    bias_d = None if bias is None else [None if b is None else dev_bf16(b) for b in bias]
    if y_col_pad:
        T, ld = y_bits.shape
        yw = torch.zeros((T, ld + y_col_pad), dtype=torch.bfloat16, device="cuda")
        yw[:, :ld] = dev_bf16(y_bits)
        y = yw[:, :ld]
    else:
        y = dev_bf16(y_bits)
    meta = _meta(ids, inp.lora_b[0].shape[0])
    eg.lora_expand(dev_f32(xin), B, y, meta, offset, add_inputs, bias_d)
    torch.cuda.synchronize()
    assert int(meta.error_word.item()) & (1 << 30) == 0, "a pipeline wait timed out"
    return host_bits(y)


def _expand_case(oracle_mod, inp, ids=None, xin=None, offset=0, add_inputs=True,
                 bias="workload", y_extra=0, y_col_pad=0):
    ids = inp.ids if ids is None else ids
    S, T, r = inp.buf.shape
    if xin is None:
        xin = np.random.default_rng(7).standard_normal((S, T, r)).astype(np.float32)
    bias = inp.lora_bias if bias == "workload" else bias
    slices = list(inp.workload.slices)
    width = offset + sum(slices) + y_extra
    y0 = W.normal_bf16(np.random.default_rng(8), (T, width), 1.0)
    got = _run_expand(inp, ids, xin, y0, slices, offset, add_inputs, bias, y_col_pad)
    ref = oracle_mod.expand(xin, inp.lora_b, ids, y0, slices, offset, add_inputs, bias)
    assert_close(bits_to_f64(got), ref, EXPAND_ATOL, EXPAND_RTOL, "expand")
    none = (ids < 0) | (ids >= inp.lora_b[0].shape[0])
    np.testing.assert_array_equal(got[none], y0[none])                   # rows untouched
    np.testing.assert_array_equal(got[:, :offset], y0[:, :offset])       # columns untouched
    np.testing.assert_array_equal(got[:, offset + sum(slices):], y0[:, offset + sum(slices):])
    return got


# "2" requires the tcgen05 kernel (a call it does not fit fails), so these
# cases cannot pass on the mma.sync kernel by accident.
EXPAND_PATHS = [pytest.param("2", id="tcgen05"), pytest.param("0", id="mma_sync")]


@pytest.mark.parametrize("path", EXPAND_PATHS)
@pytest.mark.parametrize("name,T", [("tiny", None), ("decode", None), ("prefill", 1536),
                                    ("mlp", 512), ("large", 384)])
def test_expand_workloads_reduced(oracle_mod, knob, path, name, T):
    knob(LORA_PUNICA_EXPAND_TC=path)
    inp = W.generate(name, num_tokens=T)
    _expand_case(oracle_mod, inp)


@pytest.mark.parametrize("T,r,L,slices,offset,y_extra", [
    (1, 16, 1, (128,), 0, 0),
    (70, 8, 3, (200, 56), 0, 8),          # ragged column chunk, rank 8
    (300, 24, 4, (64, 64, 64), 16, 0),    # padded rank, offset
    (129, 128, 2, (1024, 136), 8, 24),    # rank 128
    (50, 32, 5, (16,) * 8, 0, 0),         # eight slices
])
@pytest.mark.parametrize("path", [pytest.param("1", id="tcgen05_where_fits"),
                                  pytest.param("0", id="mma_sync")])
def test_expand_shapes(oracle_mod, knob, path, T, r, L, slices, offset, y_extra):
    knob(LORA_PUNICA_EXPAND_TC=path)
    rng_bias = [True, False][T % 2]
    inp = _custom(T, 64, r, L, slices, seed=T + r, bias=rng_bias)
    _expand_case(oracle_mod, inp, offset=offset, y_extra=y_extra)


@pytest.mark.parametrize("T,r,L,slices,offset,y_extra", [
    (1, 16, 1, (128,), 0, 0),
    (70, 8, 3, (192, 64), 0, 16),         # rank 8
    (300, 24, 4, (64, 64, 64), 16, 0),    # padded rank, offset
    (129, 128, 2, (1024, 192), 16, 32),   # rank 128, two tiles + 1
    (50, 32, 5, (64,) * 8, 0, 0),         # eight slices of one chunk
    (257, 64, 7, (4096, 64), 48, 0),      # rank 64, two full tiles + 1
])
def test_expand_tc_shapes(oracle_mod, knob, T, r, L, slices, offset, y_extra):
    """The tcgen05 kernel, required, on shapes it takes (slice widths that
    are multiples of 64; y, its row stride and offset 32-byte aligned)."""
    knob(LORA_PUNICA_EXPAND_TC="2")
    inp = _custom(T, 64, r, L, slices, seed=T + r + 1, bias=bool(T % 2))
    _expand_case(oracle_mod, inp, offset=offset, y_extra=y_extra)


def test_expand_tc_required_rejects_what_it_cannot_take(knob):
    """With the tcgen05 kernel required, a slice width that is not a multiple
    of 64 and outputs that are not 32-byte aligned are refused on the host."""
    eg = _eg()
    knob(LORA_PUNICA_EXPAND_TC="2")
    for slices, offset, code in (((192, 96), 0, "size"), ((64,), 3, "align"), ((64,), 8, "align")):
        inp = _custom(40, 64, 16, 2, slices, seed=3)
        B = [dev_bf16(b) for b in inp.lora_b]
        y = torch.zeros((40, offset + sum(slices)), dtype=torch.bfloat16, device="cuda")
        meta = _meta(inp.ids, 2)
        x = torch.zeros((len(slices), 40, 16), dtype=torch.float32, device="cuda")
        with pytest.raises(RuntimeError, match=code):
            eg.lora_expand(x, B, y, meta, offset, True)


@pytest.mark.parametrize("slices,offset", [((100, 7), 0), ((64, 64), 3), ((13,), 5)])
def test_expand_unaligned_scalar_path(oracle_mod, slices, offset):
    inp = _custom(90, 64, 16, 3, slices, seed=21, bias=True)
    _expand_case(oracle_mod, inp, offset=offset, y_extra=1)


@pytest.mark.parametrize("path", EXPAND_PATHS)
def test_expand_long_segments(oracle_mod, knob, path):
    """Sequences of hundreds of tokens per LoRA: many full 128-token tiles."""
    knob(LORA_PUNICA_EXPAND_TC=path)
    slices, offset = ((384, 192, 64), 16) if path == "2" else ((384, 136, 8), 8)
    w = W.Workload("longx", 31, 2500, 64, 64, 5, slices, "zipf_seq", p_none=0.2,
                   seq_len=(150, 700), bias=True)
    inp = W.generate(w)
    _expand_case(oracle_mod, inp, offset=offset, y_extra=offset)


@pytest.mark.parametrize("path", EXPAND_PATHS)
def test_expand_overwrite_mode(oracle_mod, knob, path):
    knob(LORA_PUNICA_EXPAND_TC=path)
    inp = _custom(333, 64, 32, 4, (256, 128), seed=22, bias=True)
    _expand_case(oracle_mod, inp, add_inputs=False, offset=16, y_extra=16)
    if path == "0":
        _expand_case(oracle_mod, inp, add_inputs=False, offset=3, y_extra=1)   # scalar path


def test_expand_partial_bias_and_strided_y(oracle_mod):
    inp = _custom(150, 64, 16, 3, (128, 64, 64), seed=23, bias=True)
    bias = [inp.lora_bias[0], None, inp.lora_bias[2]]
    _expand_case(oracle_mod, inp, bias=bias, y_col_pad=40)


def test_expand_no_lora_batch_untouched(oracle_mod):
    inp = _custom(500, 64, 16, 3, (256,), seed=24, bias=True)
    _expand_case(oracle_mod, inp, ids=np.full(500, -1, np.int32))


def test_expand_invalid_ids_skipped(oracle_mod):
    inp = _custom(100, 64, 16, 3, (128,), seed=25)
    ids = inp.ids.copy()
    ids[::5] = 3
    _expand_case(oracle_mod, inp, ids=ids)


# ------------------------------------------------------------- composition

@pytest.mark.parametrize("name,T", [("tiny", None), ("decode", None), ("mlp", 256)])
def test_add_lora_linear_matches_oracle_composition(oracle_mod, name, T):
    eg = _eg()
    inp = W.generate(name, num_tokens=T)
    w = inp.workload
    x = dev_bf16(inp.x)
    y = dev_bf16(inp.y)
    A = [dev_bf16(a) for a in inp.lora_a]
    B = [dev_bf16(b) for b in inp.lora_b]
    bias = None if inp.lora_bias is None else [dev_bf16(b) for b in inp.lora_bias]
    meta = _meta(inp.ids, w.max_loras)
    eg.add_lora_linear(y, x, A, B, bias, w.scale, w.slices, meta)
    torch.cuda.synchronize()
    buf = oracle_mod.shrink(inp.x, inp.lora_a, inp.ids, w.scale, inp.buf).astype(np.float32)
    ref = oracle_mod.expand(buf, inp.lora_b, inp.ids, inp.y, w.slices, 0, True, inp.lora_bias)
    assert_close(bits_to_f64(host_bits(y)), ref, EXPAND_ATOL, EXPAND_RTOL, "add_lora_linear")


def test_shrink_expand_every_lora_of_the_largest_table(oracle_mod):
    """max_loras = LORA_MAX_LORAS (1025 bins) with every id in use and ids
    spread over the batch: the segment tables hold all bins."""
    import expand_gemm_gb300 as eg
    L = eg.LORA_MAX_LORAS
    rng = np.random.default_rng(1024)
    T = 3000
    ids = rng.permutation(np.concatenate([np.arange(L), rng.integers(-1, L, T - L)]))
    inp = _custom(T, 64, 16, L, [64, 24], seed=77, bias=True)
    inp.ids[:] = ids.astype(np.int32)
    _shrink_case(oracle_mod, inp, scale=0.5)
    _expand_case(oracle_mod, inp)
