"""GPU parity of the embedding LoRA (expand over a bf16 input, add_inputs
passed through) and of the logits LoRA (shrink + expand driven by a second
metadata instance over the sampler ids), against the oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import (EXPAND_ATOL, EXPAND_RTOL, SHRINK_ATOL, SHRINK_RTOL, assert_close,
                         bits_to_f64, dev_bf16, dev_f32, dev_i32, host_bits)

pytestmark = pytest.mark.gpu


def _meta(ids, L):
    import expand_gemm_gb300 as eg
    meta = eg.LoRAKernelMeta.make(L, len(ids), "cuda")
    meta.prepare_tensors(dev_i32(ids))
    return meta


def _f32_of_bits(bits):
    return bits_to_f64(bits).astype(np.float32)      # bf16 -> fp32 is exact


def _check_embedding(oracle_mod, ids, x_bits, lora_b, y_bits, L, add_inputs):
    import expand_gemm_gb300 as eg
    meta = _meta(ids, L)
    y = dev_bf16(y_bits)
    eg.add_lora_embedding(y, dev_bf16(x_bits), dev_bf16(lora_b), meta, add_inputs)
    torch.cuda.synchronize()
    got = host_bits(y)
    ref = oracle_mod.expand(_f32_of_bits(x_bits)[None], [lora_b], ids, y_bits,
                            (lora_b.shape[1],), 0, add_inputs, None)
    assert_close(bits_to_f64(got), ref, EXPAND_ATOL, EXPAND_RTOL, "embedding y")
    none = (ids < 0) | (ids >= L)
    np.testing.assert_array_equal(got[none], y_bits[none])
    return got, meta


@pytest.mark.parametrize("add_inputs", [True, False])
def test_embedding_workload(oracle_mod, add_inputs):
    inp = W.generate("embedding")
    w = inp.workload
    _check_embedding(oracle_mod, inp.ids, inp.x, inp.lora_b[0], inp.y, w.max_loras, add_inputs)


@pytest.mark.parametrize("T,r,n,L", [
    (1, 16, 4096, 2),          # single token
    (37, 8, 200, 3),           # rank 8, ragged columns
    (300, 24, 136, 5),         # padded rank, two tiles per LoRA
    (513, 64, 1024, 4),        # rank 64
    (130, 128, 520, 6),        # rank 128, ragged tail chunk
    (64, 16, 100, 3),          # width not a multiple of 8: scalar epilogue
])
def test_embedding_shapes(oracle_mod, T, r, n, L):
    rng = np.random.Generator(np.random.PCG64(T * 7 + r))
    ids = rng.integers(-1, L, size=T).astype(np.int32)
    x = W.normal_bf16(rng, (T, r), 1.0)
    B = W.normal_bf16(rng, (L, n, r), 0.02)
    y = W.normal_bf16(rng, (T, n), 1.0)
    for add_inputs in (True, False):
        _check_embedding(oracle_mod, ids, x, B, y, L, add_inputs)


def test_bf16_input_matches_fp32_input_bitwise():
    """The fp32 expand rounds its input to bf16 before the tensor cores; on
    inputs that are already bf16 values both entries feed the same operands
    to the same deterministic kernel, so y agrees bit for bit (bias and
    several slices included)."""
    import expand_gemm_gb300 as eg
    rng = np.random.Generator(np.random.PCG64(11))
    T, r, L, slices = 300, 32, 5, (256, 72, 512)
    ids = rng.integers(-1, L, size=T).astype(np.int32)
    x = W.normal_bf16(rng, (len(slices), T, r), 1.0)
    B = [W.normal_bf16(rng, (L, n, r), 0.02) for n in slices]
    bias = [W.normal_bf16(rng, (L, n), 0.01) for n in slices]
    y0 = W.normal_bf16(rng, (T, 8 + sum(slices)), 1.0)
    meta = _meta(ids, L)
    outs = []
    for xt in (dev_bf16(x), dev_f32(_f32_of_bits(x))):
        y = dev_bf16(y0)
        eg.lora_expand(xt, [dev_bf16(b) for b in B], y, meta, 8, True,
                       [dev_bf16(b) for b in bias])
        torch.cuda.synchronize()
        outs.append(host_bits(y))
    np.testing.assert_array_equal(outs[0], outs[1])


def test_logits_workload_with_a_second_metadata_instance(oracle_mod):
    """A linear layer over the tokens (token metadata) and the logits over
    the sampled positions (prompt metadata) in one stream: each metadata
    instance drives its own calls."""
    import expand_gemm_gb300 as eg
    lin = W.generate(W.Workload("tok", 40, 512, 1024, 16, 8, (512, 512), "zipf_seq",
                                p_none=0.2, seq_len=(16, 64)))
    lg = W.generate("logits")
    wl, wg = lin.workload, lg.workload
    tok_meta = _meta(lin.ids, wl.max_loras)
    prm_meta = _meta(lg.ids, wg.max_loras)
    y_lin = dev_bf16(lin.y)
    eg.add_lora_linear(y_lin, dev_bf16(lin.x), [dev_bf16(a) for a in lin.lora_a],
                       [dev_bf16(b) for b in lin.lora_b], None, wl.scale, wl.slices, tok_meta)
    y_lg = dev_bf16(lg.y)
    buf = torch.zeros((wg.num_tokens, wg.rank), dtype=torch.float32, device="cuda")
    eg.add_lora_logits(y_lg, dev_bf16(lg.x), dev_bf16(lg.lora_a[0]), dev_bf16(lg.lora_b[0]),
                       wg.scale, prm_meta, buffer=buf)
    torch.cuda.synchronize()

    b = oracle_mod.shrink(lin.x, lin.lora_a, lin.ids, wl.scale, lin.buf)
    ref = oracle_mod.expand(b.astype(np.float32), lin.lora_b, lin.ids, lin.y, wl.slices, 0, True)
    assert_close(bits_to_f64(host_bits(y_lin)), ref, EXPAND_ATOL, EXPAND_RTOL, "linear y")

    b = oracle_mod.shrink(lg.x, lg.lora_a, lg.ids, wg.scale, lg.buf)
    assert_close(buf.cpu().numpy()[None], b, SHRINK_ATOL, SHRINK_RTOL, "logits buffer")
    ref = oracle_mod.expand(b.astype(np.float32), lg.lora_b, lg.ids, lg.y, wg.slices, 0, True)
    got = host_bits(y_lg)
    assert_close(bits_to_f64(got), ref, EXPAND_ATOL, EXPAND_RTOL, "logits y")
    np.testing.assert_array_equal(got[lg.ids < 0], lg.y[lg.ids < 0])


def test_logits_fewer_rows_than_tokens(oracle_mod):
    """One logits row per sequence (its last token), ids taken per
    sequence, while the token metadata covers every token."""
    import expand_gemm_gb300 as eg
    rng = np.random.Generator(np.random.PCG64(5))
    L, H, r, V = 4, 512, 8, 1000
    seq_ids = rng.integers(-1, L, size=12).astype(np.int32)
    x = W.normal_bf16(rng, (12, H), 1.0)
    A = W.normal_bf16(rng, (L, r, H), 0.02)
    B = W.normal_bf16(rng, (L, V, r), 0.02)
    y0 = W.normal_bf16(rng, (12, V), 1.0)
    meta = _meta(seq_ids, L)
    y = dev_bf16(y0)
    eg.add_lora_logits(y, dev_bf16(x), dev_bf16(A), dev_bf16(B), 0.5, meta)
    torch.cuda.synchronize()
    b = oracle_mod.shrink(x, [A], seq_ids, 0.5, np.zeros((1, 12, r), np.float32))
    ref = oracle_mod.expand(b.astype(np.float32), [B], seq_ids, y0, (V,), 0, True)
    assert_close(bits_to_f64(host_bits(y)), ref, EXPAND_ATOL, EXPAND_RTOL, "logits y")
