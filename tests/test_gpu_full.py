"""Full-size parity: every workload at its stated size, run through the same
C-ABI calls (and therefore the same launch configuration) the benchmark
times.  The metadata is compared bit-exactly in full; shrink and expand on
a sample of tokens that the oracle computes one by one (each token's result
depends only on its own row and id, so a sub-batch gives the same values).
"""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import (EXPAND_ATOL, EXPAND_RTOL, SHRINK_ATOL, SHRINK_RTOL, assert_close,
                         bits_to_f64, dev_bf16, dev_i32, host_bits)

pytestmark = pytest.mark.gpu


def _sample(ids, n, seed):
    rng = np.random.default_rng(seed)
    T = ids.shape[0]
    pick = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    pick |= {0, T - 1}
    # the first and last token of every segment of equal ids
    edges = np.nonzero(np.diff(ids) != 0)[0]
    pick |= set(edges[:64].tolist()) | set((edges[:64] + 1).tolist())
    return np.array(sorted(pick), np.int64)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "mlp", "large", "none"])
def test_full_size_workload(oracle_mod, name):
    import expand_gemm_gb300 as eg
    inp = W.generate(name)
    w = inp.workload
    T = w.num_tokens
    x = dev_bf16(inp.x)
    A = [dev_bf16(a) for a in inp.lora_a]
    B = [dev_bf16(b) for b in inp.lora_b]
    bias = None if inp.lora_bias is None else [dev_bf16(b) for b in inp.lora_bias]
    y = dev_bf16(inp.y)
    buf = torch.zeros(inp.buf.shape, dtype=torch.float32, device="cuda")
    ids_d = dev_i32(inp.ids)

    meta = eg.LoRAKernelMeta.make(w.max_loras, T, "cuda")
    meta.prepare_tensors(ids_d)
    eg.lora_shrink(x, A, buf, meta, w.scale)
    eg.lora_expand(buf, B, y, meta, w.offset_start, w.add_inputs, bias)
    torch.cuda.synchronize()

    o = oracle_mod.meta_prepare(inp.ids, w.max_loras)
    assert int(meta.no_lora_flag.item()) == int(o.no_lora_flag[0])
    np.testing.assert_array_equal(meta.active_lora_ids.cpu().numpy(), o.active_lora_ids)
    np.testing.assert_array_equal(meta.num_tokens_per_lora.cpu().numpy(), o.num_tokens_per_lora)
    np.testing.assert_array_equal(meta.lora_token_start_loc.cpu().numpy(), o.lora_token_start_loc)
    if not o.no_lora_flag[0]:
        np.testing.assert_array_equal(meta.token_indices_sorted_by_lora_ids[:T].cpu().numpy(),
                                      o.token_indices_sorted_by_lora_ids[:T])

    # no pipeline wait of any kernel timed out (bit 30 of the error word)
    assert int(meta.error_word.item()) & (1 << 30) == 0
    buf_h = buf.cpu().numpy()
    y_h = host_bits(y)
    if name == "none":
        assert (buf_h == 0).all()
        np.testing.assert_array_equal(y_h, inp.y)
        return

    sel = _sample(inp.ids, 256, seed=w.seed)
    ids_s = inp.ids[sel]
    zeros = np.zeros((w.num_slices, sel.size, w.rank), np.float32)
    ref_buf = oracle_mod.shrink(inp.x[sel], inp.lora_a, ids_s, w.scale, zeros)
    assert_close(buf_h[:, sel], ref_buf, SHRINK_ATOL, SHRINK_RTOL, "shrink[%s]" % name)
    ref_y = oracle_mod.expand(ref_buf.astype(np.float32), inp.lora_b, ids_s, inp.y[sel],
                              w.slices, w.offset_start, w.add_inputs, inp.lora_bias)
    assert_close(bits_to_f64(y_h[sel]), ref_y, EXPAND_ATOL, EXPAND_RTOL, "expand[%s]" % name)
    # rows of tokens without a LoRA are bit-identical to the input
    none = inp.ids < 0
    np.testing.assert_array_equal(y_h[none], inp.y[none])
    assert (buf_h[:, none] == 0).all()
