"""The seeded input generator draws what each workload states."""
import numpy as np
import pytest

import workloads as W


def _ids(name, seed=None):
    w = W.WORKLOADS[name]
    return w, W.token_ids(w, np.random.Generator(np.random.PCG64(w.seed if seed is None else seed)))


def test_determinism():
    a = W.generate("tiny")
    b = W.generate("tiny")
    assert np.array_equal(a.ids, b.ids) and np.array_equal(a.x, b.x)
    assert all(np.array_equal(p, q) for p, q in zip(a.lora_a, b.lora_a))
    c = W.generate("tiny", seed=99)
    assert not np.array_equal(a.x, c.x)


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_uniform_ids_cover_range(name):
    w, ids = _ids(name)
    assert ids.min() >= -1 and ids.max() < w.max_loras
    assert set(np.unique(ids)) == set(range(-1, w.max_loras))


def test_mlp_ids_ten_percent_none():
    fr = []
    for seed in range(20):
        w, ids = _ids("mlp", seed)
        fr.append((ids == -1).mean())
        assert ids.max() < w.max_loras
    assert abs(np.mean(fr) - 0.1) < 0.01


def test_sequence_ids_are_constant_runs_with_zipf_skew():
    counts = np.zeros(16)
    for seed in range(40):
        w, ids = _ids("prefill", seed)
        assert ids.shape == (w.num_tokens,)
        runs = np.split(ids, np.nonzero(np.diff(ids))[0] + 1)
        # every run is a whole number of sequences, each at most 1024 long
        for r in runs:
            vals, c = np.unique(r, return_counts=True)
            counts[vals[vals >= 0]] += c[vals >= 0]
    # Zipf(1.1): id 0 carries the most tokens, the top id is far behind
    assert counts[0] == counts.max() and counts[0] > 4 * counts[15]


def test_large_starts_with_decode_tokens():
    w, ids = _ids("large")
    assert ids.shape == (16384,) and w.n_decode == 64
    assert ids.max() < 64 and ids.min() >= -1


def test_bf16_rounding_ties_to_even():
    # 1 + 2^-8 is halfway between bf16 neighbours 1 and 1 + 2^-7: rounds to even (1.0)
    vals = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0], np.float32)
    bits = W.bf16_bits(vals)
    assert bits.tolist() == [0x3F80, 0x3F82, 0xC020, 0x0000]


def test_unique_bytes_counts_active_rows_and_loras():
    w = W.WORKLOADS["decode"]
    ids = np.array([-1, 0, 0, 3] + [-1] * 252, np.int32)
    ub = W.unique_bytes(w, ids)
    assert ub["t_active"] == 3 and ub["distinct"] == 2
    assert ub["shrink"] == 3 * 4096 * 2 + 2 * 3 * 16 * 4096 * 2 + 2 * 3 * 3 * 16 * 4
    assert ub["expand"] == 3 * 3 * 16 * 4 + 2 * 12288 * 16 * 2 + 3 * 12288 * 2 * 2
    # shrink and expand in one kernel: the expand's read of the buffer goes
    assert ub["linear"] == ub["shrink"] + ub["expand"] - 3 * 3 * 16 * 4


def test_embedding_workload_has_a_bf16_rank_wide_input_and_no_a():
    inp = W.generate("embedding")
    w = inp.workload
    assert inp.x.shape == (w.num_tokens, w.rank) and inp.x.dtype == np.uint16
    assert inp.lora_a == [] and inp.lora_b[0].shape == (w.max_loras, 4096, w.rank)
    ub = W.unique_bytes(w, inp.ids)
    assert ub["shrink"] == 0 and ub["flops_shrink"] == 0
    t, d = ub["t_active"], ub["distinct"]
    assert ub["expand"] == t * w.rank * 2 + d * 4096 * w.rank * 2 + t * 4096 * 4


def test_logits_workload_is_one_vocabulary_wide_slice():
    inp = W.generate("logits")
    w = inp.workload
    assert w.slices == (32000,) and inp.y.shape == (256, 32000)
    assert inp.lora_a[0].shape == (8, 16, 4096)
