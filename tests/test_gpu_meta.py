"""GPU parity of lora_meta_prepare against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import dev_i32

pytestmark = pytest.mark.gpu

SENTINEL = 0x5A5A5A5A


def _gpu_meta(ids: np.ndarray, L: int, max_tokens: int | None = None):
    import expand_gemm_gb300 as eg
    T = ids.shape[0]
    meta = eg.LoRAKernelMeta.make(L, max_tokens or max(T, 1), "cuda")
    for t in (meta.token_lora_mapping, meta.token_indices_sorted_by_lora_ids,
              meta.active_lora_ids, meta.num_tokens_per_lora, meta.lora_token_start_loc,
              meta.no_lora_flag, meta.error_word):
        t.fill_(SENTINEL)
    meta.prepare_tensors(dev_i32(ids))
    torch.cuda.synchronize()
    return meta


def _check(ids: np.ndarray, L: int, oracle_mod, max_tokens=None):
    T = ids.shape[0]
    g = _gpu_meta(ids, L, max_tokens)
    o = oracle_mod.meta_prepare(ids, L, oracle_mod.Meta(L, max(T, 1), fill=SENTINEL))
    flag = int(g.no_lora_flag.item())
    assert flag == int(o.no_lora_flag[0])
    np.testing.assert_array_equal(g.active_lora_ids.cpu().numpy(), o.active_lora_ids)
    np.testing.assert_array_equal(g.num_tokens_per_lora.cpu().numpy(), o.num_tokens_per_lora)
    np.testing.assert_array_equal(g.lora_token_start_loc.cpu().numpy(), o.lora_token_start_loc)
    assert int(g.error_word.item()) == o.invalid_ids
    if flag:
        # early exit: neither side writes the copy or the permutation
        assert (g.token_lora_mapping.cpu().numpy() == SENTINEL).all()
        assert (g.token_indices_sorted_by_lora_ids.cpu().numpy() == SENTINEL).all()
    else:
        np.testing.assert_array_equal(g.token_indices_sorted_by_lora_ids[:T].cpu().numpy(),
                                      o.token_indices_sorted_by_lora_ids[:T])
        np.testing.assert_array_equal(g.token_lora_mapping[:T].cpu().numpy(),
                                      o.token_lora_mapping[:T])
    return g


@pytest.mark.parametrize("seed,T,L,p_none", [
    (0, 1, 1, 0.0), (1, 31, 3, 0.2), (2, 32, 4, 0.0), (3, 33, 4, 0.5),
    (4, 1000, 7, 0.1), (5, 1023, 16, 0.0), (6, 1025, 64, 0.3), (7, 4097, 2, 0.9),
    (8, 16384, 64, 0.2), (9, 65536, 1024, 0.05), (10, 70001, 300, 0.0),
    (11, 5, 1024, 0.0),
    (12, 16384, 1024, 0.1),     # the largest batch the kernel stages in shared memory
    (13, 16385, 1024, 0.1)])    # one past it: read from global memory
def test_meta_random_maps(oracle_mod, seed, T, L, p_none):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, L, size=T).astype(np.int32)
    ids[rng.random(T) < p_none] = -1
    _check(ids, L, oracle_mod)


def test_meta_sorted_runs_and_single_id(oracle_mod):
    ids = np.repeat(np.array([3, -1, 0, 3, 2], np.int32), [100, 7, 300, 1, 64])
    _check(ids, 4, oracle_mod)
    _check(np.full(777, 2, np.int32), 3, oracle_mod)


def test_meta_worked_example_maps(oracle_mod):
    rng = np.random.default_rng(0)
    for ids_, counts in (([-1, 0, 1, 2], [3, 10, 5, 2]), ([-1, 0, 2, 1], [3, 10, 5, 2])):
        m = np.repeat(np.array(ids_, np.int32), counts)
        rng.shuffle(m)
        g = _check(m, 3, oracle_mod)
        if ids_[2] == 1:
            assert g.lora_token_start_loc.cpu().tolist() == [0, 3, 13, 18, 20]


def test_meta_no_lora_and_empty(oracle_mod):
    g = _check(np.full(4096, -1, np.int32), 8, oracle_mod)
    assert g.no_lora()
    g = _check(np.zeros(0, np.int32), 8, oracle_mod, max_tokens=16)
    assert g.no_lora()


def test_meta_read_no_lora_follows_each_batch(oracle_mod):
    """The host read (lora_meta_read_no_lora) sees the flag of the batch the
    last prepare wrote, in stream order, with no explicit synchronisation."""
    import expand_gemm_gb300 as eg
    from gpu_helpers import dev_i32
    meta = eg.LoRAKernelMeta.make(4, 64, "cuda")
    for ids, want in (([-1] * 64, True), ([-1] * 63 + [2], False), ([], True),
                      ([9, -1], True), ([0], False)):
        meta.prepare_tensors(dev_i32(np.array(ids, np.int32)))
        assert meta.no_lora() is want, ids


def test_meta_invalid_ids_counted(oracle_mod):
    ids = np.array([0, 9, -1, 2, -7, 0, 3, 3, 1 << 30], np.int32)
    g = _check(ids, 3, oracle_mod)
    assert int(g.error_word.item()) == 5   # 9, -7, 3, 3 and 1<<30 with L = 3


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "mlp", "large", "none"])
def test_meta_workload_maps(oracle_mod, name):
    w = W.WORKLOADS[name]
    rng = np.random.default_rng(w.seed)
    ids = W.token_ids(w, rng)
    _check(ids, w.max_loras, oracle_mod)


def test_meta_reuse_across_batches(oracle_mod):
    """Buffers reused for a smaller batch after a larger one (stale tail)."""
    import expand_gemm_gb300 as eg
    L = 8
    meta = eg.LoRAKernelMeta.make(L, 5000, "cuda")
    rng = np.random.default_rng(5)
    for T in (5000, 300, 0, 4999, 1):
        ids = rng.integers(-1, L, size=T).astype(np.int32)
        meta.prepare_tensors(dev_i32(ids))
        torch.cuda.synchronize()
        o = oracle_mod.meta_prepare(ids, L)
        assert int(meta.no_lora_flag.item()) == int(o.no_lora_flag[0])
        np.testing.assert_array_equal(meta.active_lora_ids.cpu().numpy(), o.active_lora_ids)
        np.testing.assert_array_equal(meta.num_tokens_per_lora.cpu().numpy(), o.num_tokens_per_lora)
        np.testing.assert_array_equal(meta.lora_token_start_loc.cpu().numpy(), o.lora_token_start_loc)
        if not o.no_lora_flag[0]:
            np.testing.assert_array_equal(meta.token_indices_sorted_by_lora_ids[:T].cpu().numpy(),
                                          o.token_indices_sorted_by_lora_ids[:T])


def _maps(T, L, seed):
    """A per-token map with invalid ids, a run-ordered (sequence) map and
    the all -1 map, each of T tokens over L LoRAs."""
    rng = np.random.default_rng(seed)
    per_token = rng.integers(-1, L, size=T).astype(np.int32)
    per_token[rng.random(T) < 0.01] = L + 3                      # invalid
    per_token[rng.random(T) < 0.01] = -7                         # invalid
    runs = np.repeat(rng.integers(-1, L, size=T // 100 + 1), 100)[:T].astype(np.int32)
    return [per_token, runs, np.full(T, -1, np.int32)]


@pytest.mark.parametrize("multi,cluster", [("0", "0"), ("1", "0"), ("1", "1")])
@pytest.mark.parametrize("T,L", [(513, 8), (1000, 1024), (2048, 8), (2049, 8), (4096, 64),
                                 (4097, 33), (8192, 16), (8193, 1024), (16384, 64),
                                 (20000, 1024), (32768, 64), (32769, 8), (70001, 300)])
def test_meta_single_and_multi_cta(oracle_mod, knob, multi, cluster, T, L):
    """The single-CTA kernel, the multi-CTA kernel (batches above 512
    tokens: one CTA per 256 tokens up to 4096, per 1024 above, each
    counting the whole map itself) and its cluster form (4097 to 32768
    tokens: up to 8 CTAs that read each other's run counts) give the
    oracle's metadata bit for bit, on per-token maps with invalid ids,
    run-ordered maps and the all -1 map."""
    knob(LORA_PUNICA_META_MULTI=multi, LORA_PUNICA_META_CLUSTER=cluster)
    for ids in _maps(T, L, seed=T + L):
        _check(ids, L, oracle_mod)
