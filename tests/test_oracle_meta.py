"""Pins of the oracle's metadata step (LoRAKernelMeta.prepare_tensors).

Each test checks the oracle against something other than itself: the worked
example printed on the page (tests/golden/meta_worked_example.txt), the
library definitions the page's code uses (stable sort, sorted unique with
counts, cumsum) on random maps, Python's stable ``sorted`` by brute force on
every tiny map, and invariants.
"""
import collections
import itertools
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = [int(t) for t in v.split()]
    return out


def _map_from_counts(ids, counts, seed):
    m = np.repeat(np.array(ids, np.int32), counts)
    np.random.default_rng(seed).shuffle(m)
    return m


def test_worked_example_scan(oracle_mod):
    """Counts [3,10,5,2] must give start_loc [0,3,13,18,20] (printed example)."""
    g = _golden("meta_worked_example.txt")
    L = g["max_loras"][0]
    counts = g["printed_num_tokens_per_lora"]
    # Ascending ids -1,0,1,2 carrying the printed counts in that order.
    m = _map_from_counts([-1, 0, 1, 2], counts, seed=1)
    meta = oracle_mod.meta_prepare(m, L)
    assert meta.no_lora_flag[0] == 0
    assert meta.active_lora_ids.tolist() == [-1, 0, 1, 2]
    assert meta.num_tokens_per_lora.tolist() == counts
    assert meta.lora_token_start_loc.tolist() == g["printed_lora_token_start_loc"]


def test_worked_example_printed_id_order(oracle_mod):
    """The printed ids [-1,0,2,1] with counts [3,10,5,2] come out ascending."""
    g = _golden("meta_worked_example.txt")
    L = g["max_loras"][0]
    m = _map_from_counts(g["printed_active_lora_ids"],
                         g["printed_num_tokens_per_lora"], seed=2)
    meta = oracle_mod.meta_prepare(m, L)
    assert meta.active_lora_ids.tolist() == [-1, 0, 1, 2]
    assert meta.num_tokens_per_lora.tolist() == [3, 10, 2, 5]
    assert meta.lora_token_start_loc.tolist() == [0, 3, 13, 15, 20]


def test_all_no_lora_sets_flag_and_only_resets(oracle_mod):
    L, T = 5, 37
    meta = oracle_mod.meta_prepare(np.full(T, -1, np.int32), L,
                                   oracle_mod.Meta(L, 64, fill=12345))
    assert meta.no_lora_flag[0] == 1
    assert meta.active_lora_ids.tolist() == [-1] * (L + 1)
    assert meta.num_tokens_per_lora.tolist() == [0] * (L + 1)
    assert meta.lora_token_start_loc.tolist() == [0] * (L + 2)
    # early exit: mapping copy and permutation are not written
    assert (meta.token_lora_mapping == 12345).all()
    assert (meta.token_indices_sorted_by_lora_ids == 12345).all()


def test_empty_batch_is_no_lora(oracle_mod):
    meta = oracle_mod.meta_prepare(np.zeros(0, np.int32), 3)
    assert meta.no_lora_flag[0] == 1   # torch.all of an empty tensor is True
    assert meta.num_tokens_per_lora.tolist() == [0] * 4


def _brute(m, L):
    """Stable sort, sorted unique and cumsum from Python built-ins."""
    T = len(m)
    if T == 0 or all(v == -1 for v in m):
        return None
    perm = sorted(range(T), key=lambda t: m[t])          # Timsort is stable
    cnt = collections.Counter(m)
    ids = sorted(cnt)
    counts = [cnt[i] for i in ids]
    starts = [0] + list(itertools.accumulate(counts))
    pad = L + 1 - len(ids)
    return (perm, ids + [-1] * pad, counts + [0] * pad,
            starts + [0] * (L + 2 - len(starts)))


@pytest.mark.parametrize("L", [1, 2, 3])
def test_brute_force_every_tiny_map(oracle_mod, L):
    for T in range(0, 6 if L < 3 else 5):
        for m in itertools.product(range(-1, L), repeat=T):
            m = list(m)
            meta = oracle_mod.meta_prepare(np.array(m, np.int32), L,
                                           oracle_mod.Meta(L, 8))
            ref = _brute(m, L)
            if ref is None:
                assert meta.no_lora_flag[0] == 1, m
                continue
            perm, ids, counts, starts = ref
            assert meta.no_lora_flag[0] == 0, m
            assert meta.token_indices_sorted_by_lora_ids[:T].tolist() == perm, m
            assert meta.token_lora_mapping[:T].tolist() == m
            assert meta.active_lora_ids.tolist() == ids, m
            assert meta.num_tokens_per_lora.tolist() == counts, m
            assert meta.lora_token_start_loc.tolist() == starts, m


@pytest.mark.parametrize("seed,T,L", [(0, 1000, 7), (1, 4096, 64), (2, 333, 1),
                                      (3, 20000, 128), (4, 5, 100)])
def test_random_maps_match_library_routines(oracle_mod, seed, T, L):
    rng = np.random.default_rng(seed)
    m = rng.integers(-1, L, size=T).astype(np.int32)
    meta = oracle_mod.meta_prepare(m, L)
    if (m == -1).all():
        assert meta.no_lora_flag[0] == 1
        return
    perm = np.argsort(m, kind="stable")
    ids, counts = np.unique(m, return_counts=True)
    csum = np.cumsum(counts)
    k = ids.size
    assert meta.no_lora_flag[0] == 0
    np.testing.assert_array_equal(meta.token_indices_sorted_by_lora_ids[:T], perm)
    np.testing.assert_array_equal(meta.active_lora_ids[:k], ids)
    assert (meta.active_lora_ids[k:] == -1).all()
    np.testing.assert_array_equal(meta.num_tokens_per_lora[:k], counts)
    assert (meta.num_tokens_per_lora[k:] == 0).all()
    assert meta.lora_token_start_loc[0] == 0
    np.testing.assert_array_equal(meta.lora_token_start_loc[1:k + 1], csum)
    assert (meta.lora_token_start_loc[k + 1:] == 0).all()


@pytest.mark.parametrize("seed", range(4))
def test_invariants(oracle_mod, seed):
    rng = np.random.default_rng(100 + seed)
    T, L = int(rng.integers(1, 3000)), int(rng.integers(1, 40))
    m = rng.integers(-1, L, size=T).astype(np.int32)
    m[rng.random(T) < 0.5] = -1
    meta = oracle_mod.meta_prepare(m, L)
    if meta.no_lora_flag[0]:
        return
    perm = meta.token_indices_sorted_by_lora_ids[:T]
    assert sorted(perm.tolist()) == list(range(T))                # permutation
    keys = m[perm]
    assert (np.diff(keys) >= 0).all()                             # sorted
    same = np.diff(keys) == 0
    assert (np.diff(perm)[same] > 0).all()                        # stable
    k = int((meta.num_tokens_per_lora > 0).sum())
    c = meta.num_tokens_per_lora[:k]
    s = meta.lora_token_start_loc
    assert c.sum() == T
    np.testing.assert_array_equal(np.diff(s[:k + 1]), c)
    for j in range(k):                                           # segments
        seg = perm[s[j]:s[j + 1]]
        assert (m[seg] == meta.active_lora_ids[j]).all()


def test_invalid_ids_are_counted_and_binned_as_no_lora(oracle_mod):
    L = 3
    m = np.array([0, 7, -1, 2, -5, 0, 3], np.int32)
    meta = oracle_mod.meta_prepare(m, L)
    assert meta.invalid_ids == 3
    assert meta.no_lora_flag[0] == 0
    assert meta.active_lora_ids.tolist() == [-1, 0, 2, -1]
    assert meta.num_tokens_per_lora.tolist() == [4, 2, 1, 0]
    assert meta.lora_token_start_loc.tolist() == [0, 4, 6, 7, 0]
    assert meta.token_indices_sorted_by_lora_ids.tolist() == [1, 2, 4, 6, 0, 5, 3]
    assert meta.token_lora_mapping.tolist() == m.tolist()   # raw copy
    only_bad = oracle_mod.meta_prepare(np.array([9, -2], np.int32), L)
    assert only_bad.no_lora_flag[0] == 1 and only_bad.invalid_ids == 2
