"""Pins of the oracle's shrink and expand (PunicaWrapperGPU.add_shrink /
add_expand semantics, bias as in PunicaWrapperTPU._apply_bias).

The pins are chosen so that a plausible slip in the oracle -- a dropped
scale, a transposed operand, a wrong slice, id, row stride or column offset,
a missing bias mask -- fails at least one of them: exact widening of every
bf16 pattern (checked against torch), one-hot closed forms, special cases
that reduce to a single numpy matmul, and the page's own executable
statement of the bias step rewritten with numpy array ops.
"""
import numpy as np
import pytest
import torch

import workloads as W


def _bits(a):
    return W.bf16_bits(np.asarray(a, np.float32))


def _f64(bits):
    """bf16 bits -> float64 through torch (an independent conversion)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def test_bf16_widening_every_pattern(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.bf16_to_f64(bits)
    ref = _f64(bits)
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    np.testing.assert_array_equal(got[~nan], ref[~nan])


# ----------------------------------------------------------------- shrink

def _shrink_case(seed, T=24, H=40, r=6, L=3, S=2):
    rng = np.random.default_rng(seed)
    ids = rng.integers(-1, L, size=T).astype(np.int32)
    x = _bits(rng.standard_normal((T, H)))
    A = [_bits(rng.standard_normal((L, r, H)) * 0.1) for _ in range(S)]
    buf = rng.standard_normal((S, T, r)).astype(np.float32)
    return ids, x, A, buf


def test_shrink_one_hot_closed_form(oracle_mod):
    """x[t] = e_h picks A[s][id][i][h] * scale for every slice and row."""
    T, H, r, L, S = 12, 10, 4, 3, 3
    rng = np.random.default_rng(0)
    A = [_bits(rng.standard_normal((L, r, H))) for _ in range(S)]
    hs = rng.integers(0, H, size=T)
    ids = np.array([t % (L + 1) - 1 for t in range(T)], np.int32)
    x = np.zeros((T, H), np.float32)
    x[np.arange(T), hs] = 1.0
    buf = np.zeros((S, T, r), np.float32)
    out = oracle_mod.shrink(_bits(x), A, ids, 0.5, buf)
    for t in range(T):
        for s in range(S):
            if ids[t] < 0:
                assert (out[s, t] == 0).all()
            else:
                want = 0.5 * _f64(A[s][ids[t], :, hs[t]])
                np.testing.assert_array_equal(out[s, t], want)


def test_shrink_single_id_is_one_matmul(oracle_mod):
    """All tokens on one LoRA: buf[s] += scale * X @ A[s][id]^T (numpy)."""
    T, H, r, L, S = 33, 70, 5, 4, 2
    rng = np.random.default_rng(1)
    x = _bits(rng.standard_normal((T, H)))
    A = [_bits(rng.standard_normal((L, r, H))) for _ in range(S)]
    buf = rng.standard_normal((S, T, r)).astype(np.float32)
    ids = np.full(T, 2, np.int32)
    out = oracle_mod.shrink(x, A, ids, 1.25, buf)
    for s in range(S):
        ref = buf[s].astype(np.float64) + 1.25 * (_f64(x) @ _f64(A[s][2]).T)
        np.testing.assert_allclose(out[s], ref, rtol=1e-13, atol=1e-13)


def test_shrink_grouped_matmul_and_untouched_rows(oracle_mod):
    ids, x, A, buf = _shrink_case(2)
    out = oracle_mod.shrink(x, A, ids, -0.75, buf)
    X = _f64(x)
    for s in range(len(A)):
        for lid in range(A[0].shape[0]):
            rows = np.nonzero(ids == lid)[0]
            ref = buf[s, rows].astype(np.float64) - 0.75 * (X[rows] @ _f64(A[s][lid]).T)
            np.testing.assert_allclose(out[s, rows], ref, rtol=1e-13, atol=1e-13)
        none = ids == -1
        np.testing.assert_array_equal(out[s, none], buf[s, none].astype(np.float64))


def test_shrink_scale_zero_returns_buffer(oracle_mod):
    ids, x, A, buf = _shrink_case(3)
    out = oracle_mod.shrink(x, A, ids, 0.0, buf)
    np.testing.assert_array_equal(out, buf.astype(np.float64))


def test_shrink_strided_x_rows(oracle_mod):
    """A row stride larger than H reads the same rows as a compact copy."""
    ids, x, A, buf = _shrink_case(4)
    T, H = x.shape
    wide = np.zeros((T, H + 13), np.uint16)
    wide[:, 5:5 + H] = x
    got = oracle_mod.shrink(wide[:, 5:5 + H], A, ids, 1.0, buf)
    ref = oracle_mod.shrink(np.ascontiguousarray(x), A, ids, 1.0, buf)
    np.testing.assert_array_equal(got, ref)


def test_shrink_tiny_brute_force(oracle_mod):
    """Pure-Python loops on a tiny case."""
    ids, x, A, buf = _shrink_case(5, T=5, H=7, r=3, L=2, S=2)
    out = oracle_mod.shrink(x, A, ids, 2.0, buf)
    X = _f64(x)
    for s in range(2):
        As = _f64(A[s])
        for t in range(5):
            for i in range(3):
                want = float(buf[s, t, i])
                if ids[t] >= 0:
                    acc = 0.0
                    for h in range(7):
                        acc += X[t, h] * As[ids[t], i, h]
                    want += 2.0 * acc
                assert abs(out[s, t, i] - want) <= 1e-12 * (1 + abs(want))


# ----------------------------------------------------------------- expand

def _apply_bias_numpy(indices, output, slices, bias, offset0):
    """PunicaWrapperTPU._apply_bias restated with numpy array ops:
    gather bias[indices], zero it where the index is -1, pad it out to the
    slice's columns, add."""
    out = output.copy()
    off = offset0
    for s, n in enumerate(slices):
        if bias is not None and bias[s] is not None:
            b = _f64(bias[s])[np.maximum(indices, 0)]
            b = np.where(indices[:, None] == -1, 0.0, b)
            b = np.pad(b, ((0, 0), (off, out.shape[1] - off - n)))
            out = out + b
        off += n
    return out


def _expand_case(seed, T=20, r=5, L=3, slices=(6, 9, 4), ld_extra=3, bias=True):
    rng = np.random.default_rng(seed)
    ids = rng.integers(-1, L, size=T).astype(np.int32)
    xin = rng.standard_normal((len(slices), T, r)).astype(np.float32)
    B = [_bits(rng.standard_normal((L, n, r))) for n in slices]
    bi = [_bits(rng.standard_normal((L, n))) for n in slices] if bias else None
    y = _bits(rng.standard_normal((T, sum(slices) + ld_extra)))
    return ids, xin, B, bi, y


def test_expand_zero_weights_gives_input_plus_bias(oracle_mod):
    ids, xin, B, bi, y = _expand_case(10)
    Bz = [np.zeros_like(b) for b in B]
    slices = [b.shape[1] for b in B]
    out = oracle_mod.expand(xin, Bz, ids, y, slices, offset_start=2,
                            add_inputs=True, lora_bias=bi)
    ref = _apply_bias_numpy(ids, _f64(y), slices, bi, 2)
    np.testing.assert_array_equal(out, ref)


def test_expand_one_hot_closed_form(oracle_mod):
    """x[s][t] = e_k picks B[s][id][:, k] into the slice's columns."""
    T, r, L, slices = 9, 4, 3, (5, 3)
    rng = np.random.default_rng(11)
    ids = np.array([t % (L + 1) - 1 for t in range(T)], np.int32)
    ks = rng.integers(0, r, size=(len(slices), T))
    xin = np.zeros((len(slices), T, r), np.float32)
    for s in range(len(slices)):
        xin[s, np.arange(T), ks[s]] = 1.0
    B = [_bits(rng.standard_normal((L, n, r))) for n in slices]
    y = np.zeros((T, 10), np.uint16)
    out = oracle_mod.expand(xin, B, ids, y, slices, offset_start=1)
    for t in range(T):
        row = np.zeros(10)
        if ids[t] >= 0:
            off = 1
            for s, n in enumerate(slices):
                row[off:off + n] = _f64(B[s][ids[t], :, ks[s, t]])
                off += n
        np.testing.assert_array_equal(out[t], row)


@pytest.mark.parametrize("add_inputs", [True, False])
def test_expand_single_id_is_one_matmul(oracle_mod, add_inputs):
    T, r, L, slices = 17, 6, 2, (8, 5)
    rng = np.random.default_rng(12)
    xin = rng.standard_normal((2, T, r)).astype(np.float32)
    B = [_bits(rng.standard_normal((L, n, r))) for n in slices]
    bi = [None, _bits(rng.standard_normal((L, 5)))]
    y = _bits(rng.standard_normal((T, 16)))
    ids = np.full(T, 1, np.int32)
    out = oracle_mod.expand(xin, B, ids, y, slices, offset_start=3,
                            add_inputs=add_inputs, lora_bias=bi)
    Y = _f64(y)
    ref = Y.copy()
    off = 3
    for s, n in enumerate(slices):
        v = xin[s].astype(np.float64) @ _f64(B[s][1]).T
        if bi[s] is not None:
            v = v + _f64(bi[s][1])[None, :]
        ref[:, off:off + n] = (Y[:, off:off + n] if add_inputs else 0.0) + v
        off += n
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)


def test_expand_mixed_ids_grouped_matmul_plus_bias(oracle_mod):
    ids, xin, B, bi, y = _expand_case(13)
    slices = [b.shape[1] for b in B]
    out = oracle_mod.expand(xin, B, ids, y, slices, offset_start=0,
                            add_inputs=True, lora_bias=bi)
    ref = _apply_bias_numpy(ids, _f64(y), slices, bi, 0)
    off = 0
    for s, n in enumerate(slices):
        for lid in range(B[0].shape[0]):
            rows = np.nonzero(ids == lid)[0]
            ref[rows, off:off + n] += xin[s, rows].astype(np.float64) @ _f64(B[s][lid]).T
        off += n
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)
    none = ids == -1
    np.testing.assert_array_equal(out[none], _f64(y)[none])


def test_expand_overwrite_leaves_other_columns(oracle_mod):
    ids, xin, B, bi, y = _expand_case(14, bias=False)
    slices = [b.shape[1] for b in B]
    a = oracle_mod.expand(xin, B, ids, y, slices, offset_start=2, add_inputs=False)
    b = oracle_mod.expand(xin, B, ids, np.zeros_like(y), slices, offset_start=2,
                          add_inputs=True)
    Y = _f64(y)
    act = ids >= 0
    cols = slice(2, 2 + sum(slices))
    np.testing.assert_array_equal(a[act, cols], b[act, cols])
    np.testing.assert_array_equal(a[:, :2], Y[:, :2])
    np.testing.assert_array_equal(a[:, 2 + sum(slices):], Y[:, 2 + sum(slices):])
    np.testing.assert_array_equal(a[~act], Y[~act])
