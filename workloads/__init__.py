"""Seeded synthetic inputs for the multi-LoRA shrink/expand path.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it without sharing any computation.

Five workloads of one linear LoRA layer (sizes and distributions as stated
for each below), an all-no-LoRA batch, and one workload each for the logits
and the embedding LoRA.  Values: x ~ N(0, 1), A and B ~ N(0, 0.02^2), bias ~
N(0, 0.01^2), y_in ~ N(0, 1), each rounded to bf16 (round to nearest even)
and stored as raw uint16 bit patterns; the shrink buffer starts at zero.
LoRA ids: per token uniform, or per sequence drawn from a truncated Zipf law
P(k) ~ (k + 1)^-1.1 over the LoRA count, with a stated fraction of -1 (no
LoRA).  Sequence lengths are uniform in a range; the last sequence is cut so
that the lengths sum to T.  The generator is numpy's PCG64 seeded with the
workload's index.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    num_tokens: int          # T
    hidden: int              # H
    rank: int                # r
    max_loras: int           # L
    slices: tuple            # n_s per slice
    ids: str                 # "uniform", "uniform_p", "zipf_seq", "mixed", "none"
    p_none: float = 0.0      # probability of id -1 (per token or per sequence)
    seq_len: tuple = (0, 0)  # inclusive range of sequence lengths
    n_decode: int = 0        # leading one-token sequences ("mixed")
    bias: bool = False
    scale: float = 1.0
    offset_start: int = 0
    add_inputs: bool = True
    # "linear": shrink + expand of one LoRA layer; "logits": the same over
    # the logits rows (one id per sampled position, the vocabulary as the one
    # slice); "embedding": expand only, from a bf16 [T, r] input (the
    # embedding LoRA's A rows looked up per token), no A.
    kind: str = "linear"
    description: str = field(default="", compare=False)

    @property
    def num_slices(self) -> int:
        return len(self.slices)

    @property
    def y_ld(self) -> int:
        return self.offset_start + sum(self.slices)


WORKLOADS = {
    "tiny": Workload(
        "tiny", 0, 64, 256, 8, 4, (256,), "uniform", bias=True, scale=0.5,
        description="64 tokens, hidden 256, rank 8, 4 LoRAs, 1 slice of 256, "
                    "ids uniform in {-1..3}, bias, scale 0.5"),
    "decode": Workload(
        "decode", 1, 256, 4096, 16, 8, (4096, 4096, 4096), "uniform",
        description="256 one-token sequences, hidden 4096, rank 16, 8 LoRAs, "
                    "3 slices (q/k/v) of 4096, ids uniform in {-1..7}"),
    "prefill": Workload(
        "prefill", 2, 8192, 4096, 64, 16, (4096,), "zipf_seq", p_none=0.1,
        seq_len=(128, 1024),
        description="8192 tokens in sequences of length U[128,1024], one "
                    "Zipf(1.1) id per sequence over 16 LoRAs, 10% of "
                    "sequences -1; hidden 4096, rank 64, 1 slice of 4096"),
    "mlp": Workload(
        "mlp", 3, 2048, 4096, 32, 32, (11008, 11008), "uniform_p", p_none=0.1,
        bias=True,
        description="2048 tokens, hidden 4096, rank 32, 32 LoRAs, 2 slices "
                    "(gate/up) of 11008, per-token ids uniform with 10% -1, "
                    "bias"),
    "large": Workload(
        "large", 4, 16384, 8192, 128, 64, (8192, 1024, 1024), "mixed",
        p_none=0.2, seq_len=(256, 2048), n_decode=64,
        description="16384 tokens: 64 one-token sequences then sequences of "
                    "length U[256,2048]; one Zipf(1.1) id per sequence over "
                    "64 LoRAs, 20% -1; hidden 8192, rank 128, 3 slices "
                    "8192/1024/1024"),
    "none": Workload(
        "none", 5, 16384, 8192, 128, 64, (8192, 1024, 1024), "none",
        description="large-workload shapes with every id -1 (no-LoRA batch)"),
    "logits": Workload(
        "logits", 6, 256, 4096, 16, 8, (32000,), "uniform", kind="logits",
        description="logits of 256 sampled positions (one per decode "
                    "sequence): hidden 4096, rank 16, 8 LoRAs, vocabulary "
                    "32000 as one slice, sampler ids uniform in {-1..7}"),
    "embedding": Workload(
        "embedding", 7, 2048, 16, 16, 8, (4096,), "uniform_p", p_none=0.1,
        kind="embedding",
        description="embedding LoRA of 2048 tokens: bf16 input [T, 16] (the "
                    "looked-up A rows), rank 16, 8 LoRAs, embedding width "
                    "4096, per-token ids uniform with 10% -1"),
}


def _zipf_ids(rng: np.random.Generator, n: int, num_loras: int) -> np.ndarray:
    k = np.arange(num_loras, dtype=np.float64)
    p = (k + 1.0) ** -1.1
    p /= p.sum()
    return rng.choice(num_loras, size=n, p=p).astype(np.int32)


def _seq_lengths(rng: np.random.Generator, total: int, lo: int, hi: int) -> list:
    lens = []
    left = total
    while left > 0:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, left)
        lens.append(n)
        left -= n
    return lens


def token_ids(w: Workload, rng: np.random.Generator) -> np.ndarray:
    """Per-token LoRA ids (int32, -1 = no LoRA) drawn as the workload says."""
    T, L = w.num_tokens, w.max_loras
    if w.ids == "none":
        return np.full(T, -1, np.int32)
    if w.ids == "uniform":                      # uniform over {-1, ..., L-1}
        return rng.integers(-1, L, size=T).astype(np.int32)
    if w.ids == "uniform_p":                    # -1 with p_none, else U{0..L-1}
        ids = rng.integers(0, L, size=T).astype(np.int32)
        ids[rng.random(T) < w.p_none] = -1
        return ids
    if w.ids in ("zipf_seq", "mixed"):
        lens = [1] * w.n_decode
        lens += _seq_lengths(rng, T - w.n_decode, *w.seq_len)
        n_seq = len(lens)
        seq_id = _zipf_ids(rng, n_seq, L)
        seq_id[rng.random(n_seq) < w.p_none] = -1
        return np.repeat(seq_id, lens).astype(np.int32)
    raise ValueError(w.ids)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return bf16_bits(x)


@dataclass
class Inputs:
    workload: Workload
    ids: np.ndarray                 # int32 [T]
    x: np.ndarray                   # uint16 (bf16) [T, H] ([T, r] for "embedding")
    lora_a: list                    # S x uint16 [L, r, H] (empty for "embedding")
    lora_b: list                    # S x uint16 [L, n_s, r]
    lora_bias: list | None          # S x uint16 [L, n_s] or None
    y: np.ndarray                   # uint16 (bf16) [T, y_ld]
    buf: np.ndarray                 # float32 [S, T, r], zeros


def generate(w: Workload | str, seed: int | None = None,
             num_tokens: int | None = None) -> Inputs:
    """Draw one batch of inputs for workload ``w``.

    ``num_tokens`` overrides T (the id law is unchanged); ``seed`` overrides
    the workload's own seed.  Draw order is fixed: ids, x, A, B, bias, y
    (no A for an embedding workload).
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    if num_tokens is not None:
        from dataclasses import replace
        w = replace(w, num_tokens=int(num_tokens),
                    n_decode=min(w.n_decode, int(num_tokens)))
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    T, H, r, L, S = w.num_tokens, w.hidden, w.rank, w.max_loras, w.num_slices
    ids = token_ids(w, rng)
    x = normal_bf16(rng, (T, H), 1.0)
    if w.kind == "embedding":
        lora_a = []
    else:
        lora_a = [normal_bf16(rng, (L, r, H), 0.02) for _ in range(S)]
    lora_b = [normal_bf16(rng, (L, n, r), 0.02) for n in w.slices]
    lora_bias = [normal_bf16(rng, (L, n), 0.01) for n in w.slices] if w.bias else None
    y = normal_bf16(rng, (T, w.y_ld), 1.0)
    buf = np.zeros((S, T, r), np.float32)
    return Inputs(w, ids, x, lora_a, lora_b, lora_bias, y, buf)


def unique_bytes(w: Workload, ids: np.ndarray) -> dict:
    """Algorithmic (unique) HBM bytes of one shrink and one expand call.

    Counted from the id map: x rows of tokens with an id (once, not per
    slice); A, B and bias of the LoRAs that occur; the fp32 buffer read and
    written by shrink (+=) and read by expand; y read and written for rows
    with an id (write only when add_inputs is false).  "linear" is both
    calls in one kernel, the buffer read and written once.
    """
    L = w.max_loras
    act = (ids >= 0) & (ids < L)
    t_act = int(act.sum())
    d = int(np.unique(ids[act]).size)
    S, r, H = w.num_slices, w.rank, w.hidden
    n_tot = sum(w.slices)
    if w.kind == "embedding":                  # expand only, bf16 input
        shrink, x_bytes = 0, S * t_act * r * 2
    else:
        shrink = t_act * H * 2 + d * S * r * H * 2 + 2 * S * t_act * r * 4
        x_bytes = S * t_act * r * 4
    expand = (x_bytes + d * n_tot * r * 2
              + (d * n_tot * 2 if w.bias else 0)
              + t_act * n_tot * 2 * (2 if w.add_inputs else 1))
    flops_shrink = 0 if w.kind == "embedding" else 2 * t_act * S * r * H
    flops_expand = 2 * t_act * n_tot * r
    # shrink and expand in one kernel: the buffer is read and written once
    linear = shrink + expand - (0 if w.kind == "embedding" else x_bytes)
    return {"t_active": t_act, "distinct": d, "shrink": shrink, "expand": expand,
            "linear": linear,
            "flops_shrink": flops_shrink, "flops_expand": flops_expand}
