"""Seeded synthetic inputs for the masked-attention hot path.

This module holds input generators only: mask patterns and Q/K/V tensors.
It contains none of the method's arithmetic (no encoding, no attention), so
that both the CPU oracle tests and the CUDA path can draw the same inputs
from it without sharing any computation.

Mask patterns follow the ones the STOF pages name (causal, sliding window,
random / BigBird, Longformer): "Accelerating Sparse Transformer Inference on
GPU", gist.science technical summary, Problem statement and Experimental
results.  The shapes are the five workloads of this library:

    window48_L256    B=1  H=2  L=256   d=64  fp16  causal AND 0 <= i-j < 48
    bigbird_L512     B=16 H=12 L=512   d=64  fp16  64-blocks: 3 sliding + 2 global + 3 random
    causal_L2048     B=8  H=12 L=2048  d=64  bf16  j <= i
    longformer_L4096 B=4  H=16 L=4096  d=64  bf16  |i-j| <= 256, plus 32 global tokens
    bernoulli_L16384 B=1  H=32 L=16384 d=128 bf16  j <= i AND (j == i OR u(h,i,j) < 0.1)

The last mask is defined through a counter-based hash (SplitMix64, Sebastiano
Vigna's published mixer) so that any row can be produced independently, on
the host (here, numpy) or on the device (a separate CUDA generator), without
materialising all 8.6 GB on the host.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "WORKLOAD_ORDER", "mask_index", "mask_rows", "make_mask", "workload_rule",
    "make_qkv", "splitmix64", "bernoulli_threshold", "random_mask", "to_float64",
]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    d: int
    dtype: str          # "fp16" or "bf16"
    pattern: str
    n_masks: int
    stride_b: int       # mask index of (b, h) = b * stride_b + h * stride_h
    stride_h: int
    seed: int = 0
    describe: str = ""

    @property
    def mask_bytes(self) -> int:
        return self.n_masks * self.L * self.L


WORKLOADS: dict[str, Workload] = {
    "window48_L256": Workload(
        "window48_L256", 1, 2, 256, 64, "fp16", "window48", 1, 0, 0,
        describe="causal AND sliding window 48: valid iff 0 <= i-j < 48"),
    "bigbird_L512": Workload(
        "bigbird_L512", 16, 12, 512, 64, "fp16", "bigbird64", 1, 0, 0,
        describe="BigBird at 64-blocks: sliding {I-1,I,I+1}, global blocks {0,1}, 3 random"),
    "causal_L2048": Workload(
        "causal_L2048", 8, 12, 2048, 64, "bf16", "causal", 1, 0, 0,
        describe="causal: valid iff j <= i"),
    "longformer_L4096": Workload(
        "longformer_L4096", 4, 16, 4096, 64, "bf16", "longformer", 1, 0, 0,
        describe="|i-j| <= 256 OR i in G OR j in G, G = 32 seeded positions"),
    "bernoulli_L16384": Workload(
        "bernoulli_L16384", 1, 32, 16384, 128, "bf16", "causal_bernoulli", 32, 32, 1,
        describe="per head: j <= i AND (j == i OR u(h,i,j) < 0.1), u from SplitMix64"),
}
WORKLOAD_ORDER = ["window48_L256", "bigbird_L512", "causal_L2048", "longformer_L4096",
                  "bernoulli_L16384"]

BERNOULLI_P = 0.1


def mask_index(w: Workload, b: int, h: int) -> int:
    return b * w.stride_b + h * w.stride_h


# --------------------------------------------------------------------------
# SplitMix64 (Vigna): state x, z = x + 0x9E3779B97F4A7C15, then two
# xor-shift-multiply rounds and a final xor-shift.  All arithmetic mod 2^64.
# --------------------------------------------------------------------------
_SM_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_SM_M1 = np.uint64(0xBF58476D1CE4E5B9)
_SM_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + _SM_GAMMA
        z = (z ^ (z >> np.uint64(30))) * _SM_M1
        z = (z ^ (z >> np.uint64(27))) * _SM_M2
        return z ^ (z >> np.uint64(31))


def bernoulli_threshold(p: float) -> int:
    """Integer T with  ((z >> 11) * 2^-53 < p)  <=>  ((z >> 11) < T)."""
    return int(math.ceil(p * float(1 << 53)))


def _bernoulli_rows(h: int, rows: np.ndarray, L: int, seed: int, p: float, ncols: int | None = None) -> np.ndarray:
    rows = np.asarray(rows, dtype=np.uint64)
    j = np.arange(L if ncols is None else ncols, dtype=np.uint64)
    ctr = (np.uint64(h) << np.uint64(48)) | (rows[:, None] << np.uint64(24)) | j[None, :]
    z = splitmix64(np.uint64(seed) ^ ctr)
    keep = (z >> np.uint64(11)) < np.uint64(bernoulli_threshold(p))
    ii = rows.astype(np.int64)[:, None]
    jj = j.astype(np.int64)[None, :]
    return ((jj <= ii) & ((jj == ii) | keep)).astype(np.uint8)


def _bigbird_blocks(L: int, blk: int, seed: int) -> np.ndarray:
    """Block-level BigBird layout [nb, nb] of 0/1.

    Block rows 0 and 1 are global (attend everywhere); every block row attends
    block columns 0 and 1 (global), its sliding neighbours {I-1, I, I+1}
    (clipped at the edges) and 3 further blocks drawn without replacement, in
    block-row order, from those not chosen yet (fewer if fewer remain).
    """
    nb = L // blk
    rng = np.random.default_rng(seed)
    lay = np.zeros((nb, nb), dtype=np.uint8)
    for I in range(nb):
        chosen = {0, 1} | {J for J in (I - 1, I, I + 1) if 0 <= J < nb}
        if I in (0, 1):
            chosen = set(range(nb))
        rest = [J for J in range(nb) if J not in chosen]
        if rest:
            pick = rng.choice(np.array(rest), size=min(3, len(rest)), replace=False)
            chosen |= {int(J) for J in pick}
        lay[I, sorted(chosen)] = 1
    return lay


def _longformer_globals(L: int, seed: int) -> np.ndarray:
    return np.sort(np.random.default_rng(seed).choice(L, 32, replace=False))


def mask_rows(w: Workload, m: int, rows, ncols: int | None = None) -> np.ndarray:
    """Rows `rows` of mask number m, as uint8 [len(rows), L] of 0/1; with
    `ncols`, only the first ncols key columns ([len(rows), ncols])."""
    rows = np.asarray(rows, dtype=np.int64)
    L = w.L
    i = rows[:, None]
    j = np.arange(L if ncols is None else ncols, dtype=np.int64)[None, :]
    if w.pattern == "window48":
        return ((i - j >= 0) & (i - j < 48)).astype(np.uint8)
    if w.pattern == "causal":
        return (j <= i).astype(np.uint8)
    if w.pattern == "bigbird64":
        lay = _bigbird_blocks(L, 64, w.seed)
        return lay[(rows // 64)[:, None], (j[0] // 64)[None, :]].astype(np.uint8)
    if w.pattern == "longformer":
        g = np.zeros(L, dtype=bool)
        g[_longformer_globals(L, w.seed)] = True
        out = (np.abs(i - j) <= 256) | g[rows][:, None] | g[j[0]][None, :]
        return out.astype(np.uint8)
    if w.pattern == "causal_bernoulli":
        return _bernoulli_rows(m, rows, L, w.seed, BERNOULLI_P, ncols)
    raise ValueError(w.pattern)


def workload_rule(w: Workload):
    """The workload's mask as a rule -- band (lo, hi) on i - j, global rows,
    global columns, block pattern -- or None when it has no such form (the
    per-element Bernoulli mask).  Bool arrays, block edge in elements:
    {"band_lo", "band_hi", "global_rows", "global_cols", "blocks", "block"}."""
    L = w.L
    rule = {"band_lo": 1, "band_hi": 0, "global_rows": None, "global_cols": None, "blocks": None, "block": 0}
    if w.pattern == "window48":
        rule.update(band_lo=0, band_hi=47)
    elif w.pattern == "causal":
        rule.update(band_lo=0, band_hi=(1 << 31) - 1)
    elif w.pattern == "longformer":
        g = np.zeros(L, dtype=bool)
        g[_longformer_globals(L, w.seed)] = True
        rule.update(band_lo=-256, band_hi=256, global_rows=g, global_cols=g)
    elif w.pattern == "bigbird64":
        rule.update(blocks=_bigbird_blocks(L, 64, w.seed).astype(bool), block=64)
    else:
        return None
    return rule


def make_mask(w: Workload, max_bytes: int = 1 << 30) -> np.ndarray:
    """Whole mask tensor uint8 [n_masks, L, L] (refuses very large ones)."""
    if w.mask_bytes > max_bytes:
        raise ValueError(f"{w.name}: mask is {w.mask_bytes} bytes; generate rows or on the device")
    out = np.empty((w.n_masks, w.L, w.L), dtype=np.uint8)
    for m in range(w.n_masks):
        for r0 in range(0, w.L, 1024):
            rows = np.arange(r0, min(w.L, r0 + 1024))
            out[m, r0:r0 + len(rows)] = mask_rows(w, m, rows)
    return out


def random_mask(n_masks: int, lq: int, lk: int, p: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (rng.random((n_masks, lq, lk)) < p).astype(np.uint8)


def make_qkv(B: int, H: int, L: int, d: int, dtype: str, seed: int = 0):
    """Q, K, V ~ iid N(0,1) drawn in fp32 (in that order) from one numpy
    Generator(PCG64, seed), then rounded to nearest even in fp16 or bf16.
    Returns CPU torch tensors [B, H, L, d]."""
    import torch
    rng = np.random.default_rng(seed)
    tdt = {"fp16": torch.float16, "bf16": torch.bfloat16}[dtype]
    out = []
    for _ in range(3):
        x = rng.standard_normal((B, H, L, d), dtype=np.float32)
        out.append(torch.from_numpy(x).to(tdt))
    return tuple(out)


def to_float64(t) -> np.ndarray:
    """Exact fp16/bf16 -> float64 values as a numpy array."""
    return t.double().numpy()
