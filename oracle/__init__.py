"""CPU oracle for the STOF masked-attention hot path (test infrastructure).

Only the tests, the package's smoke check and the benchmark's CPU-baseline
leg may import this package.  The library under test never does, and the two
share no code.  The arithmetic lives in ``stof_oracle.c`` (plain C, fp64,
direct loops); this module compiles it with gcc on first use and marshals
numpy arrays in and out.

What each function follows ("Accelerating Sparse Transformer Inference on
GPU", gist.science technical summary):
  - ``attention``: masked softmax attention by its definition, fp64, exact
    masking (Methodology 1, two-level storage format: "exact masking without
    materialising the sparse matrix"; Problem statement: skipping instead of
    resetting scores).  A fully masked query row gives 0.
  - ``encode`` / ``decode``: the two-level format by brute force
    (Methodology 1: OT classes empty / full / partial, pointer arrays for
    full and partial OTs, one uint64 per 8x8 IT of a partial OT).
  - ``oproj``: the operator after the MHA, the output projection with bias
    and residual, by its definition in fp64 (Methodology 2, operator fusion
    module: fusion carried past the MHA layer): heads concatenated along
    the reduction axis, y = O_cat W^T + bias + residual.  A numpy matmul is
    its one library step.
  - ``layer_norm`` / ``oproj_ln``: the LayerNorm that closes a post-norm
    transformer sublayer (the operator after the projection and residual),
    by its definition in fp64: per token, subtract the mean over the
    features, divide by sqrt(population variance + eps), scale by gamma and
    add beta; ``oproj_ln`` is ``layer_norm(oproj(...))``.
  - ``unpack_bits``: a bit-packed mask (least significant bit first along
    the key axis) back to bytes, by explicit shifts.
  - ``rule_mask``: the dense mask a parametric rule stands for, by its
    definition: the union of a diagonal band, global rows, global columns
    and a block pattern (Problem statement and Experimental results: the
    causal, sliding-window, Longformer and BigBird families).

Pins (tests/test_oracle_pins.py) tie every function to something other than
itself: library dense attention, closed forms, tiny brute force, round trips
and hand-derived fixtures under tests/golden/.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "stof_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libstof_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile stof_oracle.c into libstof_oracle.so (plain gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.stof_oracle_attention.argtypes = [i64, i64, i32, dbl, P, P, P, P, P, i32]
            lib.stof_oracle_attention.restype = i32
            lib.stof_oracle_encode_count.argtypes = [P, i32, i32, i32, i32, i32, P]
            lib.stof_oracle_encode_count.restype = i32
            lib.stof_oracle_encode.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, P, P]
            lib.stof_oracle_encode.restype = i32
            lib.stof_oracle_decode.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P]
            lib.stof_oracle_decode.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return os.cpu_count() or 1


def attention(q, k, v, mask, scale: float, n_threads: int | None = None) -> np.ndarray:
    """One head: q [n_q, d], k/v [lk, d] (float64), mask [n_q, lk] (0/1 bytes)."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    n_q, d = q.shape
    lk = k.shape[0]
    assert k.shape == (lk, d) and v.shape == (lk, d) and mask.shape == (n_q, lk)
    o = np.empty((n_q, d), dtype=np.float64)
    rc = lib.stof_oracle_attention(n_q, lk, d, float(scale), _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(mask), _ptr(o), n_threads or default_threads())
    if rc != 0:
        raise ValueError("oracle attention: bad arguments")
    return o


def _padded(mask, bm: int, bn: int) -> np.ndarray:
    """mask [n_masks, lq, lk] extended with invalid (0) elements to whole
    OTs on both sides.  The two-level format tiles the whole matrix with
    BM x BN outer tiles ("Accelerating Sparse Transformer Inference on
    GPU", gist.science technical summary, Methodology 1, two-level storage
    format); the pages only use sides that are whole numbers of tiles, and
    for other sides this is the plain reading: the last OT row and column
    are padded, and padding is never a valid element."""
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    n_masks, lq, lk = mask.shape
    lqp, lkp = -(-lq // bm) * bm, -(-lk // bn) * bn
    if (lqp, lkp) == (lq, lk):
        return mask
    out = np.zeros((n_masks, lqp, lkp), dtype=np.uint8)
    out[:, :lq, :lk] = mask
    return out


def encode_count(mask, bm: int, bn: int):
    """(n_full, n_part, nnz) of mask [n_masks, lq, lk] (sides padded to whole OTs)."""
    lib = _load()
    mask = _padded(mask, bm, bn)
    n_masks, lq, lk = mask.shape
    counts = np.zeros(3, dtype=np.int64)
    if lib.stof_oracle_encode_count(_ptr(mask), n_masks, lq, lk, bm, bn, _ptr(counts)) != 0:
        raise ValueError("oracle encode: bad shape")
    return int(counts[0]), int(counts[1]), int(counts[2])


def encode(mask, bm: int, bn: int) -> dict:
    """Brute-force two-level encoding of mask [n_masks, lq, lk]; sides that
    are not whole numbers of OTs are padded to one with invalid elements
    (_padded); lq and lk of the result are the mask's own."""
    lib = _load()
    lq0, lk0 = np.shape(mask)[1:]
    mask = _padded(mask, bm, bn)
    n_masks, lq, lk = mask.shape
    n_full, n_part, nnz = encode_count(mask, bm, bn)
    n_rows = n_masks * (lq // bm)
    fmt = dict(
        n_masks=n_masks, lq=lq, lk=lk, bm=bm, bn=bn, n_tr=lq // bm, n_tc=lk // bn,
        full_row_ptr=np.zeros(n_rows + 1, dtype=np.int32),
        full_col_idx=np.zeros(max(n_full, 1), dtype=np.int32),
        part_row_ptr=np.zeros(n_rows + 1, dtype=np.int32),
        part_col_idx=np.zeros(max(n_part, 1), dtype=np.int32),
        bitmaps=np.zeros((max(n_part, 1), bm // 8, bn // 8), dtype=np.uint64),
        n_full=n_full, n_part=n_part, nnz=nnz)
    rc = lib.stof_oracle_encode(_ptr(mask), n_masks, lq, lk, bm, bn,
                                _ptr(fmt["full_row_ptr"]), _ptr(fmt["full_col_idx"]),
                                _ptr(fmt["part_row_ptr"]), _ptr(fmt["part_col_idx"]),
                                _ptr(fmt["bitmaps"]))
    if rc != 0:
        raise ValueError("oracle encode: bad shape")
    fmt["full_col_idx"] = fmt["full_col_idx"][:n_full]
    fmt["part_col_idx"] = fmt["part_col_idx"][:n_part]
    fmt["bitmaps"] = fmt["bitmaps"][:n_part]
    fmt["lq"], fmt["lk"] = lq0, lk0
    return fmt


def decode(fmt: dict) -> np.ndarray:
    """Dense 0/1 mask [n_masks, lq, lk] rebuilt from a format dict."""
    lib = _load()
    n_masks, lq0, lk0, bm, bn = (fmt[x] for x in ("n_masks", "lq", "lk", "bm", "bn"))
    lq, lk = -(-lq0 // bm) * bm, -(-lk0 // bn) * bn     # decoded on the padded sides, then cropped
    out = np.empty((n_masks, lq, lk), dtype=np.uint8)
    arrs = [np.ascontiguousarray(fmt[x], dtype=t) for x, t in (
        ("full_row_ptr", np.int32), ("full_col_idx", np.int32), ("part_row_ptr", np.int32),
        ("part_col_idx", np.int32), ("bitmaps", np.uint64))]
    arrs = [a if a.size else np.zeros(1, a.dtype) for a in arrs]
    rc = lib.stof_oracle_decode(n_masks, lq, lk, bm, bn, *[_ptr(a) for a in arrs], _ptr(out))
    if rc != 0:
        raise ValueError("oracle decode: bad shape")
    return out[:, :lq0, :lk0]


def attention_bhld(q, k, v, mask_of, scale: float, heads=None, rows=None,
                   n_threads: int | None = None) -> dict:
    """Multi-head helper.  q, k, v: float64 [B, H, L, d]; mask_of(b, h, rows)
    returns the uint8 mask rows [len(rows), L] of head (b, h).  Returns
    {(b, h): o [len(rows), d]} over `heads` (default: all) and `rows`
    (default: all)."""
    B, H, L, d = q.shape
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    rows = np.arange(L) if rows is None else np.asarray(rows)
    out = {}
    for (b, h) in heads:
        m = mask_of(b, h, rows)
        out[(b, h)] = attention(q[b, h, rows], k[b, h], v[b, h], m, scale, n_threads)
    return out


def oproj(o, w, bias=None, residual=None) -> np.ndarray:
    """y[b, l, n] = sum_{h, c} o[b, h, l, c] w[n, h d + c] + bias[n] + residual[b, l, n],
    fp64.  o: [B, H, L, d]; w: [N, H d]; bias: [N] or None; residual: [B, L, N] or None."""
    o = np.asarray(o, np.float64)
    B, H, L, d = o.shape
    o_cat = o.transpose(0, 2, 1, 3).reshape(B, L, H * d)   # token-major, heads side by side
    y = o_cat @ np.asarray(w, np.float64).T
    if bias is not None:
        y = y + np.asarray(bias, np.float64)
    if residual is not None:
        y = y + np.asarray(residual, np.float64)
    return y


def layer_norm(x, gamma=None, beta=None, eps: float = 1e-5) -> np.ndarray:
    """LayerNorm over the last axis, fp64: (x - mean) / sqrt(var + eps) * gamma
    + beta, with mean and var (population variance, divisor n) of each row;
    gamma, beta: [n] or None (1 and 0)."""
    x = np.asarray(x, np.float64)
    n = x.shape[-1]
    mean = x.sum(axis=-1, keepdims=True) / n
    dev = x - mean
    var = (dev * dev).sum(axis=-1, keepdims=True) / n
    y = dev / np.sqrt(var + eps)
    if gamma is not None:
        y = y * np.asarray(gamma, np.float64)
    if beta is not None:
        y = y + np.asarray(beta, np.float64)
    return y


def oproj_ln(o, w, bias=None, residual=None, gamma=None, beta=None, eps: float = 1e-5) -> np.ndarray:
    """layer_norm(oproj(o, w, bias, residual), gamma, beta, eps), fp64."""
    return layer_norm(oproj(o, w, bias, residual), gamma, beta, eps)


def unpack_bits(bits, lk: int) -> np.ndarray:
    """uint8 [..., lk / 8] -> uint8 [..., lk]: element 8 jb + c = bit c of byte jb."""
    bits = np.asarray(bits, np.uint8)
    out = np.zeros(bits.shape[:-1] + (lk,), np.uint8)
    for c in range(8):
        out[..., c::8] = (bits >> c) & 1
    return out


def rule_mask(lq: int, lk: int, band_lo: int, band_hi: int, global_rows=None, global_cols=None,
              blocks=None, block: int = 0, rows=None) -> np.ndarray:
    """uint8 [lq, lk]: element (i, j) is 1 iff band_lo <= i - j <= band_hi,
    or global_rows[i], or global_cols[j], or blocks[i // block, j // block]
    (bool arrays; None for an empty set).  With `rows`, only those query
    rows ([len(rows), lk])."""
    rows = np.arange(lq, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    i = rows[:, None]
    j = np.arange(lk, dtype=np.int64)[None, :]
    m = (i - j >= band_lo) & (i - j <= band_hi)
    if global_rows is not None:
        m = m | np.asarray(global_rows, bool)[rows][:, None]
    if global_cols is not None:
        m = m | np.asarray(global_cols, bool)[None, :]
    if blocks is not None:
        b = np.asarray(blocks, bool)
        m = m | b[i // block, j // block]
    return m.astype(np.uint8)
