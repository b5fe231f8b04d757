"""Seeded random configurations of the encoders against the oracle's
brute-force encoder: mask counts, lengths (whole tiles or not, Lq != Lk),
OT shapes from 8 to 256, densities from empty to full with full rows and
columns mixed in, and every input path -- the dense mask in device memory,
in pinned host memory, through the no-allocation entry point, and
bit-packed when Lk is a multiple of 8 -- and random parametric rules on
such lengths.  Each format must equal the oracle's bit for bit
("Accelerating Sparse Transformer Inference on GPU", gist.science
technical summary, Methodology 1, two-level storage format)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof
from tests.conftest import assert_format_equal

pytestmark = pytest.mark.gpu

N_CASES = 40
SIDES = [8, 16, 24, 32, 40, 64, 96, 128, 136, 200, 256]


def _case(seed):
    rng = np.random.default_rng(5000 + seed)
    n = int(rng.integers(1, 4))
    lq = int(rng.integers(1, 700))
    lk = lq if rng.random() < 0.4 else int(rng.integers(1, 700))
    if rng.random() < 0.5:
        lk = max(8, lk - lk % 8)  # bit-packed input possible
    bm, bn = int(rng.choice(SIDES)), int(rng.choice(SIDES))
    density = float(rng.choice([0.0, 0.01, 0.3, 0.9, 1.0]))
    mask = (rng.random((n, lq, lk)) < density).astype(np.uint8)
    for _ in range(int(rng.integers(0, 4))):  # whole rows and columns, so full OTs occur
        m, i, j = int(rng.integers(n)), int(rng.integers(lq)), int(rng.integers(lk))
        mask[m, max(0, i - 40):i + 40, :] = 1
        mask[m, :, max(0, j - 40):j + 40] = 1
    return mask, bm, bn


def _noalloc(mask, bm, bn, ws):
    fn = stof.load_library().stof_encode_mask_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(stof.stof_format), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    n, lq, lk = mask.shape
    fmt = stof.stof_format()
    status = fn(mask.data_ptr(), n, lq, lk, bm, bn, ws.data_ptr(), ws.numel(), ctypes.byref(fmt),
                torch.cuda.current_stream().cuda_stream)
    assert status == stof.STOF_OK, stof.stof_status_string(status)
    return fmt


def _arrays(fmt, ws):
    stof.stof_format_sync(fmt)
    arrs = {k: v.cpu().numpy() for k, v in stof.format_arrays(fmt, ws).items()}
    arrs["bitmaps"] = arrs["bitmaps"].view("uint64")
    return arrs


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_encoder_configuration(gpu_lib, seed):
    mask, bm, bn = _case(seed)
    n, lq, lk = mask.shape
    want = oracle.encode(mask, bm, bn)
    ws_bytes = stof.stof_encode_workspace_bytes(n, lq, lk, bm, bn)
    dev = torch.from_numpy(mask).cuda()
    host = torch.empty(mask.shape, dtype=torch.uint8, pin_memory=True)
    host.copy_(torch.from_numpy(mask))
    paths = {"device": lambda ws: stof.stof_encode_mask(dev, bm, bn, ws),
             "host": lambda ws: stof.stof_encode_mask(host, bm, bn, ws),
             "noalloc": lambda ws: _noalloc(dev, bm, bn, ws)}
    if lk % 8 == 0:
        bits = torch.from_numpy(np.ascontiguousarray(np.packbits(mask != 0, axis=-1, bitorder="little"))).cuda()
        paths["bits"] = lambda ws: stof.stof_encode_mask_bits(bits, lk, bm, bn, ws)
    for name, encode in paths.items():
        ws = torch.full((ws_bytes,), 0x5A, dtype=torch.uint8, device="cuda")
        fmt = encode(ws)
        arrs = _arrays(fmt, ws)
        try:
            assert_format_equal(fmt, arrs, want)
        except AssertionError as e:
            raise AssertionError(f"{name} path, mask {mask.shape}, OT {bm}x{bn}: {e}") from e


N_RULE_CASES = 24


def _rule_case(seed):
    """Random rules (band, global rows and columns, and a block pattern when a
    block edge divides both lengths) on lengths that need not be whole OTs."""
    rng = np.random.default_rng(7000 + seed)
    n = int(rng.integers(1, 4))
    lq, lk = int(rng.integers(1, 900)), int(rng.integers(1, 900))
    if rng.random() < 0.4:
        lq, lk = 8 * max(1, lq // 8), 8 * max(1, lk // 8)
    bm, bn = int(rng.choice(SIDES)), int(rng.choice(SIDES))
    blocks = [b for b in (8, 16, 24, 32, 64) if lq % b == 0 and lk % b == 0]
    rules = []
    for _ in range(n):
        lo = int(rng.integers(-lk, lq))
        r = {"band_lo": lo, "band_hi": lo + int(rng.integers(-3, 300)), "global_rows": None, "global_cols": None,
             "blocks": None, "block": 0}
        if rng.random() < 0.5:
            r["global_rows"] = rng.random(lq) < 0.03
        if rng.random() < 0.5:
            r["global_cols"] = rng.random(lk) < 0.03
        if blocks and rng.random() < 0.5:
            blk = int(rng.choice(blocks))
            r["blocks"], r["block"] = rng.random((lq // blk, lk // blk)) < 0.15, blk
        rules.append(r)
    return rules, lq, lk, bm, bn


@pytest.mark.parametrize("seed", range(N_RULE_CASES))
def test_random_rule_configuration(gpu_lib, seed):
    rules, lq, lk, bm, bn = _rule_case(seed)
    bits = lambda a: None if a is None else stof.bitset_words(a)  # noqa: E731
    dev = [stof.MaskRule(r["band_lo"], r["band_hi"], bits(r["global_rows"]), bits(r["global_cols"]),
                         bits(r["blocks"]), r["block"]) for r in rules]
    ws = torch.full((stof.stof_encode_workspace_bytes(len(rules), lq, lk, bm, bn),), 0x5A, dtype=torch.uint8,
                    device="cuda")
    fmt = stof.stof_encode_rules(dev, lq, lk, bm, bn, ws)
    masks = np.stack([oracle.rule_mask(lq, lk, **r) for r in rules])
    assert_format_equal(fmt, _arrays(fmt, ws), oracle.encode(masks, bm, bn))
