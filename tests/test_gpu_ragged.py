"""Sequence lengths that are not a whole number of outer tiles.

The two-level format tiles the whole matrix with BM x BN outer tiles
("Accelerating Sparse Transformer Inference on GPU", gist.science technical
summary, Methodology 1, two-level storage format); a side that is not a
whole number of tiles is read as padded to one with invalid elements.  The
encoders must then give, bit for bit, the oracle's encoding of the padded
mask (so the last OT row and column are never full), and every attention
kernel must match the oracle on the L real rows and write nothing past them."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof, synth
from tests.conftest import TOL, assert_format_equal, gpu_encode

pytestmark = pytest.mark.gpu

# lk % 16 == 0 (16-byte loads), lk % 8 == 0 (8-byte loads), odd lk (byte loads)
SHAPES = [(250, 256), (256, 1000), (1000, 1000), (77, 77), (129, 200), (8, 9), (1, 1), (300, 1024 + 8)]


@pytest.mark.parametrize("lq,lk", SHAPES)
@pytest.mark.parametrize("bm,bn", [(128, 128), (64, 128), (16, 16), (24, 40)])
def test_dense_encoder_pads_to_whole_tiles(gpu_lib, lq, lk, bm, bn):
    rng = np.random.default_rng(lq * 7 + lk + bm + bn)
    masks = (rng.random((3, lq, lk)) < 0.3).astype(np.uint8)
    masks[0] = 1                                           # every element valid: edge OTs still partial
    masks[1, :, : lk // 2] = 0
    fmt, ws, arrs = gpu_encode(torch.from_numpy(masks).cuda(), bm, bn)
    want = oracle.encode(masks, bm, bn)
    assert (fmt.n_tr, fmt.n_tc, fmt.lq, fmt.lk) == (want["n_tr"], want["n_tc"], lq, lk)
    assert_format_equal(fmt, arrs, want)
    assert fmt.nnz == int(masks.sum())
    # an OT that reaches past a side is never full
    n_tr, n_tc = want["n_tr"], want["n_tc"]
    frp, fci = arrs["full_row_ptr"], arrs["full_col_idx"]
    for row in range(3 * n_tr):
        I = row % n_tr
        cols = fci[frp[row]:frp[row + 1]]
        if (I + 1) * bm > lq:
            assert cols.size == 0
        assert not np.any((cols + 1) * bn > lk)


@pytest.mark.parametrize("lq,lk", [(250, 256), (1000, 1000), (77, 130), (1, 1)])
def test_rule_encoder_pads_to_whole_tiles(gpu_lib, lq, lk):
    rng = np.random.default_rng(lq + 3 * lk)
    rules = [
        {"band_lo": 0, "band_hi": 40, "global_rows": rng.random(lq) < 0.05, "global_cols": rng.random(lk) < 0.05,
         "blocks": None, "block": 0},
        {"band_lo": -(1 << 31), "band_hi": (1 << 31) - 1, "global_rows": None, "global_cols": None, "blocks": None,
         "block": 0},
    ]
    bits = lambda a: None if a is None else stof.bitset_words(a)  # noqa: E731
    dev = [stof.MaskRule(r["band_lo"], r["band_hi"], bits(r["global_rows"]), bits(r["global_cols"]), None, 0)
           for r in rules]
    ws = torch.empty(stof.stof_encode_workspace_bytes(2, lq, lk, 128, 128), dtype=torch.uint8, device="cuda")
    fmt = stof.stof_encode_rules(dev, lq, lk, 128, 128, ws)
    stof.stof_format_sync(fmt)
    arrs = {k: v.cpu().numpy() for k, v in stof.format_arrays(fmt, ws).items()}
    arrs["bitmaps"] = arrs["bitmaps"].view("uint64")
    want = oracle.encode(np.stack([oracle.rule_mask(lq, lk, **r) for r in rules]), 128, 128)
    assert_format_equal(fmt, arrs, want)


@pytest.mark.parametrize("lq,lk", [(250, 256), (1000, 1000), (77, 136), (1, 8), (129, 2056)])
@pytest.mark.parametrize("bm,bn", [(128, 128), (64, 128), (16, 16)])
def test_bit_packed_encoder_pads_to_whole_tiles(gpu_lib, lq, lk, bm, bn):
    """The bit-packed encoder on sides that are not whole OTs (lk a multiple
    of 8, so a row is lk / 8 whole bytes): the same format as the oracle's
    encoding of the padded dense mask."""
    rng = np.random.default_rng(lq + lk + bm)
    masks = (rng.random((2, lq, lk)) < 0.4).astype(np.uint8)
    masks[0] = 1
    bits = torch.from_numpy(np.packbits(masks, axis=2, bitorder="little")).cuda()
    ws = torch.empty(stof.stof_encode_workspace_bytes(2, lq, lk, bm, bn), dtype=torch.uint8, device="cuda")
    fmt = stof.stof_encode_mask_bits(bits, lk, bm, bn, ws)
    stof.stof_format_sync(fmt)
    arrs = {k: v.cpu().numpy() for k, v in stof.format_arrays(fmt, ws).items()}
    arrs["bitmaps"] = arrs["bitmaps"].view("uint64")
    assert_format_equal(fmt, arrs, oracle.encode(masks, bm, bn))


def test_bit_packed_rows_must_be_whole_bytes(gpu_lib):
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(stof.StofError) as e:
        stof.stof_encode_mask_bits(torch.zeros(1, 64, 9, dtype=torch.uint8, device="cuda"), 77, 16, 16, ws)
    assert e.value.status == stof.STOF_ERR_SHAPE


# (kernel, plan) pairs: the row-wise kernel, the block-wise kernel one CTA per
# query tile, and (d = 64) persistent with two and with four softmax warpgroups
def _plans(d):
    out = [("row", stof.stof_plan(stof.STOF_KERNEL_ROWWISE, 0, 0, 0, 0)),
           ("tile", stof.stof_plan(stof.STOF_KERNEL_BLOCKWISE, 3, 0, 0, 0))]
    if d == 64:
        out += [("persist", stof.stof_plan(stof.STOF_KERNEL_BLOCKWISE, 4, 1, 0, 0)),
                ("persist4", stof.stof_plan(stof.STOF_KERNEL_BLOCKWISE, 4, 1, 0, 0, 0, 4))]
    return out


@pytest.mark.parametrize("L", [1, 9, 77, 200, 1000, 1100])
@pytest.mark.parametrize("d", [64, 128])
def test_attention_on_ragged_lengths(gpu_lib, L, d):
    """Per-head masks (causal with random holes, a fully masked row, one
    head fully valid) on L real rows; outputs against the oracle for every
    head and row, and a NaN guard after the last head's rows stays as it
    was (nothing is written past the tensor)."""
    B, H = 1, 3
    rng = np.random.default_rng(L + d)
    masks = (rng.random((H, L, L)) < 0.4).astype(np.uint8) * np.tril(np.ones((L, L), np.uint8))[None]
    masks[:, np.arange(L), np.arange(L)] = 1
    masks[2] = 1
    if L > 5:
        masks[1, 5] = 0
    q, k, v = synth.make_qkv(B, H, L, d, "bf16", seed=L)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    scale = 1 / math.sqrt(d)
    q64, k64, v64 = (synth.to_float64(t) for t in (q, k, v))
    ref = oracle.attention_bhld(q64, k64, v64, lambda b, h, rows: masks[h][rows], scale)
    guard = 4096
    for name, plan in _plans(d):
        fmt, ws, _ = gpu_encode(torch.from_numpy(masks).cuda(), 128, 128)
        buf = torch.full((B * H * L * d + guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
        o = buf[: B * H * L * d].view(B, H, L, d)
        stof.stof_mha_fwd_plan(qd, kd, vd, fmt, scale, 0, 1, plan, o)
        torch.cuda.synchronize()
        stof.stof_format_sync(fmt)
        assert fmt.device_error == 0, name
        assert torch.isnan(buf[B * H * L * d:]).all(), name
        for (b, h), o_ref in ref.items():
            assert np.abs(o[b, h].double().cpu().numpy() - o_ref).max() <= TOL["bf16"], (name, h)
        if L > 5:
            assert torch.all(o[0, 1, 5] == 0), name


def test_ragged_length_auto_and_tuned(gpu_lib):
    """AUTO on a ragged length (analytic, then after stof_tune) matches the
    oracle, and the tuner admits its candidates there."""
    B, H, L, d = 1, 2, 1000, 64
    mask = np.tril(np.ones((L, L), np.uint8))[None]
    q, k, v = synth.make_qkv(B, H, L, d, "fp16", seed=4)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    mdev = torch.from_numpy(mask).cuda()
    fmt, ws, _ = gpu_encode(mdev, 128, 128)
    q64, k64, v64 = (synth.to_float64(t) for t in (q, k, v))
    ref = oracle.attention_bhld(q64, k64, v64, lambda b, h, rows: mask[0][rows], 0.125)
    stof.stof_tune_clear()
    for tuned in (False, True):
        if tuned:
            wst = torch.empty(stof.stof_tune_workspace_bytes(1, L), dtype=torch.uint8, device="cuda")
            res = stof.stof_tune(mdev, qd, kd, vd, 0.125, 0, 0, wst, torch.empty_like(qd))
            assert sum(t > 0 for t in res.cand_ms) >= 10
        o = torch.full_like(qd, float("nan"))
        stof.stof_mha_fwd(qd, kd, vd, fmt, 0.125, 0, 0, stof.STOF_KERNEL_AUTO, o)
        torch.cuda.synchronize()
        for (b, h), o_ref in ref.items():
            assert np.abs(o[b, h].double().cpu().numpy() - o_ref).max() <= TOL["fp16"]
    stof.stof_tune_clear()
