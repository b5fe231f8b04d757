"""GPU encoder from parametric masks (stof_encode_rules) against the
brute-force oracle encoder applied to the dense mask the rule defines:
bit-exact pointer arrays, tile lists and bitmaps.  Mask families from
"Accelerating Sparse Transformer Inference on GPU" (gist.science technical
summary, Problem statement and Experimental results: causal, sliding
window, Longformer, BigBird)."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof, synth
from tests.conftest import assert_format_equal

pytestmark = pytest.mark.gpu

I32_MAX = (1 << 31) - 1
I32_MIN = -(1 << 31)


def _rule_dev(rule):
    """numpy rule dict -> MaskRule with device bitsets (the tensors are kept on the object)."""
    bits = lambda a: None if a is None else stof.bitset_words(a)  # noqa: E731
    return stof.MaskRule(rule["band_lo"], rule["band_hi"], bits(rule.get("global_rows")),
                         bits(rule.get("global_cols")), bits(rule.get("blocks")), rule.get("block", 0))


def _encode_rules(rules, lq, lk, bm, bn):
    ws = torch.empty(stof.stof_encode_workspace_bytes(len(rules), lq, lk, bm, bn), dtype=torch.uint8,
                     device="cuda")
    dev = [_rule_dev(r) for r in rules]
    fmt = stof.stof_encode_rules(dev, lq, lk, bm, bn, ws)
    stof.stof_format_sync(fmt)
    arrs = {k: v.cpu().numpy() for k, v in stof.format_arrays(fmt, ws).items()}
    arrs["bitmaps"] = arrs["bitmaps"].view("uint64")
    return fmt, ws, arrs


def _oracle_masks(rules, lq, lk):
    return np.stack([oracle.rule_mask(lq, lk, **r) for r in rules])


def _random_rule(rng, lq, lk, block):
    lo = int(rng.integers(-lk, lq))
    r = {"band_lo": lo, "band_hi": lo + int(rng.integers(-3, 200)), "global_rows": None, "global_cols": None,
         "blocks": None, "block": 0}
    if rng.random() < 0.5:
        r["global_rows"] = rng.random(lq) < 0.03
    if rng.random() < 0.5:
        r["global_cols"] = rng.random(lk) < 0.03
    if rng.random() < 0.5:
        r["blocks"] = rng.random((lq // block, lk // block)) < 0.15
        r["block"] = block
    return r


@pytest.mark.parametrize("name", ["window48_L256", "bigbird_L512", "causal_L2048", "longformer_L4096"])
@pytest.mark.parametrize("ot", [128, 64, 16])
def test_workload_rules_bit_exact(gpu_lib, name, ot):
    w = synth.WORKLOADS[name]
    fmt, ws, arrs = _encode_rules([synth.workload_rule(w)], w.L, w.L, ot, ot)
    assert_format_equal(fmt, arrs, oracle.encode(synth.make_mask(w), ot, ot))


@pytest.mark.parametrize("bm,bn", [(8, 8), (16, 16), (8, 16), (24, 8), (32, 64), (128, 128), (256, 256),
                                   (128, 64), (40, 200)])
@pytest.mark.parametrize("seed", [0, 1])
def test_random_rules_bit_exact(gpu_lib, bm, bn, seed):
    rng = np.random.default_rng(100 * seed + bm + bn)
    block = math.gcd(math.lcm(bm, 8), math.lcm(bn, 8))          # a block edge dividing both sizes
    lq, lk = bm * 5, bn * 7
    lq, lk = math.lcm(lq, block), math.lcm(lk, block)
    rules = [_random_rule(rng, lq, lk, block) for _ in range(3)]
    fmt, ws, arrs = _encode_rules(rules, lq, lk, bm, bn)
    assert_format_equal(fmt, arrs, oracle.encode(_oracle_masks(rules, lq, lk), bm, bn))


def test_band_extremes_and_empty_rules(gpu_lib):
    L = 512
    rules = [
        {"band_lo": I32_MIN, "band_hi": I32_MAX},            # everything valid: all full tiles
        {"band_lo": 1, "band_hi": 0},                        # nothing valid: no tiles
        {"band_lo": 0, "band_hi": I32_MAX},                  # causal
        {"band_lo": I32_MIN, "band_hi": -1},                 # strictly upper triangle
        {"band_lo": L, "band_hi": I32_MAX},                  # band entirely outside the matrix
    ]
    rules = [dict(global_rows=None, global_cols=None, blocks=None, block=0, **r) for r in rules]
    fmt, ws, arrs = _encode_rules(rules, L, L, 128, 128)
    want = oracle.encode(_oracle_masks(rules, L, L), 128, 128)
    assert_format_equal(fmt, arrs, want)
    assert fmt.n_full > 0 and fmt.nnz == L * L + L * (L + 1) // 2 + L * (L - 1) // 2


def test_long_sequence_rules_need_no_mask(gpu_lib):
    """An 8192-long Longformer-style rule (window +-256, 64 global tokens) and
    BigBird-style 64-blocks, with no 64 MB mask anywhere on the device."""
    L = 8192
    rng = np.random.default_rng(7)
    g = np.zeros(L, bool)
    g[rng.choice(L, 64, replace=False)] = True
    rules = [{"band_lo": -256, "band_hi": 256, "global_rows": g, "global_cols": g, "blocks": None, "block": 0},
             {"band_lo": 0, "band_hi": 63, "global_rows": None, "global_cols": None,
              "blocks": rng.random((L // 64, L // 64)) < 0.01, "block": 64}]
    fmt, ws, arrs = _encode_rules(rules, L, L, 128, 128)
    assert_format_equal(fmt, arrs, oracle.encode(_oracle_masks(rules, L, L), 128, 128))


def test_attention_from_rules_equals_attention_from_the_dense_mask(gpu_lib):
    w = synth.WORKLOADS["longformer_L4096"]
    mask = torch.from_numpy(synth.make_mask(w)).cuda()
    ws_d = torch.empty(stof.stof_encode_workspace_bytes(1, w.L, w.L, 128, 128), dtype=torch.uint8, device="cuda")
    fd = stof.stof_encode_mask(mask, 128, 128, ws_d)
    stof.stof_format_sync(fd)
    fr, ws_r, _ = _encode_rules([synth.workload_rule(w)], w.L, w.L, 128, 128)
    q, k, v = (t[:1, :4].contiguous().cuda() for t in synth.make_qkv(w.B, w.H, w.L, w.d, w.dtype, seed=w.seed))
    outs = []
    for f in (fd, fr):
        o = torch.empty_like(q)
        stof.stof_mha_fwd(q, k, v, f, 1 / math.sqrt(w.d), 0, 0, stof.STOF_KERNEL_BLOCKWISE, o)
        outs.append(o)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


def test_rules_differ_per_mask_and_heads_pick_their_mask(gpu_lib):
    """Two heads with different rules (mask_stride_h = 1): each head's output
    equals the oracle attention under its own rule."""
    L, d = 256, 64
    rules = [{"band_lo": 0, "band_hi": 31, "global_rows": None, "global_cols": None, "blocks": None, "block": 0},
             {"band_lo": -40, "band_hi": 40, "global_rows": None, "global_cols": np.arange(L) % 50 == 0,
              "blocks": None, "block": 0}]
    fmt, ws, _ = _encode_rules(rules, L, L, 128, 128)
    q, k, v = synth.make_qkv(1, 2, L, d, "fp16", seed=3)
    o = torch.empty_like(q).cuda()
    stof.stof_mha_fwd(q.cuda(), k.cuda(), v.cuda(), fmt, 0.125, 0, 1, stof.STOF_KERNEL_BLOCKWISE, o)
    torch.cuda.synchronize()
    masks = _oracle_masks(rules, L, L)
    qf, kf, vf = (synth.to_float64(t) for t in (q, k, v))
    for h in range(2):
        ref = oracle.attention(qf[0, h], kf[0, h], vf[0, h], masks[h], 0.125)
        assert np.abs(o[0, h].double().cpu().numpy() - ref).max() <= 2e-3


def test_maximum_rule_count(gpu_lib):
    """STOF_MAX_RULES (64) masks, each with its own rule."""
    rng = np.random.default_rng(64)
    L, blk = 256, 32
    rules = [_random_rule(rng, L, L, blk) for _ in range(stof.STOF_MAX_RULES)]
    fmt, ws, arrs = _encode_rules(rules, L, L, 64, 64)
    assert_format_equal(fmt, arrs, oracle.encode(_oracle_masks(rules, L, L), 64, 64))


@pytest.mark.parametrize("kern", ["block", "row"])
def test_64k_tokens_from_a_rule(gpu_lib, kern):
    """A 65,536-token causal sliding window (4096 keys) with 16 global
    tokens, two heads, d = 128: the mask would be 4 GB as bytes and is never
    materialised.  Sampled OT rows of the format bit-exact against the
    oracle's encoding of the same rows; sampled query rows of O against the
    oracle (the first, the last and seeded others)."""
    L, H, d = 65536, 2, 128
    rng = np.random.default_rng(64)
    g = np.zeros(L, bool)
    g[rng.choice(L, 16, replace=False)] = True
    rule = {"band_lo": 0, "band_hi": 4095, "global_rows": g, "global_cols": g, "blocks": None, "block": 0}
    fmt, ws, arrs = _encode_rules([rule], L, L, 128, 128)
    frp, prp = arrs["full_row_ptr"], arrs["part_row_ptr"]
    for I in [0, 1, 31, 32, 511] + [int(x) for x in rng.choice(512, 4, replace=False)]:
        want = oracle.encode(oracle.rule_mask(L, L, rows=np.arange(I * 128, I * 128 + 128), **rule)[None], 128, 128)
        assert frp[I + 1] - frp[I] == want["n_full"] and prp[I + 1] - prp[I] == want["n_part"]
        assert np.array_equal(arrs["full_col_idx"][frp[I]:frp[I + 1]], want["full_col_idx"])
        assert np.array_equal(arrs["part_col_idx"][prp[I]:prp[I + 1]], want["part_col_idx"])
        assert np.array_equal(arrs["bitmaps"][prp[I]:prp[I + 1]], want["bitmaps"])
    q, k, v = synth.make_qkv(1, H, L, d, "bf16", seed=65)
    o = torch.full((1, H, L, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    which = stof.STOF_KERNEL_BLOCKWISE if kern == "block" else stof.STOF_KERNEL_ROWWISE
    stof.stof_mha_fwd(q.cuda(), k.cuda(), v.cuda(), fmt, 1 / math.sqrt(d), 0, 0, which, o)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(32), rng.choice(L, 96, replace=False), np.arange(L - 32, L),
                                     np.flatnonzero(g)]))
    q64, k64, v64 = (synth.to_float64(t) for t in (q, k, v))
    ref = oracle.attention_bhld(q64, k64, v64, lambda b, h, r: oracle.rule_mask(L, L, rows=r, **rule),
                                1 / math.sqrt(d), rows=rows)
    og = o.double().cpu().numpy()
    for (b, h), o_ref in ref.items():
        assert np.abs(og[b, h, rows] - o_ref).max() <= 1.5e-2
