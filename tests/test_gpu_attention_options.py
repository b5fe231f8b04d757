"""The block-wise kernels' two sampled softmax options against the fp64
oracle, and the exp split's FMA-pipe exp2 against exp2.

The exp split evaluates one key pair in eight with a polynomial exp2 on the
FMA pipe instead of the special-function unit; the four-warpgroup layout of
the persistent d = 64 kernel gives each softmax thread half a tile row and
swaps the halves' row max through shared memory.  Both are candidates of
the tuner's parameter sampling (gist.science technical summary,
Methodology 2, two-stage tuning, stage 2) and must compute the masked
softmax of the block-wise kernel (same page, Methodology 1, block-wise
kernel) within the same tolerance."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof, synth
from tests.conftest import TOL, gpu_encode

pytestmark = pytest.mark.gpu

# (d, ring depth, persistent, exp split, softmax warpgroups)
OPTIONS = [(64, 4, 1, 1, 0), (64, 4, 1, 0, 4), (64, 3, 0, 1, 0), (128, 3, 0, 1, 0)]


def test_fma_exp2_against_exp2(gpu_lib):
    """Relative error at most 3e-6 over the softmax's argument range
    [-125, 8] (the polynomial's 2.9e-6 plus fp32 rounding); exactly 2^k at
    integers, exactly 1 at 0, exactly 0 below -125 and at -inf."""
    x = np.concatenate([np.linspace(-125.0, 8.0, 4_000_001), np.arange(-125, 9)]).astype(np.float32)
    y = torch.empty(x.size, dtype=torch.float32, device="cuda")
    stof.stof_ex2_fma(torch.from_numpy(x).cuda(), y)
    got = y.cpu().numpy().astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(got - ref) / ref) <= 3e-6
    ints = np.arange(-125, 9)
    assert np.array_equal(got[-ints.size:], np.exp2(ints.astype(np.float64)))
    special = np.array([0.0, -0.0, -np.inf, -125.25, -126.0, -1000.0, -3.0e38], np.float32)
    ys = torch.empty(special.size, dtype=torch.float32, device="cuda")
    stof.stof_ex2_fma(torch.from_numpy(special).cuda(), ys)
    assert ys.cpu().tolist() == [1.0, 1.0, 0.0, 0.0, 0.0, 0.0, 0.0]


@pytest.mark.parametrize("d,stages,persistent,esplit,swg", OPTIONS)
@pytest.mark.parametrize("dtype,sign", [("fp16", 1.0), ("bf16", 1.0), ("fp16", -1.0)])
@pytest.mark.parametrize("L", [128, 640])
def test_options_match_the_oracle(gpu_lib, d, stages, persistent, esplit, swg, dtype, sign, L):
    """Per-head masks with a fully masked row, a row with a single valid key,
    a query tile without listed OTs (L = 640), all-full OTs next to partial
    ones; negative scale included; with L = 128 every query tile has one
    listed OT, so one pair of warpgroups has no tile of the item."""
    B, H = 1, 3
    rng = np.random.default_rng(L + d + 10 * esplit + swg + (5 if sign < 0 else 0) + (7 if dtype == "bf16" else 0))
    masks = (rng.random((B * H, L, L)) < 0.3).astype(np.uint8)
    masks[0, :, : min(L, 256)] = 1                      # full OTs in head 0
    masks[1, 5] = 0                                     # fully masked row
    masks[1, 9] = 0
    masks[1, 9, 77] = 1                                 # a single valid key
    if L > 128:
        masks[2, 128:256] = 0                           # a query tile without listed OTs
    q, k, v = synth.make_qkv(B, H, L, d, dtype, seed=17)
    fmt, ws, _ = gpu_encode(torch.from_numpy(masks).cuda(), 128, 128)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qd, float("nan"))
    scale = sign / math.sqrt(d)
    plan = stof.stof_plan(stof.STOF_KERNEL_BLOCKWISE, stages, persistent, 0, 0, esplit, swg)
    stof.stof_mha_fwd_plan(qd, kd, vd, fmt, scale, H, 1, plan, o)
    torch.cuda.synchronize()
    stof.stof_format_sync(fmt)
    assert fmt.device_error == 0
    q64, k64, v64 = (synth.to_float64(t) for t in (q, k, v))
    ref = oracle.attention_bhld(q64, k64, v64, lambda b, h, rows: masks[b * H + h][rows], scale)
    for (b, h), o_ref in ref.items():
        assert np.abs(o[b, h].double().cpu().numpy() - o_ref).max() <= TOL[dtype]
    assert torch.all(o[0, 1, 5] == 0)
    assert torch.allclose(o[0, 1, 9].float(), vd[0, 1, 77].float())
    if L > 128:
        assert torch.all(o[0, 2, 128:256] == 0)


def test_four_warpgroups_over_many_items(gpu_lib):
    """The four-warpgroup persistent kernel with more query tiles than SMs
    and items of 1 to 40 listed OTs (causal, L = 5120), sampled heads and rows
    against the oracle; and the same P as the default layout, the row sums
    added in another order: outputs within one bf16 step of each other, or
    1e-5 apart where the merge of the two pairs' partial outputs cancels."""
    B, H, L, d = 1, 4, 5120, 64
    mask = np.tril(np.ones((L, L), np.uint8))[None]
    q, k, v = synth.make_qkv(B, H, L, d, "bf16", seed=23)
    fmt, ws, _ = gpu_encode(torch.from_numpy(mask).cuda(), 128, 128)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    outs = []
    for swg in (0, 4):
        o = torch.full_like(qd, float("nan"))
        stof.stof_mha_fwd_plan(qd, kd, vd, fmt, 0.125, 0, 0, stof.stof_plan(1, 4, 1, 0, 0, 0, swg), o)
        outs.append(o)
    torch.cuda.synchronize()
    stof.stof_format_sync(fmt)
    assert fmt.device_error == 0
    a, b = outs[0].float(), outs[1].float()
    assert torch.all((a - b).abs() <= torch.maximum(a.abs(), b.abs()) * 2 ** -7 + 1e-5)
    rows = np.unique(np.concatenate([np.arange(130), np.arange(L - 130, L), np.random.default_rng(3).choice(L, 200)]))
    q64, k64, v64 = (synth.to_float64(t) for t in (q, k, v))
    ref = oracle.attention_bhld(q64, k64, v64, lambda b, h, r: mask[0][r], 0.125, heads=[(0, 0), (0, 3)], rows=rows)
    for (b, h), o_ref in ref.items():
        assert np.abs(outs[1][b, h, rows].double().cpu().numpy() - o_ref).max() <= TOL["bf16"]
