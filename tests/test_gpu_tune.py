"""Measured parameter choice with a result cache (gist.science technical
summary, Methodology 2, two-stage tuning, stage 2 "parameter sampling":
kernel parameters are sampled by running them and the outcomes cached).
The candidates are the row-wise kernel on 128x128 OTs with 1, 2 or 4 rows
per warp and the block-wise kernel on 128x128 OTs with ring depths 2-4, one
CTA per query tile or persistent CTAs (d = 64), the exp split, four softmax
warpgroups (persistent, d = 64), and on 128x64 OTs; the chosen one must also
be correct, and stof_mha_fwd(AUTO) must run it once it is cached."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof, synth
from tests.conftest import TOL, gpu_encode

pytestmark = pytest.mark.gpu


def test_tune_picks_the_fastest_candidate_and_caches_it(gpu_lib):
    B, H, L, d = 1, 4, 1024, 64
    mask = np.tril(np.ones((L, L), np.uint8))[None]          # causal, shared by the heads
    q, k, v = synth.make_qkv(B, H, L, d, "bf16", seed=8)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qd)
    mdev = torch.from_numpy(mask).cuda()
    ws = torch.empty(stof.stof_tune_workspace_bytes(1, L), dtype=torch.uint8, device="cuda")
    stof.stof_tune_clear()
    res = stof.stof_tune(mdev, qd, kd, vd, 1 / math.sqrt(d), 0, 0, ws, o)
    ms = list(res.cand_ms)
    assert all(t > 0 for t in ms)                            # d = 64 admits every candidate
    assert list(res.cand_stages) == [0, 0, 0, 3, 2, 4, 4, 3, 2, 4, 3, 4, 4]
    # 128x64: 9 OTs per row -> persistent
    assert list(res.cand_persistent) == [0, 0, 0, 0, 0, 0, 1, 1, 1, 1, 0, 1, 1]
    assert list(res.cand_rows_per_warp) == [1, 2, 4] + [0] * 10
    assert list(res.cand_exp_split) == [0] * 10 + [1, 1, 0]
    assert list(res.cand_softmax_warpgroups) == [0, 0, 0] + [2] * 9 + [4]
    best = int(np.argmin(ms))
    assert res.kernel == res.cand_kernel[best] and res.bn == res.cand_bn[best]
    assert res.stages == res.cand_stages[best] and res.persistent == res.cand_persistent[best]
    assert res.rows_per_warp == res.cand_rows_per_warp[best]
    assert res.exp_split == res.cand_exp_split[best]
    assert res.softmax_warpgroups == res.cand_softmax_warpgroups[best]
    assert res.ms == pytest.approx(ms[best])
    assert res.density == pytest.approx((L + 1) / (2 * L))
    hit = stof.stof_tune_lookup(L, d, res.density * 1.05)    # same half-octave bucket
    assert hit is not None and hit.kernel == res.kernel and hit.bn == res.bn
    assert stof.stof_tune_lookup(2 * L, d, res.density) is None
    assert stof.stof_tune_lookup(L, 128, res.density) is None
    # the chosen configuration computes the right thing
    fmt, ws2, _ = gpu_encode(mdev, 128, res.bn)
    o2 = torch.full_like(qd, float("nan"))
    stof.stof_mha_fwd(qd, kd, vd, fmt, 1 / math.sqrt(d), 0, 0, res.kernel, o2)
    torch.cuda.synchronize()
    q64, k64, v64 = (synth.to_float64(t) for t in (q, k, v))
    ref = oracle.attention_bhld(q64, k64, v64, lambda b, h, rows: mask[0][rows], 1 / math.sqrt(d),
                                heads=[(0, 0), (0, 3)])
    for (b, h), o_ref in ref.items():
        assert np.abs(o2[b, h].double().cpu().numpy() - o_ref).max() <= TOL["bf16"]
    stof.stof_tune_clear()
    assert stof.stof_tune_lookup(L, d, res.density) is None


@pytest.mark.parametrize("d", [64, 128])
def test_auto_runs_the_cached_measurement(gpu_lib, d):
    """Without a cache entry AUTO follows the analytic model; after stof_tune
    it runs the fastest measured candidate on the format's OT width (kernel,
    ring depth, variant), and the result still matches the oracle."""
    B, H, L = 1, 2, 512
    mask = synth.random_mask(1, L, L, 0.05, seed=77)
    q, k, v = synth.make_qkv(B, H, L, d, "fp16", seed=78)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    mdev = torch.from_numpy(mask).cuda()
    scale = 1 / math.sqrt(d)
    fmt, ws, _ = gpu_encode(mdev, 128, 128)
    stof.stof_tune_clear()
    plan = stof.stof_mha_plan(fmt, B, H, L, d, stof.STOF_KERNEL_AUTO)
    density = fmt.nnz / (L * L)
    assert plan.source == stof.STOF_PLAN_ANALYTIC and plan.kernel == stof.stof_select_kernel(density, L, d)
    o = torch.empty_like(qd)
    wst = torch.empty(stof.stof_tune_workspace_bytes(1, L), dtype=torch.uint8, device="cuda")
    res = stof.stof_tune(mdev, qd, kd, vd, scale, 0, 0, wst, o)
    ms = [t if (t > 0 and res.cand_bn[i] == 128) else float("inf") for i, t in enumerate(res.cand_ms)]
    best = int(np.argmin(ms))
    if d == 128:
        assert all(res.cand_ms[i] < 0 for i in (5, 6, 7, 8, 11, 12))    # d = 64-only candidates
    plan = stof.stof_mha_plan(fmt, B, H, L, d, stof.STOF_KERNEL_AUTO)
    assert plan.source == stof.STOF_PLAN_TUNED
    assert plan.kernel == res.cand_kernel[best]
    if plan.kernel == stof.STOF_KERNEL_BLOCKWISE:
        assert (plan.stages, plan.persistent) == (res.cand_stages[best], res.cand_persistent[best])
        assert (plan.exp_split, plan.softmax_warpgroups) == (res.cand_exp_split[best],
                                                             res.cand_softmax_warpgroups[best])
    else:
        assert plan.rows_per_warp == res.cand_rows_per_warp[best]
    o2 = torch.full_like(qd, float("nan"))
    stof.stof_mha_fwd(qd, kd, vd, fmt, scale, 0, 0, stof.STOF_KERNEL_AUTO, o2)
    torch.cuda.synchronize()
    q64, k64, v64 = (synth.to_float64(t) for t in (q, k, v))
    ref = oracle.attention_bhld(q64, k64, v64, lambda b, h, rows: mask[0][rows], scale)
    for (b, h), o_ref in ref.items():
        assert np.abs(o2[b, h].double().cpu().numpy() - o_ref).max() <= TOL["fp16"]
    stof.stof_tune_clear()
    assert stof.stof_mha_plan(fmt, B, H, L, d, stof.STOF_KERNEL_AUTO).source == stof.STOF_PLAN_ANALYTIC


@pytest.mark.parametrize("d,stages,persistent,esplit,swg", [
    (64, 2, 0, 0, 0), (64, 3, 0, 0, 0), (64, 4, 0, 0, 0), (64, 2, 1, 0, 0), (64, 3, 1, 0, 0), (64, 4, 1, 0, 0),
    (128, 2, 0, 0, 0), (128, 3, 0, 0, 0),
    (64, 3, 0, 1, 0), (64, 4, 1, 1, 0), (128, 3, 0, 1, 0),       # exp split
    (64, 4, 1, 0, 4)])                                           # four softmax warpgroups
def test_every_tuned_configuration_matches_the_oracle(gpu_lib, d, stages, persistent, esplit, swg):
    """Each block-wise configuration the tuner samples (ring depth, variant,
    exp split, softmax warpgroups), run through stof_mha_fwd_plan: per-head
    causal masks with random holes, a fully masked row and a query tile
    without listed OTs, more query tiles than SMs for d = 64."""
    B, H, L = (2, 10, 1024) if d == 64 else (1, 4, 512)
    rng = np.random.default_rng(90 + stages + 10 * persistent + d + 100 * esplit + swg)
    masks = (rng.random((B * H, L, L)) < 0.2).astype(np.uint8) * np.tril(np.ones((L, L), np.uint8))[None]
    masks[:, np.arange(L), np.arange(L)] = 1
    masks[3, 300] = 0
    masks[1, :128] = 0
    q, k, v = synth.make_qkv(B, H, L, d, "bf16", seed=91)
    fmt, ws, _ = gpu_encode(torch.from_numpy(masks).cuda(), 128, 128)
    plan = stof.stof_plan(stof.STOF_KERNEL_BLOCKWISE, stages, persistent, 0, 0, esplit, swg)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qd, float("nan"))
    scale = 1 / math.sqrt(d)
    stof.stof_mha_fwd_plan(qd, kd, vd, fmt, scale, H, 1, plan, o)
    torch.cuda.synchronize()
    stof.stof_format_sync(fmt)
    assert fmt.device_error == 0
    q64, k64, v64 = (synth.to_float64(t) for t in (q, k, v))
    heads = [(0, 0), (0, 1), (0, 3)] + ([(1, H - 1)] if B > 1 else [])
    ref = oracle.attention_bhld(q64, k64, v64, lambda b, h, rows: masks[b * H + h][rows], scale, heads=heads)
    for (b, h), o_ref in ref.items():
        assert np.abs(o[b, h].double().cpu().numpy() - o_ref).max() <= TOL["bf16"]
    assert torch.all(o[0, 3, 300] == 0) and torch.all(o[0, 1, :128] == 0)


def test_configurations_the_sizes_do_not_admit_are_refused(gpu_lib):
    L = 256
    fmt, ws, _ = gpu_encode(torch.ones(1, L, L, dtype=torch.uint8, device="cuda"), 128, 128)
    q = torch.zeros(1, 1, L, 128, dtype=torch.bfloat16, device="cuda")
    # d = 128: ring depth 4, persistent CTAs, four softmax warpgroups, the exp split off its ring depth
    for stages, persistent, esplit, swg in ((4, 0, 0, 0), (2, 1, 0, 0), (5, 0, 0, 0), (3, 0, 0, 4), (4, 1, 0, 4),
                                            (2, 0, 1, 0)):
        with pytest.raises(stof.StofError) as e:
            stof.stof_mha_fwd_plan(q, q, q, fmt, 0.1, 0, 0,
                                   stof.stof_plan(1, stages, persistent, 0, 0, esplit, swg), q.clone())
        assert e.value.status == stof.STOF_ERR_UNSUPPORTED
    # d = 64: four warpgroups only persistent at ring depth 4 and without the exp split
    q64 = torch.zeros(1, 1, L, 64, dtype=torch.bfloat16, device="cuda")
    for stages, persistent, esplit, swg in ((4, 0, 0, 4), (3, 1, 0, 4), (4, 1, 1, 4), (3, 1, 1, 0)):
        with pytest.raises(stof.StofError) as e:
            stof.stof_mha_fwd_plan(q64, q64, q64, fmt, 0.1, 0, 0,
                                   stof.stof_plan(1, stages, persistent, 0, 0, esplit, swg), q64.clone())
        assert e.value.status == stof.STOF_ERR_UNSUPPORTED


@pytest.mark.parametrize("rpw", [1, 2, 4])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bm,bn,L,density", [(128, 128, 384, 0.05), (128, 128, 512, 0.6), (8, 8, 136, 0.2),
                                             (64, 32, 320, 0.02)])
def test_rowwise_rows_per_warp_match_the_oracle(gpu_lib, rpw, d, bm, bn, L, density):
    """The row-wise kernel with 1, 2 or 4 query rows per warp (the rows of a
    warp have different OT and key counts; with 3 heads and L = 136 the last
    warp is ragged), per-head masks with a fully masked row and empty tile
    columns."""
    B, H = 1, 3
    masks = synth.random_mask(B * H, L, L, density, seed=L + rpw + d)
    masks[1, 5] = 0
    masks[2, :, : L // 3] = 0
    masks[0, 7, :] = 1                                  # one dense row among sparse ones
    q, k, v = synth.make_qkv(B, H, L, d, "fp16", seed=12)
    fmt, ws, _ = gpu_encode(torch.from_numpy(masks).cuda(), bm, bn)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qd, float("nan"))
    scale = 1 / math.sqrt(d)
    stof.stof_mha_fwd_plan(qd, kd, vd, fmt, scale, H, 1, stof.stof_plan(stof.STOF_KERNEL_ROWWISE, 0, 0, 0, rpw), o)
    torch.cuda.synchronize()
    stof.stof_format_sync(fmt)
    assert fmt.device_error == 0
    q64, k64, v64 = (synth.to_float64(t) for t in (q, k, v))
    ref = oracle.attention_bhld(q64, k64, v64, lambda b, h, rows: masks[b * H + h][rows], scale)
    for (b, h), o_ref in ref.items():
        assert np.abs(o[b, h].double().cpu().numpy() - o_ref).max() <= TOL["fp16"]
    assert torch.all(o[0, 1, 5] == 0)


def test_auto_ignores_a_cached_kernel_the_format_cannot_run(gpu_lib):
    """A tuned entry for (L, d, density bucket) made on 128x128 OTs does not
    apply to a format of 64x128 OTs when it names the block-wise kernel: AUTO
    then follows the analytic model (which falls back to the row-wise kernel
    for such OTs) instead of failing."""
    B, H, L, d = 1, 2, 512, 64
    mask = np.tril(np.ones((L, L), np.uint8))[None]
    q, k, v = (t.cuda() for t in synth.make_qkv(B, H, L, d, "bf16", seed=5))
    mdev = torch.from_numpy(mask).cuda()
    wst = torch.empty(stof.stof_tune_workspace_bytes(1, L), dtype=torch.uint8, device="cuda")
    stof.stof_tune_clear()
    res = stof.stof_tune(mdev, q, k, v, 0.125, 0, 0, wst, torch.empty_like(q))
    f128, _, _ = gpu_encode(mdev, 128, 128)
    f64, _, _ = gpu_encode(mdev, 64, 128)
    p128 = stof.stof_mha_plan(f128, B, H, L, d, stof.STOF_KERNEL_AUTO)
    p64 = stof.stof_mha_plan(f64, B, H, L, d, stof.STOF_KERNEL_AUTO)
    assert p128.source == stof.STOF_PLAN_TUNED
    if p128.kernel == stof.STOF_KERNEL_BLOCKWISE:
        assert p64.source == stof.STOF_PLAN_ANALYTIC and p64.kernel == stof.STOF_KERNEL_ROWWISE
    o = torch.full_like(q, float("nan"))
    stof.stof_mha_fwd(q, k, v, f64, 0.125, 0, 0, stof.STOF_KERNEL_AUTO, o)   # runs, does not raise
    torch.cuda.synchronize()
    assert torch.isfinite(o).all()
    stof.stof_tune_clear()
