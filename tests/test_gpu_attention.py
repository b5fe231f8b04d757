"""Masked MHA forward on the GPU (both kernels, forced and automatic)
against the fp64 CPU oracle ("Accelerating Sparse Transformer Inference on
GPU", gist.science technical summary, Methodology 1: exact masking;
row-wise and block-wise kernels).  Tolerance: max |O - O_oracle| <= 2e-3
for fp16 inputs and <= 1.5e-2 for bf16 inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof, synth
from tests.conftest import TOL, gpu_encode

pytestmark = pytest.mark.gpu

KERNELS = {"row": stof.STOF_KERNEL_ROWWISE, "block": stof.STOF_KERNEL_BLOCKWISE}


def _run(q, k, v, mask_dev, bm, bn, sb, sh, which, scale=None):
    B, H, L, d = q.shape
    fmt, ws, _ = gpu_encode(mask_dev, bm, bn)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qd, float("nan"))
    scale = 1 / math.sqrt(d) if scale is None else scale
    stof.stof_mha_fwd(qd, kd, vd, fmt, scale, sb, sh, which, o)
    torch.cuda.synchronize()
    return o.cpu(), fmt


def _check(o_gpu, q, k, v, mask_of, dtype, heads=None, rows=None, scale=None, rel=False):
    """Max |O - O_oracle| <= TOL[dtype].  With rel=True (stress inputs
    outside the N(0,1) workloads, where |O| can exceed 1 and bf16 output
    rounding alone reaches 2^-6 |O|) the bound is TOL[dtype] * max(1, |O|)."""
    B, H, L, d = q.shape
    scale = 1 / math.sqrt(d) if scale is None else scale
    q64, k64, v64 = (synth.to_float64(t) for t in (q, k, v))
    ref = oracle.attention_bhld(q64, k64, v64, mask_of, scale, heads=heads, rows=rows)
    og = o_gpu.double().numpy()
    worst = 0.0
    for (b, h), o_ref in ref.items():
        got = og[b, h] if rows is None else og[b, h, rows]
        assert np.all(np.isfinite(got))
        err = np.abs(got - o_ref)
        if rel:
            err = err / np.maximum(1.0, np.abs(o_ref))
        worst = max(worst, float(err.max()))
    assert worst <= TOL[dtype], f"max abs error {worst} > {TOL[dtype]}"
    return worst


def _mask_of_np(mask, sb, sh):
    return lambda b, h, rows: mask[b * sb + h * sh][rows]


@pytest.mark.parametrize("kern", ["row", "block"])
@pytest.mark.parametrize("name", ["window48_L256", "bigbird_L512", "causal_L2048", "longformer_L4096"])
def test_workloads_full_size(gpu_lib, name, kern):
    w = synth.WORKLOADS[name]
    mask = synth.make_mask(w)
    q, k, v = synth.make_qkv(w.B, w.H, w.L, w.d, w.dtype, seed=w.seed)
    o, fmt = _run(q, k, v, torch.from_numpy(mask).cuda(), 128, 128, w.stride_b, w.stride_h, KERNELS[kern])
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    if len(heads) > 6:  # oracle on a seeded sample of heads; the GPU ran them all
        idx = np.random.default_rng(1).choice(len(heads), 6, replace=False)
        heads = [heads[i] for i in sorted(idx)]
    _check(o, q, k, v, _mask_of_np(mask, w.stride_b, w.stride_h), w.dtype, heads=heads)
    assert fmt.device_error == 0


@pytest.mark.parametrize("kern", ["row", "block"])
def test_bernoulli_L16384_full_size_sampled(gpu_lib, kern):
    w = synth.WORKLOADS["bernoulli_L16384"]
    L = w.L
    mask = torch.empty(w.n_masks, L, L, dtype=torch.uint8, device="cuda")
    stof.stof_synth_causal_bernoulli_mask(mask, w.n_masks, L, w.seed,
                                          synth.bernoulli_threshold(synth.BERNOULLI_P))
    q, k, v = synth.make_qkv(w.B, w.H, w.L, w.d, w.dtype, seed=w.seed)
    o, fmt = _run(q, k, v, mask, 128, 128, w.stride_b, w.stride_h, KERNELS[kern])
    del mask
    torch.cuda.empty_cache()
    # 8 heads (the first, the last and 6 seeded others), 1024 query rows of
    # each: the first 128, the last 128 and 768 seeded others
    rng = np.random.default_rng(2)
    heads = [(0, 0), (0, 31)] + [(0, int(h)) for h in rng.choice(np.arange(1, 31), 6, replace=False)]
    mid = rng.choice(np.arange(128, L - 128), 768, replace=False)
    rows = np.unique(np.concatenate([np.arange(128), mid, np.arange(L - 128, L)]))
    assert len(rows) == 1024
    _check(o, q, k, v, lambda b, h, r: synth.mask_rows(w, b * w.stride_b + h * w.stride_h, r),
           w.dtype, heads=heads, rows=rows)


@pytest.mark.parametrize("kern,bn", [("row", 128), ("block", 128), ("block", 64)])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("density", [0.02, 0.3, 0.9])
def test_random_masks_small(gpu_lib, kern, bn, d, dtype, density):
    # several OTs per row and column, per-head masks, a fully masked row
    B, H, L = 2, 3, 384
    mask = synth.random_mask(B * H, L, L, density, seed=d + int(density * 100))
    mask[1, 5] = 0
    mask[2, :, :200] = 0          # empty and partly-empty tile columns
    q, k, v = synth.make_qkv(B, H, L, d, dtype, seed=3)
    o, _ = _run(q, k, v, torch.from_numpy(mask).cuda(), 128, bn, H, 1, KERNELS[kern])
    _check(o, q, k, v, _mask_of_np(mask, H, 1), dtype)
    assert torch.all(o[0, 1, 5] == 0)


@pytest.mark.parametrize("bm,bn", [(16, 16), (64, 32), (8, 8)])
def test_rowwise_other_tile_sizes(gpu_lib, bm, bn):
    B, H, L, d = 1, 2, 256, 64
    mask = synth.random_mask(1, L, L, 0.2, seed=bm + bn)
    q, k, v = synth.make_qkv(B, H, L, d, "fp16", seed=4)
    o, _ = _run(q, k, v, torch.from_numpy(mask).cuda(), bm, bn, 0, 0, stof.STOF_KERNEL_ROWWISE)
    _check(o, q, k, v, _mask_of_np(mask, 0, 0), "fp16")


@pytest.mark.parametrize("kern,bn", [("row", 128), ("block", 128), ("block", 64)])
@pytest.mark.parametrize("d", [64, 128])
def test_edge_cases(gpu_lib, kern, bn, d):
    B, H, L = 1, 4, 256
    q, k, v = synth.make_qkv(B, H, L, d, "bf16", seed=6)
    q = (q.float() * 8).to(torch.bfloat16)  # sharp softmax
    masks = np.zeros((4, L, L), np.uint8)
    masks[0] = 1                                       # all valid: dense attention
    js = np.random.default_rng(7).integers(0, L, L)
    masks[1, np.arange(L), js] = 1                     # one valid key per row
    masks[2, :128] = 0                                 # first OT row empty
    masks[2, 128:, 5] = 1
    # mask 3 all zero: every row fully masked
    o, _ = _run(q, k, v, torch.from_numpy(masks).cuda(), 128, bn, 0, 1, KERNELS[kern])
    assert torch.equal(o[0, 1], v[0, 1, js])           # exactly that V row
    assert torch.all(o[0, 2, :128] == 0)
    assert torch.equal(o[0, 2, 128:], v[0, 2, 5].expand(128, d))
    assert torch.all(o[0, 3] == 0)
    _check(o, q, k, v, _mask_of_np(masks, 0, 1), "bf16", heads=[(0, 0)], rel=True)


@pytest.mark.parametrize("bn", [128, 64])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_blockwise_many_items_of_every_size(gpu_lib, bn, dtype):
    """d = 64 runs persistent CTAs that take query tiles from a counter:
    more query tiles than SMs, with 0, 1, 2, ... listed tiles each (odd and
    even counts, full and partial tiles), per-head masks."""
    B, H, L, d = 2, 20, 1024, 64
    n_tr, n_tc = L // 128, L // bn
    rng = np.random.default_rng(11 + bn)
    masks = np.zeros((B * H, L, L), np.uint8)
    for m in range(B * H):
        for I in range(n_tr):
            cnt = (m * n_tr + I) % (n_tc + 1)              # every tile count, 0 .. n_tc
            for J in rng.choice(n_tc, cnt, replace=False):
                blk = masks[m, I * 128:(I + 1) * 128, J * bn:(J + 1) * bn]
                blk[:] = 1 if rng.random() < 0.3 else (rng.random(blk.shape) < 0.3)
    q, k, v = synth.make_qkv(B, H, L, d, dtype, seed=12)
    o, fmt = _run(q, k, v, torch.from_numpy(masks).cuda(), 128, bn, H, 1, stof.STOF_KERNEL_BLOCKWISE)
    assert fmt.n_full > 0 and fmt.n_part > 0
    assert B * H * n_tr > 152
    empty = masks.reshape(B, H, L, L).sum(axis=-1) == 0
    assert torch.all(o[torch.from_numpy(empty)] == 0)  # rows of query tiles without tiles
    _check(o, q, k, v, _mask_of_np(masks, H, 1), dtype,
           heads=[(0, 0), (0, 7), (0, 19), (1, 0), (1, 11), (1, 19)])


def test_blockwise_d64_long_query_tiles_sampled(gpu_lib):
    """d = 64 with many listed OTs per query tile (about 64 here) runs a CTA
    per query tile instead of the persistent kernel; sampled rows against
    the oracle."""
    B, H, L, d = 1, 2, 16384, 64
    rng = np.random.default_rng(21)
    mask = np.tril(rng.integers(0, 2, (L, L), dtype=np.uint8))[None]   # causal, half the keys dropped
    mask[0, np.arange(L), np.arange(L)] = 1
    q, k, v = synth.make_qkv(B, H, L, d, "bf16", seed=22)
    o, fmt = _run(q, k, v, torch.from_numpy(mask).cuda(), 128, 128, 0, 0, stof.STOF_KERNEL_BLOCKWISE)
    assert (fmt.n_full + fmt.n_part) / (L // 128) >= 48
    rows = np.unique(np.concatenate([np.arange(64), rng.choice(L, 192, replace=False), np.arange(L - 64, L)]))
    _check(o, q, k, v, _mask_of_np(mask, 0, 0), "bf16", rows=rows)


@pytest.mark.parametrize("name", ["bigbird_L512", "longformer_L4096"])
def test_blockwise_128x64_tiles_full_size(gpu_lib, name):
    # 128 x 64 OTs: half-width key tiles, 1 KB bitmaps, N = 64 score MMAs
    w = synth.WORKLOADS[name]
    mask = synth.make_mask(w)
    q, k, v = synth.make_qkv(w.B, w.H, w.L, w.d, w.dtype, seed=w.seed)
    o, fmt = _run(q, k, v, torch.from_numpy(mask).cuda(), 128, 64, w.stride_b, w.stride_h,
                  stof.STOF_KERNEL_BLOCKWISE)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    idx = np.random.default_rng(5).choice(len(heads), min(4, len(heads)), replace=False)
    _check(o, q, k, v, _mask_of_np(mask, w.stride_b, w.stride_h), w.dtype,
           heads=[heads[i] for i in sorted(idx)])
    assert fmt.device_error == 0


def test_blockwise_other_tiles_refused(gpu_lib):
    mask = torch.ones(1, 256, 256, dtype=torch.uint8, device="cuda")
    q = torch.zeros(1, 1, 256, 64, dtype=torch.float16, device="cuda")
    for bm, bn in ((64, 64), (128, 32), (128, 256)):
        fmt, ws, _ = gpu_encode(mask, bm, bn)
        with pytest.raises(stof.StofError) as e:
            stof.stof_mha_fwd(q, q, q, fmt, 0.125, 0, 0, stof.STOF_KERNEL_BLOCKWISE, q.clone())
        assert e.value.status == stof.STOF_ERR_UNSUPPORTED


def test_auto_selection_runs_the_selected_kernel(gpu_lib):
    w = synth.WORKLOADS["window48_L256"]
    mask = torch.from_numpy(synth.make_mask(w)).cuda()
    q, k, v = synth.make_qkv(w.B, w.H, w.L, w.d, w.dtype)
    o, fmt = _run(q, k, v, mask, 128, 128, 0, 0, stof.STOF_KERNEL_AUTO)
    _check(o, q, k, v, lambda b, h, r: mask.cpu().numpy()[0][r], w.dtype)
    assert fmt.synced == 1


def test_unsynced_auto_is_refused(gpu_lib):
    mask = torch.ones(1, 128, 128, dtype=torch.uint8, device="cuda")
    ws = torch.empty(stof.stof_encode_workspace_bytes(1, 128, 128, 128, 128), dtype=torch.uint8, device="cuda")
    fmt = stof.stof_encode_mask(mask, 128, 128, ws)
    q = torch.zeros(1, 1, 128, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(stof.StofError) as e:
        stof.stof_mha_fwd(q, q, q, fmt, 0.125, 0, 0, stof.STOF_KERNEL_AUTO, q.clone())
    assert e.value.status == stof.STOF_ERR_NOT_SYNCED


def test_concurrent_calls_with_different_formats(gpu_lib):
    """Calls with different formats may overlap on the GPU (each d = 64
    persistent launch keeps its work counter in its own format's workspace):
    two heads' worth of work on two streams at once, each against the oracle."""
    B, H, L, d = 1, 8, 1024, 64
    masks = [synth.random_mask(1, L, L, p, seed=30 + i) for i, p in enumerate((0.1, 0.6))]
    encoded = [gpu_encode(torch.from_numpy(m).cuda(), 128, 128) for m in masks]
    qkv = [tuple(t.cuda() for t in synth.make_qkv(B, H, L, d, "fp16", seed=40 + i)) for i in range(2)]
    outs = [torch.full_like(qkv[i][0], float("nan")) for i in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    torch.cuda.synchronize()
    for rep in range(3):
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                q, k, v = qkv[i]
                stof.stof_mha_fwd(q, k, v, encoded[i][0], 0.125, 0, 0, stof.STOF_KERNEL_BLOCKWISE, outs[i],
                                  stream=streams[i])
    torch.cuda.synchronize()
    for i in range(2):
        q, k, v = (t.cpu() for t in qkv[i])
        _check(outs[i].cpu(), q, k, v, _mask_of_np(masks[i], 0, 0), "fp16", heads=[(0, 0), (0, 7)], scale=0.125)


@pytest.mark.parametrize("kern,bn", [("row", 128), ("block", 128), ("block", 64)])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("sign", [-1.0, 0.0])
def test_nonpositive_scale(gpu_lib, kern, bn, d, sign):
    """scale <= 0 is a legal softmax temperature: with a negative scale the
    row max of the scaled scores is the scaled minimum, and a zero scale gives
    the plain mean of the valid V rows.  Per-head masks with a fully masked
    row and a query tile without listed OTs."""
    B, H, L = 1, 3, 384
    mask = synth.random_mask(B * H, L, L, 0.3, seed=41 + d)
    mask[1, 5] = 0
    mask[2, :128] = 0                 # query tile 0 of head 2: no listed OT
    q, k, v = synth.make_qkv(B, H, L, d, "fp16", seed=43)
    scale = sign / math.sqrt(d)
    o, fmt = _run(q, k, v, torch.from_numpy(mask).cuda(), 128, bn, H, 1, KERNELS[kern], scale=scale)
    assert fmt.device_error == 0
    _check(o, q, k, v, _mask_of_np(mask, H, 1), "fp16", scale=scale)
    assert torch.all(o[0, 1, 5] == 0) and torch.all(o[0, 2, :128] == 0)
