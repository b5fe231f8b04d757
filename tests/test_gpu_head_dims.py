"""Head dimensions 32 and 256 (the row-wise kernel's alone) against the fp64
oracle: the masked softmax of "Accelerating Sparse Transformer Inference on
GPU" (gist.science technical summary, Problem statement), with 1, 2 or 4
query rows per warp (2 at most for d = 256), AUTO, a length that is not a
whole number of tiles and two sequences; the block-wise kernel refuses
these sizes."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof, synth
from tests.conftest import TOL, gpu_encode

pytestmark = pytest.mark.gpu


def _run(d, Lq, Lk, dtype, plan=None, which=stof.STOF_KERNEL_AUTO, seed=0):
    B, H = 1, 3
    rng = np.random.default_rng(seed + d)
    masks = (rng.random((H, Lq, Lk)) < 0.2).astype(np.uint8)
    masks[0, :, : min(Lk, 128)] = 1
    masks[1, 5] = 0
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Lq, d, generator=g).to(dt)
    k = torch.randn(B, H, Lk, d, generator=g).to(dt)
    v = torch.randn(B, H, Lk, d, generator=g).to(dt)
    fmt, ws, _ = gpu_encode(torch.from_numpy(masks).cuda(), 128, 128)
    n = B * H * Lq * d
    buf = torch.full((n + 1024,), float("nan"), dtype=dt, device="cuda")
    o = buf[:n].view(B, H, Lq, d)
    scale = 1 / math.sqrt(d)
    if plan is not None:
        stof.stof_mha_fwd_plan(q.cuda(), k.cuda(), v.cuda(), fmt, scale, 0, 1, plan, o)
    else:
        stof.stof_mha_fwd_cross(q.cuda(), k.cuda(), v.cuda(), fmt, scale, 0, 1, which, o)
    torch.cuda.synchronize()
    stof.stof_format_sync(fmt)
    assert fmt.device_error == 0
    assert torch.isnan(buf[n:]).all()
    q64, k64, v64 = (t.double().numpy() for t in (q, k, v))
    for h in range(H):
        ref = oracle.attention(q64[0, h], k64[0, h], v64[0, h], masks[h], scale)
        assert np.abs(o[0, h].double().cpu().numpy() - ref).max() <= TOL[dtype], h
    assert torch.all(o[0, 1, 5] == 0)


@pytest.mark.parametrize("d", [32, 256])
@pytest.mark.parametrize("rpw", [0, 1, 2, 4])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_row_wise_rows_per_warp(gpu_lib, d, rpw, dtype):
    plan = stof.stof_plan(stof.STOF_KERNEL_ROWWISE, 0, 0, 0, rpw)
    if d == 256 and rpw == 4:
        with pytest.raises(stof.StofError) as e:
            _run(d, 384, 384, dtype, plan=plan)
        assert e.value.status == stof.STOF_ERR_UNSUPPORTED
        return
    _run(d, 384, 384, dtype, plan=plan, seed=rpw)


@pytest.mark.parametrize("d", [32, 256])
@pytest.mark.parametrize("Lq,Lk", [(200, 200), (77, 300), (1000, 129)])
def test_auto_and_two_sequences(gpu_lib, d, Lq, Lk):
    _run(d, Lq, Lk, "bf16", seed=Lq)


@pytest.mark.parametrize("d", [32, 256])
def test_block_wise_refuses_these_sizes(gpu_lib, d):
    with pytest.raises(stof.StofError) as e:
        _run(d, 256, 256, "bf16", which=stof.STOF_KERNEL_BLOCKWISE)
    assert e.value.status == stof.STOF_ERR_UNSUPPORTED


def test_tuner_keeps_to_the_row_wise_kernel(gpu_lib):
    L, d = 256, 256
    mask = np.tril(np.ones((L, L), np.uint8))[None]
    q, k, v = (t.cuda() for t in synth.make_qkv(1, 2, L, d, "bf16", seed=3))
    wst = torch.empty(stof.stof_tune_workspace_bytes(1, L), dtype=torch.uint8, device="cuda")
    stof.stof_tune_clear()
    res = stof.stof_tune(torch.from_numpy(mask).cuda(), q, k, v, 0.0625, 0, 0, wst, torch.empty_like(q))
    ms = list(res.cand_ms)
    assert ms[0] > 0 and ms[1] > 0 and ms[2] < 0       # row-wise 1 and 2 rows per warp; 4 refused
    assert all(t < 0 for t in ms[3:])                  # no block-wise candidate at d = 256
    assert res.kernel == stof.STOF_KERNEL_ROWWISE
    stof.stof_tune_clear()
