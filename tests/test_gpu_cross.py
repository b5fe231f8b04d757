"""Attention of Lq query rows over Lk keys (stof_mha_fwd_cross) with
[Lq][Lk] masks: the masked softmax of "Accelerating Sparse Transformer
Inference on GPU" (gist.science technical summary, Problem statement)
where queries and keys come from two sequences.  Each kernel against the
fp64 oracle, lengths whole tiles or not, and a NaN guard after O."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof, synth
from tests.conftest import TOL, gpu_encode

pytestmark = pytest.mark.gpu

KERNELS = {"row": stof.STOF_KERNEL_ROWWISE, "block": stof.STOF_KERNEL_BLOCKWISE, "auto": stof.STOF_KERNEL_AUTO}


@pytest.mark.parametrize("Lq,Lk", [(128, 512), (512, 128), (77, 1000), (1000, 77), (256, 256), (1, 300)])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("kern", ["row", "block", "auto"])
def test_cross_attention_matches_the_oracle(gpu_lib, Lq, Lk, d, kern):
    B, H = 2, 2
    rng = np.random.default_rng(Lq * 3 + Lk + d)
    masks = (rng.random((B * H, Lq, Lk)) < 0.3).astype(np.uint8)
    masks[0, :, : min(Lk, 256)] = 1                   # full OTs next to partial ones
    if Lq > 3:
        masks[1, 3] = 0                               # a query with no valid key
    g = torch.Generator().manual_seed(Lq + Lk)
    q = torch.randn(B, H, Lq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, H, Lk, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, H, Lk, d, generator=g).to(torch.bfloat16)
    fmt, ws, _ = gpu_encode(torch.from_numpy(masks).cuda(), 128, 128)
    n = B * H * Lq * d
    buf = torch.full((n + 4096,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = buf[:n].view(B, H, Lq, d)
    scale = 1 / math.sqrt(d)
    stof.stof_mha_fwd_cross(q.cuda(), k.cuda(), v.cuda(), fmt, scale, H, 1, KERNELS[kern], o)
    torch.cuda.synchronize()
    stof.stof_format_sync(fmt)
    assert fmt.device_error == 0
    assert torch.isnan(buf[n:]).all()
    q64, k64, v64 = (t.double().numpy() for t in (q, k, v))
    for b in range(B):
        for h in range(H):
            ref = oracle.attention(q64[b, h], k64[b, h], v64[b, h], masks[b * H + h], scale)
            assert np.abs(o[b, h].double().cpu().numpy() - ref).max() <= TOL["bf16"], (b, h)
    if Lq > 3:
        assert torch.all(o[0, 1, 3] == 0)


def test_self_attention_is_the_square_case(gpu_lib):
    """stof_mha_fwd equals stof_mha_fwd_cross with Lq = Lk, bit for bit."""
    L, d = 384, 64
    masks = synth.random_mask(2, L, L, 0.2, seed=5)
    q, k, v = (t.cuda() for t in synth.make_qkv(1, 2, L, d, "bf16", seed=6))
    fmt, ws, _ = gpu_encode(torch.from_numpy(masks).cuda(), 128, 128)
    a, b = torch.empty_like(q), torch.empty_like(q)
    stof.stof_mha_fwd(q, k, v, fmt, 0.125, 0, 1, stof.STOF_KERNEL_BLOCKWISE, a)
    stof.stof_mha_fwd_cross(q, k, v, fmt, 0.125, 0, 1, stof.STOF_KERNEL_BLOCKWISE, b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_mismatched_format_is_refused(gpu_lib):
    masks = torch.ones(1, 128, 256, dtype=torch.uint8, device="cuda")
    fmt, ws, _ = gpu_encode(masks, 128, 128)
    q = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16, device="cuda")   # Lq = 256, format has 128 rows
    k = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(stof.StofError) as e:
        stof.stof_mha_fwd_cross(q, k, k, fmt, 0.1, 0, 0, stof.STOF_KERNEL_BLOCKWISE, q.clone())
    assert e.value.status == stof.STOF_ERR_SHAPE
