"""stof.MaskedAttention, the binding's one-call sequence (encode, sync,
attention) for PyTorch callers, against the fp64 oracle: per-(b, h),
per-head and shared masks, bool and uint8 masks, a second call reusing the
encoded mask, and the workspace growing for a larger mask."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof, synth
from tests.conftest import TOL

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_masks", ["bh", "h", "one"])
def test_one_call_matches_the_oracle(gpu_lib, n_masks):
    B, H, L, d = 2, 3, 300, 64
    n = {"bh": B * H, "h": H, "one": 1}[n_masks]
    masks = synth.random_mask(n, L, L, 0.3, seed=n)
    q, k, v = synth.make_qkv(B, H, L, d, "bf16", seed=7)
    att = stof.MaskedAttention()
    o = att(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(masks).cuda().bool())
    torch.cuda.synchronize()
    q64, k64, v64 = (synth.to_float64(t) for t in (q, k, v))
    for b in range(B):
        for h in range(H):
            m = masks[{"bh": b * H + h, "h": h, "one": 0}[n_masks]]
            ref = oracle.attention(q64[b, h], k64[b, h], v64[b, h], m, 1 / math.sqrt(d))
            assert np.abs(o[b, h].double().cpu().numpy() - ref).max() <= TOL["bf16"]


def test_reuse_and_grow(gpu_lib):
    att = stof.MaskedAttention()
    small = torch.from_numpy(synth.random_mask(1, 128, 128, 0.5, seed=1)).cuda()
    big = torch.from_numpy(synth.random_mask(1, 1000, 1000, 0.1, seed=2)).cuda()
    q, k, v = (t.cuda() for t in synth.make_qkv(1, 1, 128, 128, "fp16", seed=3))
    o1 = att(q, k, v, small).clone()
    o2 = att(q, k, v)                        # the encoded mask again
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    ws_small = att.workspace.numel()
    qc, kc, vc = synth.make_qkv(1, 1, 1000, 128, "fp16", seed=4)
    ob = att(qc.cuda(), kc.cuda(), vc.cuda(), big)
    torch.cuda.synchronize()
    assert att.workspace.numel() > ws_small
    q64, k64, v64 = (synth.to_float64(t) for t in (qc, kc, vc))
    ref = oracle.attention(q64[0, 0], k64[0, 0], v64[0, 0], big.cpu().numpy()[0], 1 / math.sqrt(128))
    assert np.abs(ob[0, 0].double().cpu().numpy() - ref).max() <= TOL["fp16"]
