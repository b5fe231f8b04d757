"""Measured parameter choice with a result cache (gist.science technical
summary, Methodology 2, two-stage tuning, stage 2 "parameter sampling":
kernel parameters are sampled by running them and the outcomes cached).
The candidates are the row-wise kernel on 128x128 OTs and the block-wise
kernel on 128x128 and 128x64 OTs; the chosen one must also be correct."""
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
    best = int(np.argmin(ms))
    assert res.kernel == res.cand_kernel[best] and res.bn == res.cand_bn[best]
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
