"""Seeded random configurations of the whole attention path against the fp64
oracle: lengths (whole tiles or not, Lq != Lk), head sizes 32-256, OT sizes,
kernels and variants, dtypes, the scale's sign, mask densities and how masks are shared
between batch elements and heads (mask strides).  Each case encodes its
masks on the GPU, runs the attention and compares every output row with
"Accelerating Sparse Transformer Inference on GPU" (gist.science technical
summary, Problem statement: softmax over the valid keys only, 0 for a row
without one) as the oracle computes it."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof
from tests.conftest import TOL, gpu_encode

pytestmark = pytest.mark.gpu

N_CASES = 48
TILES = [(128, 128), (128, 64), (64, 64), (16, 16), (8, 24), (32, 128)]


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    c = dict(B=int(rng.integers(1, 3)), H=int(rng.integers(1, 4)), d=int(rng.choice([32, 64, 64, 128, 128, 256])),
             dtype=str(rng.choice(["bf16", "fp16"])), sign=float(rng.choice([1.0, 1.0, -1.0])),
             density=float(rng.choice([0.02, 0.2, 0.6, 1.0])))
    c["Lq"] = int(rng.integers(1, 700))
    c["Lk"] = c["Lq"] if rng.random() < 0.6 else int(rng.integers(1, 700))
    c["bm"], c["bn"] = TILES[int(rng.integers(len(TILES)))]
    blockwise_ok = c["bm"] == 128 and c["bn"] in (64, 128) and c["d"] in (64, 128)
    kinds = ["row", "auto"] + (["block", "persist", "persist4", "esplit"] if blockwise_ok else [])
    c["kind"] = str(rng.choice(kinds))
    if c["kind"] in ("persist", "persist4") and c["d"] != 64:
        c["kind"] = "block"
    if c["kind"] == "persist4" and c["bn"] != 128:
        c["kind"] = "persist"
    if c["kind"] == "esplit" and c["bn"] != 128:
        c["kind"] = "block"
    # masks: one per (b, h), one per head shared by the batch, or one for all
    c["share"] = str(rng.choice(["per_head", "per_h_only", "one"]))
    return c


def _plan(c):
    K = stof.STOF_KERNEL_BLOCKWISE
    return {"row": stof.stof_plan(stof.STOF_KERNEL_ROWWISE, 0, 0, 0, 0),
            "block": stof.stof_plan(K, 0, 0, 0, 0),
            "persist": stof.stof_plan(K, 4, 1, 0, 0),
            "persist4": stof.stof_plan(K, 4, 1, 0, 0, 0, 4),
            "esplit": stof.stof_plan(K, 3, 0, 0, 0, 1, 0)}.get(c["kind"])


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_configuration(gpu_lib, seed):
    c = _case(seed)
    B, H, Lq, Lk, d = c["B"], c["H"], c["Lq"], c["Lk"], c["d"]
    rng = np.random.default_rng(seed)
    n_masks, sb, sh = {"per_head": (B * H, H, 1), "per_h_only": (H, 0, 1), "one": (1, 0, 0)}[c["share"]]
    masks = (rng.random((n_masks, Lq, Lk)) < c["density"]).astype(np.uint8)
    if Lq > 2 and rng.random() < 0.5:
        masks[0, 2] = 0                                  # a row without a valid key
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}[c["dtype"]]
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Lq, d, generator=g).to(dt)
    k = torch.randn(B, H, Lk, d, generator=g).to(dt)
    v = torch.randn(B, H, Lk, d, generator=g).to(dt)
    fmt, ws, _ = gpu_encode(torch.from_numpy(masks).cuda(), c["bm"], c["bn"])
    n = B * H * Lq * d
    buf = torch.full((n + 2048,), float("nan"), dtype=dt, device="cuda")
    o = buf[:n].view(B, H, Lq, d)
    scale = c["sign"] / math.sqrt(d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    plan = _plan(c)
    if Lq == Lk and plan is not None:
        stof.stof_mha_fwd_plan(qd, kd, vd, fmt, scale, sb, sh, plan, o)
    else:
        which = {"row": stof.STOF_KERNEL_ROWWISE, "auto": stof.STOF_KERNEL_AUTO}.get(c["kind"],
                                                                                   stof.STOF_KERNEL_BLOCKWISE)
        stof.stof_mha_fwd_cross(qd, kd, vd, fmt, scale, sb, sh, which, o)
    torch.cuda.synchronize()
    stof.stof_format_sync(fmt)
    assert fmt.device_error == 0, c
    assert torch.isnan(buf[n:]).all(), c
    q64, k64, v64 = (t.double().numpy() for t in (q, k, v))
    got = o.double().cpu().numpy()
    for b in range(B):
        for h in range(H):
            ref = oracle.attention(q64[b, h], k64[b, h], v64[b, h], masks[b * sb + h * sh], scale)
            # the fixed tolerance of the other parity tests, plus the output's own
            # rounding where |O| reaches past 1 (half a step: 2^-9 |O| bf16, 2^-12 fp16)
            u = 2.0 ** -9 if c["dtype"] == "bf16" else 2.0 ** -12
            assert np.all(np.abs(got[b, h] - ref) <= TOL[c["dtype"]] + u * np.abs(ref)), (c, b, h)
