"""Tolerance feasibility: the output is rounded once to fp16 / bf16, so even
an exact kernel differs from the fp64 oracle by |round(O) - O|.  For each
workload this computes that floor on sampled rows (always the first rows,
where causal masks leave few keys and |O| is largest) and checks it is
below the tolerance the GPU path is held to (2e-3 fp16, 1.5e-2 bf16):
otherwise a kernel failing the bound would not be distinguishable from the
rounding itself.  Masks and inputs are those of the five workloads."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import synth
from tests.conftest import TOL

TORCH_DT = {"fp16": torch.float16, "bf16": torch.bfloat16}


def _floor(w, heads, rows):
    q, k, v = synth.make_qkv(w.B, w.H, w.L, w.d, w.dtype, seed=w.seed)
    q64, k64, v64 = (synth.to_float64(t) for t in (q, k, v))
    worst = 0.0
    for (b, h) in heads:
        m = synth.mask_index(w, b, h)
        mask = synth.mask_rows(w, m, rows)
        o = oracle.attention(q64[b, h, rows], k64[b, h], v64[b, h], mask, 1 / math.sqrt(w.d))
        rounded = torch.from_numpy(o).to(TORCH_DT[w.dtype]).double().numpy()
        worst = max(worst, float(np.abs(rounded - o).max()))
    return worst


@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_output_rounding_floor_is_below_the_tolerance(name):
    w = synth.WORKLOADS[name]
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([np.arange(min(64, w.L)), rng.choice(w.L, min(64, w.L), replace=False)]))
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    floor = _floor(w, heads, rows)
    print(f"{name}: rounding floor {floor:.3g} (tolerance {TOL[w.dtype]})")
    assert floor < TOL[w.dtype]
