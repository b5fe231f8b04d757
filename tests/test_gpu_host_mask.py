"""A mask in pinned host memory, which the encoder reads over the host link
with no device copy: the format is the one the oracle's encoder gives
("Accelerating Sparse Transformer Inference on GPU", gist.science technical
summary, Methodology 1, two-level storage format) and, byte for byte, the one
encoded from the same mask in device memory; attention through
MaskedAttention with a host mask equals that with a device mask."""
import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof, synth
from tests.conftest import assert_format_equal, gpu_encode

pytestmark = pytest.mark.gpu


def _pinned(a):
    t = torch.empty(a.shape, dtype=torch.uint8, pin_memory=True)
    t.copy_(torch.from_numpy(np.ascontiguousarray(a)))
    return t


@pytest.mark.parametrize("n,lq,lk,bm,bn", [(3, 512, 512, 128, 128), (2, 300, 520, 128, 64), (4, 1000, 777, 64, 64),
                                          (1, 96, 4096, 16, 16)])
def test_host_mask_same_format(gpu_lib, n, lq, lk, bm, bn):
    mask = synth.random_mask(n, lq, lk, 0.2, seed=lq + lk)
    mask[0, : min(lq, 128), : min(lk, 128)] = 1  # a full OT where the sizes allow one
    ws_bytes = stof.stof_encode_workspace_bytes(n, lq, lk, bm, bn)
    ws_h = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    fmt_h = stof.stof_encode_mask(_pinned(mask), bm, bn, ws_h)
    stof.stof_format_sync(fmt_h)
    assert fmt_h.device_error == 0
    fmt_d, ws_d, arrs = gpu_encode(torch.from_numpy(mask).cuda(), bm, bn)
    assert_format_equal(fmt_d, arrs, oracle.encode(mask, bm, bn))
    ws_d0 = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    fmt_d0 = stof.stof_encode_mask(torch.from_numpy(mask).cuda(), bm, bn, ws_d0)
    stof.stof_format_sync(fmt_d0)
    assert (fmt_h.n_full, fmt_h.n_part, fmt_h.nnz) == (fmt_d0.n_full, fmt_d0.n_part, fmt_d0.nnz)
    assert torch.equal(ws_h, ws_d0)  # every byte of the two workspaces


def test_masked_attention_with_host_mask(gpu_lib):
    B, H, L, d = 1, 4, 640, 128
    masks = synth.random_mask(H, L, L, 0.15, seed=11)
    q, k, v = (t.cuda() for t in synth.make_qkv(B, H, L, d, "bf16", seed=5))
    o_dev = stof.MaskedAttention()(q, k, v, torch.from_numpy(masks).cuda())
    o_host = stof.MaskedAttention()(q, k, v, _pinned(masks))
    torch.cuda.synchronize()
    assert torch.equal(o_dev, o_host)
