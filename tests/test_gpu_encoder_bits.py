"""Encoder from a bit-packed mask (one bit per element, least significant
bit first along the key axis): the format must equal, bit for bit, the
brute-force oracle encoding of the same mask unpacked ("Accelerating Sparse
Transformer Inference on GPU", gist.science technical summary, Methodology
1, two-level storage format; scifaro.com summary, Results, long sequences
within memory)."""
import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof, synth
from tests.conftest import assert_format_equal

pytestmark = pytest.mark.gpu


def _encode_bits(mask_np, bm, bn):
    bits = np.packbits(mask_np != 0, axis=-1, bitorder="little")
    n, lq, lk = mask_np.shape
    dbits = torch.from_numpy(np.ascontiguousarray(bits)).cuda()
    ws = torch.empty(stof.stof_encode_workspace_bytes(n, lq, lk, bm, bn), dtype=torch.uint8, device="cuda")
    ws.fill_(0x5A)
    fmt = stof.stof_encode_mask_bits(dbits, lk, bm, bn, ws)
    stof.stof_format_sync(fmt)
    arrs = {k: v.cpu().numpy() for k, v in stof.format_arrays(fmt, ws).items()}
    arrs["bitmaps"] = arrs["bitmaps"].view("uint64")
    return fmt, ws, arrs


@pytest.mark.parametrize("name", ["window48_L256", "bigbird_L512", "causal_L2048", "longformer_L4096"])
@pytest.mark.parametrize("bm,bn", [(128, 128), (128, 64), (16, 16)])
def test_workload_masks_bit_exact(gpu_lib, name, bm, bn):
    mask = synth.make_mask(synth.WORKLOADS[name])
    fmt, ws, arrs = _encode_bits(mask, bm, bn)
    assert_format_equal(fmt, arrs, oracle.encode(mask, bm, bn))


# tile widths whose byte count is a multiple of 16, of 8 only, and neither
@pytest.mark.parametrize("bm,bn", [(8, 128), (32, 256), (8, 64), (24, 192), (8, 8), (16, 24), (40, 200)])
@pytest.mark.parametrize("density", [0.0, 0.01, 0.5, 0.995, 1.0])
def test_random_masks_bit_exact(gpu_lib, bm, bn, density):
    mask = synth.random_mask(3, bm * 5, bn * 7, density, seed=bm * 3 + bn + int(density * 1000))
    fmt, ws, arrs = _encode_bits(mask, bm, bn)
    assert_format_equal(fmt, arrs, oracle.encode(mask, bm, bn))


def test_single_bits_pin_bit_order(gpu_lib):
    masks = np.zeros((64, 8, 16), np.uint8)
    for b in range(64):
        masks[b, b // 8, 8 + b % 8] = 1
    fmt, ws, arrs = _encode_bits(masks, 8, 16)
    words = arrs["bitmaps"].reshape(64, 2)
    assert np.all(words[:, 0] == 0)
    assert [int(x) for x in words[:, 1]] == [1 << b for b in range(64)]


def test_device_packer_and_bit_generator_match_numpy(gpu_lib):
    w = synth.WORKLOADS["bernoulli_L16384"]
    n, L = 2, 1024
    thr = synth.bernoulli_threshold(synth.BERNOULLI_P)
    dense = torch.empty(n, L, L, dtype=torch.uint8, device="cuda")
    stof.stof_synth_causal_bernoulli_mask(dense, n, L, w.seed, thr)
    packed = stof.stof_synth_pack_bits(dense)
    want = np.packbits(dense.cpu().numpy() != 0, axis=-1, bitorder="little")
    assert np.array_equal(packed.cpu().numpy(), want)
    direct = torch.empty(n, L, L // 8, dtype=torch.uint8, device="cuda")
    stof.stof_synth_causal_bernoulli_mask_bits(direct, n, L, w.seed, thr)
    assert np.array_equal(direct.cpu().numpy(), want)


def test_bernoulli_L16384_full_size_bits_equal_dense(gpu_lib):
    """The 16k workload from its 1.07 GB bit-packed form: every array equals
    the encoding of the dense mask (which the dense tests pin to the oracle);
    sampled OT rows also against the oracle directly."""
    w = synth.WORKLOADS["bernoulli_L16384"]
    L = w.L
    thr = synth.bernoulli_threshold(synth.BERNOULLI_P)
    bits = torch.empty(w.n_masks, L, L // 8, dtype=torch.uint8, device="cuda")
    stof.stof_synth_causal_bernoulli_mask_bits(bits, w.n_masks, L, w.seed, thr)
    ws_b = torch.empty(stof.stof_encode_workspace_bytes(w.n_masks, L, L, 128, 128), dtype=torch.uint8,
                       device="cuda")
    fb = stof.stof_encode_mask_bits(bits, L, 128, 128, ws_b)
    stof.stof_format_sync(fb)
    del bits
    torch.cuda.empty_cache()
    ab = stof.format_arrays(fb, ws_b)
    for m, I in ((0, 0), (31, 127), (7, 93)):
        band = synth.mask_rows(w, m, np.arange(I * 128, I * 128 + 128))[None]
        want = oracle.encode(band, 128, 128)
        r = m * 128 + I
        prp = ab["part_row_ptr"].cpu().numpy()
        assert np.array_equal(ab["part_col_idx"][prp[r]:prp[r + 1]].cpu().numpy(), want["part_col_idx"])
        assert np.array_equal(ab["bitmaps"][prp[r]:prp[r + 1]].cpu().numpy().view("uint64"), want["bitmaps"])
    dense = torch.empty(w.n_masks, L, L, dtype=torch.uint8, device="cuda")
    stof.stof_synth_causal_bernoulli_mask(dense, w.n_masks, L, w.seed, thr)
    ws_d = torch.empty_like(ws_b)
    fd = stof.stof_encode_mask(dense, 128, 128, ws_d)
    stof.stof_format_sync(fd)
    del dense
    torch.cuda.empty_cache()
    assert (fb.n_full, fb.n_part, fb.nnz) == (fd.n_full, fd.n_part, fd.nnz)
    ad = stof.format_arrays(fd, ws_d)
    for key in ("full_row_ptr", "part_row_ptr", "part_col_idx", "bitmaps"):
        assert torch.equal(ab[key], ad[key]), key
