"""GPU mask encoder against the brute-force oracle encoder: bit-exact
pointer arrays, tile lists and bitmaps ("Accelerating Sparse Transformer
Inference on GPU", gist.science technical summary, Methodology 1,
two-level storage format)."""
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof, synth
from tests.conftest import assert_format_equal, gpu_encode

pytestmark = pytest.mark.gpu


def _dev(mask):
    return torch.from_numpy(np.ascontiguousarray(mask)).cuda()


@pytest.mark.parametrize("name", ["window48_L256", "bigbird_L512", "causal_L2048", "longformer_L4096"])
@pytest.mark.parametrize("ot", [128, 64, 16])
def test_workload_masks_bit_exact(gpu_lib, name, ot):
    w = synth.WORKLOADS[name]
    mask = synth.make_mask(w)
    fmt, ws, arrs = gpu_encode(_dev(mask), ot, ot)
    assert_format_equal(fmt, arrs, oracle.encode(mask, ot, ot))


@pytest.mark.parametrize("bm,bn", [(8, 8), (16, 16), (8, 16), (24, 8), (32, 64), (128, 128),
                                   (256, 256), (40, 200)])
@pytest.mark.parametrize("density", [0.0, 0.01, 0.5, 0.995, 1.0])
def test_random_masks_bit_exact(gpu_lib, bm, bn, density):
    lq = bm * 5
    lk = bn * 7
    mask = synth.random_mask(3, lq, lk, density, seed=bm * 7 + bn + int(density * 1000))
    fmt, ws, arrs = gpu_encode(_dev(mask), bm, bn)
    assert_format_equal(fmt, arrs, oracle.encode(mask, bm, bn))


def test_many_chunks_long_lookback(gpu_lib):
    # 2 x 64 OT rows x 4 chunks per row at 8x8 OTs: deep chained prefix sums
    mask = synth.random_mask(2, 512, 4096, 0.002, seed=5)
    fmt, ws, arrs = gpu_encode(_dev(mask), 8, 8)
    assert_format_equal(fmt, arrs, oracle.encode(mask, 8, 8))


def test_single_bits_pin_bit_order(gpu_lib):
    masks = np.zeros((64, 8, 16), np.uint8)
    for b in range(64):
        masks[b, b // 8, 8 + b % 8] = 1
    fmt, ws, arrs = gpu_encode(_dev(masks), 8, 16)
    assert fmt.n_part == 64 and fmt.n_full == 0 and fmt.nnz == 64
    words = arrs["bitmaps"].reshape(64, 2)
    assert np.all(words[:, 0] == 0)
    assert [int(x) for x in words[:, 1]] == [1 << b for b in range(64)]


def test_nonzero_bytes_count_as_valid(gpu_lib):
    mask = synth.random_mask(1, 64, 64, 0.5, seed=1) * np.uint8(200)
    fmt, ws, arrs = gpu_encode(_dev(mask), 16, 16)
    assert_format_equal(fmt, arrs, oracle.encode((mask != 0).astype(np.uint8), 16, 16))


def test_reuse_workspace_gives_same_result(gpu_lib):
    mask = synth.random_mask(2, 256, 256, 0.3, seed=9)
    dmask = _dev(mask)
    ws = torch.empty(stof.stof_encode_workspace_bytes(2, 256, 256, 32, 32), dtype=torch.uint8, device="cuda")
    ws.fill_(0xAB)  # garbage from an earlier user
    want = oracle.encode(mask, 32, 32)
    for _ in range(2):
        fmt = stof.stof_encode_mask(dmask, 32, 32, ws)
        stof.stof_format_sync(fmt)
        arrs = {k: v.cpu().numpy() for k, v in stof.format_arrays(fmt, ws).items()}
        arrs["bitmaps"] = arrs["bitmaps"].view("uint64")
        assert_format_equal(fmt, arrs, want)


def test_device_mask_generator_matches_numpy(gpu_lib):
    w = synth.WORKLOADS["bernoulli_L16384"]
    L = 1024
    n = 3
    out = torch.empty(n, L, L, dtype=torch.uint8, device="cuda")
    stof.stof_synth_causal_bernoulli_mask(out, n, L, w.seed, synth.bernoulli_threshold(synth.BERNOULLI_P))
    small = synth.Workload("t", 1, n, L, 128, "bf16", "causal_bernoulli", n, n, 1)
    for m in range(n):
        assert np.array_equal(out[m].cpu().numpy(), synth.mask_rows(small, m, np.arange(L)))


def _check_band(w, arrs, m, I):
    """OT row I of mask m of the 16k workload: the GPU's column lists,
    bitmaps and row-pointer increments against the oracle encoding of the
    same 128 mask rows regenerated on the host.  The mask is causal, so
    columns past the band's last row are zero and are not regenerated."""
    bm = 128
    ncols = (I + 1) * bm
    band = np.zeros((1, bm, w.L), np.uint8)
    band[0, :, :ncols] = synth.mask_rows(w, m, np.arange(I * bm, (I + 1) * bm), ncols=ncols)
    want = oracle.encode(band, bm, bm)
    r = m * (w.L // bm) + I
    frp, prp = arrs["full_row_ptr"], arrs["part_row_ptr"]
    assert frp[r + 1] - frp[r] == want["n_full"] and prp[r + 1] - prp[r] == want["n_part"], (m, I)
    assert np.array_equal(arrs["full_col_idx"][frp[r]:frp[r + 1]], want["full_col_idx"]), (m, I)
    assert np.array_equal(arrs["part_col_idx"][prp[r]:prp[r + 1]], want["part_col_idx"]), (m, I)
    assert np.array_equal(arrs["bitmaps"][prp[r]:prp[r + 1]], want["bitmaps"]), (m, I)
    return want["nnz"]


def test_bernoulli_L16384_full_size_every_ot_row(gpu_lib):
    """The 16k workload at full size (8.6 GB mask made on the device), every
    OT row of all 32 masks bit-exact against the oracle: row pointers (first
    entry 0 and every increment), full and partial column lists and all
    541 MB of bitmaps.  The host regenerates each 128-row band from the
    seeded generator, so no 8.6 GB host copy is needed."""
    from concurrent.futures import ThreadPoolExecutor
    w = synth.WORKLOADS["bernoulli_L16384"]
    L = w.L
    mask = torch.empty(w.n_masks, L, L, dtype=torch.uint8, device="cuda")
    stof.stof_synth_causal_bernoulli_mask(mask, w.n_masks, L, w.seed,
                                          synth.bernoulli_threshold(synth.BERNOULLI_P))
    fmt, ws, arrs = gpu_encode(mask, 128, 128)
    del mask, ws
    torch.cuda.empty_cache()
    assert fmt.device_error == 0
    frp, prp = arrs["full_row_ptr"], arrs["part_row_ptr"]
    n_rows = w.n_masks * (L // 128)
    assert len(frp) == n_rows + 1 and frp[0] == 0 and prp[0] == 0
    assert frp[-1] == fmt.n_full and prp[-1] == fmt.n_part
    bands = [(m, I) for m in range(w.n_masks) for I in range(L // 128)]
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        nnz = sum(ex.map(lambda mi: _check_band(w, arrs, *mi), bands))
    assert nnz == fmt.nnz
