"""GPU mask encoder against the brute-force oracle encoder: bit-exact
pointer arrays, tile lists and bitmaps ("Accelerating Sparse Transformer
Inference on GPU", gist.science technical summary, Methodology 1,
two-level storage format)."""
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


def test_bernoulli_L16384_full_size_sampled(gpu_lib):
    """The 16k workload at full size (8.6 GB mask made on the device):
    sampled OT rows bit-exact against the oracle, global counts against an
    independent count."""
    w = synth.WORKLOADS["bernoulli_L16384"]
    L = w.L
    mask = torch.empty(w.n_masks, L, L, dtype=torch.uint8, device="cuda")
    stof.stof_synth_causal_bernoulli_mask(mask, w.n_masks, L, w.seed,
                                          synth.bernoulli_threshold(synth.BERNOULLI_P))
    rng = np.random.default_rng(0)
    rows = [(0, 0), (31, 127), (5, 64)] + [(int(m), int(I)) for m, I in
                                           zip(rng.integers(0, 32, 3), rng.integers(0, 128, 3))]
    for m, I in rows[:2]:  # the device generator agrees with the host one here
        band = synth.mask_rows(w, m, np.arange(I * 128, I * 128 + 128))
        assert np.array_equal(mask[m, I * 128:(I + 1) * 128].cpu().numpy(), band)
    fmt, ws, arrs = gpu_encode(mask, 128, 128)
    assert fmt.nnz == int(mask.sum(dtype=torch.int64).item())
    frp, prp = arrs["full_row_ptr"], arrs["part_row_ptr"]
    assert np.all(np.diff(frp) >= 0) and np.all(np.diff(prp) >= 0)
    assert frp[-1] == fmt.n_full and prp[-1] == fmt.n_part
    for m, I in rows:
        band = synth.mask_rows(w, m, np.arange(I * 128, I * 128 + 128))[None]
        want = oracle.encode(band, 128, 128)
        r = m * 128 + I
        fc = arrs["full_col_idx"][frp[r]:frp[r + 1]]
        pc = arrs["part_col_idx"][prp[r]:prp[r + 1]]
        assert np.array_equal(fc, want["full_col_idx"])
        assert np.array_equal(pc, want["part_col_idx"])
        assert np.array_equal(arrs["bitmaps"][prp[r]:prp[r + 1]], want["bitmaps"])
    del mask, ws
    torch.cuda.empty_cache()
