"""The no-allocation encoder entry point, stof_encode_mask_noalloc.

It exists for callers that cannot allocate device memory when they encode,
such as code running inside a memory pool or allocator callback, or a
runtime that plans every buffer ahead of time: its scratch lives in a
static device array of the library instead of the caller's workspace.  Its
output must be identical to the regular encoder's, also on a second call
in a row (the static scratch keeps the previous call's words, so the call
must clear them).  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from sparse_mask_transformer_gb300 import stof, synth
from tests.conftest import gpu_encode

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    fn = stof.load_library().stof_encode_mask_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(stof.stof_format), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _encode_noalloc(mask, bm, bn):
    n_masks, lq, lk = mask.shape
    ws = torch.empty(stof.stof_encode_workspace_bytes(n_masks, lq, lk, bm, bn), dtype=torch.uint8,
                     device=mask.device)
    fmt = stof.stof_format()
    status = _noalloc_fn()(mask.data_ptr(), n_masks, lq, lk, bm, bn, ws.data_ptr(), ws.numel(),
                           ctypes.byref(fmt), torch.cuda.current_stream().cuda_stream)
    assert status == stof.STOF_OK, stof.stof_status_string(status)
    stof.stof_format_sync(fmt)
    arrs = {k: v.cpu().numpy() for k, v in stof.format_arrays(fmt, ws).items()}
    arrs["bitmaps"] = arrs["bitmaps"].view("uint64")
    return fmt, arrs


def _assert_same(a_fmt, a, b_fmt, b):
    assert (a_fmt.n_full, a_fmt.n_part, a_fmt.nnz) == (b_fmt.n_full, b_fmt.n_part, b_fmt.nnz)
    assert a_fmt.device_error == 0 and b_fmt.device_error == 0
    for k in ("full_row_ptr", "part_row_ptr", "full_col_idx", "part_col_idx", "bitmaps"):
        assert np.array_equal(a[k], b[k]), k


def test_noalloc_encoder_matches_regular_encoder_two_calls_in_a_row(gpu_lib):
    """Masks A, B, A of one geometry (same chunk count) in a row: the
    look-back words that A leaves in the shared scratch are wrong prefixes
    for B, so a call that did not clear them would give B a wrong format."""
    cases = [
        (torch.from_numpy(synth.make_mask(synth.WORKLOADS["causal_L2048"])).cuda(),
         torch.from_numpy(synth.random_mask(1, 2048, 2048, 0.5, seed=13)).cuda(), 128, 128),
        (torch.from_numpy(synth.random_mask(3, 512, 4096, 0.01, seed=11)).cuda(),           # 768 chunks
         torch.from_numpy(synth.random_mask(3, 512, 4096, 0.3, seed=12)).cuda(), 8, 8),
    ]
    for mask_a, mask_b, bm, bn in cases:
        refs = {id(m): gpu_encode(m, bm, bn) for m in (mask_a, mask_b)}
        assert refs[id(mask_a)][0].n_part != refs[id(mask_b)][0].n_part
        for mask in (mask_a, mask_b, mask_a):
            ref_fmt, _, ref = refs[id(mask)]
            fmt, got = _encode_noalloc(mask, bm, bn)
            _assert_same(fmt, got, ref_fmt, ref)


def test_noalloc_encoder_on_sides_that_are_not_whole_tiles(gpu_lib):
    """A 1000 x 777 mask (edge chunks with byte-guarded loads, rows not
    8-byte aligned) gives the regular encoder's format."""
    mask = torch.from_numpy(synth.random_mask(2, 1000, 777, 0.2, seed=21)).cuda()
    ref_fmt, _, ref = gpu_encode(mask, 128, 128)
    fmt, got = _encode_noalloc(mask, 128, 128)
    _assert_same(fmt, got, ref_fmt, ref)


def test_noalloc_encoder_rejects_sizes_beyond_its_scratch(gpu_lib):
    # 5 masks of 65536^2 at 128x128 need 5 * 512 * 64 = 163840 chunks > 131072;
    # rejected on the host before any device access (the pointers are never used)
    fmt = stof.stof_format()
    fake = 1 << 20
    status = _noalloc_fn()(fake, 5, 65536, 65536, 128, 128, fake, 1 << 62, ctypes.byref(fmt), None)
    assert status == stof.STOF_ERR_SHAPE
