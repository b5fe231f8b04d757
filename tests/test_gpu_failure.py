"""Failure handling on the GPU without a fault: every pipeline wait in the
kernels is bounded in wall time and reports through a device error word.
stof_check_bounded_wait runs that same wait on a barrier nothing arrives on;
the test watches it give up, checks the status reaches the host (directly,
and through a format's error word and stof_format_sync), and that the
context then still runs attention correctly."""
import ctypes
import math
import time

import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof, synth
from tests.conftest import TOL, gpu_encode

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports(gpu_lib):
    err = torch.zeros(1, dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    stof.stof_check_bounded_wait(err, 0.2)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(err.item()) & stof.STOF_DEVERR_PIPE_TIMEOUT
    assert 0.19 <= elapsed < 5.0


def test_device_error_word_reaches_format_sync_and_context_survives(gpu_lib):
    w = synth.WORKLOADS["window48_L256"]
    mask = synth.make_mask(w)
    fmt, ws, _ = gpu_encode(torch.from_numpy(mask).cuda(), 128, 128)
    # the timeout lands in the format's device error word (counts_dev[3])
    st = gpu_lib.stof_check_bounded_wait(ctypes.c_void_p(fmt.counts_dev + 24), ctypes.c_double(0.1), None)
    assert st == stof.STOF_OK
    with pytest.raises(stof.StofError) as e:
        stof.stof_format_sync(fmt)
    assert e.value.status == stof.STOF_ERR_DEVICE
    assert fmt.device_error & stof.STOF_DEVERR_PIPE_TIMEOUT
    # a fresh encode clears the word, and attention still matches the oracle
    fmt2, ws2, _ = gpu_encode(torch.from_numpy(mask).cuda(), 128, 128)
    assert fmt2.device_error == 0
    q, k, v = synth.make_qkv(w.B, w.H, w.L, w.d, w.dtype, seed=w.seed)
    o = torch.empty_like(q).cuda()
    stof.stof_mha_fwd(q.cuda(), k.cuda(), v.cuda(), fmt2, 1 / math.sqrt(w.d), 0, 0,
                      stof.STOF_KERNEL_BLOCKWISE, o)
    torch.cuda.synchronize()
    qf, kf, vf = (synth.to_float64(t) for t in (q, k, v))
    for h in range(w.H):
        ref = oracle.attention(qf[0, h], kf[0, h], vf[0, h], mask[0], 1 / math.sqrt(w.d))
        assert np.abs(o[0, h].double().cpu().numpy() - ref).max() <= TOL[w.dtype]
