"""Concurrent use of the library: calls from two host threads, each on its
own CUDA stream with its own format and workspace, give the same outputs,
bit for bit, as the same calls made one after the other.  The shared state
the calls touch is host-side (the tensor-map cache, the once-per-device
kernel set-up, the tuning cache) and the persistent kernel's work counter,
which lives in each format's own workspace."""
import math
import threading

import numpy as np
import pytest
import torch

from sparse_mask_transformer_gb300 import stof, synth

pytestmark = pytest.mark.gpu


def _job(seed, L, d, which):
    masks = torch.from_numpy(synth.random_mask(2, L, L, 0.3, seed=seed)).cuda()
    q, k, v = (t.cuda() for t in synth.make_qkv(1, 2, L, d, "bf16", seed=seed))
    ws = torch.empty(stof.stof_encode_workspace_bytes(2, L, L, 128, 128), dtype=torch.uint8, device="cuda")
    return dict(masks=masks, q=q, k=k, v=v, ws=ws, o=torch.empty_like(q), d=d, which=which)


def _run(job, stream, repeats):
    with torch.cuda.stream(stream):
        for _ in range(repeats):
            fmt = stof.stof_encode_mask(job["masks"], 128, 128, job["ws"], stream=stream)
            stof.stof_format_sync(fmt, stream)
            stof.stof_mha_fwd(job["q"], job["k"], job["v"], fmt, 1 / math.sqrt(job["d"]), 0, 1, job["which"],
                              job["o"], stream=stream)
        stream.synchronize()
        stof.stof_format_sync(fmt, stream)
        assert fmt.device_error == 0


@pytest.mark.parametrize("which", [stof.STOF_KERNEL_BLOCKWISE, stof.STOF_KERNEL_ROWWISE, stof.STOF_KERNEL_AUTO])
def test_two_threads_two_streams(gpu_lib, which):
    jobs = [_job(1, 1024, 64, which), _job(2, 768, 128, which), _job(3, 1000, 64, which)]
    # serial references
    refs = []
    for j in jobs:
        _run(j, torch.cuda.current_stream(), 1)
        refs.append(j["o"].clone())
        j["o"].zero_()
    # concurrent: one thread and one stream per job, several rounds each
    errors = []

    def worker(j):
        try:
            _run(j, torch.cuda.Stream(), 5)
        except Exception as e:  # reported below, in the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(j,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors
    torch.cuda.synchronize()
    for j, ref in zip(jobs, refs):
        assert torch.equal(j["o"], ref)
