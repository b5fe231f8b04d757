import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    """Parse a `key = value` fixture; repeated keys collect into lists."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            out.setdefault(key, []).append(val)
    return {k: (v[0] if len(v) == 1 and k != "case" else v) for k, v in out.items()}


# ---------------------------------------------------------------- GPU helpers
# Used by the -m gpu tests only; they call the library through its C ABI.

TOL = {"fp16": 2e-3, "bf16": 1.5e-2}  # max |O_gpu - O_oracle|, fp32 accumulation


@pytest.fixture(scope="session")
def gpu_lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mask_transformer_gb300 import build, stof
    build.build()
    return stof.load_library()


def gpu_encode(mask_dev, bm, bn):
    """Encode a device mask; return (fmt, workspace, host dict of arrays)."""
    import torch
    from sparse_mask_transformer_gb300 import stof
    n_masks, lq, lk = mask_dev.shape
    ws = torch.empty(stof.stof_encode_workspace_bytes(n_masks, lq, lk, bm, bn),
                     dtype=torch.uint8, device=mask_dev.device)
    fmt = stof.stof_encode_mask(mask_dev, bm, bn, ws)
    stof.stof_format_sync(fmt)
    arrs = {k: v.cpu().numpy() for k, v in stof.format_arrays(fmt, ws).items()}
    arrs["bitmaps"] = arrs["bitmaps"].view("uint64")
    return fmt, ws, arrs


def assert_format_equal(fmt, arrs, want):
    import numpy as np
    assert (fmt.n_full, fmt.n_part, fmt.nnz) == (want["n_full"], want["n_part"], want["nnz"])
    assert fmt.device_error == 0
    for k in ("full_row_ptr", "part_row_ptr", "full_col_idx", "part_col_idx"):
        assert np.array_equal(arrs[k], want[k]), k
    assert np.array_equal(arrs["bitmaps"], want["bitmaps"].reshape(arrs["bitmaps"].shape))
