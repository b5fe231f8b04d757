"""Output projection after the MHA with the fused bias + residual epilogue
(gist.science technical summary, Methodology 2: fusion carried past the MHA
layer) against the fp64 oracle.  Tolerance from the arithmetic: inputs are
exact fp16/bf16 values and sums accumulate in fp32 (relative error of the
sum far below the output's rounding), so the error is the output's single
rounding: |y - y_ref| <= 2^-8 (|y_ref| + 1) for bf16 and 2^-11 (|y_ref| + 1)
for fp16."""
import numpy as np
import pytest
import torch

import oracle
from sparse_mask_transformer_gb300 import stof, synth

pytestmark = pytest.mark.gpu

TOL_REL = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11}
DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def _case(B, H, L, d, N, dtype, bias=True, residual=True, seed=0):
    g = torch.Generator().manual_seed(seed)
    o = torch.randn(B, H, L, d, generator=g).to(DT[dtype])
    w = (torch.randn(N, H * d, generator=g) / (H * d) ** 0.5).to(DT[dtype])
    b = (0.1 * torch.randn(N, generator=g)).to(DT[dtype]) if bias else None
    r = torch.randn(B, L, N, generator=g).to(DT[dtype]) if residual else None
    err = torch.zeros(1, dtype=torch.int64, device="cuda")
    guard = 4096  # after y: must stay as it is (no row past L of the last batch element is stored)
    buf = torch.full((B * L * N + guard,), float("nan"), dtype=DT[dtype], device="cuda")
    y = buf[: B * L * N].view(B, L, N)
    cuda = lambda t: None if t is None else t.cuda()
    stof.stof_oproj_fwd(o.cuda(), w.cuda(), cuda(b), cuda(r), y, err)
    torch.cuda.synchronize()
    assert torch.isnan(buf[B * L * N:]).all()
    f64 = lambda t: None if t is None else t.double().numpy()
    want = oracle.oproj(f64(o), f64(w), f64(b), f64(r))
    got = y.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - want) <= TOL_REL[dtype] * (np.abs(want) + 1.0))
    assert int(err.item()) == 0
    return got, want


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [64, 128])
def test_small_shapes(gpu_lib, dtype, d):
    _case(2, 3, 256, d, 512, dtype, seed=d)


@pytest.mark.parametrize("bias,residual", [(False, False), (True, False), (False, True)])
def test_without_bias_or_residual(gpu_lib, bias, residual):
    _case(1, 2, 128, 64, 256, "bf16", bias=bias, residual=residual, seed=3)


def test_bert_base_layer_shape(gpu_lib):
    # BERT-base attention output: 12 heads x 64 = 768 features, 512 tokens x 16
    _case(16, 12, 512, 64, 768, "bf16", seed=4)


def test_more_tiles_than_sms(gpu_lib):
    # 8 x 1024 tokens / 128 x 1024 / 256 = 256 output tiles: more than one per SM, so CTAs loop
    _case(8, 8, 1024, 128, 1024, "fp16", seed=5)


def test_identity_weight_concatenates_heads(gpu_lib):
    B, H, L, d = 1, 4, 128, 64
    o = torch.randn(B, H, L, d, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    w = torch.eye(H * d).to(torch.bfloat16)
    y = torch.empty(B, L, H * d, dtype=torch.bfloat16, device="cuda")
    stof.stof_oproj_fwd(o.cuda(), w.cuda(), None, None, y)
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), o.transpose(1, 2).reshape(B, L, H * d))


@pytest.mark.parametrize("B,L,d", [(2, 100, 64), (3, 300, 128), (1, 1, 64), (2, 129, 64)])
def test_lengths_that_are_not_whole_tiles(gpu_lib, B, L, d):
    """Any sequence length: the last 128-token tile of each batch element
    runs past L (zeros read there, nothing stored)."""
    _case(B, 2, L, d, 256, "bf16", seed=L)


def test_shape_errors(gpu_lib):
    o = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(200, 128, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(1, 128, 200, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(stof.StofError) as e:
        stof.stof_oproj_fwd(o, w, None, None, y)
    assert e.value.status == stof.STOF_ERR_SHAPE          # N not a multiple of 256


# ---------------------------------------------------------------- with the LayerNorm that follows

def _ln_case(B, H, L, d, N, dtype, affine=True, offset=0.0, eps=1e-5, seed=0):
    """stof_oproj_ln_fwd against oracle.oproj_ln.  Error bound from the
    arithmetic: the pre-norm value z is rounded once to the input type
    (relative error u = 2^-8 for bf16, 2^-11 for fp16) before its statistics
    are taken, which moves a normalised value by at most
    u (|z_i| + mean|z| (1 + |y'_i|)) / sigma (y' = (z_i - mean) / sigma),
    scaled by |gamma_i|; the output's own rounding adds u |y|.  The test
    allows twice that sum."""
    u = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11}[dtype]
    g = torch.Generator().manual_seed(seed)
    o = torch.randn(B, H, L, d, generator=g).to(DT[dtype])
    w = (torch.randn(N, H * d, generator=g) / (H * d) ** 0.5).to(DT[dtype])
    b = (0.1 * torch.randn(N, generator=g)).to(DT[dtype])
    r = (torch.randn(B, L, N, generator=g) + offset).to(DT[dtype])
    gamma = (1 + 0.5 * torch.randn(N, generator=g)).to(DT[dtype]) if affine else None
    beta = (0.2 * torch.randn(N, generator=g)).to(DT[dtype]) if affine else None
    err = torch.zeros(1, dtype=torch.int64, device="cuda")
    y = torch.full((B, L, N), float("nan"), dtype=DT[dtype], device="cuda")
    ws = torch.empty(stof.stof_oproj_ln_workspace_bytes(B, L, N), dtype=torch.uint8, device="cuda")
    cuda = lambda t: None if t is None else t.cuda()  # noqa: E731
    stof.stof_oproj_ln_fwd(o.cuda(), w.cuda(), b.cuda(), r.cuda(), cuda(gamma), cuda(beta), eps, y, ws, err)
    torch.cuda.synchronize()
    f64 = lambda t: None if t is None else t.double().numpy()  # noqa: E731
    z = oracle.oproj(f64(o), f64(w), f64(b), f64(r))
    want = oracle.oproj_ln(f64(o), f64(w), f64(b), f64(r), f64(gamma), f64(beta), eps)
    got = y.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    mean = z.mean(axis=-1, keepdims=True)
    sigma = np.sqrt(z.var(axis=-1, keepdims=True) + eps)
    m_abs = np.abs(z).mean(axis=-1, keepdims=True)
    g_abs = np.abs(f64(gamma)) if gamma is not None else 1.0
    bound = 2 * u * (np.abs(want) + g_abs * (np.abs(z) + m_abs * (1 + np.abs((z - mean) / sigma))) / sigma)
    assert np.all(np.abs(got - want) <= bound), float(np.max(np.abs(got - want) / bound))
    assert int(err.item()) == 0


def test_ln_length_not_whole_tiles(gpu_lib):
    _ln_case(2, 4, 200, 64, 512, "bf16", seed=12)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_ln_bert_base_layer_shape(gpu_lib, dtype):
    _ln_case(16, 12, 512, 64, 768, dtype, seed=5)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("affine", [True, False])
def test_ln_llama_width(gpu_lib, dtype, affine):
    _ln_case(1, 32, 256, 128, 4096, dtype, affine=affine, seed=6)


def test_ln_rows_far_from_zero_mean(gpu_lib):
    # residual stream offset by 40: the statistics must not cancel
    _ln_case(2, 4, 128, 64, 512, "fp16", offset=40.0, seed=7)


def test_ln_constant_row_gives_beta(gpu_lib):
    """O = 0 and no bias: z is the residual; a constant residual row has no
    deviation, so its output is beta exactly."""
    B, H, L, d, N = 1, 2, 128, 64, 256
    o = torch.zeros(B, H, L, d, dtype=torch.bfloat16, device="cuda")
    w = torch.randn(N, H * d, device="cuda").to(torch.bfloat16)
    r = torch.randn(B, L, N, device="cuda").to(torch.bfloat16)
    r[0, 3] = 2.5
    beta = torch.randn(N, device="cuda").to(torch.bfloat16)
    gamma = torch.randn(N, device="cuda").to(torch.bfloat16)
    y = torch.empty(B, L, N, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(stof.stof_oproj_ln_workspace_bytes(B, L, N), dtype=torch.uint8, device="cuda")
    stof.stof_oproj_ln_fwd(o, w, None, r, gamma, beta, 1e-5, y, ws)
    torch.cuda.synchronize()
    assert torch.equal(y[0, 3], beta)


def test_ln_argument_errors(gpu_lib):
    B, H, L, d, N = 1, 2, 128, 64, 256
    o = torch.zeros(B, H, L, d, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(N, H * d, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(B, L, N, dtype=torch.bfloat16, device="cuda")
    need = stof.stof_oproj_ln_workspace_bytes(B, L, N)
    big = torch.empty(need + 16, dtype=torch.uint8, device="cuda")
    ws = big[:need]
    for eps, wsp, status in ((0.0, ws, stof.STOF_ERR_INVALID_ARG), (float("nan"), ws, stof.STOF_ERR_INVALID_ARG),
                             (1e-5, ws[:-8], stof.STOF_ERR_WORKSPACE),
                             (1e-5, big[8:8 + need], stof.STOF_ERR_ALIGNMENT)):
        with pytest.raises(stof.StofError) as e:
            stof.stof_oproj_ln_fwd(o, w, None, None, None, None, eps, y, wsp)
        assert e.value.status == status


@pytest.mark.parametrize("seed", range(24))
def test_random_shapes(gpu_lib, seed):
    """Seeded random batch sizes, head counts, lengths (whole token tiles or
    not), head sizes, widths, dtypes and epilogue parts, with and without
    the LayerNorm, each within the error bound of its case above."""
    rng = np.random.default_rng(9000 + seed)
    B, H, L = int(rng.integers(1, 4)), int(rng.integers(1, 17)), int(rng.integers(1, 700))
    d, N = int(rng.choice([64, 128])), 256 * int(rng.integers(1, 9))
    dtype = str(rng.choice(["bf16", "fp16"]))
    bias, residual = bool(rng.random() < 0.7), bool(rng.random() < 0.7)
    if rng.random() < 0.5:
        _case(B, H, L, d, N, dtype, bias=bias, residual=residual, seed=seed)
    else:
        _ln_case(B, H, L, d, N, dtype, affine=bool(rng.random() < 0.7), offset=float(rng.choice([0.0, 30.0])),
                 seed=seed)
