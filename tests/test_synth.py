"""Input generators: published test vectors and structural properties."""
import numpy as np

from sparse_mask_transformer_gb300 import synth


def test_splitmix64_reference_outputs():
    # SplitMix64 seeded with 0 (state advances by 0x9E3779B97F4A7C15 per call):
    # its first two outputs in Vigna's reference implementation.
    gamma = 0x9E3779B97F4A7C15
    out = synth.splitmix64(np.array([0, gamma], dtype=np.uint64))
    assert int(out[0]) == 0xE220A8397B1DCDAF
    assert int(out[1]) == 0x6E789E6AA1B965F4


def test_bernoulli_threshold_is_exact():
    t = synth.bernoulli_threshold(0.1)
    assert (t - 1) * 2.0 ** -53 < 0.1 <= t * 2.0 ** -53


def test_bernoulli_mask_structure():
    w = synth.WORKLOADS["bernoulli_L16384"]
    rows = np.array([0, 1, 2, 100, 8191, 16383])
    for h in (0, 31):
        m = synth.mask_rows(w, h, rows)
        assert m.shape == (len(rows), w.L)
        for r, i in enumerate(rows):
            assert m[r, i] == 1 and not m[r, i + 1:].any()
        below = m[-1, :16383]
        assert 0.09 < below.mean() < 0.11
    a = synth.mask_rows(w, 0, rows)
    b = synth.mask_rows(w, 1, rows)
    assert not np.array_equal(a, b)  # per-head masks differ


def test_bigbird_layout():
    w = synth.WORKLOADS["bigbird_L512"]
    lay = synth._bigbird_blocks(512, 64, 0)
    assert lay[0].all() and lay[1].all() and lay[:, 0].all() and lay[:, 1].all()
    for I in range(8):
        for J in (I - 1, I, I + 1):
            if 0 <= J < 8:
                assert lay[I, J]
    assert lay.sum() == 62  # rows 2 and 7 have one block left over
    m = synth.make_mask(w)
    assert m.shape == (1, 512, 512) and abs(m.mean() - 62 / 64) < 1e-12


def test_longformer_mask():
    w = synth.WORKLOADS["longformer_L4096"]
    g = synth._longformer_globals(4096, 0)
    assert len(set(g.tolist())) == 32
    m = synth.make_mask(w)[0]
    assert m[g].all() and m[:, g].all()
    i = 2000
    if i not in set(g.tolist()):
        assert m[i, i - 256] and m[i, i + 256]


def test_qkv_are_seeded_and_rounded():
    q, k, v = synth.make_qkv(1, 2, 16, 8, "bf16", seed=0)
    q2, _, _ = synth.make_qkv(1, 2, 16, 8, "bf16", seed=0)
    assert (q == q2).all() and not (q == k).all()
    assert str(q.dtype) == "torch.bfloat16"
