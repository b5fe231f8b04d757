"""Pins for the CPU oracle: each check ties an oracle function to something
other than itself (a library routine, a closed form, a hand-derived fixture,
a tiny brute force, or a round trip), chosen so that a dropped term, a wrong
sign or index, or a transposed operand fails at least one of them.

Method: "Accelerating Sparse Transformer Inference on GPU" (gist.science
technical summary), Methodology 1, Unified MHA module: exact masking over a
two-level format (outer tiles empty / full / partial, one uint64 per 8x8
inner tile of a partial outer tile).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from sparse_mask_transformer_gb300 import synth
from tests.conftest import read_golden


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, mask, scale):
    """torch's own fp64 attention (library routine) for one head."""
    tq, tk, tv = (torch.from_numpy(x)[None, None] for x in (q, k, v))
    am = torch.from_numpy(mask.astype(bool))[None, None]
    return F.scaled_dot_product_attention(tq, tk, tv, attn_mask=am, scale=scale)[0, 0].numpy()


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("n_q,lk,d", [(1, 1, 64), (37, 53, 64), (64, 200, 128), (5, 300, 16)])
def test_all_ones_mask_is_dense_attention(n_q, lk, d):
    q, k, v = _rand((n_q, d), 1), _rand((lk, d), 2), _rand((lk, d), 3)
    scale = 1 / math.sqrt(d)
    o = oracle.attention(q, k, v, np.ones((n_q, lk), np.uint8), scale)
    tq, tk, tv = (torch.from_numpy(x)[None, None] for x in (q, k, v))
    ref = F.scaled_dot_product_attention(tq, tk, tv, scale=scale)[0, 0].numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)
    # and against the textbook two-pass softmax written with numpy ops
    s = scale * q @ k.T
    p = np.exp(s - s.max(axis=1, keepdims=True))
    np.testing.assert_allclose(o, (p @ v) / p.sum(axis=1, keepdims=True), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("density", [0.05, 0.3, 0.9])
def test_random_mask_matches_library_masked_attention(density):
    n_q, lk, d = 96, 160, 64
    q, k, v = _rand((n_q, d), 4), _rand((lk, d), 5), _rand((lk, d), 6)
    mask = (np.random.default_rng(7).random((n_q, lk)) < density).astype(np.uint8)
    mask[3] = 0  # one fully masked row
    scale = 0.125
    o = oracle.attention(q, k, v, mask, scale)
    rows = mask.any(axis=1)
    ref = _sdpa(q, k, v, mask, scale)
    np.testing.assert_allclose(o[rows], ref[rows], rtol=1e-11, atol=1e-12)
    assert np.all(o[~rows] == 0.0)


def test_causal_matches_library_is_causal():
    L, d = 130, 32
    q, k, v = _rand((L, d), 8), _rand((L, d), 9), _rand((L, d), 10)
    o = oracle.attention(q, k, v, np.tril(np.ones((L, L), np.uint8)), 0.3)
    tq, tk, tv = (torch.from_numpy(x)[None, None] for x in (q, k, v))
    ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=0.3)[0, 0].numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_mask_orientation_is_query_by_key():
    # a non-symmetric mask: transposing it must change the answer
    L, d = 24, 8
    q, k, v = _rand((L, d), 11), _rand((L, d), 12), _rand((L, d), 13)
    m = np.triu(np.ones((L, L), np.uint8))
    o = oracle.attention(q, k, v, m, 1.0)
    np.testing.assert_allclose(o, _sdpa(q, k, v, m, 1.0), rtol=1e-12, atol=1e-12)
    assert not np.allclose(o, oracle.attention(q, k, v, m.T.copy(), 1.0))


def test_single_valid_key_returns_that_value_row_exactly():
    n_q, lk, d = 50, 70, 64
    q, k, v = _rand((n_q, d), 14) * 30, _rand((lk, d), 15), _rand((lk, d), 16)
    mask = np.zeros((n_q, lk), np.uint8)
    js = np.random.default_rng(17).integers(0, lk, n_q)
    mask[np.arange(n_q), js] = 1
    o = oracle.attention(q, k, v, mask, 0.125)
    assert np.array_equal(o, v[js])  # softmax of one element is exactly 1


def test_key_order_does_not_matter():
    # permuting the keys (rows of K and V with the mask's columns) is a
    # relabelling of the sum over valid keys: O is unchanged
    n_q, lk, d = 40, 90, 32
    q, k, v = _rand((n_q, d), 40), _rand((lk, d), 41), _rand((lk, d), 42)
    mask = (np.random.default_rng(43).random((n_q, lk)) < 0.3).astype(np.uint8)
    perm = np.random.default_rng(44).permutation(lk)
    o = oracle.attention(q, k, v, mask, 0.2)
    o_p = oracle.attention(q, k[perm], v[perm], mask[:, perm], 0.2)
    assert np.allclose(o, o_p, rtol=0, atol=1e-13)


def test_output_is_linear_in_values():
    # the softmax weights do not depend on V: O(a V1 + b V2) = a O(V1) + b O(V2)
    n_q, lk, d = 30, 70, 16
    q, k = _rand((n_q, d), 45), _rand((lk, d), 46)
    v1, v2 = _rand((lk, d), 47), _rand((lk, d), 48)
    mask = (np.random.default_rng(49).random((n_q, lk)) < 0.4).astype(np.uint8)
    o = oracle.attention(q, k, 2.5 * v1 - 0.75 * v2, mask, 0.3)
    want = 2.5 * oracle.attention(q, k, v1, mask, 0.3) - 0.75 * oracle.attention(q, k, v2, mask, 0.3)
    assert np.allclose(o, want, rtol=0, atol=1e-12)


def test_shifting_every_key_by_one_vector_changes_nothing():
    # k_j + c adds scale * q_i . c to every score of row i: softmax is
    # invariant to a per-row constant, so O is unchanged (shifts of ~1000
    # and more, beyond exp's fp64 range: only a max-subtracting softmax
    # survives them)
    n_q, lk, d = 25, 60, 16
    q, k, v = _rand((n_q, d), 50) * 4, _rand((lk, d), 51), _rand((lk, d), 52)
    c = _rand((d,), 53) * 200
    mask = (np.random.default_rng(54).random((n_q, lk)) < 0.5).astype(np.uint8)
    o = oracle.attention(q, k, v, mask, 0.5)
    assert np.abs(0.5 * (q @ c)).max() > 800
    o_s = oracle.attention(q, k + c, v, mask, 0.5)
    assert np.allclose(o, o_s, rtol=0, atol=1e-9)


def test_fully_masked_rows_are_zero():
    q, k, v = _rand((4, 8), 18), _rand((9, 8), 19), _rand((9, 8), 20)
    o = oracle.attention(q, k, v, np.zeros((4, 9), np.uint8), 1.0)
    assert np.array_equal(o, np.zeros((4, 8)))


@pytest.mark.parametrize("L", [8, 16, 24])
def test_tiny_brute_force_unstabilised_formula(L):
    # o_i = sum_j m_ij e^{s_ij} v_j / sum_j m_ij e^{s_ij}, pure Python loops
    d = 4
    q, k, v = _rand((L, d), 21 + L), _rand((L, d), 22 + L), _rand((L, d), 23 + L)
    mask = (np.random.default_rng(24 + L).random((L, L)) < 0.4).astype(np.uint8)
    mask[0] = 0
    scale = 0.7
    o = oracle.attention(q, k, v, mask, scale)
    for i in range(L):
        num = [0.0] * d
        den = 0.0
        for j in range(L):
            if mask[i, j]:
                w = math.exp(scale * sum(q[i, t] * k[j, t] for t in range(d)))
                den += w
                for t in range(d):
                    num[t] += w * v[j, t]
        want = [x / den for x in num] if den > 0 else [0.0] * d
        np.testing.assert_allclose(o[i], want, rtol=1e-12, atol=1e-13)


def test_large_scores_stay_finite():
    # the max-shift keeps exp() in range where the unstabilised form overflows
    q = np.full((2, 4), 40.0)
    k = np.array([[40.0] * 4, [39.0] * 4, [-5.0] * 4])
    v = np.array([[1.0, 0, 0, 0], [0, 1.0, 0, 0], [0, 0, 1.0, 0]])
    o = oracle.attention(q, k, v, np.ones((2, 3), np.uint8), 1.0)
    w1 = math.exp(-160.0)  # s = 6400, 6240, -800
    np.testing.assert_allclose(o[0], [1 / (1 + w1), w1 / (1 + w1), 0, 0], rtol=1e-15, atol=1e-300)


def test_golden_tiny_attention():
    g = read_golden("attention_tiny.txt")
    q = np.array([[float(x) for x in g["q"].split()]])
    k = np.array([[float(x) for x in r.split()] for r in g["k"].split(";")])
    v = np.array([[float(x) for x in r.split()] for r in g["v"].split(";")])
    for case in g["case"]:
        m, want = case.split("->")
        mask = np.array([[int(x) for x in m.split()]], np.uint8)
        o = oracle.attention(q, k, v, mask, float(g["scale"]))
        np.testing.assert_allclose(o[0], [float(x) for x in want.split()], rtol=1e-14, atol=1e-14)


def test_threads_do_not_change_results():
    q, k, v = _rand((301, 64), 25), _rand((77, 64), 26), _rand((77, 64), 27)
    mask = (np.random.default_rng(28).random((301, 77)) < 0.5).astype(np.uint8)
    a = oracle.attention(q, k, v, mask, 0.125, n_threads=1)
    b = oracle.attention(q, k, v, mask, 0.125, n_threads=7)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- encoder

def _golden_format(name):
    g = read_golden(name)
    ints = lambda s: np.array([int(x, 0) for x in s.split()], dtype=np.int64)
    return g, dict(
        full_row_ptr=ints(g["full_row_ptr"]), full_col_idx=ints(g["full_col_idx"]),
        part_row_ptr=ints(g["part_row_ptr"]), part_col_idx=ints(g["part_col_idx"]),
        bitmaps=np.array([int(x, 16) for x in g["bitmaps"].split()], dtype=np.uint64))


@pytest.mark.parametrize("name", ["encode_causal16_ot8.txt", "encode_upper16x32_ot8x16.txt"])
def test_golden_encodings(name):
    g, want = _golden_format(name)
    lq, lk, bm, bn = (int(g[x]) for x in ("lq", "lk", "bm", "bn"))
    i = np.arange(lq)[:, None]
    j = np.arange(lk)[None, :]
    mask = ((j <= i) if g["pattern"] == "causal" else (j >= i)).astype(np.uint8)[None]
    fmt = oracle.encode(mask, bm, bn)
    for key in ("full_row_ptr", "full_col_idx", "part_row_ptr", "part_col_idx"):
        assert fmt[key].tolist() == want[key].tolist(), key
    assert fmt["bitmaps"].reshape(-1).tolist() == want["bitmaps"].tolist()
    assert fmt["nnz"] == int(g["nnz"])
    assert np.array_equal(oracle.decode(fmt), mask)


def test_every_single_bit_position():
    # 64 masks of one 8x8 tile, one valid element each: the tile is partial
    # and its word has exactly the bit of that element (row-major, bit 0 =
    # top-left).  Read back through the hand-derived rule r = b // 8, c = b % 8.
    for b in range(64):
        mask = np.zeros((1, 8, 16), np.uint8)
        mask[0, b // 8, 8 + b % 8] = 1  # second IT column: pins the IT order too
        fmt = oracle.encode(mask, 8, 16)
        assert fmt["n_full"] == 0 and fmt["n_part"] == 1 and fmt["nnz"] == 1
        words = fmt["bitmaps"].reshape(-1)
        assert int(words[0]) == 0
        assert int(words[1]) == 1 << b
        assert np.array_equal(oracle.decode(fmt), mask)


def test_tile_classes_from_hand_built_masks():
    mask = np.zeros((2, 32, 32), np.uint8)
    mask[0, 0:16, 16:32] = 1          # mask 0: OT(0,1) full at 16x16
    mask[0, 20, 3] = 1                # mask 0: OT(1,0) partial, one element
    mask[1] = 1                       # mask 1: all four OTs full
    fmt = oracle.encode(mask, 16, 16)
    assert fmt["full_row_ptr"].tolist() == [0, 1, 1, 3, 5]
    assert fmt["full_col_idx"].tolist() == [1, 0, 1, 0, 1]
    assert fmt["part_row_ptr"].tolist() == [0, 0, 1, 1, 1]
    assert fmt["part_col_idx"].tolist() == [0]
    words = fmt["bitmaps"][0]         # [2][2] ITs; element (20,3) -> IT(0,0), r=4, c=3
    assert int(words[0, 0]) == 1 << (8 * 4 + 3)
    assert int(words.sum()) == 1 << 35
    assert fmt["nnz"] == 256 + 1 + 32 * 32
    assert oracle.encode_count(np.zeros((1, 64, 64), np.uint8), 32, 32) == (0, 0, 0)


@pytest.mark.parametrize("bm,bn", [(8, 8), (16, 16), (8, 16), (24, 8), (32, 64)])
@pytest.mark.parametrize("density", [0.0, 0.02, 0.5, 0.98, 1.0])
def test_encode_decode_round_trip_random(bm, bn, density):
    mask = synth.random_mask(3, 96, 128, density, seed=int(density * 100) + bm + bn)
    fmt = oracle.encode(mask, bm, bn)
    assert np.array_equal(oracle.decode(fmt), mask)
    assert fmt["nnz"] == int(mask.sum())
    n_tiles = 3 * (96 // bm) * (128 // bn)
    assert fmt["n_full"] + fmt["n_part"] <= n_tiles
    assert np.all(np.diff(fmt["full_row_ptr"]) >= 0) and np.all(np.diff(fmt["part_row_ptr"]) >= 0)


def test_window48_tile_counts_closed_form():
    # valid iff 0 <= i - j < 48.  At 16x16 an OT(I,J) spans i - j in
    # [16(I-J) - 15, 16(I-J) + 15]: full iff I-J in {1, 2} (15 + 14 = 29),
    # partial iff I-J in {0, 3} (16 + 13 = 29), empty otherwise (198).
    # At 128x128: OT(0,0), OT(1,1) partial (diagonal), OT(1,0) partial
    # (i - j spans [1, 255]), OT(0,1) empty.
    w = synth.WORKLOADS["window48_L256"]
    mask = synth.make_mask(w)
    assert oracle.encode_count(mask, 16, 16) == (29, 29, 11160)
    assert oracle.encode_count(mask, 128, 128) == (0, 3, 11160)
    assert 11160 == sum(min(i + 1, 48) for i in range(256))


def test_causal_tile_counts_closed_form():
    # causal L = 2048 at 128x128, n = 16 OT rows: n(n-1)/2 = 120 full tiles
    # strictly below the diagonal, n = 16 partial diagonal tiles; nnz = L(L+1)/2
    w = synth.WORKLOADS["causal_L2048"]
    mask = synth.make_mask(w)
    assert oracle.encode_count(mask, 128, 128) == (120, 16, 2048 * 2049 // 2)
    fmt = oracle.encode(mask, 128, 128)
    assert np.array_equal(oracle.decode(fmt), mask)
    assert fmt["full_row_ptr"].tolist() == [I * (I - 1) // 2 for I in range(17)]
    assert fmt["part_col_idx"].tolist() == list(range(16))


@pytest.mark.parametrize("name", ["window48_L256", "bigbird_L512", "causal_L2048", "longformer_L4096"])
def test_workload_masks_round_trip(name):
    w = synth.WORKLOADS[name]
    mask = synth.make_mask(w)
    fmt = oracle.encode(mask, 128, 128)
    assert np.array_equal(oracle.decode(fmt), mask)
    assert fmt["nnz"] == int(mask.sum())


def test_oproj_brute_force_tiny():
    # the definition written out as loops on a tiny case
    rng = np.random.default_rng(11)
    B, H, L, d, N = 2, 3, 4, 2, 5
    o = rng.standard_normal((B, H, L, d))
    w = rng.standard_normal((N, H * d))
    bias = rng.standard_normal(N)
    res = rng.standard_normal((B, L, N))
    y = oracle.oproj(o, w, bias, res)
    for b in range(B):
        for l in range(L):
            for n in range(N):
                acc = bias[n] + res[b, l, n]
                for h in range(H):
                    for c in range(d):
                        acc += o[b, h, l, c] * w[n, h * d + c]
                assert abs(y[b, l, n] - acc) < 1e-12


def test_oproj_identity_weight_concatenates_heads():
    # W = I: y is the heads' outputs side by side (plus bias and residual)
    rng = np.random.default_rng(12)
    B, H, L, d = 1, 4, 3, 8
    o = rng.standard_normal((B, H, L, d))
    y = oracle.oproj(o, np.eye(H * d), np.zeros(H * d), None)
    for h in range(H):
        assert np.array_equal(y[0, :, h * d:(h + 1) * d], o[0, h])
    assert np.array_equal(oracle.oproj(o, np.zeros((5, H * d)), np.arange(5.0), None)[0, 2], np.arange(5.0))


def test_unpack_bits_inverts_numpy_packbits():
    rng = np.random.default_rng(13)
    m = (rng.random((3, 5, 64)) < 0.3).astype(np.uint8)
    assert np.array_equal(oracle.unpack_bits(np.packbits(m, axis=-1, bitorder="little"), 64), m)
    one = np.zeros((1, 16), np.uint8)
    one[0, 9] = 1                                  # key 9 = bit 1 of byte 1
    assert list(np.packbits(one, axis=-1, bitorder="little")[0]) == [0, 2]
    assert np.array_equal(oracle.unpack_bits(np.array([[0, 2]], np.uint8), 16), one)


# ---------------------------------------------------------------- parametric masks

def test_rule_mask_bands_match_numpy_triangles():
    """A band on i - j is a pair of numpy triangles: causal = tril, a causal
    window of w keys = tril - tril(-w), a symmetric window = triu(tril(w), -w)."""
    L = 97
    ones = np.ones((L, L), np.uint8)
    assert np.array_equal(oracle.rule_mask(L, L, 0, (1 << 31) - 1), np.tril(ones))
    assert np.array_equal(oracle.rule_mask(L, L, 0, 47), np.tril(ones) - np.tril(ones, -48))
    assert np.array_equal(oracle.rule_mask(L, L, -5, 5), np.triu(np.tril(ones, 5), -5))
    assert np.array_equal(oracle.rule_mask(L, L, -(1 << 31), (1 << 31) - 1), ones)
    assert not oracle.rule_mask(L, L, 1, 0).any()                     # empty band
    rect = oracle.rule_mask(40, 72, -3, 10)                            # non-square: i - j on the full grid
    assert np.array_equal(rect, np.triu(np.tril(np.ones((40, 72), np.uint8), 3), -10))


def test_rule_mask_sets_match_their_definitions():
    rng = np.random.default_rng(5)
    lq, lk, blk = 64, 128, 16
    gr, gc = rng.random(lq) < 0.2, rng.random(lk) < 0.1
    blocks = rng.random((lq // blk, lk // blk)) < 0.3
    empty = dict(band_lo=1, band_hi=0)
    assert np.array_equal(oracle.rule_mask(lq, lk, global_rows=gr, **empty),
                          np.repeat(gr[:, None], lk, 1).astype(np.uint8))
    assert np.array_equal(oracle.rule_mask(lq, lk, global_cols=gc, **empty),
                          np.repeat(gc[None, :], lq, 0).astype(np.uint8))
    assert np.array_equal(oracle.rule_mask(lq, lk, blocks=blocks, block=blk, **empty),
                          np.kron(blocks, np.ones((blk, blk))).astype(np.uint8))
    both = oracle.rule_mask(lq, lk, 0, 3, global_rows=gr, global_cols=gc, blocks=blocks, block=blk)
    union = (oracle.rule_mask(lq, lk, 0, 3) | oracle.rule_mask(lq, lk, global_rows=gr, **empty)
             | oracle.rule_mask(lq, lk, global_cols=gc, **empty)
             | oracle.rule_mask(lq, lk, blocks=blocks, block=blk, **empty))
    assert np.array_equal(both, union)


@pytest.mark.parametrize("name", ["window48_L256", "bigbird_L512", "causal_L2048", "longformer_L4096"])
def test_workload_rules_reproduce_the_workload_masks(name):
    """The rule form of each structured workload equals its element generator
    (two independent descriptions of the same mask)."""
    w = synth.WORKLOADS[name]
    assert np.array_equal(oracle.rule_mask(w.L, w.L, **synth.workload_rule(w)), synth.make_mask(w)[0])
    assert synth.workload_rule(synth.WORKLOADS["bernoulli_L16384"]) is None


# ---------------------------------------------------------------- LayerNorm after the projection

def test_layer_norm_matches_the_library_routine():
    import torch
    rng = np.random.default_rng(31)
    x = rng.standard_normal((7, 96)) * 3 + 5
    g, b = rng.standard_normal(96), rng.standard_normal(96)
    for eps in (1e-5, 1e-12, 0.3):
        want = torch.nn.functional.layer_norm(torch.from_numpy(x), (96,), torch.from_numpy(g),
                                              torch.from_numpy(b), eps).numpy()
        assert np.allclose(oracle.layer_norm(x, g, b, eps), want, rtol=0, atol=1e-12)


def test_layer_norm_closed_forms():
    # a constant row has zero deviation: the output is beta
    b = np.arange(6.0)
    assert np.array_equal(oracle.layer_norm(np.full((1, 6), 4.25), np.ones(6), b, 1e-5)[0], b)
    # +a, -a alternating: mean 0, variance a^2, so y = +-a / sqrt(a^2 + eps)
    a, eps = 2.0, 0.25
    x = np.array([[a, -a, a, -a]])
    want = np.array([a, -a, a, -a]) / np.sqrt(a * a + eps)
    assert np.allclose(oracle.layer_norm(x, None, None, eps)[0], want, rtol=1e-15, atol=0)
    # gamma scales and beta shifts each feature
    g = np.array([1.0, 2.0, -1.0, 0.5])
    assert np.allclose(oracle.layer_norm(x, g, np.ones(4), eps)[0], want * g + 1, rtol=1e-15, atol=0)


def test_layer_norm_invariances():
    rng = np.random.default_rng(32)
    x = rng.standard_normal((3, 64))
    y = oracle.layer_norm(x, None, None, 0.0)
    # shift invariance, positive scale invariance (eps = 0), zero mean and unit variance
    assert np.allclose(oracle.layer_norm(x + 7.5, None, None, 0.0), y, atol=1e-12)
    assert np.allclose(oracle.layer_norm(x * 3.0, None, None, 0.0), y, atol=1e-12)
    assert np.allclose(y.mean(axis=-1), 0, atol=1e-14)
    assert np.allclose((y * y).mean(axis=-1), 1, atol=1e-12)


def test_oproj_ln_is_layer_norm_of_the_projection():
    rng = np.random.default_rng(33)
    o = rng.standard_normal((2, 3, 4, 8))
    w = rng.standard_normal((16, 24))
    bias, res = rng.standard_normal(16), rng.standard_normal((2, 4, 16))
    g, b = rng.standard_normal(16), rng.standard_normal(16)
    z = oracle.oproj(o, w, bias, res)
    assert np.array_equal(oracle.oproj_ln(o, w, bias, res, g, b, 1e-5), oracle.layer_norm(z, g, b, 1e-5))


def test_rule_mask_rows_are_rows_of_the_whole_mask():
    rng = np.random.default_rng(34)
    L = 96
    r = dict(band_lo=-5, band_hi=9, global_rows=rng.random(L) < 0.1, global_cols=rng.random(L) < 0.1,
             blocks=rng.random((L // 8, L // 8)) < 0.2, block=8)
    rows = np.array([0, 7, 8, 50, 95])
    assert np.array_equal(oracle.rule_mask(L, L, rows=rows, **r), oracle.rule_mask(L, L, **r)[rows])


@pytest.mark.parametrize("lq,lk,bm,bn", [(250, 256, 128, 128), (77, 130, 16, 24), (1, 1, 8, 8), (129, 200, 64, 128)])
def test_padded_sides_closed_forms(lq, lk, bm, bn):
    """A side that is not a whole number of OTs is read as padded with invalid
    elements: an all-valid lq x lk mask then has floor(lq/bm) * floor(lk/bn)
    full OTs, every other OT of the ceil(lq/bm) x ceil(lk/bn) grid partial,
    and lq * lk valid elements; decoding gives the mask back."""
    mask = np.ones((1, lq, lk), np.uint8)
    f = oracle.encode(mask, bm, bn)
    n_tr, n_tc = -(-lq // bm), -(-lk // bn)
    assert (f["n_tr"], f["n_tc"], f["lq"], f["lk"]) == (n_tr, n_tc, lq, lk)
    assert f["n_full"] == (lq // bm) * (lk // bn)
    assert f["n_part"] == n_tr * n_tc - f["n_full"]
    assert f["nnz"] == lq * lk
    assert np.array_equal(oracle.decode(f), mask)
    rng = np.random.default_rng(lq + lk)
    m2 = (rng.random((2, lq, lk)) < 0.3).astype(np.uint8)
    assert np.array_equal(oracle.decode(oracle.encode(m2, bm, bn)), m2)
