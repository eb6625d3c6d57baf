"""Pins for the fp64 CPU oracle: values the pages print, closed forms,
invariants, brute force on tiny inputs and library second opinions.

Each test is chosen so that a plausible mistake in the oracle (a dropped
scale, a transposed operand, an off-by-one in a mask, a wrong head block, an
unbiased variance, a missing residual) fails at least one of them.
"""

import math
import os

import numpy as np
import pytest

import oracle
from synth import inputs as synth
from tests import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows[key] = vals
    return rows


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- printed values

def test_softmax_printed_values():
    g = _golden("softmax_1_2_3.txt")
    s = np.array([float(x) for x in g["scores"]])
    w = oracle.softmax(s)
    printed = np.array([float(x) for x in g["weights_3dp"]])
    assert np.array_equal(np.round(w, 3), printed)
    assert abs(w.sum() - 1.0) < 1e-15
    w10 = oracle.softmax(np.array([float(x) for x in g["scores_x10"]]))
    # "close to 1" on the last entry; ordering preserved.
    assert w10[-1] > 0.9999 and w10[0] < w10[1] < w10[2]


def test_worked_example_reconstruction():
    g = _golden("worked_example_zuo.txt")
    d_k = int(g["d_k"][0])
    q = np.array([float(x) for x in g["q"]]).reshape(1, 1, 1, d_k)
    k = np.array([float(x) for x in g["k"]]).reshape(1, 3, 1, d_k)
    v = np.array([float(x) for x in g["v"]]).reshape(1, 3, 1, 2)
    out, w = oracle.attn_rows(q, k, v, 1.0 / math.sqrt(d_k), [(0, 0, 0)], weights=True)
    assert np.array_equal(np.round(w[0], 4), [float(x) for x in g["printed_weights_4dp"]])
    assert np.array_equal(np.round(out[0], 4), [float(x) for x in g["printed_output_4dp"]])
    # Without the 1/sqrt(d_k) scale the printed digits are NOT reproduced.
    out_noscale, w_noscale = oracle.attn_rows(q, k, v, 1.0, [(0, 0, 0)], weights=True)
    assert not np.array_equal(np.round(w_noscale[0], 4), [float(x) for x in g["printed_weights_4dp"]])


def test_causal_pattern_matches_printed_triu():
    rows = []
    with open(os.path.join(GOLDEN, "causal_mask_5x5.txt"), encoding="utf-8") as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([tok == "-inf" for tok in line.split()])
    masked = np.array(rows)
    rng = np.random.default_rng(11)
    n = 5
    q, k, v = _rand(rng, 1, n, 1, 4), _rand(rng, 1, n, 1, 4), _rand(rng, 1, n, 1, 3)
    sel = [(0, t, 0) for t in range(n)]
    _, w = oracle.attn_rows(q, k, v, 0.5, sel, mask_kind=oracle.MASK_CAUSAL, weights=True)
    assert np.all(w[masked] == 0.0)
    assert np.all(w[~masked] > 0.0)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("mask_kind", [0, 1, 2, 3])
def test_zero_query_gives_mean_of_visible_values(mask_kind):
    rng = np.random.default_rng(1)
    B, h, n, d = 2, 3, 7, 5
    q = np.zeros((B, n, h, d))
    k, v = _rand(rng, B, n, h, d), _rand(rng, B, n, h, d)
    key_lens = np.array([4, 7], dtype=np.int32)
    out = oracle.attn(q, k, v, 0.3, mask_kind, key_lens if mask_kind & 2 else None)
    for b in range(B):
        for t in range(n):
            last = n
            if mask_kind & 1:
                last = min(last, t + 1)
            if mask_kind & 2:
                last = min(last, key_lens[b])
            expect = v[b, :last].mean(axis=0)  # [h, d]
            np.testing.assert_allclose(out[b, t], expect, rtol=0, atol=1e-14)


def test_single_key_returns_that_value():
    rng = np.random.default_rng(2)
    q, k, v = _rand(rng, 2, 5, 3, 4), _rand(rng, 2, 1, 3, 4), _rand(rng, 2, 1, 3, 6)
    out = oracle.attn(q, k, v, 0.5)
    np.testing.assert_array_equal(out, np.broadcast_to(v, out.shape))


def test_causal_first_row_is_first_value():
    # Masking by a score of 0 instead of -inf would give row 0 weight on every key.
    rng = np.random.default_rng(3)
    q, k, v = _rand(rng, 1, 6, 2, 4), _rand(rng, 1, 6, 2, 4), _rand(rng, 1, 6, 2, 4)
    out = oracle.attn(q, k, v, 0.5, oracle.MASK_CAUSAL)
    np.testing.assert_array_equal(out[0, 0], v[0, 0])


def test_large_scale_selects_argmax():
    rng = np.random.default_rng(4)
    q, k, v = _rand(rng, 1, 4, 1, 8), _rand(rng, 1, 9, 1, 8), _rand(rng, 1, 9, 1, 3)
    out = oracle.attn(q, k, v, 1e4)
    for t in range(4):
        j = int(np.argmax(k[0, :, 0] @ q[0, t, 0]))
        np.testing.assert_allclose(out[0, t, 0], v[0, j, 0], atol=1e-12)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("mask_kind", [0, 1, 2, 3])
def test_weights_nonnegative_rows_sum_to_one_and_masked_are_zero(mask_kind):
    rng = np.random.default_rng(5)
    B, h, n, d = 3, 2, 9, 4
    q, k, v = _rand(rng, B, n, h, d), _rand(rng, B, n, h, d), _rand(rng, B, n, h, d)
    key_lens = np.array([1, 5, 9], dtype=np.int32)
    sel = [(b, t, i) for b in range(B) for t in range(n) for i in range(h)]
    out, w = oracle.attn_rows(q, k, v, 0.7, sel, mask_kind,
                              key_lens if mask_kind & 2 else None, weights=True)
    assert np.all(w >= 0.0)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-14)
    for r, (b, t, i) in enumerate(sel):
        for j in range(n):
            invisible = (mask_kind & 1 and j > t) or (mask_kind & 2 and j >= key_lens[b])
            if invisible:
                assert w[r, j] == 0.0
            else:
                assert w[r, j] > 0.0
        # Convex combination of the value rows: inside their per-column range.
        vis = [j for j in range(n) if w[r, j] > 0]
        lo = v[b, vis, i].min(axis=0)
        hi = v[b, vis, i].max(axis=0)
        assert np.all(out[r] >= lo - 1e-14) and np.all(out[r] <= hi + 1e-14)


def test_permutation_equivariance_unmasked_self_attention():
    rng = np.random.default_rng(6)
    B, h, n, d = 2, 3, 8, 4
    x = _rand(rng, B, n, h, d)
    q, k, v = x, x * 0.5 + 0.1, _rand(rng, B, n, h, d)
    perm = rng.permutation(n)
    out = oracle.attn(q, k, v, 0.4)
    out_p = oracle.attn(q[:, perm], k[:, perm], v[:, perm], 0.4)
    np.testing.assert_allclose(out_p, out[:, perm], atol=1e-13)


def test_causal_future_perturbation_leaves_past_unchanged():
    rng = np.random.default_rng(7)
    B, h, n, d = 1, 2, 10, 4
    q, k, v = _rand(rng, B, n, h, d), _rand(rng, B, n, h, d), _rand(rng, B, n, h, d)
    out = oracle.attn(q, k, v, 0.5, oracle.MASK_CAUSAL)
    t0 = 4
    k2, v2 = k.copy(), v.copy()
    k2[:, t0 + 1:] = 1e4 * rng.standard_normal(k2[:, t0 + 1:].shape)
    v2[:, t0 + 1:] = -1e4
    out2 = oracle.attn(q, k2, v2, 0.5, oracle.MASK_CAUSAL)
    np.testing.assert_array_equal(out2[:, :t0 + 1], out[:, :t0 + 1])
    assert not np.array_equal(out2[:, t0 + 1:], out[:, t0 + 1:])


def test_padding_contents_do_not_matter():
    rng = np.random.default_rng(8)
    B, h, n_q, n_k, d = 2, 2, 5, 9, 4
    q, k, v = _rand(rng, B, n_q, h, d), _rand(rng, B, n_k, h, d), _rand(rng, B, n_k, h, d)
    kl = np.array([3, 6], dtype=np.int32)
    out = oracle.attn(q, k, v, 0.5, oracle.MASK_KEY_PADDING, kl)
    k2, v2 = k.copy(), v.copy()
    for b in range(B):
        k2[b, kl[b]:] = 1e4
        v2[b, kl[b]:] = -1e4
    out2 = oracle.attn(q, k2, v2, 0.5, oracle.MASK_KEY_PADDING, kl)
    np.testing.assert_array_equal(out2, out)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("mask_kind", [0, 1, 2, 3])
@pytest.mark.parametrize("shape", [(2, 2, 3, 3, 4, 4), (1, 3, 5, 5, 3, 6), (2, 1, 8, 8, 2, 1),
                                   (2, 2, 4, 7, 5, 3)])
def test_brute_force_tiny(mask_kind, shape):
    B, h, n_q, n_k, d_k, d_v = shape
    if mask_kind & 1 and n_q != n_k:
        pytest.skip("causal needs n_q == n_k")
    rng = np.random.default_rng(100 + 7 * mask_kind + n_k)
    q, k, v = _rand(rng, B, n_q, h, d_k), _rand(rng, B, n_k, h, d_k), _rand(rng, B, n_k, h, d_v)
    kl = rng.integers(1, n_k + 1, size=B).astype(np.int32)
    scale = 1.0 / math.sqrt(d_k)
    out = oracle.attn(q, k, v, scale, mask_kind, kl if mask_kind & 2 else None)
    ref = np.array(brute.attention(q.tolist(), k.tolist(), v.tolist(), scale,
                                   causal=bool(mask_kind & 1),
                                   key_lens=kl.tolist() if mask_kind & 2 else None))
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- library second opinion

@pytest.mark.parametrize("mask_kind", [0, 1, 2, 3])
def test_against_torch_fp64(mask_kind):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(9)
    B, h, n, d_k, d_v = 3, 4, 33, 16, 8
    q, k, v = _rand(rng, B, n, h, d_k), _rand(rng, B, n, h, d_k), _rand(rng, B, n, h, d_v)
    kl = np.array([1, 17, 33], dtype=np.int32)
    scale = 0.25
    out = oracle.attn(q, k, v, scale, mask_kind, kl if mask_kind & 2 else None)
    tq, tk, tv = (torch.from_numpy(a).permute(0, 2, 1, 3) for a in (q, k, v))  # [B, h, n, d]
    s = torch.matmul(tq, tk.transpose(-2, -1)) * scale
    bias = torch.zeros(B, 1, n, n, dtype=torch.float64)
    if mask_kind & 1:
        bias = bias + torch.triu(torch.full((n, n), float("-inf"), dtype=torch.float64), 1)
    if mask_kind & 2:
        for b in range(B):
            bias[b, :, :, kl[b]:] = float("-inf")
    ref = torch.matmul(torch.softmax(s + bias, dim=-1), tv).permute(0, 2, 1, 3).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_matmul_against_numpy():
    rng = np.random.default_rng(10)
    a, w = _rand(rng, 17, 23), _rand(rng, 23, 9)
    np.testing.assert_allclose(oracle.matmul(a, w), a @ w, rtol=0, atol=1e-12)
    # Not the transposed product.
    w2 = _rand(rng, 23, 23)
    assert not np.allclose(oracle.matmul(a[:, :23], w2), a[:, :23] @ w2.T)


def test_layernorm_closed_forms_and_torch():
    torch = pytest.importorskip("torch")
    d = 8
    gamma, beta = np.linspace(0.5, 2.0, d), np.linspace(-1, 1, d)
    # Constant row: z - mu = 0, so y = beta exactly.
    np.testing.assert_array_equal(oracle.layernorm(np.full((1, d), 3.25), gamma, beta, 1e-6)[0], beta)
    # Alternating +a/-a: mean 0, biased variance a^2 -> y = gamma*(+-a)/sqrt(a^2+eps) + beta.
    a, eps = 2.0, 1e-6
    z = np.array([[a, -a] * (d // 2)])
    expect = gamma * z[0] / math.sqrt(a * a + eps) + beta
    np.testing.assert_allclose(oracle.layernorm(z, gamma, beta, eps)[0], expect, atol=1e-15)
    # The biased (divide by d) variance: an unbiased one would give sqrt(d/(d-1)) larger output.
    rng = np.random.default_rng(12)
    z = _rand(rng, 5, d) * 3 + 1
    ref = torch.nn.functional.layer_norm(torch.from_numpy(z), (d,), torch.from_numpy(gamma),
                                         torch.from_numpy(beta), eps).numpy()
    np.testing.assert_allclose(oracle.layernorm(z, gamma, beta, eps), ref, atol=1e-12)


# ---------------------------------------------------------------- MHA sublayer

def _mha_torch(torch, x_q, x_kv, wq, wk, wv, wo, gamma, beta, eps, h, mask_kind, kl):
    T = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    xq, xkv = T(x_q), T(x_kv)
    B, n_q, dm = xq.shape
    n_k = xkv.shape[1]
    Q = (xq @ T(wq)).view(B, n_q, h, -1).transpose(1, 2)
    K = (xkv @ T(wk)).view(B, n_k, h, -1).transpose(1, 2)
    V = (xkv @ T(wv)).view(B, n_k, h, -1).transpose(1, 2)
    s = Q @ K.transpose(-2, -1) / math.sqrt(Q.shape[-1])
    bias = torch.zeros(B, 1, n_q, n_k, dtype=torch.float64)
    if mask_kind & 1:
        bias = bias + torch.triu(torch.full((n_q, n_k), float("-inf"), dtype=torch.float64), 1)
    if mask_kind & 2:
        for b in range(B):
            bias[b, :, :, int(kl[b]):] = float("-inf")
    A = (torch.softmax(s + bias, -1) @ V).transpose(1, 2).reshape(B, n_q, -1)
    z = xq + A @ T(wo)
    return torch.nn.functional.layer_norm(z, (dm,), T(gamma), T(beta), eps).numpy()


@pytest.mark.parametrize("cross,mask_kind", [(False, 0), (False, 1), (True, 2)])
def test_mha_against_torch_fp64(cross, mask_kind):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(13)
    B, n_q, dm, h, dk = 2, 6, 16, 4, 4
    n_k = 9 if cross else n_q
    x_q = _rand(rng, B, n_q, dm)
    x_kv = _rand(rng, B, n_k, dm) if cross else x_q
    ws = [_rand(rng, dm, h * dk) / 4 for _ in range(3)] + [_rand(rng, h * dk, dm) / 4]
    gamma, beta = rng.uniform(0.5, 1.5, dm), rng.uniform(-0.5, 0.5, dm)
    kl = np.array([3, 9], dtype=np.int32) if mask_kind & 2 else None
    y = oracle.mha(x_q, x_kv, *ws, gamma, beta, 1e-6, h, mask_kind, kl)
    ref = _mha_torch(torch, x_q, x_kv, *ws, gamma, beta, 1e-6, h, mask_kind, kl)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-11)
    sel = [(1, 0), (0, n_q - 1), (1, 3)]
    yr = oracle.mha_rows(x_q, x_kv, *ws, gamma, beta, 1e-6, h, sel, mask_kind, kl)
    for r, (b, t) in enumerate(sel):
        np.testing.assert_allclose(yr[r], y[b, t], rtol=0, atol=1e-12)


def test_mha_reductions():
    rng = np.random.default_rng(14)
    B, n, dm = 2, 5, 6
    x = _rand(rng, B, n, dm)
    eye = np.eye(dm)
    g, b0 = np.ones(dm), np.zeros(dm)
    # One head, identity projections: y = LN(X + Attn(X, X, X)) with scale 1/sqrt(d_model).
    y = oracle.mha(x, x, eye, eye, eye, eye, g, b0, 1e-6, 1)
    a = oracle.attn(x[:, :, None, :], x[:, :, None, :], x[:, :, None, :], 1 / math.sqrt(dm))[:, :, 0]
    np.testing.assert_allclose(y, oracle.layernorm(x + a, g, b0, 1e-6), atol=1e-13)
    # W^O = 0: the sublayer reduces to LN(X) (the residual is kept).
    y0 = oracle.mha(x, x, eye, eye, eye, np.zeros((dm, dm)), g, b0, 1e-6, 1)
    np.testing.assert_allclose(y0, oracle.layernorm(x, g, b0, 1e-6), atol=1e-14)
    # Relabelling the heads (column blocks of W^Q/W^K/W^V, row blocks of W^O) changes nothing.
    h, dk = 3, 2
    ws = [_rand(rng, dm, h * dk) for _ in range(3)] + [_rand(rng, h * dk, dm)]
    perm = [2, 0, 1]
    cols = np.concatenate([np.arange(p * dk, (p + 1) * dk) for p in perm])
    y1 = oracle.mha(x, x, *ws, g, b0, 1e-6, h)
    y2 = oracle.mha(x, x, ws[0][:, cols], ws[1][:, cols], ws[2][:, cols], ws[3][cols, :],
                    g, b0, 1e-6, h)
    np.testing.assert_allclose(y1, y2, atol=1e-13)
    # ...but mismatching the head blocks of W^O does change it.
    y3 = oracle.mha(x, x, ws[0][:, cols], ws[1][:, cols], ws[2][:, cols], ws[3], g, b0, 1e-6, h)
    assert not np.allclose(y1, y3, atol=1e-6)


# ---------------------------------------------------------------- generator statistics

def test_generator_scaled_score_variance_is_one():
    # The pages' scaling argument: with i.i.d. N(0,1) components, q.k has
    # variance d_k, so q.k / sqrt(d_k) has variance 1.
    d_k = 64
    q = synth.draw_normal(0, synth.STREAM_Q, (4096, d_k))
    k = synth.draw_normal(0, synth.STREAM_K, (4096, d_k))
    s = (q * k).sum(axis=1) / math.sqrt(d_k)
    assert abs(s.var() - 1.0) < 0.05
    assert abs(q.mean()) < 0.01 and abs(q.var() - 1.0) < 0.01


def test_generator_rounding_and_key_lengths():
    x = synth.draw_normal(3, 0, (1000,))
    bits = synth.round_to_bf16_bits(x)
    back = synth.bf16_bits_to_f64(bits)
    assert np.all(np.abs(back - x) <= np.abs(x) * 2.0 ** -8)
    # Exactly representable values survive unchanged.
    exact = np.array([1.0, -2.5, 0.15625, 3.0 * 2 ** -20])
    np.testing.assert_array_equal(synth.bf16_bits_to_f64(synth.round_to_bf16_bits(exact)), exact)
    # Round-to-nearest-even at a tie: 1 + 2^-8 sits halfway between 1 and 1 + 2^-7.
    assert synth.bf16_bits_to_f64(synth.round_to_bf16_bits(np.array([1 + 2.0 ** -8])))[0] == 1.0
    kl = synth.draw_key_lens(2, synth.STREAM_KEYLEN, 20000, 64, 256)
    assert kl.min() == 64 and kl.max() == 256
    assert np.array_equal(kl, synth.draw_key_lens(2, synth.STREAM_KEYLEN, 20000, 64, 256))


# ---------------------------------------------------------------- positional encoding

def test_pos_encoding_printed_table():
    rows = []
    with open(os.path.join(GOLDEN, "pe_table_5x4.txt"), encoding="utf-8") as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    pe = oracle.pos_encoding(1, 5, 4)[0]
    # Within one unit of the last printed digit: the page prints cos(0.01) =
    # 0.99995000... as 0.9999 (correct rounding gives 1.0000); every other entry
    # matches to the printed four decimals.
    np.testing.assert_allclose(pe, np.array(rows), rtol=0, atol=1e-4)
    mismatched = np.round(pe, 4) != np.array(rows)
    assert mismatched.sum() == 1 and mismatched[1, 3]


def test_pos_encoding_relative_shift_is_a_rotation():
    # For each frequency pair, PE(pos + k) is PE(pos) rotated by the angle k * w_i:
    # a linear map that depends only on k (the pages' motivation for sin/cos pairs).
    d, k = 16, 7
    pe = oracle.pos_encoding(1, 64, d)[0]
    for i in range(d // 2):
        w = 10000.0 ** (-2.0 * i / d)
        rot = np.array([[math.cos(k * w), -math.sin(k * w)], [math.sin(k * w), math.cos(k * w)]])
        pair = pe[:, 2 * i:2 * i + 2]
        np.testing.assert_allclose(pair[k:], pair[:-k] @ rot, atol=1e-12)


def test_pos_encoding_embedding_scale_and_offset():
    rng = np.random.default_rng(15)
    emb = rng.standard_normal((2, 6, 8))
    full = oracle.pos_encoding(2, 6, 8, emb=emb, emb_scale=math.sqrt(8), pos0=3)
    pe = oracle.pos_encoding(1, 9, 8)[0]
    np.testing.assert_allclose(full, emb * math.sqrt(8) + pe[3:9][None], atol=1e-14)
    # Position 0: sin(0) = 0 on even dimensions, cos(0) = 1 on odd ones.
    np.testing.assert_array_equal(oracle.pos_encoding(1, 1, 8)[0, 0], [0, 1] * 4)


# ---------------------------------------------------------------- feed-forward sublayer

def _ffn_case(rng, rows, dm, dff):
    return dict(x=_rand(rng, rows, dm), w1=_rand(rng, dm, dff) / 2, b1=_rand(rng, dff) / 2,
                w2=_rand(rng, dff, dm) / 2, b2=_rand(rng, dm), gamma=rng.uniform(0.5, 1.5, dm),
                beta=rng.uniform(-0.5, 0.5, dm))


def test_ffn_brute_force_tiny():
    """Non-square W1 (d_ff != d_model) and non-trivial biases / gamma / beta: a
    transposed operand, a dropped bias or a misplaced ReLU fails this."""
    rng = np.random.default_rng(21)
    c = _ffn_case(rng, 4, 5, 7)
    y = oracle.ffn(c["x"], c["w1"], c["b1"], c["w2"], c["b2"], c["gamma"], c["beta"], 1e-6)
    for r in range(4):
        ref = brute.feed_forward_row(list(c["x"][r]), c["w1"].tolist(), list(c["b1"]),
                                     c["w2"].tolist(), list(c["b2"]), list(c["gamma"]),
                                     list(c["beta"]), 1e-6)
        np.testing.assert_allclose(y[r], ref, rtol=0, atol=1e-12)
    # Some pre-activations are negative here, so the ReLU is exercised.
    pre = c["x"] @ c["w1"] + c["b1"]
    assert (pre < 0).any() and (pre > 0).any()


def test_ffn_against_torch_fp64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(22)
    c = _ffn_case(rng, 2 * 6, 16, 40)
    y = oracle.ffn(c["x"].reshape(2, 6, 16), c["w1"], c["b1"], c["w2"], c["b2"], c["gamma"],
                   c["beta"], 1e-6)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    F = torch.nn.functional
    hid = F.relu(T(c["x"]) @ T(c["w1"]) + T(c["b1"]))
    ref = F.layer_norm(T(c["x"]) + hid @ T(c["w2"]) + T(c["b2"]), (16,), T(c["gamma"]),
                       T(c["beta"]), 1e-6).numpy()
    np.testing.assert_allclose(y.reshape(12, 16), ref, rtol=0, atol=1e-12)


def test_ffn_closed_forms():
    rng = np.random.default_rng(23)
    dm = 6
    x = _rand(rng, 5, dm)
    g, b0 = np.ones(dm), np.zeros(dm)
    # A very negative b1 switches every hidden unit off: y = LN(x + b2).
    b2 = _rand(rng, dm)
    y = oracle.ffn(x, _rand(rng, dm, 9), np.full(9, -1e6), _rand(rng, 9, dm), b2, g, b0, 1e-6)
    np.testing.assert_allclose(y, oracle.layernorm(x + b2, g, b0, 1e-6), atol=1e-13)
    # W1 = W2 = I, no biases: y = LN(x + max(0, x)).
    eye = np.eye(dm)
    y = oracle.ffn(x, eye, np.zeros(dm), eye, np.zeros(dm), g, b0, 1e-6)
    np.testing.assert_allclose(y, oracle.layernorm(x + np.maximum(x, 0.0), g, b0, 1e-6), atol=1e-13)


def test_ffn_is_position_wise():
    """[hex4c59] §前馈网络为什么放在注意力后面？: a row never reads another row."""
    rng = np.random.default_rng(24)
    c = _ffn_case(rng, 6, 8, 12)
    args = (c["w1"], c["b1"], c["w2"], c["b2"], c["gamma"], c["beta"], 1e-6)
    y = oracle.ffn(c["x"], *args)
    x2 = c["x"].copy()
    x2[[0, 5]] = _rand(rng, 2, 8) * 10
    y2 = oracle.ffn(x2, *args)
    np.testing.assert_array_equal(y[1:5], y2[1:5])
    perm = rng.permutation(6)
    np.testing.assert_array_equal(oracle.ffn(c["x"][perm], *args), y[perm])


def test_encoder_layer_reduction():
    """With W^O = 0 and W2 = 0, b2 = 0, both sublayers reduce to LayerNorm, so the
    layer gives LN(LN(x)) = LN(x) up to the epsilon (gamma = 1, beta = 0)."""
    rng = np.random.default_rng(25)
    B, n, dm, h = 2, 5, 8, 2
    x = _rand(rng, B, n, dm)
    g, b0 = np.ones(dm), np.zeros(dm)
    ws = [_rand(rng, dm, dm) for _ in range(3)]
    y1 = oracle.mha(x, x, *ws, np.zeros((dm, dm)), g, b0, 1e-6, h)
    y = oracle.ffn(y1, _rand(rng, dm, 16), _rand(rng, 16), np.zeros((16, dm)), np.zeros(dm), g, b0,
                   1e-6)
    np.testing.assert_allclose(y, oracle.layernorm(x, g, b0, 1e-6), atol=1e-5)


# ---------------------------------------------------------------- attention backward

def _fwd_objective(q, k, v, dout, scale, mask_kind, kl):
    return float(np.sum(dout * oracle.attn(q, k, v, scale, mask_kind, kl)))


@pytest.mark.parametrize("mask_kind", [0, 1, 2, 3])
def test_attn_bwd_matches_finite_differences(mask_kind):
    """Central differences of <dO, Attention(Q, K, V)> through the pinned forward
    oracle: an independent check of every term of the chain rule (a dropped
    softmax-Jacobian term, a sign or a transposed operand fails it)."""
    rng = np.random.default_rng(31 + mask_kind)
    B, n, h, dk_, dv_ = 2, 5, 2, 3, 4
    q, k = _rand(rng, B, n, h, dk_), _rand(rng, B, n, h, dk_)
    v, dout = _rand(rng, B, n, h, dv_), _rand(rng, B, n, h, dv_)
    kl = np.array([3, 5], dtype=np.int32) if mask_kind & 2 else None
    scale = 0.7
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, dout, scale, mask_kind, kl)
    eps = 1e-6
    for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += eps
            minus[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = plus
            fp = _fwd_objective(args["q"], args["k"], args["v"], dout, scale, mask_kind, kl)
            args[name] = minus
            fm = _fwd_objective(args["q"], args["k"], args["v"], dout, scale, mask_kind, kl)
            fd[idx] = (fp - fm) / (2 * eps)
        np.testing.assert_allclose(grad, fd, rtol=0, atol=2e-8, err_msg=name)


@pytest.mark.parametrize("mask_kind", [0, 1, 2])
def test_attn_bwd_against_torch_autograd(mask_kind):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(41)
    B, n_q, n_k, h, d = 2, 6, 6 if mask_kind & 1 else 9, 3, 4
    q, k, v = _rand(rng, B, n_q, h, d), _rand(rng, B, n_k, h, d), _rand(rng, B, n_k, h, d)
    dout = _rand(rng, B, n_q, h, d)
    kl = np.array([4, n_k], dtype=np.int32) if mask_kind & 2 else None
    scale = 0.5
    dq, dk, dv, lse = oracle.attn_bwd(q, k, v, dout, scale, mask_kind, kl)
    Q, K, V = (torch.from_numpy(a.transpose(0, 2, 1, 3).copy()).requires_grad_() for a in (q, k, v))
    s = Q @ K.transpose(-1, -2) * scale
    bias = torch.zeros(B, 1, n_q, n_k, dtype=torch.float64)
    if mask_kind & 1:
        bias = bias + torch.triu(torch.full((n_q, n_k), float("-inf"), dtype=torch.float64), 1)
    if mask_kind & 2:
        for b in range(B):
            bias[b, :, :, int(kl[b]):] = float("-inf")
    O = torch.softmax(s + bias, -1) @ V
    O.backward(torch.from_numpy(dout.transpose(0, 2, 1, 3).copy()))
    back = lambda t: t.grad.numpy().transpose(0, 2, 1, 3)
    np.testing.assert_allclose(dq, back(Q), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, back(K), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, back(V), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(s + bias, -1).detach().numpy(), rtol=0, atol=1e-12)


def test_attn_bwd_invariants_and_closed_forms():
    rng = np.random.default_rng(42)
    B, n, h, d = 2, 7, 2, 5
    q, k, v, dout = (_rand(rng, B, n, h, d) for _ in range(4))
    kl = np.array([4, 7], dtype=np.int32)
    dq, dk, dv, lse = oracle.attn_bwd(q, k, v, dout, 0.4, 2, kl)
    # Shifting every key of a head by one vector shifts each score row by a constant:
    # the softmax ignores it, so the key gradients of a head sum to zero.
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    # Each weight row sums to 1, so the value gradients sum to the output gradients.
    np.testing.assert_allclose(dv.sum(axis=1), dout.sum(axis=1), atol=1e-12)
    # Padded keys receive no gradient.
    assert np.all(dk[0, 4:] == 0.0) and np.all(dv[0, 4:] == 0.0)
    # One key: O = v_1 whatever q and k are, so dQ = dK = 0 and dV = sum of dO.
    dq1, dk1, dv1, lse1 = oracle.attn_bwd(q, k[:, :1], v[:, :1], dout, 0.4)
    assert np.all(dq1 == 0.0) and np.all(dk1 == 0.0)
    np.testing.assert_allclose(dv1[:, 0], dout.sum(axis=1), atol=1e-12)
    np.testing.assert_allclose(lse1, 0.4 * np.einsum("bthc,bhc->bht", q, k[:, 0]), atol=1e-12)
    # Causal: key j only receives gradient from queries t >= j (the last key only from the last query).
    dqc, dkc, dvc, _ = oracle.attn_bwd(q, k, v, dout, 0.4, 1)
    # ...so dV of the last key is the last query's weight on it times that query's dO.
    sel = [(b, n - 1, i) for b in range(B) for i in range(h)]
    _, wts = oracle.attn_rows(q, k, v, 0.4, sel, 1, weights=True)
    for r, (b, t, i) in enumerate(sel):
        np.testing.assert_allclose(dvc[b, n - 1, i], wts[r, n - 1] * dout[b, n - 1, i], atol=1e-13)
    dout2 = dout.copy()
    dout2[:, n - 1] = 0.0
    _, dk2, dv2, _ = oracle.attn_bwd(q, k, v, dout2, 0.4, 1)
    assert np.all(dv2[:, n - 1] == 0.0) and np.all(dk2[:, n - 1] == 0.0)


def test_attn_lse_brute_force():
    rng = np.random.default_rng(43)
    q, k, v = (_rand(rng, 1, 4, 1, 3) for _ in range(3))
    _, _, _, lse = oracle.attn_bwd(q, k, v, np.zeros_like(v), 0.9, 1)
    for t in range(4):
        scores = [0.9 * math.fsum(q[0, t, 0] * k[0, j, 0]) for j in range(t + 1)]
        top = max(scores)
        ref = top + math.log(math.fsum(math.exp(s - top) for s in scores))
        assert abs(lse[0, 0, t] - ref) < 1e-13
