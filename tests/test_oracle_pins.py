"""Pins for the fp64 oracle: the pages' worked examples, closed forms,
invariants and an independent library routine. CPU only.

Each check is chosen so that a plausible mistake in the oracle (a wrong
scale, masking after the softmax, a transposed operand, a wrong head block,
an off-by-one in the causal or padding test) fails at least one of them.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import MASK_CAUSAL, MASK_KEY_PADDING, MASK_NONE

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


def _one(q, k, v, mask=MASK_NONE, **kw):
    """Wrap single-head [n, d] arrays as [1, 1, n, d]."""
    q, k, v = (np.asarray(a, dtype=np.float64)[None, None] for a in (q, k, v))
    out, w = oracle.attention(q, k, v, mask, return_weights=True, **kw)
    return out[0, 0], w[0, 0]


# ---------------------------------------------------------------- worked examples

def test_three_token_unmasked_matches_printed_run():
    g = _load("three_token_verification.json")
    out, w = _one(g["q"], g["k"], g["v"])
    tol = g["tolerance"]
    assert np.sqrt(2.0) == pytest.approx(g["scale_sqrt_dk"], abs=tol)
    np.testing.assert_allclose(w[0], g["unmasked_row0_weights"], atol=tol, rtol=0)
    np.testing.assert_allclose(out[0], g["unmasked_row0_output"], atol=tol, rtol=0)


def test_three_token_causal_matches_printed_run():
    g = _load("three_token_verification.json")
    out, w = _one(g["q"], g["k"], g["v"], MASK_CAUSAL)
    tol = g["tolerance"]
    np.testing.assert_allclose(w, g["causal_weights"], atol=tol, rtol=0)
    np.testing.assert_allclose(out, g["causal_outputs"], atol=tol, rtol=0)


def test_mask_goes_before_softmax_not_after():
    """Zeroing future weights after the softmax leaves row 0 summing to 0.401112
    (the page's negative example); the oracle must not do that."""
    g = _load("three_token_verification.json")
    _, w_unmasked = _one(g["q"], g["k"], g["v"])
    wrong = np.array([w_unmasked[0, 0], 0.0, 0.0])
    assert wrong.sum() == pytest.approx(g["wrong_post_softmax_mask_row0_sum"], abs=1e-6)
    np.testing.assert_allclose(wrong @ np.asarray(g["v"]), g["wrong_post_softmax_mask_row0_output"],
                               atol=1e-6)
    out, w = _one(g["q"], g["k"], g["v"], MASK_CAUSAL)
    assert w[0].sum() == pytest.approx(1.0, abs=1e-15)
    assert not np.allclose(out[0], g["wrong_post_softmax_mask_row0_output"], atol=1e-3)


def test_two_token_worked_example():
    g = _load("two_token_worked_example.json")
    q, k = np.asarray(g["q"]), np.asarray(g["k"])
    # the page's step 2 (Q K^T) and step 3 (divide by sqrt(d_k)) on its own matrices
    np.testing.assert_allclose(q @ k.T, g["scores_qkt"], atol=0)
    np.testing.assert_allclose(q @ k.T / np.sqrt(2.0), g["scaled_scores"], atol=g["tolerance_scores"])
    out, w = _one(g["q"], g["k"], g["v"])
    np.testing.assert_allclose(w, g["weights"], atol=g["tolerance"])
    np.testing.assert_allclose(out, g["output"], atol=g["tolerance"])
    # exact values, re-derived from the closed form of a 2-key softmax (logistic function)
    for i in range(2):
        s = q[i] @ k.T / np.sqrt(2.0)
        p0 = 1.0 / (1.0 + np.exp(s[1] - s[0]))
        assert w[i, 0] == pytest.approx(p0, abs=1e-14)


# ---------------------------------------------------------------- closed forms

def test_scale_is_inverse_sqrt_dk():
    """With two keys the log weight ratio is the scaled logit difference, which
    pins the factor 1/sqrt(d_k) (not 1/d_k, not 1)."""
    rng = np.random.default_rng(7)
    for d_k in (2, 16, 64, 128):
        q = rng.standard_normal((1, d_k))
        k = rng.standard_normal((2, d_k))
        v = rng.standard_normal((2, 3))
        _, w = _one(q, k, v)
        expect = (q[0] @ k[0] - q[0] @ k[1]) / np.sqrt(d_k)
        assert np.log(w[0, 0] / w[0, 1]) == pytest.approx(expect, abs=1e-12)


def test_explicit_scale_is_used():
    rng = np.random.default_rng(8)
    q, k, v = rng.standard_normal((1, 4)), rng.standard_normal((2, 4)), rng.standard_normal((2, 2))
    _, w = _one(q, k, v, scale=0.3)
    assert np.log(w[0, 0] / w[0, 1]) == pytest.approx(0.3 * (q[0] @ (k[0] - k[1])), abs=1e-12)


def test_output_is_weights_times_v_and_q_k_not_transposed():
    """Asymmetric shapes (n_q != n_k, d_k != d_v) catch a transposed operand."""
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 1, 3, 5))
    k = rng.standard_normal((1, 1, 7, 5))
    v = rng.standard_normal((1, 1, 7, 2))
    out, w = oracle.attention(q, k, v, return_weights=True)
    assert out.shape == (1, 1, 3, 2) and w.shape == (1, 1, 3, 7)
    np.testing.assert_allclose(out[0, 0], w[0, 0] @ v[0, 0], atol=1e-14)
    # each weight row is a normalised exponential of that query's logits
    s = q[0, 0] @ k[0, 0].T / np.sqrt(5.0)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    np.testing.assert_allclose(w[0, 0], e / e.sum(axis=1, keepdims=True), atol=1e-14)


# ---------------------------------------------------------------- invariants

def _rand(seed, B=2, h=3, n_q=9, n_k=9, d_k=8, d_v=6):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, h, n_q, d_k)), rng.standard_normal((B, h, n_k, d_k)),
            rng.standard_normal((B, h, n_k, d_v)))


@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING,
                                  MASK_CAUSAL | MASK_KEY_PADDING])
def test_rows_sum_to_one_and_masked_weights_are_zero(mask):
    q, k, v = _rand(11)
    lens = np.array([4, 9], dtype=np.int32)
    out, w = oracle.attention(q, k, v, mask, kv_lens=lens, return_weights=True)
    n = q.shape[2]
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    for b in range(2):
        allowed = np.ones((n, n), dtype=bool)
        if mask & MASK_CAUSAL:
            allowed &= j <= i
        if mask & MASK_KEY_PADDING:
            allowed &= j < lens[b]
        assert np.all(w[b][:, ~allowed] == 0.0)          # future / pad weights exactly 0
        assert np.all(w[b][:, allowed] > 0.0)
        np.testing.assert_allclose(w[b].sum(axis=-1), 1.0, atol=1e-14)


@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING,
                                  MASK_CAUSAL | MASK_KEY_PADDING])
def test_zero_query_gives_mean_of_allowed_values(mask):
    _, k, v = _rand(12)
    q = np.zeros((2, 3, 9, 8))
    lens = np.array([5, 2], dtype=np.int32)
    out = oracle.attention(q, k, v, mask, kv_lens=lens)
    for b in range(2):
        for i in range(9):
            hi = 9
            if mask & MASK_CAUSAL:
                hi = min(hi, i + 1)
            if mask & MASK_KEY_PADDING:
                hi = min(hi, lens[b])
            np.testing.assert_allclose(out[b, :, i], v[b, :, :hi].mean(axis=1), atol=1e-13)


def test_causal_row_zero_is_v0():
    q, k, v = _rand(13)
    out = oracle.attention(q, k, v, MASK_CAUSAL)
    np.testing.assert_array_equal(out[:, :, 0], v[:, :, 0])


def test_joint_key_value_permutation_leaves_output_unchanged():
    q, k, v = _rand(14, n_q=5, n_k=11)
    perm = np.random.default_rng(0).permutation(11)
    a = oracle.attention(q, k, v)
    b = oracle.attention(q, k[:, :, perm], v[:, :, perm])
    np.testing.assert_allclose(a, b, atol=1e-13)
    # key padding: permuting within the valid prefix changes nothing either
    lens = np.array([6, 11], dtype=np.int32)
    p6 = np.concatenate([np.random.default_rng(1).permutation(6), np.arange(6, 11)])
    a = oracle.attention(q, k, v, MASK_KEY_PADDING, kv_lens=lens)
    b = oracle.attention(q, k[:, :, p6], v[:, :, p6], MASK_KEY_PADDING, kv_lens=lens)
    np.testing.assert_allclose(a, b, atol=1e-13)


def test_query_permutation_permutes_outputs():
    q, k, v = _rand(15, n_q=7, n_k=5)
    perm = np.random.default_rng(2).permutation(7)
    a = oracle.attention(q, k, v)
    b = oracle.attention(q[:, :, perm], k, v)
    np.testing.assert_allclose(a[:, :, perm], b, atol=1e-13)


def test_single_key_and_constant_values():
    q, k, v = _rand(16, n_q=4, n_k=1)
    np.testing.assert_allclose(oracle.attention(q, k, v), np.broadcast_to(v, (2, 3, 4, 6)), atol=0)
    q, k, v = _rand(17, n_q=4, n_k=6)
    c = np.broadcast_to(np.arange(6.0)[None, None, None, :] - 2.5, v.shape).copy()
    np.testing.assert_allclose(oracle.attention(q, k, c), np.broadcast_to(c[:, :, :1], (2, 3, 4, 6)),
                               atol=1e-13)


def test_common_key_shift_leaves_output_unchanged():
    """K + 1 u^T adds q.u to every logit of a row; the softmax ignores it."""
    q, k, v = _rand(18)
    u = np.random.default_rng(3).standard_normal(8)
    for mask in (MASK_NONE, MASK_CAUSAL):
        a = oracle.attention(q, k, v, mask)
        b = oracle.attention(q, k + u, v, mask)
        np.testing.assert_allclose(a, b, atol=1e-12)


def test_empty_key_set_gives_zero_rows():
    q, k, v = _rand(19)
    out, w = oracle.attention(q, k, v, MASK_KEY_PADDING, kv_lens=np.array([0, 3], np.int32),
                              return_weights=True)
    assert np.all(out[0] == 0.0) and np.all(w[0] == 0.0)
    assert np.all(np.isfinite(out))
    # out-of-range lengths are clamped to [0, n_k]
    a = oracle.attention(q, k, v, MASK_KEY_PADDING, kv_lens=np.array([-5, 100], np.int32))
    assert np.all(a[0] == 0.0)
    np.testing.assert_allclose(a[1], oracle.attention(q, k, v)[1], atol=0)


def test_large_logits_do_not_overflow():
    """The max-subtraction keeps exp finite for logits far beyond exp's range."""
    q = np.full((1, 1, 2, 4), 300.0)
    k = np.full((1, 1, 3, 4), 300.0)
    k[0, 0, 1] = 299.0
    v = np.eye(3)[None, None]
    out, w = oracle.attention(q, k, v, return_weights=True)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(w.sum(-1), 1.0, atol=1e-15)


def test_rows_entry_equals_full_attention_rows():
    q, k, v = _rand(20, n_q=12, n_k=12)
    lens = np.array([7, 12], dtype=np.int32)
    for mask in (MASK_NONE, MASK_CAUSAL, MASK_CAUSAL | MASK_KEY_PADDING):
        full = oracle.attention(q, k, v, mask, kv_lens=lens)
        rows = np.array([0, 5, 11, 3])
        for b in range(2):
            for hh in range(3):
                got = oracle.attention_rows(q[b, hh, rows], rows, k[b, hh], v[b, hh],
                                            causal=bool(mask & MASK_CAUSAL),
                                            kv_len=int(lens[b]) if mask & MASK_KEY_PADDING else None)
                np.testing.assert_allclose(got, full[b, hh, rows], atol=0)


def test_variance_of_unscaled_logits_is_dk():
    """Var(q.k) = d_k for iid unit-variance components; after 1/sqrt(d_k) it is 1
    ("[논문 리뷰]Attention Is All You Need", section 3.2.1, the variance argument).
    Checked on the generator's bf16 N(0,1) draws through two-key weight ratios."""
    import synthetic
    rng = np.random.default_rng(21)
    d_k, n = 64, 20000
    qb = synthetic.bf16_bits_to_f64(synthetic.normal_bf16(rng, (n, d_k)))
    kb = synthetic.bf16_bits_to_f64(synthetic.normal_bf16(rng, (n, 2, d_k)))
    q = qb[:, None, None, :].reshape(n, 1, 1, d_k)
    k = kb.reshape(n, 1, 2, d_k)
    v = np.zeros((n, 1, 2, 1))
    _, w = oracle.attention(q, k, v, return_weights=True)
    # log(w0/w1) = (q.k0 - q.k1)/sqrt(d_k) has variance 2 (difference of two unit-variance logits)
    z = np.log(w[:, 0, 0, 0] / w[:, 0, 0, 1])
    assert np.var(z) == pytest.approx(2.0, rel=0.05)


# ---------------------------------------------------------------- library special case

def _torch_sdpa(q, k, v, mask, lens):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    B, h, n_q, _ = q.shape
    n_k = k.shape[2]
    allowed = torch.ones((B, 1, n_q, n_k), dtype=torch.bool)
    if mask & MASK_CAUSAL:
        allowed &= torch.tril(torch.ones((n_q, n_k), dtype=torch.bool))
    if mask & MASK_KEY_PADDING:
        allowed &= (torch.arange(n_k)[None, :] < torch.as_tensor(lens)[:, None])[:, None, None, :]
    return F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                          torch.from_numpy(v), attn_mask=allowed).numpy()


@pytest.mark.parametrize("shape", [(2, 3, 9, 9, 8, 8), (1, 2, 5, 13, 16, 4), (3, 1, 17, 17, 64, 64)])
@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING,
                                  MASK_CAUSAL | MASK_KEY_PADDING])
def test_matches_torch_fp64_sdpa(shape, mask):
    B, h, n_q, n_k, d_k, d_v = shape
    if mask & MASK_CAUSAL and n_q != n_k:
        pytest.skip("causal defined for n_q == n_k")
    rng = np.random.default_rng(hash(shape) % 2**32)
    q = rng.standard_normal((B, h, n_q, d_k))
    k = rng.standard_normal((B, h, n_k, d_k))
    v = rng.standard_normal((B, h, n_k, d_v))
    lens = rng.integers(1, n_k + 1, size=B).astype(np.int32)
    ours = oracle.attention(q, k, v, mask, kv_lens=lens)
    ref = _torch_sdpa(q, k, v, mask, lens)
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- multi-head

def _mha_case(seed, B=2, n_q=6, n_k=6, d_model=16, h=4, d=4):
    rng = np.random.default_rng(seed)
    x_q = rng.standard_normal((B, n_q, d_model))
    x_kv = x_q if n_k == n_q else rng.standard_normal((B, n_k, d_model))
    ws = [rng.standard_normal((d_model, h * d)) * 0.3 for _ in range(3)]
    w_o = rng.standard_normal((h * d, d_model)) * 0.3
    return x_q, x_kv, ws, w_o


@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING])
def test_mha_equals_independent_heads_then_output_projection(mask):
    """MultiHead = Concat(head_1..head_h) W^O with head_i on column block i."""
    x_q, x_kv, (w_q, w_k, w_v), w_o = _mha_case(31)
    h, d = 4, 4
    lens = np.array([3, 6], dtype=np.int32)
    got, concat = oracle.mha(x_q, x_kv, w_q, w_k, w_v, w_o, h, mask, kv_lens=lens, return_concat=True)
    heads = []
    for i in range(h):
        cols = slice(i * d, (i + 1) * d)
        Qi, Ki, Vi = x_q @ w_q[:, cols], x_kv @ w_k[:, cols], x_kv @ w_v[:, cols]
        heads.append(oracle.attention(Qi[:, None], Ki[:, None], Vi[:, None], mask, kv_lens=lens)[:, 0])
    expect_concat = np.concatenate(heads, axis=-1)
    np.testing.assert_allclose(concat, expect_concat, atol=1e-13)
    np.testing.assert_allclose(got, expect_concat @ w_o, atol=1e-12)


@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING])
@pytest.mark.parametrize("cross", [False, True])
def test_mha_matches_torch_multi_head_attention_forward(mask, cross):
    """torch's fp64 multi_head_attention_forward (weights transposed into its
    y = x W^T convention, no biases) is an independent implementation."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    if cross and mask & MASK_CAUSAL:
        pytest.skip("causal defined for self-attention")
    B, n_q, n_k, d_model, h = 2, 6, (9 if cross else 6), 16, 4
    x_q, x_kv, (w_q, w_k, w_v), w_o = _mha_case(32, B=B, n_q=n_q, n_k=n_k, d_model=d_model, h=h)
    lens = np.array([n_k - 2, n_k], dtype=np.int32)
    ours = oracle.mha(x_q, x_kv, w_q, w_k, w_v, w_o, h, mask, kv_lens=lens)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    attn_mask = None
    if mask & MASK_CAUSAL:
        attn_mask = ~torch.tril(torch.ones((n_q, n_k), dtype=torch.bool))  # True = not allowed
    kpm = None
    if mask & MASK_KEY_PADDING:
        kpm = torch.arange(n_k)[None, :] >= T(lens)[:, None]
    ref, _ = F.multi_head_attention_forward(
        T(x_q.transpose(1, 0, 2)), T(x_kv.transpose(1, 0, 2)), T(x_kv.transpose(1, 0, 2)),
        d_model, h, None, None, None, None, False, 0.0, T(w_o.T), None, training=False,
        key_padding_mask=kpm, need_weights=False, attn_mask=attn_mask,
        use_separate_proj_weight=True, q_proj_weight=T(w_q.T), k_proj_weight=T(w_k.T),
        v_proj_weight=T(w_v.T))
    np.testing.assert_allclose(ours, ref.numpy().transpose(1, 0, 2), rtol=1e-11, atol=1e-11)


# ---------------------------------------------------------------- restricted self-attention
# "[논문 리뷰]Attention Is All You Need" (kimjiil.github.io), section "[4] Why
# Self-Attention", Table 1: restricted self-attention considers only the r
# positions around each query (O(r n d)). The oracle takes the window per
# side: keys j in [i - left, i + right].

def _rand_self(seed, B=2, h=2, n=11, d_k=5, d_v=3):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, h, n, d_k)), rng.standard_normal((B, h, n, d_k)),
            rng.standard_normal((B, h, n, d_v)), rng)


def test_window_of_zero_width_returns_each_query_its_own_value():
    q, k, v, _ = _rand_self(1)
    out = oracle.attention(q, k, v, window=(0, 0))
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-15)


@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING])
def test_window_covering_every_key_is_unrestricted_attention(mask):
    q, k, v, rng = _rand_self(2)
    lens = rng.integers(1, 12, size=2).astype(np.int32)
    full = oracle.attention(q, k, v, mask, kv_lens=lens)
    for window in [(10, 10), (50, 50), (None, 10), (10, None)]:
        np.testing.assert_array_equal(oracle.attention(q, k, v, mask, kv_lens=lens, window=window),
                                      full)


@pytest.mark.parametrize("left,right", [(0, 0), (1, 1), (2, 0), (0, 3), (3, 1), (4, 4)])
@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING])
def test_window_zero_query_gives_mean_of_window_values(left, right, mask):
    """Q = 0 makes every allowed logit 0, so each output row is the plain mean
    of v_j over j in [i - left, i + right] (clipped to the keys, the causal
    limit and the key length): an off-by-one in either bound changes it."""
    n = 13
    _, k, v, _ = _rand_self(3, B=2, h=1, n=n)
    q = np.zeros_like(k)
    lens = np.array([n, 7], dtype=np.int32)
    out = oracle.attention(q, k, v, mask, kv_lens=lens, window=(left, right))
    for b in range(2):
        klen = lens[b] if mask & MASK_KEY_PADDING else n
        for i in range(n):
            lo = max(0, i - left)
            hi = min(i + right, klen - 1, i if mask & MASK_CAUSAL else n - 1)
            want = v[b, 0, lo:hi + 1].mean(axis=0) if hi >= lo else np.zeros(v.shape[-1])
            np.testing.assert_allclose(out[b, 0, i], want, rtol=0, atol=1e-14)


@pytest.mark.parametrize("n,r", [(16, 2), (40, 5), (9, 0), (7, 3)])
def test_radius_window_visits_the_table_1_number_of_pairs(n, r):
    """A radius-r window over n positions connects sum_i (min(n-1, i+r) -
    max(0, i-r) + 1) pairs, which is (2r+1) n - r (r+1) when n > 2r: the
    O(r n) count of Table 1. The nonzero weights of the oracle count them."""
    q, k, v, _ = _rand_self(4, B=1, h=1, n=n)
    _, w = oracle.attention(q, k, v, return_weights=True, window=(r, r))
    pairs = int(np.count_nonzero(w))
    assert pairs == sum(min(n - 1, i + r) - max(0, i - r) + 1 for i in range(n))
    if n > 2 * r:
        assert pairs == (2 * r + 1) * n - r * (r + 1)
    np.testing.assert_allclose(w.sum(axis=-1), 1.0, rtol=0, atol=1e-14)


def test_causal_window_equals_left_only_window():
    q, k, v, _ = _rand_self(5)
    np.testing.assert_array_equal(oracle.attention(q, k, v, MASK_CAUSAL, window=(3, 5)),
                                  oracle.attention(q, k, v, MASK_NONE, window=(3, 0)))


def test_window_rows_entry_matches_full_window_attention():
    q, k, v, _ = _rand_self(6, B=1, h=1, n=21)
    full = oracle.attention(q, k, v, window=(4, 2))
    rows = np.array([0, 5, 20, 13], dtype=np.int32)
    got = oracle.attention_rows(q[0, 0, rows], rows, k[0, 0], v[0, 0], causal=False,
                                window=(4, 2))
    np.testing.assert_array_equal(got, full[0, 0, rows])


def test_window_needs_equal_query_and_key_lengths():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 1, 4, 3))
    kv = rng.standard_normal((1, 1, 5, 3))
    with pytest.raises(ValueError):
        oracle.attention(q, kv, kv, window=(1, 1))


@pytest.mark.parametrize("left,right,mask", [(2, 2, MASK_NONE), (0, 4, MASK_NONE),
                                             (3, 0, MASK_CAUSAL), (5, 1, MASK_KEY_PADDING),
                                             (1, 6, MASK_CAUSAL | MASK_KEY_PADDING)])
def test_window_matches_torch_fp64_sdpa_with_band_mask(left, right, mask):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    B, h, n = 3, 2, 19
    q, k, v, rng = _rand_self(8 + left * 7 + right, B=B, h=h, n=n, d_k=8, d_v=6)
    lens = rng.integers(1, n + 1, size=B).astype(np.int32)
    i = torch.arange(n)[:, None]
    j = torch.arange(n)[None, :]
    allowed = ((j >= i - left) & (j <= i + right))[None, None].expand(B, 1, n, n).clone()
    if mask & MASK_CAUSAL:
        allowed &= (j <= i)[None, None]
    if mask & MASK_KEY_PADDING:
        allowed &= (torch.arange(n)[None, :] < torch.as_tensor(lens)[:, None])[:, None, None, :]
    ref = F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                         torch.from_numpy(v), attn_mask=allowed).numpy()
    ours = oracle.attention(q, k, v, mask, kv_lens=lens, window=(left, right))
    live = allowed.any(dim=-1).numpy()[:, 0]          # rows with at least one key
    np.testing.assert_allclose(ours[np.broadcast_to(live[:, None], ours.shape[:3])],
                               ref[np.broadcast_to(live[:, None], ref.shape[:3])],
                               rtol=1e-12, atol=1e-12)
    assert np.all(ours[np.broadcast_to(~live[:, None], ours.shape[:3])] == 0.0)


# ---------------------------------------------------------------- incremental decoding (KV cache)
# "Attention Is All You Need 해부" (sj-techlog), section "KV cache는 추론의 같은
# 계산을 반복하지 않게 한다": the new token's query only, against the cached
# keys/values of all earlier positions and its own.

def test_decode_one_token_at_a_time_reproduces_the_printed_causal_run():
    """Feeding the page's 3 tokens one at a time through the cache gives the
    printed causal outputs row by row ([10, 0], [3.302385, 6.697615],
    [7.517449, 7.517449])."""
    g = _load("three_token_verification.json")
    q = np.asarray(g["q"], dtype=np.float64)[None, None]
    k = np.asarray(g["k"], dtype=np.float64)[None, None]
    v = np.asarray(g["v"], dtype=np.float64)[None, None]
    tol = g["tolerance"]
    for t in range(3):
        out = oracle.decode(q[:, :, t:t + 1], k, v, cache_lens=[t + 1])
        np.testing.assert_allclose(out[0, 0, 0], g["causal_outputs"][t], atol=tol, rtol=0)


@pytest.mark.parametrize("n_q", [1, 3, 8])
def test_decode_equals_the_last_rows_of_causal_attention(n_q):
    """With L cached rows, the n_q newest tokens' outputs are rows L - n_q ..
    L - 1 of causal self-attention over the first L positions (bottom-right
    alignment); rows past L in the cache are never read."""
    rng = np.random.default_rng(11 + n_q)
    B, h, n_max, d = 3, 2, 23, 6
    q_all = rng.standard_normal((B, h, n_max, d))
    k = rng.standard_normal((B, h, n_max, d))
    v = rng.standard_normal((B, h, n_max, d))
    lens = np.array([23, 15, n_q], dtype=np.int32)
    q = np.stack([q_all[b, :, lens[b] - n_q:lens[b]] for b in range(B)])
    k_junk, v_junk = k.copy(), v.copy()
    for b in range(B):  # garbage past each entry's length must not matter
        k_junk[b, :, lens[b]:] = 1e6
        v_junk[b, :, lens[b]:] = -1e6
    out = oracle.decode(q, k_junk, v_junk, cache_lens=lens)
    for b in range(B):
        L = lens[b]
        full = oracle.attention(q_all[b:b + 1, :, :L], k[b:b + 1, :, :L], v[b:b + 1, :, :L],
                                MASK_CAUSAL)
        np.testing.assert_allclose(out[b], full[0, :, L - n_q:L], rtol=0, atol=1e-12)


def test_decode_more_queries_than_cached_rows_gives_zero_rows_first():
    rng = np.random.default_rng(21)
    q = rng.standard_normal((2, 1, 4, 5))
    k = rng.standard_normal((2, 1, 6, 5))
    v = rng.standard_normal((2, 1, 6, 5))
    out = oracle.decode(q, k, v, cache_lens=[2, 0])
    assert np.all(out[0, 0, :2] == 0.0) and np.all(out[1] == 0.0)
    np.testing.assert_allclose(out[0, 0, 2], v[0, 0, 0], rtol=0, atol=1e-15)  # position 0
    assert np.all(np.abs(out[0, 0, 3]) > 0)


def test_decode_matches_torch_fp64_sdpa_with_bottom_right_causal_mask():
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    rng = np.random.default_rng(31)
    B, h, n_q, n_max, d = 2, 3, 5, 37, 8
    q = rng.standard_normal((B, h, n_q, d))
    k = rng.standard_normal((B, h, n_max, d))
    v = rng.standard_normal((B, h, n_max, d))
    lens = np.array([37, 20], dtype=np.int32)
    ours = oracle.decode(q, k, v, cache_lens=lens)
    for b in range(B):
        L = int(lens[b])
        pos = torch.arange(L - n_q, L)[:, None]
        allowed = (torch.arange(L)[None, :] <= pos)[None, None]
        ref = F.scaled_dot_product_attention(torch.from_numpy(q[b:b + 1]),
                                             torch.from_numpy(k[b:b + 1, :, :L]),
                                             torch.from_numpy(v[b:b + 1, :, :L]),
                                             attn_mask=allowed).numpy()
        np.testing.assert_allclose(ours[b:b + 1], ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- encoder sub-layers
# "[논문 리뷰]Attention Is All You Need", sections 3.1 (output = LayerNorm(x +
# Sublayer(x))) and 3.3 (FFN(x) = max(0, x W_1 + b_1) W_2 + b_2);
# "Attention Is All You Need 해부", section "4. residual connection과
# LayerNorm": LayerNorm(x) = gamma (x - mu) / sqrt(sigma^2 + eps) + beta over
# one token's features.

def test_layernorm_rows_have_zero_mean_and_the_eps_shrunk_unit_variance():
    rng = np.random.default_rng(41)
    x = rng.standard_normal((7, 33)) * 3.0 + 5.0
    eps = 1e-3
    out = oracle.layernorm(x, np.ones(33), np.zeros(33), eps)
    np.testing.assert_allclose(out.mean(axis=1), 0.0, atol=1e-13)
    var = x.var(axis=1)
    np.testing.assert_allclose(out.var(axis=1), var / (var + eps), rtol=1e-12)


def test_layernorm_constant_row_gives_beta_and_gamma_beta_are_affine():
    rng = np.random.default_rng(42)
    d = 16
    gamma, beta = rng.standard_normal(d), rng.standard_normal(d)
    const = np.full((2, d), 3.25)
    np.testing.assert_allclose(oracle.layernorm(const, gamma, beta, 1e-6), np.broadcast_to(beta, (2, d)),
                               atol=1e-15)
    x = rng.standard_normal((5, d))
    plain = oracle.layernorm(x, np.ones(d), np.zeros(d), 1e-6)
    np.testing.assert_allclose(oracle.layernorm(x, gamma, beta, 1e-6), plain * gamma + beta,
                               rtol=0, atol=1e-14)


def test_ffn_with_identity_weights_is_relu_of_the_shifted_input():
    """W_1 = W_2 = I, b_2 = 0: FFN(x) = max(0, x + b_1) (the max(0, .) of the
    formula, not a smooth activation; an off-by-one bias or a missing ReLU fails)."""
    rng = np.random.default_rng(43)
    d = 12
    x = rng.standard_normal((6, d))
    b_1 = rng.standard_normal(d) * 0.5
    out = oracle.ffn(x, np.eye(d), b_1, np.eye(d), np.zeros(d))
    np.testing.assert_allclose(out, np.maximum(0.0, x + b_1), rtol=0, atol=1e-15)


def test_ffn_and_layernorm_match_torch_fp64():
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    rng = np.random.default_rng(44)
    x = rng.standard_normal((3, 5, 32))
    w_1, b_1 = rng.standard_normal((32, 128)) * 0.2, rng.standard_normal(128) * 0.1
    w_2, b_2 = rng.standard_normal((128, 32)) * 0.2, rng.standard_normal(32) * 0.1
    t = torch.from_numpy
    ref = F.linear(F.relu(F.linear(t(x), t(w_1.T.copy()), t(b_1))), t(w_2.T.copy()), t(b_2))
    np.testing.assert_allclose(oracle.ffn(x, w_1, b_1, w_2, b_2), ref.numpy(), rtol=1e-12,
                               atol=1e-12)
    g, b = rng.standard_normal(32), rng.standard_normal(32)
    ref = F.layer_norm(t(x), (32,), t(g), t(b), eps=1e-5)
    np.testing.assert_allclose(oracle.layernorm(x, g, b, 1e-5), ref.numpy(), rtol=1e-12,
                               atol=1e-12)


def _encoder_case(seed, B=2, n=7, d_model=16, h=4, d_ff=32):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, n, d_model))
    ws = [rng.standard_normal((d_model, d_model)) * 0.3 for _ in range(4)]
    g_1, be_1 = 1 + 0.1 * rng.standard_normal(d_model), 0.1 * rng.standard_normal(d_model)
    w_1, b_1 = rng.standard_normal((d_model, d_ff)) * 0.3, 0.1 * rng.standard_normal(d_ff)
    w_2, b_2 = rng.standard_normal((d_ff, d_model)) * 0.3, 0.1 * rng.standard_normal(d_model)
    g_2, be_2 = 1 + 0.1 * rng.standard_normal(d_model), 0.1 * rng.standard_normal(d_model)
    return x, ws, (g_1, be_1, w_1, b_1, w_2, b_2, g_2, be_2), h


@pytest.mark.parametrize("mask", [MASK_NONE, MASK_KEY_PADDING])
def test_encoder_layer_is_two_post_ln_sublayers(mask):
    x, ws, p, h = _encoder_case(45)
    g_1, be_1, w_1, b_1, w_2, b_2, g_2, be_2 = p
    lens = np.array([7, 3], dtype=np.int32)
    out, y = oracle.encoder_layer(x, *ws, *p, h, mask, kv_lens=lens, eps=1e-6, return_mid=True)
    att = oracle.mha(x, x, *ws, h, mask, kv_lens=lens)
    np.testing.assert_allclose(y, oracle.layernorm(x + att, g_1, be_1, 1e-6), rtol=0, atol=1e-13)
    np.testing.assert_allclose(out, oracle.layernorm(y + oracle.ffn(y, w_1, b_1, w_2, b_2), g_2,
                                                     be_2, 1e-6), rtol=0, atol=1e-13)


def test_encoder_layer_matches_torch_transformer_encoder_layer():
    """torch's post-LN TransformerEncoderLayer (ReLU, no dropout, zero
    attention biases) with the same weights, in fp64."""
    torch = pytest.importorskip("torch")
    x, ws, p, h = _encoder_case(46)
    g_1, be_1, w_1, b_1, w_2, b_2, g_2, be_2 = p
    d_model, d_ff = x.shape[2], w_1.shape[1]
    layer = torch.nn.TransformerEncoderLayer(d_model, h, d_ff, dropout=0.0, activation="relu",
                                             layer_norm_eps=1e-6, batch_first=True,
                                             norm_first=False, dtype=torch.float64)
    t = torch.from_numpy
    with torch.no_grad():
        layer.self_attn.in_proj_weight.copy_(t(np.concatenate([w.T for w in ws[:3]], axis=0)))
        layer.self_attn.in_proj_bias.zero_()
        layer.self_attn.out_proj.weight.copy_(t(ws[3].T.copy()))
        layer.self_attn.out_proj.bias.zero_()
        layer.linear1.weight.copy_(t(w_1.T.copy()))
        layer.linear1.bias.copy_(t(b_1))
        layer.linear2.weight.copy_(t(w_2.T.copy()))
        layer.linear2.bias.copy_(t(b_2))
        layer.norm1.weight.copy_(t(g_1))
        layer.norm1.bias.copy_(t(be_1))
        layer.norm2.weight.copy_(t(g_2))
        layer.norm2.bias.copy_(t(be_2))
    layer.eval()
    with torch.no_grad():
        ref = layer(t(x)).numpy()
    np.testing.assert_allclose(oracle.encoder_layer(x, *ws, *p, h, eps=1e-6), ref, rtol=1e-10,
                               atol=1e-10)


def test_oracle_refuses_bf16_bit_patterns():
    """A bf16 tensor's uint16 bits are not its values: the oracle refuses them."""
    bits = np.zeros((1, 1, 4, 64), dtype=np.uint16)
    with pytest.raises(TypeError):
        oracle.attention(bits, bits, bits)
    with pytest.raises(TypeError):
        oracle.attention_rows(bits[0, 0], np.arange(4), bits[0, 0], bits[0, 0], causal=False)
