"""Pins of the fused LM-head oracle (oracle/lm_head.py), on the CPU.

Each check ties the oracle to something other than its own formula: a
permutation head reduces the step to row selection and the already-pinned row
verify; a rank-one head with hand-picked integers has a closed form; linearity
and the shape rules hold exactly; the fp32 perturbation bound holds for the
accumulation orders a kernel may use.
"""
import numpy as np
import pytest

from oracle import lm_head, sampler


def _bf16(x):
    """Round float64 values to bf16 (round to nearest even) and back."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _perm_head(V, shift):
    perm = (np.arange(V) + shift) % V                # a cyclic shift: not its own inverse
    W = np.zeros((V, V))
    W[np.arange(V), perm] = 1.0
    return W, perm


def test_permutation_head_is_row_selection():
    rng = np.random.default_rng(1)
    B, K, V = 3, 2, 64
    h = _bf16(rng.normal(0, 2, (B, K + 1, V)))
    W, perm = _perm_head(V, 5)
    z = lm_head.lm_head_logits(h, W)
    assert np.array_equal(z, h[..., perm])
    # a transposed operand selects by the inverse permutation and fails this pin
    assert not np.array_equal(h @ W, h[..., perm])


@pytest.mark.parametrize("T", [0.0, 0.7, 1.3])
def test_permutation_head_verify_equals_row_verify(T):
    rng = np.random.default_rng(2)
    B, K, V = 4, 3, 48
    W, perm = _perm_head(V, 7)
    ht = _bf16(rng.normal(0, 2, (B, K + 1, V)))
    hd = _bf16(0.6 * ht[:, :K] + 0.4 * rng.normal(0, 2, (B, K, V)))
    dtok = rng.integers(0, V, (B, K))
    Ts, ks, Ps = np.full(B, T), np.array([0, 5, 0, 12]), np.array([1.0, 0.9, 0.8, 1.0])
    got = lm_head.verify_from_hidden(ht, W, (hd, W), dtok, Ts, ks, Ps, 11, 3)
    want = sampler.verify_batch(ht[..., perm], hd[..., perm], dtok, Ts, ks, Ps, 11, 3)
    for g, w in zip(got, want):
        assert g.n_accepted == w.n_accepted
        assert np.array_equal(g.tokens, w.tokens)


def test_rank_one_head_closed_form():
    # W[v] = c_v * a with a = e0 + e1 and h = (3, 4, 0, 0): h . a = 7, so z_v = 7 c_v
    c = np.array([2.0, -1.0, 0.5, 3.0, 0.0])
    a = np.array([1.0, 1.0, 0.0, 0.0])
    W = c[:, None] * a[None, :]
    h = np.array([3.0, 4.0, 0.0, 0.0])
    assert np.array_equal(lm_head.lm_head_logits(h, W), np.array([14.0, -7.0, 3.5, 21.0, 0.0]))
    # greedy over that row picks the largest c (id 3)
    tok, _ = sampler.sample_row(lm_head.lm_head_logits(h, W), 0.0, 0, 1.0, 0.5)
    assert tok == 3


def test_linearity_and_shapes():
    rng = np.random.default_rng(3)
    V, d = 7, 5                                       # non-square: a transposition cannot pass
    W = rng.integers(-4, 5, (V, d)).astype(np.float64)
    h1 = rng.integers(-8, 9, (2, 3, d)).astype(np.float64)
    h2 = rng.integers(-8, 9, (2, 3, d)).astype(np.float64)
    z = lm_head.lm_head_logits(h1 + h2, W)
    assert z.shape == (2, 3, V)
    assert np.array_equal(z, lm_head.lm_head_logits(h1, W) + lm_head.lm_head_logits(h2, W))
    assert np.array_equal(lm_head.lm_head_logits(3.0 * h1, W), 3.0 * lm_head.lm_head_logits(h1, W))
    with pytest.raises(ValueError):
        lm_head.lm_head_logits(h1, W.T)


def test_fp32_accumulation_stays_within_bound():
    rng = np.random.default_rng(4)
    d, V = 4096, 24
    h = _bf16(rng.normal(0, 1, d))
    W = _bf16(rng.normal(0, 0.05, (V, d)))
    z = lm_head.lm_head_logits(h, W)
    bound = lm_head.logit_error_bound(h, W)
    prods = (h[None, :] * W).astype(np.float32)       # exact: bf16 x bf16 fits fp32
    orders = {
        "forward": np.cumsum(prods, axis=1, dtype=np.float32)[:, -1],
        "reverse": np.cumsum(prods[:, ::-1], axis=1, dtype=np.float32)[:, -1],
        "pairwise": np.sum(prods, axis=1, dtype=np.float32),
        "tiled": np.sum(np.sum(prods.reshape(V, 16, 256), axis=2, dtype=np.float32), axis=1,
                        dtype=np.float32),
    }
    for name, z32 in orders.items():
        err = np.abs(z32.astype(np.float64) - z)
        assert np.all(err <= bound), name
    # the bound is tight enough to matter: gamma_4095 is about 4.9e-4 of sum |h w|
    scale = np.abs(h) @ np.abs(W).T
    assert np.all(bound <= 5e-4 * scale)


def test_greedy_without_draft_and_vocab_mismatch():
    rng = np.random.default_rng(5)
    B, K, V, d = 2, 2, 16, 8
    ht = _bf16(rng.normal(0, 1, (B, K + 1, d)))
    W = _bf16(rng.normal(0, 1, (V, d)))
    dtok = rng.integers(0, V, (B, K))
    res = lm_head.verify_from_hidden(ht, W, None, dtok, np.zeros(B), np.zeros(B, int), np.ones(B), 1, 0)
    z = lm_head.lm_head_logits(ht, W)
    for b, r in enumerate(res):
        n = r.n_accepted
        assert r.tokens[n] == int(np.argmax(z[b, n]))
    with pytest.raises(ValueError):
        lm_head.verify_from_hidden(ht, W, np.zeros((B, K, V + 1)), dtok, np.ones(B), np.zeros(B, int),
                                   np.ones(B), 1, 0)


def _add_trunc(s, t):
    """fp32 addition that truncates toward zero (an accumulator without rounding)."""
    x = float(s) + float(t)                           # exact: both operands are fp32
    r = np.float32(x)
    if abs(float(r)) > abs(x):
        r = np.nextafter(r, np.float32(0.0))
    return r


def test_error_bound_is_nearly_attained():
    # h = (1, e, e, ..., e) against a row of ones, e = 0.9375 ulp(1) = 15 * 2^-27:
    # a truncating fp32 accumulator drops every e after the leading 1, so the
    # error is 4095 e, about 94% of the bound; a bound half as large would fail
    d = 4096
    e = 15.0 * 2.0 ** -27
    h = np.full(d, e)
    h[0] = 1.0
    W = np.ones((1, d))
    z = lm_head.lm_head_logits(h, W)[0]
    assert z == 1.0 + (d - 1) * e
    acc = np.float32(0.0)
    for x in h:
        acc = _add_trunc(acc, np.float32(x))
    assert acc == np.float32(1.0)
    err = z - float(acc)
    bound = lm_head.logit_error_bound(h, W)[0]
    assert 0.9 * bound <= err <= bound


def test_greedy_from_hidden_ties_take_the_lowest_id():
    # W[v] = e_(v mod 4): logits z_v = h[v mod 4] repeat with period 4, so every
    # maximum appears twice; the greedy step must take the lower id (closed form)
    V, d, K = 8, 4, 2
    W = np.zeros((V, d))
    W[np.arange(V), np.arange(V) % d] = 1.0
    ht = np.array([[[1.0, 5.0, 2.0, 0.0],      # max 5 at ids 1 and 5
                    [3.0, 0.0, 3.0, 1.0],      # max 3 at ids 0, 2, 4 and 6
                    [0.0, 0.0, 0.0, 4.0]]])    # max 4 at ids 3 and 7
    zeros, ones = np.zeros(1), np.ones(1)
    for dtok, tokens, n in (([1, 0], [1, 0, 3], 2),     # both drafts are the lowest maxima
                            ([5, 0], [1, -1, -1], 0),   # an equal maximum with a higher id is rejected
                            ([1, 2], [1, 0, -1], 1)):
        r = lm_head.verify_from_hidden(ht, W, None, np.array([dtok]), zeros, np.zeros(1, int), ones, 0, 0)[0]
        assert r.n_accepted == n and list(r.tokens) == tokens, (dtok, r.tokens)
