"""Pins of the fp64 softmax-segment oracle (causal scaled dot-product attention
of a query segment over its gathered key/value prefix), each independent of
the oracle's own arithmetic: closed forms, a brute-force evaluation of the
definition without max subtraction, the textbook library routine, and
invariances a plausible mistake would break."""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(seed, B, H, Tq, Tk, d, s=1.0):
    r = np.random.default_rng(seed)
    return (s * r.standard_normal((B, H, Tq, d)), s * r.standard_normal((B, H, Tk, d)),
            s * r.standard_normal((B, H, Tk, d)))


def test_single_token_closed_form():
    q, k, v = _rand(1, 2, 3, 1, 1, 8)
    o, lse = oracle.softmax_segment_fwd(q, k, v)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, np.einsum("bhtd,bhtd->bht", q, k) / math.sqrt(8), rtol=1e-15, atol=0)


def test_zero_queries_average_the_causal_prefix():
    _, k, v = _rand(2, 1, 2, 5, 9, 4)
    q = np.zeros((1, 2, 5, 4))
    o, lse = oracle.softmax_segment_fwd(q, k, v)
    off = 9 - 5
    for i in range(5):
        np.testing.assert_allclose(o[:, :, i], v[:, :, :off + i + 1].mean(axis=2), rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(lse[:, :, i], math.log(off + i + 1), rtol=1e-15)


def test_brute_force_definition():
    q, k, v = _rand(3, 1, 1, 4, 6, 3, s=0.7)
    o, lse = oracle.softmax_segment_fwd(q, k, v, scale=0.9)
    off = 2
    for i in range(4):
        w = [math.exp(0.9 * sum(q[0, 0, i, c] * k[0, 0, j, c] for c in range(3))) for j in range(off + i + 1)]
        z = sum(w)
        for c in range(3):
            ref = sum(w[j] * v[0, 0, j, c] for j in range(off + i + 1)) / z
            assert abs(o[0, 0, i, c] - ref) < 1e-13
        assert abs(lse[0, 0, i] - math.log(z)) < 1e-13


@pytest.mark.parametrize("Tq,Tk", [(7, 7), (5, 12), (64, 64)])
def test_library_causal_attention(Tq, Tk):
    # queries are the last Tq positions: rows Tk-Tq.. of the full causal attention over Tk tokens
    q, k, v = _rand(4, 2, 2, Tq, Tk, 16)
    o, lse = oracle.softmax_segment_fwd(q, k, v)
    qf = np.concatenate([np.zeros((2, 2, Tk - Tq, 16)), q], axis=2)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qf), torch.from_numpy(k), torch.from_numpy(v), is_causal=True).numpy()
    np.testing.assert_allclose(o, ref[:, :, Tk - Tq:], rtol=1e-12, atol=1e-13)
    s = np.einsum("bhid,bhjd->bhij", qf, k) / 4.0
    s = np.where(np.tril(np.ones((Tk, Tk), bool)), s, -np.inf)
    np.testing.assert_allclose(lse, np.log(np.exp(s).sum(axis=3))[:, :, Tk - Tq:], rtol=1e-12)


def test_key_shift_leaves_outputs_and_moves_lse():
    q, k, v = _rand(5, 1, 2, 6, 10, 8)
    c = np.random.default_rng(6).standard_normal(8)
    o1, l1 = oracle.softmax_segment_fwd(q, k, v)
    o2, l2 = oracle.softmax_segment_fwd(q, k + c, v)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, l1 + np.einsum("bhtd,d->bht", q, c) / math.sqrt(8), rtol=1e-12, atol=1e-12)


def test_dominant_key_selects_its_value():
    q, k, v = _rand(7, 1, 1, 3, 8, 4, s=0.1)
    k[0, 0, 2] = 40.0 * q[0, 0, 0] / np.linalg.norm(q[0, 0, 0]) ** 2 * 2  # score 40 for query 0 at key 2
    o, _ = oracle.softmax_segment_fwd(q, k, v)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 2], rtol=0, atol=1e-12)


def test_rows_subset_matches_full():
    q, k, v = _rand(8, 1, 2, 9, 9, 4)
    o, lse = oracle.softmax_segment_fwd(q, k, v)
    o2, lse2 = oracle.softmax_segment_fwd(q, k, v, rows=[0, 4, 8])
    np.testing.assert_array_equal(o2[:, :, [0, 4, 8]], o[:, :, [0, 4, 8]])
    assert np.isnan(o2[:, :, 1]).all() and np.isnan(lse2[:, :, 2]).all()


# ------------------------------------------------------------------ planted mistakes
def _library_ok(fn):
    """True iff fn (a softmax-segment forward) matches the textbook causal attention
    (rows of the full causal attention over the prefix) and its log-sum-exp."""
    q, k, v = _rand(9, 1, 2, 6, 11, 8)
    o, lse = fn(q, k, v)
    qf = np.concatenate([np.zeros((1, 2, 5, 8)), q], axis=2)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qf), torch.from_numpy(k), torch.from_numpy(v), is_causal=True).numpy()[:, :, 5:]
    s = np.einsum("bhid,bhjd->bhij", qf, k) / math.sqrt(8)
    s = np.where(np.tril(np.ones((11, 11), bool)), s, -np.inf)
    rl = np.log(np.exp(s).sum(axis=3))[:, :, 5:]
    return np.allclose(o, ref, rtol=1e-10, atol=1e-12) and np.allclose(lse, rl, rtol=1e-10, atol=1e-12)


def _strict_mask(q, k, v):      # j < i instead of j <= i: drop the diagonal key
    o, lse = oracle.softmax_segment_fwd(q[:, :, 1:], k[:, :, :-1], v[:, :, :-1])
    return np.concatenate([v[:, :, :1] * 0 + o[:, :, :1], o], axis=2)[:, :, :q.shape[2]], \
        np.concatenate([lse[:, :, :1], lse], axis=2)[:, :, :q.shape[2]]


SOFTMAX_MUTANTS = {
    "no_scale": lambda q, k, v: oracle.softmax_segment_fwd(q, k, v, scale=1.0),
    "queries_first_not_last": lambda q, k, v: (lambda o, l: (o, l))(*oracle.softmax_segment_fwd(
        q, k[:, :, :q.shape[2]], v[:, :, :q.shape[2]])),
    "strict_causal_mask": _strict_mask,
    "keys_values_swapped": lambda q, k, v: oracle.softmax_segment_fwd(q, v, k),
}


def test_softmax_oracle_passes_library_pin():
    assert _library_ok(oracle.softmax_segment_fwd)


@pytest.mark.parametrize("name", sorted(SOFTMAX_MUTANTS))
def test_softmax_mutant_is_rejected(name):
    assert not _library_ok(SOFTMAX_MUTANTS[name]), name
