"""Pins of the oracle's softmax-segment backward (the gradients of q, k, v of causal
scaled dot-product attention of a query segment over its key/value prefix), each
independent of the function's own arithmetic: torch fp64 autograd of the library's
scaled_dot_product_attention, central finite differences of the (separately pinned)
forward oracle, the one-key closed form, and two identities the softmax fixes
(every row's weights sum to one: the dv rows sum to the dO rows; shifting every key
by one vector leaves each row's softmax unchanged: the dk rows sum to zero)."""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(seed, B, H, Tq, Tk, d, s=1.0):
    r = np.random.default_rng(seed)
    return (s * r.standard_normal((B, H, Tq, d)), s * r.standard_normal((B, H, Tk, d)),
            s * r.standard_normal((B, H, Tk, d)), r.standard_normal((B, H, Tq, d)))


@pytest.mark.parametrize("Tq,Tk,scale", [(7, 7, None), (5, 12, None), (33, 70, 0.3)])
def test_matches_autograd_of_the_library_attention(Tq, Tk, scale):
    """The queries are the last Tq of Tk positions: prepend Tk - Tq zero query rows with
    a zero output gradient (they add nothing to dk, dv) and differentiate the library's
    causal attention."""
    B, H, d = 2, 2, 16
    q, k, v, dO = _rand(Tq * 31 + Tk, B, H, Tq, Tk, d, s=0.8)
    qf = torch.from_numpy(np.concatenate([np.zeros((B, H, Tk - Tq, d)), q], axis=2)).requires_grad_(True)
    kt, vt = torch.from_numpy(k).requires_grad_(True), torch.from_numpy(v).requires_grad_(True)
    o = torch.nn.functional.scaled_dot_product_attention(qf, kt, vt, is_causal=True, scale=scale)
    g = torch.from_numpy(np.concatenate([np.zeros((B, H, Tk - Tq, d)), dO], axis=2))
    (o * g).sum().backward()
    dq, dk, dv = oracle.softmax_segment_bwd(q, k, v, dO, scale=scale)
    np.testing.assert_allclose(dq, qf.grad[:, :, Tk - Tq:].numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_finite_differences_of_the_forward_oracle():
    B, H, Tq, Tk, d = 1, 1, 6, 9, 4
    q, k, v, dO = _rand(5, B, H, Tq, Tk, d)
    dq, dk, dv = oracle.softmax_segment_bwd(q, k, v, dO, scale=0.7)
    f = lambda q_, k_, v_: float(np.sum(oracle.softmax_segment_fwd(q_, k_, v_, scale=0.7)[0] * dO))
    h = 1e-6
    for name, x, grad, idx in (("q", q, dq, (0, 0, 2, 1)), ("q", q, dq, (0, 0, 5, 3)), ("k", k, dk, (0, 0, 0, 2)),
                               ("k", k, dk, (0, 0, 8, 0)), ("v", v, dv, (0, 0, 4, 1)), ("v", v, dv, (0, 0, 8, 3))):
        up, dn = x.copy(), x.copy()
        up[idx] += h
        dn[idx] -= h
        args_up = {"q": (up, k, v), "k": (q, up, v), "v": (q, k, up)}[name]
        args_dn = {"q": (dn, k, v), "k": (q, dn, v), "v": (q, k, dn)}[name]
        num = (f(*args_up) - f(*args_dn)) / (2 * h)
        assert abs(num - grad[idx]) < 1e-7 * max(1.0, abs(num)), (name, idx, num, grad[idx])


def test_one_key_closed_form():
    """One query over one key: o = v, so dv = dO and the scores get no gradient."""
    q, k, v, dO = _rand(6, 2, 3, 1, 1, 8)
    dq, dk, dv = oracle.softmax_segment_bwd(q, k, v, dO)
    np.testing.assert_allclose(dv, dO, rtol=0, atol=1e-15)
    assert np.all(dq == 0) and np.all(np.abs(dk) < 1e-15)


def test_softmax_identities():
    B, H, Tq, Tk, d = 2, 2, 20, 45, 8
    q, k, v, dO = _rand(7, B, H, Tq, Tk, d)
    dq, dk, dv = oracle.softmax_segment_bwd(q, k, v, dO, scale=1 / math.sqrt(d))
    np.testing.assert_allclose(dv.sum(axis=2), dO.sum(axis=2), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    # keys no query reaches past the causal limit do not exist here (Tk - Tq + Tq - 1 = Tk - 1),
    # but the first key is seen by every query: its dv row is the sum of p_i0 dO_i over all rows
    o, lse = oracle.softmax_segment_fwd(q, k, v)
    p0 = np.exp(np.einsum("bhid,bhd->bhi", q, k[:, :, 0]) / math.sqrt(d) - lse)
    np.testing.assert_allclose(dv[:, :, 0], np.einsum("bhi,bhie->bhe", p0, dO), rtol=1e-12, atol=1e-12)


def test_sampled_rows_and_last_keys_equal_the_full_computation():
    """The sampling arguments (dq of chosen rows; dk, dv of the last keys) give the same
    entries as the full computation, whose pins are above."""
    B, H, Tq, Tk, d = 1, 2, 30, 80, 8
    q, k, v, dO = _rand(8, B, H, Tq, Tk, d)
    fq, fk, fv = oracle.softmax_segment_bwd(q, k, v, dO)
    rows = [0, 7, 29]
    sq, sk, sv = oracle.softmax_segment_bwd(q, k, v, dO, rows=rows, first_key=70)
    np.testing.assert_allclose(sq[:, :, rows], fq[:, :, rows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(sk[:, :, 70:], fk[:, :, 70:], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(sv[:, :, 70:], fv[:, :, 70:], rtol=1e-13, atol=1e-14)
    assert np.isnan(sq[:, :, 1]).all() and np.isnan(sk[:, :, 69]).all()
