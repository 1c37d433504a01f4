"""The pins of the softmax-segment backward and of the per-dimension gates reject
plausible mistakes: each mutant plants one mistake in the oracle's result (on the
CPU) and must fail the autograd pin that the unmodified oracle passes (torch fp64
autograd of the library attention, resp. of the masked per-dimension form)."""
import math

import numpy as np
import pytest
import torch

import oracle


# ----------------------------------------------------------------------------- softmax backward
def _softmax_case():
    r = np.random.default_rng(5)
    B, H, Tq, Tk, d = 1, 2, 9, 21, 8
    return tuple(0.8 * r.standard_normal(s) for s in ((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, d), (B, H, Tq, d)))


def _softmax_autograd(q, k, v, dO):
    B, H, Tq, d = q.shape
    Tk = k.shape[2]
    qf = torch.from_numpy(np.concatenate([np.zeros((B, H, Tk - Tq, d)), q], axis=2)).requires_grad_(True)
    kt, vt = torch.from_numpy(k).requires_grad_(True), torch.from_numpy(v).requires_grad_(True)
    o = torch.nn.functional.scaled_dot_product_attention(qf, kt, vt, is_causal=True)
    (o * torch.from_numpy(np.concatenate([np.zeros((B, H, Tk - Tq, d)), dO], axis=2))).sum().backward()
    return qf.grad[:, :, Tk - Tq:].numpy(), kt.grad.numpy(), vt.grad.numpy()


def _softmax_ok(bwd):
    q, k, v, dO = _softmax_case()
    got, ref = bwd(q, k, v, dO), _softmax_autograd(q, k, v, dO)
    return all(np.allclose(a, b, rtol=1e-9, atol=1e-11) for a, b in zip(got, ref))


def _no_delta(q, k, v, dO):
    # dq from ds = p dp (the row term delta dropped); dk and dv as the oracle gives them
    dq, dk, dv = oracle.softmax_segment_bwd(q, k, v, dO)
    off, sc = k.shape[2] - q.shape[2], 1 / math.sqrt(q.shape[3])
    o, _ = oracle.softmax_segment_fwd(q, k, v)
    delta = np.einsum("bhte,bhte->bht", o, dO)
    # the dropped term, added back: dq_i += scale delta_i sum_j p_ij k_j
    for i in range(q.shape[2]):
        n = off + i + 1
        s = sc * np.einsum("bhjd,bhd->bhj", k[:, :, :n], q[:, :, i])
        p = np.exp(s - s.max(axis=2, keepdims=True))
        p /= p.sum(axis=2, keepdims=True)
        dq[:, :, i] += sc * delta[:, :, i, None] * np.einsum("bhj,bhjd->bhd", p, k[:, :, :n])
    return dq, dk, dv


SOFTMAX_MUTANTS = {
    "no_delta_term": _no_delta,
    "dk_without_scale": lambda q, k, v, dO: (lambda a, b, c: (a, b * math.sqrt(q.shape[3]), c))(
        *oracle.softmax_segment_bwd(q, k, v, dO)),
    "queries_first": lambda q, k, v, dO: oracle.softmax_segment_bwd(
        q, k[:, :, :q.shape[2]], v[:, :, :q.shape[2]], dO) + (),
    "dv_from_ds": lambda q, k, v, dO: (lambda a, b, c: (a, b, c + b))(*oracle.softmax_segment_bwd(q, k, v, dO)),
}


def test_unmodified_softmax_backward_passes():
    assert _softmax_ok(lambda q, k, v, dO: oracle.softmax_segment_bwd(q, k, v, dO))


@pytest.mark.parametrize("name", sorted(SOFTMAX_MUTANTS))
def test_softmax_backward_mutant_is_rejected(name):
    f = SOFTMAX_MUTANTS[name]
    if name == "queries_first":
        # the keys past Tq get no gradient at all in this mutant: compare on the full shapes
        def g(q, k, v, dO):
            dq, dk, dv = f(q, k, v, dO)
            pad = lambda x: np.concatenate([x, np.zeros((*x.shape[:2], k.shape[2] - x.shape[2], x.shape[3]))], axis=2)
            return dq, pad(dk), pad(dv)
        assert not _softmax_ok(g)
    else:
        assert not _softmax_ok(f)


# ----------------------------------------------------------------------------- per-dimension gates
def _vec_case():
    r = np.random.default_rng(9)
    B, H, T, dk, dv = 1, 2, 19, 3, 4
    q, k = r.standard_normal((B, H, T, dk)), r.standard_normal((B, H, T, dk))
    v, dO = r.standard_normal((B, H, T, dv)), r.standard_normal((B, H, T, dv))
    init, D = r.standard_normal((B, H, dk, dv)), r.standard_normal((B, H, dk, dv))
    lg = r.uniform(-0.4, 0.0, (B, H, T, dk))
    return q, k, v, dO, init, D, lg


def _vec_autograd(q, k, v, dO, init, D, lg):
    t = [torch.tensor(a, requires_grad=True) for a in (q, k, v, init, lg)]
    qt, kt, vt, it, gt = t
    G = torch.cumsum(gt, dim=2)
    T = q.shape[2]
    causal = torch.tril(torch.ones(T, T, dtype=torch.bool))
    diff = G[:, :, :, None, :] - G[:, :, None, :, :]
    W = torch.exp(torch.where(causal[..., None], diff, torch.full_like(diff, -1e300)))
    O = torch.einsum("bhti,bhsi,bhtsi->bhts", qt, kt, W) @ vt + torch.einsum("bhti,bhti,bhij->bhtj", qt, torch.exp(G), it)
    Gl = G[:, :, -1:, :]
    Sf = torch.einsum("bhsi,bhsi,bhsj->bhij", torch.exp(Gl - G), kt, vt) + torch.exp(Gl[:, :, 0, :, None]) * it
    ((O * torch.from_numpy(dO)).sum() + (Sf * torch.from_numpy(D)).sum()).backward()
    return tuple(x.grad.numpy() for x in (qt, kt, vt, gt, it))


def _vec_ok(bwd):
    c = _vec_case()
    got = bwd(*c)
    ref = _vec_autograd(*c)
    return all(np.allclose(a, b, rtol=1e-9, atol=1e-10) for a, b in zip(got, ref))


def _vec(q, k, v, dO, init, D, lg):
    return oracle.bwd_gated_vec(q, k, v, dO, lg, init=init, d_final=D)


VEC_MUTANTS = {
    # the state term sum_j D[i][j] S_T[i][j] of the last log-gate dropped
    "no_final_state_term": lambda q, k, v, dO, init, D, lg: (lambda a, b, c, g, e: (
        a, b, c, g - np.concatenate([np.zeros_like(g[:, :, :-1]), np.ones_like(g[:, :, -1:])], axis=2) *
        np.einsum("bhij,bhij->bhi", D, oracle.fwd_gated_vec(q, k, v, lg, init=init)[1])[:, :, None, :], e))(
        *_vec(q, k, v, dO, init, D, lg)),
    # every dimension given the mean gate (the scalar-gated problem)
    "shared_gate": lambda q, k, v, dO, init, D, lg: _vec(q, k, v, dO, init, D,
                                                         np.repeat(lg.mean(-1, keepdims=True), lg.shape[-1], -1)),
    # gates of dimension i applied to dimension i+1
    "rolled_gate_dims": lambda q, k, v, dO, init, D, lg: _vec(q, k, v, dO, init, D, np.roll(lg, 1, axis=-1)),
    # the log-gate gradient of token t shifted by one token
    "shifted_gate_gradient": lambda q, k, v, dO, init, D, lg: (lambda a, b, c, g, e: (
        a, b, c, np.roll(g, 1, axis=2), e))(*_vec(q, k, v, dO, init, D, lg)),
}


def test_unmodified_gated_vec_backward_passes():
    assert _vec_ok(_vec)


@pytest.mark.parametrize("name", sorted(VEC_MUTANTS))
def test_gated_vec_mutant_is_rejected(name):
    assert not _vec_ok(VEC_MUTANTS[name])
