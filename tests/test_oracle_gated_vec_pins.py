"""Pins of the oracle's per-dimension gates (one decay per token, head and key
dimension: S_t = diag(alpha_t) S_{t-1} + k_t v_t^T, o_t = S_t^T q_t).

Pinned to facts outside the function itself: torch fp64 autograd of the masked
form with per-dimension weights exp(G_t[i] - G_s[i]) (G the cumulative
log-gates), the reduction to the scalar-gated oracle when every dimension shares
the token's gate, the decomposition into independent one-dimensional
scalar-gated problems (row i of the state sees only the gates of key dimension
i), and central finite differences of the log-gate gradient across the
oracle's 64-token recompute blocks.
"""
import numpy as np
import torch

import oracle


def _rand(seed, B, H, T, dk, dv):
    r = np.random.default_rng(seed)
    return (r.standard_normal((B, H, T, dk)), r.standard_normal((B, H, T, dk)),
            r.standard_normal((B, H, T, dv)), r.standard_normal((B, H, T, dv)))


def _gates(seed, B, H, T, dk, lo=-0.3):
    return np.random.default_rng(seed).uniform(lo, 0.0, (B, H, T, dk))


def _torch_vec_loss(q, k, v, init, lg, dO, D):
    G = torch.cumsum(lg, dim=2)                                              # [B, H, T, dk]
    T = q.shape[2]
    causal = torch.tril(torch.ones(T, T, dtype=torch.bool))
    diff = G[:, :, :, None, :] - G[:, :, None, :, :]                         # [B, H, t, s, dk]
    W = torch.exp(torch.where(causal[..., None], diff, torch.full_like(diff, -1e300)))
    scores = torch.einsum("bhti,bhsi,bhtsi->bhts", q, k, W)
    O = scores @ v + torch.einsum("bhti,bhti,bhij->bhtj", q, torch.exp(G), init)
    Glast = G[:, :, -1:, :]
    Sfin = torch.einsum("bhsi,bhsi,bhsj->bhij", torch.exp(Glast - G), k, v) + torch.exp(Glast[:, :, 0, :, None]) * init
    return (O * dO).sum() + (Sfin * D).sum()


def test_gated_vec_matches_fp64_autograd_of_the_masked_form():
    """o, S_final and every gradient (q, k, v, init, each log-gate) against torch fp64
    autograd of o_t = sum_{s<=t} sum_i q_t[i] k_s[i] exp(G_t[i] - G_s[i]) v_s + the init term."""
    B, H, T, dk, dv = 1, 2, 37, 4, 3
    q, k, v, dO = _rand(101, B, H, T, dk, dv)
    r = np.random.default_rng(102)
    init, D = r.standard_normal((B, H, dk, dv)), r.standard_normal((B, H, dk, dv))
    lg = _gates(103, B, H, T, dk)
    t = [torch.tensor(a, requires_grad=True) for a in (q, k, v, init, lg)]
    loss = _torch_vec_loss(*t, torch.tensor(dO), torch.tensor(D))
    loss.backward()
    o, fin = oracle.fwd_gated_vec(q, k, v, lg, init=init)
    assert abs(float(np.sum(o * dO) + np.sum(fin * D)) - loss.item()) < 1e-9 * max(1.0, abs(loss.item()))
    dq, dk_, dv_, dlg, dinit = oracle.bwd_gated_vec(q, k, v, dO, lg, init=init, d_final=D)
    for got, ref in zip((dq, dk_, dv_, dinit, dlg), (t[0].grad, t[1].grad, t[2].grad, t[3].grad, t[4].grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-10)


def test_shared_gates_reduce_to_the_scalar_gated_oracle():
    """Every key dimension taking the token's one gate gives the (pinned) scalar-gated
    oracle; the scalar log-gate gradient is the sum of the per-dimension ones."""
    B, H, T, dk, dv = 2, 2, 45, 3, 5
    q, k, v, dO = _rand(111, B, H, T, dk, dv)
    r = np.random.default_rng(112)
    init, D = r.standard_normal((B, H, dk, dv)), r.standard_normal((B, H, dk, dv))
    g = np.random.default_rng(113).uniform(-0.4, 0.0, (B, H, T))
    gv = np.repeat(g[..., None], dk, axis=-1)
    o, fin = oracle.fwd_gated_vec(q, k, v, gv, init=init)
    ro, rfin = oracle.fwd_gated(q, k, v, g, init=init)
    np.testing.assert_allclose(o, ro, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(fin, rfin, rtol=1e-12, atol=1e-12)
    got = oracle.bwd_gated_vec(q, k, v, dO, gv, init=init, d_final=D)
    ref = oracle.bwd_gated(q, k, v, dO, g, init=init, d_final=D)
    for a, b in zip((got[0], got[1], got[2], got[4]), (ref[0], ref[1], ref[2], ref[4])):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(got[3].sum(-1), ref[3], rtol=1e-10, atol=1e-10)


def test_each_key_dimension_is_an_independent_scalar_gated_problem():
    """Row i of the state only ever sees key dimension i: the output is the sum over i
    of the scalar-gated problems (q[..., i], k[..., i], v, gate[..., i]); row i of the
    final state, the gradients of q[..., i], k[..., i], the log-gates of dimension i and
    row i of d_init come from problem i, and dv is the sum over the problems."""
    B, H, T, dk, dv = 1, 2, 70, 3, 4
    q, k, v, dO = _rand(121, B, H, T, dk, dv)
    r = np.random.default_rng(122)
    init, D = r.standard_normal((B, H, dk, dv)), r.standard_normal((B, H, dk, dv))
    lg = _gates(123, B, H, T, dk, lo=-0.5)
    o, fin = oracle.fwd_gated_vec(q, k, v, lg, init=init)
    dq, dk_, dv_, dlg, dinit = oracle.bwd_gated_vec(q, k, v, dO, lg, init=init, d_final=D)
    o_sum, dv_sum = np.zeros_like(o), np.zeros_like(dv_)
    for i in range(dk):
        sl = slice(i, i + 1)
        oi, fi = oracle.fwd_gated(q[..., sl], k[..., sl], v, lg[..., i], init=init[:, :, sl])
        gi = oracle.bwd_gated(q[..., sl], k[..., sl], v, dO, lg[..., i], init=init[:, :, sl], d_final=D[:, :, sl])
        o_sum += oi
        dv_sum += gi[2]
        np.testing.assert_allclose(fin[:, :, sl], fi, rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(dq[..., sl], gi[0], rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(dk_[..., sl], gi[1], rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(dlg[..., i], gi[3], rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(dinit[:, :, sl], gi[4], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(o, o_sum, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(dv_, dv_sum, rtol=1e-10, atol=1e-10)


def test_gated_vec_log_gate_gradient_finite_differences():
    """d(<o, dO> + <S_final, D>)/d log_gate_t[i] by central differences on the forward,
    at tokens on both sides of the 64-token recompute blocks."""
    B, H, T, dk, dv = 1, 1, 70, 3, 2
    q, k, v, dO = _rand(131, B, H, T, dk, dv)
    r = np.random.default_rng(132)
    init, D = r.standard_normal((B, H, dk, dv)), r.standard_normal((B, H, dk, dv))
    lg = _gates(133, B, H, T, dk, lo=-0.5)
    dlg = oracle.bwd_gated_vec(q, k, v, dO, lg, init=init, d_final=D)[3]
    h = 1e-6
    f = lambda g: (lambda o, fin: float(np.sum(o * dO) + np.sum(fin * D)))(*oracle.fwd_gated_vec(q, k, v, g, init=init))
    for t, i in ((0, 0), (1, 2), (31, 1), (63, 0), (64, 2), (65, 1), (69, 0)):
        up, dn = lg.copy(), lg.copy()
        up[0, 0, t, i] += h
        dn[0, 0, t, i] -= h
        num = (f(up) - f(dn)) / (2 * h)
        assert abs(num - dlg[0, 0, t, i]) < 1e-6 * max(1.0, abs(num)), (t, i)
