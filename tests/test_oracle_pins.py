"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test names what it pins.  The pages print no formula, table or worked
example, so the pins are: an exact hand-worked example (also recomputed here by
an exact rational brute force of the definition), torch fp64 autograd of the
masked quadratic form, central finite differences, closed forms for special
cases, and invariants (chunked == recurrent == quadratic for every chunk length,
associativity of the segment scan, bilinearity of the output).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from chunked_state_scan_causal_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "t4d2.json")


def _frac_arr(rows):
    return np.array([[float(Fraction(x)) for x in r] for r in rows])


def _golden():
    with open(GOLDEN) as f:
        g = json.load(f)
    inp = {k: np.array(v, dtype=np.float64)[None, None] for k, v in g["inputs"].items()}
    return g, inp


def _rand(seed, B, H, T, dk, dv, scale=1.0):
    r = np.random.default_rng(seed)
    return (r.standard_normal((B, H, T, dk)) * scale, r.standard_normal((B, H, T, dk)) * scale,
            r.standard_normal((B, H, T, dv)) * scale, r.standard_normal((B, H, T, dv)))


# ------------------------------------------------------------------ exact example
@pytest.mark.parametrize("lam", ["1", "1/2"])
def test_golden_t4d2_exact(lam):
    """Hand-worked T=4, d=2 example: every output matches bit for bit (all values are dyadic)."""
    g, x = _golden()
    case = g["cases"][lam]
    l = np.array([float(Fraction(lam))])
    o, cs, fin = oracle.fwd_recurrent(x["q"], x["k"], x["v"], lam=l, chunk=2)
    assert np.array_equal(o[0, 0], _frac_arr(case["O"]))
    assert np.array_equal(cs[0, 0, 0], _frac_arr(case["chunk_states_C2"][0]))
    assert np.array_equal(cs[0, 0, 1], _frac_arr(case["chunk_states_C2"][1]))
    assert np.array_equal(fin[0, 0], _frac_arr(case["final_state"]))
    dq, dk, dv, _ = oracle.bwd_recurrent(x["q"], x["k"], x["v"], x["dO"], lam=l)
    assert np.array_equal(dq[0, 0], _frac_arr(case["dq"]))
    assert np.array_equal(dk[0, 0], _frac_arr(case["dk"]))
    assert np.array_equal(dv[0, 0], _frac_arr(case["dv"]))
    assert float(np.sum(o * x["dO"])) == float(Fraction(case["inner_O_dO"]))
    # the chunked form (chunk 2 and chunk 3, ragged) and the quadratic form reach the same values
    for C in (1, 2, 3, 4):
        oc, csc, finc = oracle.fwd_chunked(x["q"], x["k"], x["v"], C, lam=l)
        assert np.array_equal(oc, o), C
        assert np.array_equal(finc, fin), C
        dqc, dkc, dvc, _ = oracle.bwd_chunked(x["q"], x["k"], x["v"], x["dO"], C, lam=l)
        assert np.array_equal(dqc, dq) and np.array_equal(dkc, dk) and np.array_equal(dvc, dv), C
    assert np.array_equal(oracle.fwd_quadratic(x["q"], x["k"], x["v"], lam=l), o)


def _brute_fraction(q, k, v, dO, lam):
    """Exact rational evaluation of o_t = sum_{s<=t} lam^{t-s} (q_t.k_s) v_s and its gradients."""
    T, dk = len(q), len(q[0])
    dv = len(v[0])
    dot = lambda a, b: sum(x * y for x, y in zip(a, b))
    O = [[sum(lam ** (t - s) * dot(q[t], k[s]) * v[s][b] for s in range(t + 1)) for b in range(dv)]
         for t in range(T)]
    dq = [[sum(lam ** (t - s) * dot(dO[t], v[s]) * k[s][a] for s in range(t + 1)) for a in range(dk)]
          for t in range(T)]
    dk_ = [[sum(lam ** (t - s) * dot(dO[t], v[s]) * q[t][a] for t in range(s, T)) for a in range(dk)]
           for s in range(T)]
    dv_ = [[sum(lam ** (t - s) * dot(q[t], k[s]) * dO[t][b] for t in range(s, T)) for b in range(dv)]
           for s in range(T)]
    return O, dq, dk_, dv_


def test_golden_matches_rational_brute_force():
    """The stored hand-worked values equal an exact rational brute force of the definition."""
    g, _ = _golden()
    ins = {k: [[Fraction(x) for x in r] for r in v] for k, v in g["inputs"].items()}
    for lam, case in g["cases"].items():
        O, dq, dk, dv = _brute_fraction(ins["q"], ins["k"], ins["v"], ins["dO"], Fraction(lam))
        for name, val in (("O", O), ("dq", dq), ("dk", dk), ("dv", dv)):
            assert [[Fraction(x) for x in r] for r in case[name]] == val, (lam, name)


def test_small_integer_rational_brute_force_rectangular():
    """Random small integers, d_k=3 != d_v=2, lambda=3/4: oracle equals exact rationals (<=1 ulp)."""
    r = np.random.default_rng(7)
    T, dk, dv = 6, 3, 2
    q, k = r.integers(-3, 4, (T, dk)), r.integers(-3, 4, (T, dk))
    v, dO = r.integers(-3, 4, (T, dv)), r.integers(-3, 4, (T, dv))
    lam = Fraction(3, 4)
    O, dq, dk_, dv_ = _brute_fraction(q.tolist(), k.tolist(), v.tolist(), dO.tolist(), lam)
    f = lambda a: np.array(a, dtype=np.float64)[None, None]
    l = np.array([0.75])
    o, _, _ = oracle.fwd_recurrent(f(q), f(k), f(v), lam=l)
    gq, gk, gv, _ = oracle.bwd_recurrent(f(q), f(k), f(v), f(dO), lam=l)
    for got, exp in ((o, O), (gq, dq), (gk, dk_), (gv, dv_)):
        exp = np.array([[float(x) for x in row] for row in exp])
        np.testing.assert_allclose(got[0, 0], exp, rtol=1e-15, atol=1e-15)


# ------------------------------------------------------------------ autograd / finite differences
def _torch_quadratic_loss(q, k, v, init, lam, dO):
    T = q.shape[2]
    t = torch.arange(T, dtype=torch.float64)
    diff = t[:, None] - t[None, :]
    lam_t = lam.view(1, -1, 1, 1)                      # [1, H, 1, 1]
    M = torch.where(diff >= 0, lam_t ** diff.clamp(min=0), torch.zeros((), dtype=torch.float64))
    A = (q @ k.transpose(-1, -2)) * M
    O = A @ v + (lam_t[..., 0] ** (t + 1))[..., None] * (q @ init)
    return (O * dO).sum()


@pytest.mark.parametrize("lam", [1.0, 0.5, 0.96875, 0.9998554587364197])
def test_backward_matches_fp64_autograd(lam):
    """Recurrent and chunked backward equal torch fp64 autograd of the masked quadratic form."""
    B, H, T, dk, dv = 1, 2, 45, 5, 3
    q, k, v, dO = _rand(11, B, H, T, dk, dv)
    init = np.random.default_rng(12).standard_normal((B, H, dk, dv))
    lam_h = np.array([lam, lam ** 0.5])
    tq, tk, tv, ti = (torch.tensor(a, requires_grad=True) for a in (q, k, v, init))
    loss = _torch_quadratic_loss(tq, tk, tv, ti, torch.tensor(lam_h), torch.tensor(dO))
    loss.backward()
    ref = [x.grad.numpy() for x in (tq, tk, tv, ti)]
    for got in (oracle.bwd_recurrent(q, k, v, dO, lam=lam_h, init=init),
                oracle.bwd_chunked(q, k, v, dO, 8, lam=lam_h, init=init),
                oracle.bwd_quadratic(q, k, v, dO, lam=lam_h, init=init)):
        for g, r in zip(got, ref):
            np.testing.assert_allclose(g, r, rtol=1e-10, atol=1e-10)
    o, _, _ = oracle.fwd_recurrent(q, k, v, lam=lam_h, init=init)
    lv = loss.item()
    assert abs(float(np.sum(o * dO)) - lv) < 1e-9 * max(1.0, abs(lv))


def test_backward_central_finite_differences():
    """d<O,dO>/dx by central differences matches the analytic backward on sampled entries."""
    B, H, T, dk, dv = 1, 1, 20, 4, 3
    q, k, v, dO = _rand(3, B, H, T, dk, dv)
    init = np.random.default_rng(4).standard_normal((B, H, dk, dv))
    lam = np.array([0.8])
    grads = oracle.bwd_recurrent(q, k, v, dO, lam=lam, init=init)
    args = [q, k, v, init]
    r = np.random.default_rng(5)
    h = 1e-6
    for which in range(4):
        for _ in range(4):
            idx = tuple(r.integers(0, n) for n in args[which].shape)
            up = [a.copy() for a in args]
            dn = [a.copy() for a in args]
            up[which][idx] += h
            dn[which][idx] -= h
            fu = np.sum(oracle.fwd_recurrent(*up[:3], lam=lam, init=up[3])[0] * dO)
            fd = np.sum(oracle.fwd_recurrent(*dn[:3], lam=lam, init=dn[3])[0] * dO)
            num = (fu - fd) / (2 * h)
            assert abs(num - grads[which][idx]) < 1e-6 * max(1.0, abs(num)), (which, idx)


def _torch_final_state(k, v, init, lam):
    """S_{T-1} = lambda^T init + sum_s lambda^{T-1-s} k_s v_s^T, written out per token."""
    T = k.shape[2]
    lam_t = lam.view(1, -1, 1, 1)
    w = lam_t[..., 0] ** (T - 1 - torch.arange(T, dtype=torch.float64))      # [1, H, T]
    return torch.einsum("bht,bhta,bhtc->bhac", w.expand(k.shape[0], -1, -1), k, v) + (lam_t ** T) * init


@pytest.mark.parametrize("lam", [1.0, 0.5, 0.96875])
def test_backward_with_final_state_gradient_matches_autograd(lam):
    """A gradient D arriving at the final state (from a later segment) adds <D, S_final>
    to the loss: the recurrent backward with d_final equals torch fp64 autograd of it."""
    B, H, T, dk, dv = 1, 2, 37, 4, 6
    q, k, v, dO = _rand(21, B, H, T, dk, dv)
    r = np.random.default_rng(22)
    init, D = r.standard_normal((B, H, dk, dv)), r.standard_normal((B, H, dk, dv))
    lam_h = np.array([lam, lam ** 0.25])
    tq, tk, tv, ti = (torch.tensor(a, requires_grad=True) for a in (q, k, v, init))
    lt = torch.tensor(lam_h)
    loss = _torch_quadratic_loss(tq, tk, tv, ti, lt, torch.tensor(dO)) + \
        (_torch_final_state(tk, tv, ti, lt) * torch.tensor(D)).sum()
    loss.backward()
    ref = [x.grad.numpy() for x in (tq, tk, tv, ti)]
    got = oracle.bwd_recurrent(q, k, v, dO, lam=lam_h, init=init, d_final=D)
    for g, e in zip(got, ref):
        np.testing.assert_allclose(g, e, rtol=1e-10, atol=1e-10)
    # the final state of the forward is the one the torch expression differentiates
    _, _, fin = oracle.fwd_recurrent(q, k, v, lam=lam_h, init=init)
    np.testing.assert_allclose(fin, _torch_final_state(*(torch.tensor(a) for a in (k, v, init)), lt).numpy(),
                               rtol=1e-12, atol=1e-12)


def test_final_state_gradient_finite_differences():
    """d<S_final, D>/dx by central differences matches the backward with d_final (dO = 0)."""
    B, H, T, dk, dv = 1, 1, 15, 3, 4
    q, k, v, _ = _rand(31, B, H, T, dk, dv)
    r = np.random.default_rng(32)
    init, D = r.standard_normal((B, H, dk, dv)), r.standard_normal((B, H, dk, dv))
    lam = np.array([0.85])
    grads = oracle.bwd_recurrent(q, k, v, np.zeros_like(v), lam=lam, init=init, d_final=D)
    assert np.abs(grads[0]).max() == 0.0                      # q does not reach the state
    args, h = [q, k, v, init], 1e-6
    for which in (1, 2, 3):
        for _ in range(4):
            idx = tuple(r.integers(0, n) for n in args[which].shape)
            up, dn = [a.copy() for a in args], [a.copy() for a in args]
            up[which][idx] += h
            dn[which][idx] -= h
            fu = np.sum(oracle.fwd_recurrent(*up[:3], lam=lam, init=up[3])[2] * D)
            fd = np.sum(oracle.fwd_recurrent(*dn[:3], lam=lam, init=dn[3])[2] * D)
            num = (fu - fd) / (2 * h)
            assert abs(num - grads[which][idx]) < 1e-6 * max(1.0, abs(num)), (which, idx)


def test_empty_sequence_passes_final_gradient_to_init():
    """With no tokens the initial state is the final state: d_init == d_final."""
    D = np.random.default_rng(41).standard_normal((1, 2, 3, 4))
    z = np.zeros((1, 2, 0, 3))
    _, _, _, dinit = oracle.bwd_recurrent(z, z, np.zeros((1, 2, 0, 4)), np.zeros((1, 2, 0, 4)),
                                          lam=np.array([0.7, 0.9]), d_final=D)
    np.testing.assert_array_equal(dinit, D)


@pytest.mark.parametrize("lam", [None, 0.9])
def test_segment_grad_states_one_segment_is_d_init(lam):
    """Over one segment, sum_s lambda^{s+1} q_s dO_s^T is the pinned d_init of the backward."""
    B, H, T, dk, dv = 2, 2, 29, 3, 5
    q, k, v, dO = _rand(51, B, H, T, dk, dv)
    lam_h = None if lam is None else np.array([lam, lam ** 0.5])
    W = oracle.segment_grad_states(q, dO, T, lam=lam_h)
    _, _, _, dinit = oracle.bwd_recurrent(q, k, v, dO, lam=lam_h)
    np.testing.assert_allclose(W[0], dinit, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("lam", [None, 0.93])
def test_split_sequence_backward_equals_whole(lam):
    """Sequence split into N equal segments (ranks): each starts from the forward scan of
    the segment states and receives d_final from the reverse scan of the segment gradient
    states; the concatenated gradients equal the whole-sequence backward."""
    B, H, N, L, dk, dv = 1, 2, 4, 11, 3, 4
    T = N * L
    q, k, v, dO = _rand(61, B, H, T, dk, dv)
    init = np.random.default_rng(62).standard_normal((B, H, dk, dv))
    lam_h = np.ones(H) if lam is None else np.array([lam, lam ** 0.5])
    a = lam_h[None, :] ** L                                      # per-segment multiplier, [B, H]
    U = oracle.segment_states(k, v, L, lam=lam_h)                # [N, B, H, dk, dv]
    S_in, _ = oracle.state_scan(U, seg_decay=a, init=init)
    W = oracle.segment_grad_states(q, dO, L, lam=lam_h)
    Dr, _ = oracle.state_scan(W[::-1], seg_decay=a)              # reverse exclusive scan
    D_fin = Dr[::-1]
    ref = oracle.bwd_recurrent(q, k, v, dO, lam=lam_h, init=init)
    parts = [oracle.bwd_recurrent(*(x[:, :, r * L:(r + 1) * L] for x in (q, k, v, dO)), lam=lam_h,
                                  init=S_in[r], d_final=D_fin[r]) for r in range(N)]
    for i in range(3):
        np.testing.assert_allclose(np.concatenate([p[i] for p in parts], axis=2), ref[i], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(parts[0][3], ref[3], rtol=1e-10, atol=1e-10)


# ------------------------------------------------------------------ data-dependent gates
def _gates(seed, B, H, T, lo=-0.3):
    return np.random.default_rng(seed).uniform(lo, 0.0, (B, H, T))


def test_constant_gates_reduce_to_the_scalar_decay():
    """log_gate_t = log(lambda_h) for every t gives the (pinned) per-head decay path."""
    B, H, T, dk, dv = 2, 2, 33, 3, 4
    q, k, v, dO = _rand(71, B, H, T, dk, dv)
    r = np.random.default_rng(72)
    init, D = r.standard_normal((B, H, dk, dv)), r.standard_normal((B, H, dk, dv))
    lam = np.array([0.9, 0.6])
    lg = np.broadcast_to(np.log(lam)[None, :, None], (B, H, T)).copy()
    o, fin = oracle.fwd_gated(q, k, v, lg, init=init)
    ro, _, rfin = oracle.fwd_recurrent(q, k, v, lam=lam, init=init)
    np.testing.assert_allclose(o, ro, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(fin, rfin, rtol=1e-12, atol=1e-12)
    g = oracle.bwd_gated(q, k, v, dO, lg, init=init, d_final=D)
    rg = oracle.bwd_recurrent(q, k, v, dO, lam=lam, init=init, d_final=D)
    for a, b in zip((g[0], g[1], g[2], g[4]), rg):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-11)


def _torch_gated_loss(q, k, v, init, lg, dO, D):
    G = torch.cumsum(lg, dim=-1)                                            # [B, H, T]
    T = q.shape[2]
    causal = torch.tril(torch.ones(T, T, dtype=torch.bool))
    diff = G[..., :, None] - G[..., None, :]
    M = torch.where(causal, torch.exp(torch.where(causal, diff, torch.zeros_like(diff))), torch.zeros_like(diff))
    O = ((q @ k.transpose(-1, -2)) * M) @ v + torch.exp(G)[..., None] * (q @ init)
    Sfin = torch.einsum("bht,bhta,bhtc->bhac", torch.exp(G[..., -1:] - G), k, v) + torch.exp(G[..., -1])[..., None, None] * init
    return (O * dO).sum() + (Sfin * D).sum()


def test_gated_backward_matches_fp64_autograd():
    """Gradients of <dO, o> + <D, S_final> w.r.t. q, k, v, init and every log-gate equal
    torch fp64 autograd of the masked form with mask exp(G_t - G_s), G = cumsum(log_gate)."""
    B, H, T, dk, dv = 1, 2, 41, 4, 3
    q, k, v, dO = _rand(81, B, H, T, dk, dv)
    r = np.random.default_rng(82)
    init, D = r.standard_normal((B, H, dk, dv)), r.standard_normal((B, H, dk, dv))
    lg = _gates(83, B, H, T)
    t = [torch.tensor(a, requires_grad=True) for a in (q, k, v, init, lg)]
    loss = _torch_gated_loss(*t[:4], t[4], torch.tensor(dO), torch.tensor(D))
    loss.backward()
    dq, dk_, dv_, dlg, dinit = oracle.bwd_gated(q, k, v, dO, lg, init=init, d_final=D)
    for got, ref in zip((dq, dk_, dv_, dinit, dlg), (t[0].grad, t[1].grad, t[2].grad, t[3].grad, t[4].grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-10)
    o, fin = oracle.fwd_gated(q, k, v, lg, init=init)
    assert abs(float(np.sum(o * dO) + np.sum(fin * D)) - loss.item()) < 1e-9 * max(1.0, abs(loss.item()))


def test_gated_log_gate_gradient_finite_differences():
    """d(<o, dO> + <S_final, D>)/d log_gate_t by central differences on the forward."""
    B, H, T, dk, dv = 1, 1, 70, 3, 2        # more than one 64-token recompute block
    q, k, v, dO = _rand(91, B, H, T, dk, dv)
    r = np.random.default_rng(92)
    init, D = r.standard_normal((B, H, dk, dv)), r.standard_normal((B, H, dk, dv))
    lg = _gates(93, B, H, T, lo=-0.5)
    dlg = oracle.bwd_gated(q, k, v, dO, lg, init=init, d_final=D)[3]
    h = 1e-6
    for t in (0, 1, 31, 63, 64, 65, 69):
        up, dn = lg.copy(), lg.copy()
        up[0, 0, t] += h
        dn[0, 0, t] -= h
        f = lambda g: (lambda o, fin: float(np.sum(o * dO) + np.sum(fin * D)))(*oracle.fwd_gated(q, k, v, g, init=init))
        num = (f(up) - f(dn)) / (2 * h)
        assert abs(num - dlg[0, 0, t]) < 1e-6 * max(1.0, abs(num)), t


# ------------------------------------------------------------------ chunked == recurrent == quadratic
@pytest.mark.parametrize("lam", [None, 0.5, 0.96875])
def test_chunked_equals_recurrent_every_chunk_length(lam):
    """For every C in [1, T] (ragged last chunk included) the chunked form equals the definition."""
    B, H, T, dk, dv = 1, 2, 23, 4, 6
    q, k, v, dO = _rand(21, B, H, T, dk, dv)
    init = np.random.default_rng(22).standard_normal((B, H, dk, dv))
    lam_h = None if lam is None else np.array([lam, 0.9])
    o_r, _, fin_r = oracle.fwd_recurrent(q, k, v, lam=lam_h, init=init)
    g_r = oracle.bwd_recurrent(q, k, v, dO, lam=lam_h, init=init)
    o_q = oracle.fwd_quadratic(q, k, v, lam=lam_h, init=init)
    np.testing.assert_allclose(o_q, o_r, rtol=1e-12, atol=1e-12)
    for C in range(1, T + 1):
        o_c, cs_c, fin_c = oracle.fwd_chunked(q, k, v, C, lam=lam_h, init=init)
        _, cs_r, _ = oracle.fwd_recurrent(q, k, v, lam=lam_h, init=init, chunk=C)
        np.testing.assert_allclose(o_c, o_r, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(fin_c, fin_r, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(cs_c, cs_r, rtol=1e-12, atol=1e-12)
        g_c = oracle.bwd_chunked(q, k, v, dO, C, lam=lam_h, init=init)
        for a, b in zip(g_c, g_r):
            np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-11)


# ------------------------------------------------------------------ closed forms
def test_single_token_closed_form():
    """T=1: o = (q.k) v + lambda init^T q."""
    q, k, v, _ = _rand(31, 1, 1, 1, 3, 4)
    init = np.random.default_rng(32).standard_normal((1, 1, 3, 4))
    lam = np.array([0.7])
    o, _, fin = oracle.fwd_recurrent(q, k, v, lam=lam, init=init)
    exp = np.dot(q[0, 0, 0], k[0, 0, 0]) * v[0, 0, 0] + 0.7 * init[0, 0].T @ q[0, 0, 0]
    np.testing.assert_allclose(o[0, 0, 0], exp, rtol=1e-14)
    np.testing.assert_allclose(fin[0, 0], 0.7 * init[0, 0] + np.outer(k[0, 0, 0], v[0, 0, 0]), rtol=1e-14)


@pytest.mark.parametrize("lam", [None, 0.9])
def test_final_state_closed_form(lam):
    """S_final = K^T diag(lambda^{T-1-s}) V (lambda = 1: plain K^T V)."""
    q, k, v, _ = _rand(41, 1, 1, 30, 5, 7)
    lam_h = None if lam is None else np.array([lam])
    _, _, fin = oracle.fwd_recurrent(q, k, v, lam=lam_h)
    w = np.ones(30) if lam is None else lam ** (29 - np.arange(30))
    np.testing.assert_allclose(fin[0, 0], k[0, 0].T @ (w[:, None] * v[0, 0]), rtol=1e-12)


def test_scaling_is_trilinear():
    """O(a q, b k, c v) = a b c O(q, k, v) (no normaliser, identity feature map)."""
    q, k, v, _ = _rand(51, 1, 2, 17, 4, 4)
    o, _, _ = oracle.fwd_recurrent(q, k, v, lam=np.array([0.9, 1.0]))
    o2, _, _ = oracle.fwd_recurrent(2.0 * q, -3.0 * k, 0.5 * v, lam=np.array([0.9, 1.0]))
    np.testing.assert_allclose(o2, -3.0 * o, rtol=1e-12)


@pytest.mark.parametrize("lam", [None, 0.95])
def test_bilinearity_inner_products(lam):
    """<O,dO> = <q,dq> = <k,dk> = <v,dv> (O is linear in each of q, k, v); <init,dinit> = init part."""
    B, H, T, dk, dv = 2, 1, 33, 4, 5
    q, k, v, dO = _rand(61, B, H, T, dk, dv)
    lam_h = None if lam is None else np.array([lam])
    o, _, _ = oracle.fwd_recurrent(q, k, v, lam=lam_h)
    dq, dk_, dv_, _ = oracle.bwd_recurrent(q, k, v, dO, lam=lam_h)
    ip = np.sum(o * dO)
    for a, b in ((q, dq), (k, dk_), (v, dv_)):
        assert abs(np.sum(a * b) - ip) < 1e-10 * max(1.0, abs(ip))
    init = np.random.default_rng(62).standard_normal((B, H, dk, dv))
    o_i, _, _ = oracle.fwd_recurrent(q, k, v, lam=lam_h, init=init)
    *_, dinit = oracle.bwd_recurrent(q, k, v, dO, lam=lam_h, init=init)
    assert abs(np.sum(init * dinit) - np.sum((o_i - o) * dO)) < 1e-10 * max(1.0, abs(ip))


# ------------------------------------------------------------------ segments and the scan
@pytest.mark.parametrize("lam", [None, 0.97])
def test_segment_scan_reproduces_chunk_states(lam):
    """Scan of segment-local states == the definition's state at every segment boundary."""
    B, H, T, d = 1, 3, 96, 4
    q, k, v, _ = _rand(71, B, H, T, d, d)
    init = np.random.default_rng(72).standard_normal((B, H, d, d))
    lam_h = None if lam is None else np.array([lam, 0.5, 1.0])
    L = 16
    U = oracle.segment_states(k, v, L, lam=lam_h)                 # [G, B, H, d, d]
    seg_decay = None if lam_h is None else lam_h ** L
    S, total = oracle.state_scan(U, seg_decay=None if seg_decay is None else seg_decay[None, :],
                                 init=init)
    _, cs, fin = oracle.fwd_recurrent(q, k, v, lam=lam_h, init=init, chunk=L)
    np.testing.assert_allclose(np.moveaxis(S, 0, 2), cs, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(total, fin, rtol=1e-12, atol=1e-12)
    # a single segment is the final state without init
    U1 = oracle.segment_states(k, v, T, lam=lam_h)
    _, _, fin0 = oracle.fwd_recurrent(q, k, v, lam=lam_h)
    np.testing.assert_allclose(U1[0], fin0, rtol=1e-12, atol=1e-12)


def test_scan_is_associative_under_regrouping():
    """Scanning 4 segments of 8 equals scanning 2 segments of 16 (two-level regrouping)."""
    B, H, T, d = 1, 2, 32, 3
    _, k, v, _ = _rand(81, B, H, T, d, d)
    lam = np.array([0.8, 0.99])
    U8 = oracle.segment_states(k, v, 8, lam=lam)
    U16 = oracle.segment_states(k, v, 16, lam=lam)
    # combine pairs of 8-segments by the affine composition (a2, U2) o (a1, U1) = (a1 a2, a2 U1 + U2)
    a8 = lam ** 8
    comb = a8[None, None, :, None, None] * U8[0::2] + U8[1::2]
    np.testing.assert_allclose(comb, U16, rtol=1e-12, atol=1e-12)
    S8, t8 = oracle.state_scan(U8, seg_decay=a8[None, :])
    S16, t16 = oracle.state_scan(U16, seg_decay=(lam ** 16)[None, :])
    np.testing.assert_allclose(S8[0::2], S16, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(t8, t16, rtol=1e-12, atol=1e-12)


def test_scan_closed_form_lambda_one():
    """lambda = 1: the exclusive scan is a plain prefix sum."""
    U = np.random.default_rng(91).standard_normal((7, 2, 3, 3))
    S, tot = oracle.state_scan(U)
    np.testing.assert_allclose(S[0], 0.0)
    np.testing.assert_allclose(S[1:], np.cumsum(U, axis=0)[:-1], rtol=1e-13)
    np.testing.assert_allclose(tot, U.sum(0), rtol=1e-13)


# ------------------------------------------------------------------ input recipe
def test_decay_recipe():
    lam = inputs.decay_per_head(32)
    assert lam.dtype == np.float32
    assert lam[0] == np.float32(0.96875)
    assert np.all(np.diff(lam) > 0) and lam[-1] < 1.0
    np.testing.assert_allclose(float(lam[31]), 1 - 2 ** -(5 + 31 / 4), rtol=1e-7)


def test_inputs_are_seeded_and_headwise():
    cfg = dict(inputs.WORKLOADS[2], T=256, B=2, H=3)
    a = inputs.make(cfg, "k")
    b = inputs.make(cfg, "k")
    assert torch.equal(a, b) and a.dtype == torch.bfloat16
    h = inputs.make_head64(cfg, "k", 1, 2)
    np.testing.assert_array_equal(a[1, 2].double().numpy(), h)
    # unit-norm keys (before the bf16 rounding)
    raw = inputs.head(cfg["seed"], "k", 0, 0, 256, 128, "unit_k", cfg["sigma"])
    np.testing.assert_allclose(np.linalg.norm(raw, axis=1), 1.0, rtol=1e-5)
