"""The weighted-operand forms of the chunked tensor-core kernels, restated block
by block in fp64 numpy, equal the oracle's recurrent definition.

With a per-head decay of at least 0.8 (or gates whose cumulative sums stay in a
narrow span) the kernels weight the rows of one operand per block, reduce every
score mask to a 0/1 pattern times one scalar, and apply a row weight to each
output in the store.  This checks that algebra in exact-enough arithmetic (the
GPU parity tests check the kernels): forward o and final state, the dq pass
(the forward form with roles (dO, v, k) and transposed states), and the
reverse-time dk/dv form with its state-gradient recurrence and d_init, over
several blocks, a partial last block and an initial state.
"""
import numpy as np
import pytest

import oracle


def fwd_weighted(q, k, v, lam, S0, nb):
    """Forward of one sequence ([T, d]) in the value-weighted form, blocks of nb."""
    T = q.shape[0]
    S = S0.copy()
    o = np.zeros((T, v.shape[1]))
    for t0 in range(0, T, nb):
        n = min(nb, T - t0)
        Q, K, V = q[t0:t0 + n], k[t0:t0 + n], v[t0:t0 + n]
        i = np.arange(n)
        Vw = (lam ** (n - 1 - i))[:, None] * V        # value rows weighted
        P = np.tril(Q @ K.T) * lam ** (-n)            # causal 0/1 mask times one scalar
        acc = Q @ S + P @ Vw                          # holds o_i / lambda^{i+1}
        o[t0:t0 + n] = (lam ** (i + 1))[:, None] * acc
        S = lam ** n * S + K.T @ Vw
    return o, S


def bwd_reverse_weighted(q, k, v, dO, lam, nb):
    """dk, dv and the state gradient before token 0 of one sequence in the
    dO-weighted reverse-time form (blocks of nb aligned at the start)."""
    T, d = q.shape
    R = np.zeros((d, v.shape[1]))
    dk, dv = np.zeros_like(k), np.zeros_like(v)
    starts = list(range(0, T, nb))
    for t0 in reversed(starts):
        n = min(nb, T - t0)
        Q, K, V, G = q[t0:t0 + n], k[t0:t0 + n], v[t0:t0 + n], dO[t0:t0 + n]
        i = np.arange(n)
        Gw = (lam ** (i + 1))[:, None] * G            # dO rows weighted
        w = lam ** (n - 1 - i)                        # output row weights
        P1 = np.triu(K @ Q.T) * lam ** (-n)           # anti-causal 0/1 mask times one scalar
        P2 = np.triu(V @ Gw.T) * lam ** (-n)
        dv[t0:t0 + n] = w[:, None] * (K @ R + P1 @ Gw)
        dk[t0:t0 + n] = w[:, None] * (V @ R.T + P2 @ Q)
        R = lam ** n * R + Q.T @ Gw
    return dk, dv, R


def fwd_gated_weighted(q, k, v, log_gate, nb):
    """Gated forward of one sequence in the value-weighted form: C the
    cumulative log2 gate sums, C_prev the sum before a block, C_last at its end."""
    T = q.shape[0]
    C = np.cumsum(log_gate) / np.log(2.0)
    S = np.zeros((q.shape[1], v.shape[1]))
    o = np.zeros((T, v.shape[1]))
    for t0 in range(0, T, nb):
        n = min(nb, T - t0)
        Q, K, V, c = q[t0:t0 + n], k[t0:t0 + n], v[t0:t0 + n], C[t0:t0 + n]
        cprev = C[t0 - 1] if t0 > 0 else 0.0
        clast = c[-1]
        Vw = np.exp2(clast - c)[:, None] * V
        P = np.tril(Q @ K.T) * np.exp2(cprev - clast)
        acc = Q @ S + P @ Vw                          # holds o_i / exp2(C_i - C_prev)
        o[t0:t0 + n] = np.exp2(c - cprev)[:, None] * acc
        S = np.exp2(clast - cprev) * S + K.T @ Vw
    return o


def _case(seed, T, d):
    r = np.random.default_rng(seed)
    return [r.standard_normal((T, d)) / np.sqrt(d) for _ in range(4)]


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


@pytest.mark.parametrize("lam", [0.8, 0.9, 0.999])
@pytest.mark.parametrize("T,nb", [(53, 16), (300, 128), (16, 16)])
def test_forward_and_dq_forms_equal_the_definition(lam, T, nb):
    d = 4
    q, k, v, dO = _case(int(lam * 1000) + T, T, d)
    S0 = np.random.default_rng(T).standard_normal((d, d)) * 0.1
    o, S = fwd_weighted(q, k, v, lam, S0, nb)
    lamv = np.array([lam])
    ro, _, rfin = oracle.fwd_recurrent(q[None, None], k[None, None], v[None, None], lam=lamv, init=S0[None, None])
    assert _rel(o, ro[0, 0]) < 1e-10
    assert _rel(S, rfin[0, 0]) < 1e-10
    # dq = the forward form with roles (dO, v, k) from the transposed state
    dq, _ = fwd_weighted(dO, v, k, lam, S0.T, nb)
    rq, rk, rv, rinit = oracle.bwd_recurrent(q[None, None], k[None, None], v[None, None], dO[None, None], lam=lamv,
                                             init=S0[None, None])
    assert _rel(dq, rq[0, 0]) < 1e-10


@pytest.mark.parametrize("lam", [0.8, 0.9, 0.999])
@pytest.mark.parametrize("T,nb", [(53, 16), (300, 128), (16, 16)])
def test_reverse_form_equals_the_definition(lam, T, nb):
    d = 4
    q, k, v, dO = _case(int(lam * 1000) + 7 * T, T, d)
    dk, dv, dinit = bwd_reverse_weighted(q, k, v, dO, lam, nb)
    rq, rk, rv, rinit = oracle.bwd_recurrent(q[None, None], k[None, None], v[None, None], dO[None, None],
                                             lam=np.array([lam]))
    assert _rel(dk, rk[0, 0]) < 1e-10
    assert _rel(dv, rv[0, 0]) < 1e-10
    assert _rel(dinit, rinit[0, 0]) < 1e-10


@pytest.mark.parametrize("lo,hi", [(-0.05, 0.0), (-0.03, 0.02), (-0.3, 0.0)])
def test_gated_forward_form_equals_the_definition(lo, hi):
    T, d, nb = 70, 4, 16
    q, k, v, _ = _case(5, T, d)
    g = np.random.default_rng(6).uniform(lo, hi, T)
    o = fwd_gated_weighted(q, k, v, g, nb)
    ro, _ = oracle.fwd_gated(q[None, None], k[None, None], v[None, None], g[None, None])
    assert _rel(o, ro[0, 0]) < 1e-10
