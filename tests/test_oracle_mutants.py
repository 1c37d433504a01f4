"""The pins reject plausible mistakes: each mutant below plants one mistake in the
oracle (on the CPU, by wrapping its functions) and must fail the exact
hand-worked example or the autograd pin, while the unmodified oracle passes."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "t4d2.json")


def _golden():
    with open(GOLDEN) as f:
        g = json.load(f)
    return g, {k: np.array(v, dtype=np.float64)[None, None] for k, v in g["inputs"].items()}


def _arr(rows):
    return np.array([[float(Fraction(x)) for x in r] for r in rows])


def golden_ok(fwd, bwd):
    """True iff fwd/bwd reproduce every exact value of the hand-worked example."""
    g, x = _golden()
    for lam, case in g["cases"].items():
        l = np.array([float(Fraction(lam))])
        o, cs, fin = fwd(x["q"], x["k"], x["v"], l)
        dq, dk, dv = bwd(x["q"], x["k"], x["v"], x["dO"], l)
        checks = [(o[0, 0], case["O"]), (fin[0, 0], case["final_state"]), (cs[0, 0, 1], case["chunk_states_C2"][1]),
                  (cs[0, 0, 0], case["chunk_states_C2"][0]), (dq[0, 0], case["dq"]), (dk[0, 0], case["dk"]),
                  (dv[0, 0], case["dv"])]
        if not all(np.array_equal(a, _arr(b)) for a, b in checks):
            return False
    return True


def f_ok(q, k, v, l):
    return oracle.fwd_recurrent(q, k, v, lam=l, chunk=2)


def b_ok(q, k, v, g, l):
    return oracle.bwd_recurrent(q, k, v, g, lam=l)[:3]


MUTANTS = {
    # output uses S q instead of S^T q (transposed state)
    "transposed_state": (lambda q, k, v, l: oracle.fwd_recurrent(q, v, k, lam=l, chunk=2), b_ok),
    # decay exponent off by one (lambda^{t-s+1})
    "decay_off_by_one": (lambda q, k, v, l: tuple(
        x * (l[0] if i != 1 else 1.0) for i, x in enumerate(oracle.fwd_recurrent(q, k, v, lam=l, chunk=2))), b_ok),
    # chunk states inclusive instead of exclusive
    "inclusive_chunk_states": (lambda q, k, v, l: (lambda o, cs, f: (o, np.concatenate(
        [cs[:, :, 1:], f[:, :, None]], axis=2), f))(*oracle.fwd_recurrent(q, k, v, lam=l, chunk=2)), b_ok),
    # strictly causal (s < t): the diagonal term dropped
    "dropped_diagonal": (lambda q, k, v, l: (lambda o, cs, f: (
        o - np.einsum("bhtd,bhtd->bht", q, k)[..., None] * v, cs, f))(*oracle.fwd_recurrent(q, k, v, lam=l, chunk=2)),
        b_ok),
    # sign error in dk
    "dk_sign": (f_ok, lambda q, k, v, g, l: (lambda a, b, c: (a, -b, c))(*b_ok(q, k, v, g, l))),
    # dq and dk swapped
    "dq_dk_swapped": (f_ok, lambda q, k, v, g, l: (lambda a, b, c: (b, a, c))(*b_ok(q, k, v, g, l))),
    # dv computed with R instead of R^T (transposed operand)
    "dv_transposed": (f_ok, lambda q, k, v, g, l: (lambda a, b, c: (a, b, oracle.bwd_recurrent(
        q, k, v, g, lam=l)[1]))(*b_ok(q, k, v, g, l))),
}


def test_unmodified_oracle_passes():
    assert golden_ok(f_ok, b_ok)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_rejected(name):
    fwd, bwd = MUTANTS[name]
    assert not golden_ok(fwd, bwd), name
