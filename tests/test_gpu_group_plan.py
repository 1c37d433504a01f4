"""Many short sequences: the shapes where the tensor-core path cuts every
sequence into long groups followed by a tail of shorter ones (several waves of
(group, sequence) items, handed out at run time).  H = 160, T = 1000 gives
groups of 512, 256 and 232 tokens on a 152-SM GB300: a long group, a short
one and a ragged last one, so every boundary kind of the plan is crossed.

Each (batch, head) sequence is independent, so the fp64 oracle recomputes a
few sampled sequences, taken from both ends of the item order; the others are
checked for finite values and a clean device status.  Tolerance as in
test_gpu_parity: 1e-2 of max|ref| per tensor for bf16 inputs."""
import numpy as np
import pytest
import torch

import oracle
import chunked_state_scan_causal_gb300 as la
from chunked_state_scan_causal_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 1e-2
B, H, T, D = 1, 160, 1000, 128
SAMPLE = (0, 1, 79, 158, 159)


def rel(got, ref):
    got = got.detach().double().cpu().numpy() if torch.is_tensor(got) else got
    return float(np.max(np.abs(got - ref))) / max(float(np.max(np.abs(ref))), 1e-30)


@pytest.fixture(scope="module", autouse=True)
def built():
    from chunked_state_scan_causal_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def case():
    c = inputs.random_case(31, B, H, T, D, dtype="bf16", sigma=1 / np.sqrt(D))
    dev = {k: torch.from_numpy(np.ascontiguousarray(v)).to(torch.bfloat16).cuda() for k, v in c.items()}
    r = np.random.default_rng(32)
    init = (0.1 * r.standard_normal((B, H, D, D))).astype(np.float32)
    dfin = (0.1 * r.standard_normal((B, H, D, D))).astype(np.float32)
    return c, dev, init, dfin


def sampled(a):
    return np.ascontiguousarray(a[:, list(SAMPLE)])


def f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


@pytest.mark.parametrize("with_decay", [False, True])
def test_forward_and_backward_across_long_and_short_groups(case, with_decay):
    c, dev, init, dfin = case
    lam = np.linspace(0.9, 0.999, H).astype(np.float32) if with_decay else None
    dec = None if lam is None else torch.from_numpy(lam).cuda()
    wsf, wsb = la.workspace(dev["q"], la.OP_FWD, dec), la.workspace(dev["q"], la.OP_BWD, dec)
    o, fin, _ = la.fwd(dev["q"], dev["k"], dev["v"], decay=dec, init_state=f32(init), want_final=True, ws=wsf)
    dq, dk, dv, dinit = la.bwd(dev["q"], dev["k"], dev["v"], dev["dO"], decay=dec, init_state=f32(init),
                               d_final=f32(dfin), want_dinit=True, ws=wsb)
    torch.cuda.synchronize()
    assert la.device_status(wsf) == la.OK and la.device_status(wsb) == la.OK
    for t in (o, fin, dq, dk, dv, dinit):
        assert torch.isfinite(t.float()).all()
    sl = None if lam is None else lam[list(SAMPLE)]
    qs, ks, vs, dOs = (sampled(c[w]) for w in ("q", "k", "v", "dO"))
    i64, d64 = sampled(init).astype(np.float64), sampled(dfin).astype(np.float64)
    ro, _, rfin = oracle.fwd_recurrent(qs, ks, vs, lam=sl, init=i64)
    rq, rk, rv, rinit = oracle.bwd_recurrent(qs, ks, vs, dOs, lam=sl, init=i64, d_final=d64)
    idx = list(SAMPLE)
    for name, got, ref in (("o", o[:, idx], ro), ("final", fin[:, idx], rfin), ("dq", dq[:, idx], rq),
                           ("dk", dk[:, idx], rk), ("dv", dv[:, idx], rv), ("d_init", dinit[:, idx], rinit)):
        assert rel(got, ref) < TOL, (name, rel(got, ref))


def test_gated_across_long_and_short_groups(case):
    c, dev, init, dfin = case
    lg = np.random.default_rng(33).uniform(-0.05, 0.0, (B, H, T)).astype(np.float32)
    ck = la.checkpoint_gated(dev["q"])
    o, fin = la.fwd_gated(dev["q"], dev["k"], dev["v"], f32(lg), ck, init_state=f32(init), want_final=True)
    dq, dk, dv, dlg, dinit = la.bwd_gated(dev["q"], dev["k"], dev["v"], dev["dO"], f32(lg), ck,
                                          init_state=f32(init), d_final=f32(dfin), want_dinit=True)
    torch.cuda.synchronize()
    qs, ks, vs, dOs = (sampled(c[w]) for w in ("q", "k", "v", "dO"))
    lgs = sampled(lg).astype(np.float64)
    i64, d64 = sampled(init).astype(np.float64), sampled(dfin).astype(np.float64)
    ro, rfin = oracle.fwd_gated(qs, ks, vs, lgs, init=i64)
    rq, rk, rv, rlg, rinit = oracle.bwd_gated(qs, ks, vs, dOs, lgs, init=i64, d_final=d64)
    idx = list(SAMPLE)
    for name, got, ref in (("o", o[:, idx], ro), ("final", fin[:, idx], rfin), ("dq", dq[:, idx], rq),
                           ("dk", dk[:, idx], rk), ("dv", dv[:, idx], rv), ("d_log_gate", dlg[:, idx], rlg),
                           ("d_init", dinit[:, idx], rinit)):
        assert rel(got, ref) < TOL, (name, rel(got, ref))


def test_checkpointed_backward_equals_recomputed(case):
    # the checkpoint written by the forward holds one state per group of the plan;
    # the backward from it equals the backward that recomputes them, bit for bit,
    # and both match the oracle on the sampled sequences
    c, dev, init, dfin = case
    ck = la.checkpoint(dev["q"])
    o1, _, _ = la.fwd(dev["q"], dev["k"], dev["v"], init_state=f32(init), ckpt=ck)
    a = la.bwd(dev["q"], dev["k"], dev["v"], dev["dO"], init_state=f32(init), ckpt=ck, d_final=f32(dfin))
    b = la.bwd(dev["q"], dev["k"], dev["v"], dev["dO"], init_state=f32(init), d_final=f32(dfin))
    torch.cuda.synchronize()
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x, y)
    qs, ks, vs, dOs = (sampled(c[w]) for w in ("q", "k", "v", "dO"))
    rq, rk, rv, _ = oracle.bwd_recurrent(qs, ks, vs, dOs, init=sampled(init).astype(np.float64),
                                         d_final=sampled(dfin).astype(np.float64))
    idx = list(SAMPLE)
    for got, ref in zip(a[:3], (rq, rk, rv)):
        assert rel(got[:, idx], ref) < TOL
