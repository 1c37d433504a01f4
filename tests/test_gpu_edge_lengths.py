"""Lengths at the edges of the tensor-core kernels' 128-token blocks, through the C ABI
against the fp64 oracle: one token, two, one short of a block, a block, one past,
and two blocks either side (bf16 with d = 128 and d = 64, the plain forward and
backward with an initial state and a final-state gradient, and the gated form).
Tolerance as in the parity tests: 1e-2 of max|ref| per tensor (bf16 inputs)."""
import numpy as np
import pytest
import torch

import oracle
import chunked_state_scan_causal_gb300 as la
from chunked_state_scan_causal_gb300 import inputs

pytestmark = pytest.mark.gpu
LENGTHS = [1, 2, 127, 128, 129, 255, 257]


@pytest.fixture(scope="module", autouse=True)
def built():
    from chunked_state_scan_causal_gb300 import build
    build.build()


def rel(got, ref):
    got = got.detach().double().cpu().numpy() if torch.is_tensor(got) else got
    scale = float(np.max(np.abs(ref)))
    return float(np.max(np.abs(got - ref))) / max(scale, 1e-30)


def _case(seed, B, H, T, d):
    c = inputs.random_case(seed, B, H, T, d, dtype="bf16", sigma=1 / np.sqrt(d))
    dev = {k: torch.from_numpy(np.ascontiguousarray(v)).to(torch.bfloat16).cuda() for k, v in c.items()}
    r = np.random.default_rng(seed + 1)
    init = (0.1 * r.standard_normal((B, H, d, d))).astype(np.float32)
    D = (0.1 * r.standard_normal((B, H, d, d))).astype(np.float32)
    return c, dev, init, D


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("T", LENGTHS)
def test_plain_forward_backward_at_block_edges(d, T):
    B, H = 1, 2
    c, dev, init, D = _case(300 + T + d, B, H, T, d)
    init_d, D_d = torch.from_numpy(init).cuda(), torch.from_numpy(D).cuda()
    o, fin, _ = la.fwd(dev["q"], dev["k"], dev["v"], init_state=init_d, want_final=True)
    dq, dk, dv, dinit = la.bwd(dev["q"], dev["k"], dev["v"], dev["dO"], init_state=init_d, d_final=D_d,
                               want_dinit=True)
    torch.cuda.synchronize()
    i64, D64 = init.astype(np.float64), D.astype(np.float64)
    ro, _, rfin = oracle.fwd_recurrent(c["q"], c["k"], c["v"], init=i64)
    rq, rk, rv, rinit = oracle.bwd_recurrent(c["q"], c["k"], c["v"], c["dO"], init=i64, d_final=D64)
    for name, got, ref in (("o", o, ro), ("final", fin, rfin), ("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv),
                           ("d_init", dinit, rinit)):
        assert rel(got, ref) < 1e-2, (name, rel(got, ref))
    # the checkpointed pair (the forward's group states kept for the backward)
    ck = la.checkpoint(dev["q"])
    o2, fin2, _ = la.fwd(dev["q"], dev["k"], dev["v"], init_state=init_d, want_final=True, ckpt=ck)
    g2 = la.bwd(dev["q"], dev["k"], dev["v"], dev["dO"], init_state=init_d, d_final=D_d, want_dinit=True, ckpt=ck)
    torch.cuda.synchronize()
    for name, got, ref in (("o", o2, ro), ("final", fin2, rfin), ("dq", g2[0], rq), ("dk", g2[1], rk),
                           ("dv", g2[2], rv), ("d_init", g2[3], rinit)):
        assert rel(got, ref) < 1e-2, ("ckpt " + name, rel(got, ref))


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("T", LENGTHS)
def test_gated_forward_backward_at_block_edges(d, T):
    B, H = 1, 2
    c, dev, init, D = _case(400 + T + d, B, H, T, d)
    lg = np.random.default_rng(T + d).uniform(-0.5, 0.0, (B, H, T)).astype(np.float32)
    lgd, init_d, D_d = (torch.from_numpy(x).cuda() for x in (lg, init, D))
    ck = la.checkpoint_gated(dev["q"])
    o, fin = la.fwd_gated(dev["q"], dev["k"], dev["v"], lgd, ck, init_state=init_d, want_final=True)
    dq, dk, dv, dlg, dinit = la.bwd_gated(dev["q"], dev["k"], dev["v"], dev["dO"], lgd, ck, init_state=init_d,
                                          d_final=D_d, want_dinit=True)
    torch.cuda.synchronize()
    i64, D64, lg64 = init.astype(np.float64), D.astype(np.float64), lg.astype(np.float64)
    ro, rfin = oracle.fwd_gated(c["q"], c["k"], c["v"], lg64, init=i64)
    rq, rk, rv, rlg, rinit = oracle.bwd_gated(c["q"], c["k"], c["v"], c["dO"], lg64, init=i64, d_final=D64)
    for name, got, ref in (("o", o, ro), ("final", fin, rfin), ("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv),
                           ("d_log_gate", dlg, rlg), ("d_init", dinit, rinit)):
        assert rel(got, ref) < 1e-2, (name, rel(got, ref))
