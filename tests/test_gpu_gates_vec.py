"""Per-dimension gates through the C ABI (linattn_fwd_gated_vec / linattn_bwd_gated_vec)
against the fp64 oracle: o, the final state, dq, dk, dv, d_init and the gradient of
every log-gate [B, H, T, d].

Tolerances: fp32 inputs 1e-4 of max|ref| (one fp32 walk per sequence); bf16 inputs
1e-2 (outputs rounded to bf16; the oracle sees the same bf16 inputs), the fp32
log-gate gradient and states 1e-3.  Cases: d = 64 and 128, several heads, ragged
lengths, an initial state and a final-state gradient, padded strides, shared gates
(every dimension the token's gate) against the per-token gated entry points, T = 0,
lengths 1 to 16 at the edges of the 8-token staging and the two-token updates,
sequences long enough to be cut into chunk groups joined by per-row scans, and two
whole heads of the full-size per-dimension gated workload.
"""
import numpy as np
import pytest
import torch

import oracle
import chunked_state_scan_causal_gb300 as la

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from chunked_state_scan_causal_gb300 import build
    build.build()


def rel(got, ref):
    got = got.detach().double().cpu().numpy() if torch.is_tensor(got) else got
    return float(np.max(np.abs(got - ref))) / max(float(np.max(np.abs(ref))), 1e-30)


def case(seed, B, H, T, d, dtype, lo=-0.2):
    g = torch.Generator().manual_seed(seed)
    q, k, v, dO = (torch.randn(B, H, T, d, generator=g) * s for s in (d ** -0.5, d ** -0.5, 1.0, 1.0))
    q, k, v, dO = (x.to(dtype) for x in (q, k, v, dO))
    lg = torch.rand(B, H, T, d, generator=g) * lo                     # log-gates in (lo, 0]
    init = torch.randn(B, H, d, d, generator=g)
    D = torch.randn(B, H, d, d, generator=g)
    return q, k, v, dO, lg, init, D


@pytest.mark.parametrize("d,dtype,B,H,T", [(64, torch.float32, 1, 2, 200), (128, torch.float32, 2, 1, 77),
                                           (128, torch.bfloat16, 1, 3, 150), (64, torch.bfloat16, 2, 2, 65)])
def test_gated_vec_matches_oracle(d, dtype, B, H, T):
    q, k, v, dO, lg, init, D = case(T + d, B, H, T, d, dtype)
    cu = [x.cuda() for x in (q, k, v, dO, lg, init, D)]
    o, fin = la.fwd_gated_vec(cu[0], cu[1], cu[2], cu[4], init_state=cu[5], want_final=True)
    dq, dk, dv, dlg, dinit = la.bwd_gated_vec(cu[0], cu[1], cu[2], cu[3], cu[4], init_state=cu[5], d_final=cu[6],
                                              want_dinit=True)
    torch.cuda.synchronize()
    n = lambda x: x.double().numpy()
    ro, rfin = oracle.fwd_gated_vec(n(q), n(k), n(v), n(lg), init=n(init))
    rq, rk, rv, rlg, rinit = oracle.bwd_gated_vec(n(q), n(k), n(v), n(dO), n(lg), init=n(init), d_final=n(D))
    tol = 1e-4 if dtype == torch.float32 else 1e-2
    stol = 1e-4 if dtype == torch.float32 else 1e-3
    for name, got, ref, t in (("o", o, ro, tol), ("final", fin, rfin, stol), ("dq", dq, rq, tol), ("dk", dk, rk, tol),
                              ("dv", dv, rv, tol), ("d_log_gate", dlg, rlg, stol), ("d_init", dinit, rinit, stol)):
        assert rel(got, ref) < t, (name, rel(got, ref))


def test_shared_gates_equal_the_per_token_entry_points():
    """Every key dimension taking the token's gate: the per-dimension kernels equal the
    per-token gated entry points (fp32, d = 64: the CUDA-core gated path), and the
    per-token log-gate gradient is the sum of the per-dimension ones."""
    B, H, T, d = 1, 2, 130, 64
    q, k, v, dO, _, init, D = case(7, B, H, T, d, torch.float32)
    g = torch.rand(B, H, T) * -0.3
    gv = g[..., None].expand(B, H, T, d).contiguous()
    cu = [x.cuda() for x in (q, k, v, dO, init, D)]
    gc, gvc = g.cuda(), gv.cuda()
    o_v, fin_v = la.fwd_gated_vec(cu[0], cu[1], cu[2], gvc, init_state=cu[4], want_final=True)
    ck = la.checkpoint_gated(cu[0])
    o_s, fin_s = la.fwd_gated(cu[0], cu[1], cu[2], gc, ck, init_state=cu[4], want_final=True)
    gv_out = la.bwd_gated_vec(cu[0], cu[1], cu[2], cu[3], gvc, init_state=cu[4], d_final=cu[5], want_dinit=True)
    gs_out = la.bwd_gated(cu[0], cu[1], cu[2], cu[3], gc, ck, init_state=cu[4], d_final=cu[5], want_dinit=True)
    torch.cuda.synchronize()
    for a, b in ((o_v, o_s), (fin_v, fin_s), (gv_out[0], gs_out[0]), (gv_out[1], gs_out[1]), (gv_out[2], gs_out[2]),
                 (gv_out[4], gs_out[4])):
        assert rel(a, b.double().cpu().numpy()) < 1e-4
    assert rel(gv_out[3].sum(-1), gs_out[3].double().cpu().numpy()) < 1e-4


def test_gated_vec_padded_strides():
    """Rows 136 elements apart (a padded layout) give the same results as contiguous rows."""
    B, H, T, d = 1, 2, 90, 128
    q, k, v, dO, lg, init, D = case(11, B, H, T, d, torch.bfloat16)

    def padded(x, width=136):
        buf = torch.zeros(*x.shape[:3], width, dtype=x.dtype)
        buf[..., :d] = x
        return buf.cuda()[..., :d]

    qp, kp, vp, dOp = (padded(x) for x in (q, k, v, dO))
    lgc = lg.cuda()
    o, _ = la.fwd_gated_vec(qp, kp, vp, lgc, out=padded(torch.zeros_like(q)))
    outs = [padded(torch.zeros_like(q)) for _ in range(3)]
    dq, dk, dv, dlg, _ = la.bwd_gated_vec(qp, kp, vp, dOp, lgc, outs=outs)
    torch.cuda.synchronize()
    n = lambda x: x.double().numpy()
    ro, _ = oracle.fwd_gated_vec(n(q), n(k), n(v), n(lg))
    rq, rk, rv, rlg, _ = oracle.bwd_gated_vec(n(q), n(k), n(v), n(dO), n(lg))
    for got, ref in ((o, ro), (dq, rq), (dk, rk), (dv, rv)):
        assert rel(got, ref) < 1e-2
    assert rel(dlg, rlg) < 1e-3


def test_gated_vec_empty_sequence():
    B, H, d = 1, 2, 64
    q = torch.zeros(B, H, 0, d, device="cuda")
    lg = torch.zeros(B, H, 0, d, device="cuda")
    init = torch.randn(B, H, d, d, device="cuda")
    D = torch.randn(B, H, d, d, device="cuda")
    o, fin = la.fwd_gated_vec(q, q, q, lg, init_state=init, want_final=True)
    *_, dinit = la.bwd_gated_vec(q, q, q, q, lg, init_state=init, d_final=D, want_dinit=True)
    torch.cuda.synchronize()
    assert o.numel() == 0
    assert torch.equal(fin, init) and torch.equal(dinit, D)


@pytest.mark.parametrize("d,dtype,B,H,T,lo", [(128, torch.bfloat16, 1, 2, 3000, -0.2), (64, torch.float32, 2, 3, 2500, -0.5),
                                              (128, torch.float32, 1, 1, 1025, -2.0), (64, torch.bfloat16, 1, 4, 4096, -0.05)])
def test_gated_vec_chunk_groups(d, dtype, B, H, T, lo):
    """Sequences long enough to be cut into chunk groups (one CTA per group and sequence,
    the groups joined by scans with per-row multipliers), ragged last groups, an initial
    state and a final-state gradient, against the oracle."""
    q, k, v, dO, lg, init, D = case(T + d + 5, B, H, T, d, dtype, lo=lo)
    cu = [x.cuda() for x in (q, k, v, dO, lg, init, D)]
    la.linattn_timing_enable(True)
    la.linattn_timing_collect()
    o, fin = la.fwd_gated_vec(cu[0], cu[1], cu[2], cu[4], init_state=cu[5], want_final=True)
    dq, dk, dv, dlg, dinit = la.bwd_gated_vec(cu[0], cu[1], cu[2], cu[3], cu[4], init_state=cu[5], d_final=cu[6],
                                              want_dinit=True)
    torch.cuda.synchronize()
    kinds = la.linattn_timing_collect()
    la.linattn_timing_enable(False)
    assert kinds["gated_vec_fwd"][0] >= 3 + 2, kinds  # aggregates, scan, outputs (forward), aggregates, scan (backward)
    n = lambda x: x.double().numpy()
    ro, rfin = oracle.fwd_gated_vec(n(q), n(k), n(v), n(lg), init=n(init))
    rq, rk, rv, rlg, rinit = oracle.bwd_gated_vec(n(q), n(k), n(v), n(dO), n(lg), init=n(init), d_final=n(D))
    tol = 1e-4 if dtype == torch.float32 else 1e-2
    stol = 1e-4 if dtype == torch.float32 else 1e-3
    for name, got, ref, t in (("o", o, ro, tol), ("final", fin, rfin, stol), ("dq", dq, rq, tol), ("dk", dk, rk, tol),
                              ("dv", dv, rv, tol), ("d_log_gate", dlg, rlg, stol), ("d_init", dinit, rinit, stol)):
        assert rel(got, ref) < t, (name, rel(got, ref))


def test_gated_vec_full_size_sampled_heads():
    """The per-dimension gated workload at its full size (B1 H32 T131072 d128 bf16, nine
    chunk groups per sequence, the launch configuration the benchmark times): every
    output of two whole heads, the first and the last, against the oracle."""
    from chunked_state_scan_causal_gb300 import inputs
    cfg = dict(inputs.WORKLOADS[8])
    dev = torch.device("cuda", 0)
    q, k, v, dO = (inputs.make(cfg, w).to(dev) for w in ("q", "k", "v", "dO"))
    lg = inputs.make_gates(cfg, device=dev)
    o, _ = la.fwd_gated_vec(q, k, v, lg)
    dq, dk, dv, dlg, _ = la.bwd_gated_vec(q, k, v, dO, lg)
    torch.cuda.synchronize()
    for h in (0, cfg["H"] - 1):
        n = lambda x: x[:, h:h + 1].double().cpu().numpy()
        ro, _ = oracle.fwd_gated_vec(n(q), n(k), n(v), n(lg))
        rq, rk, rv, rlg, _ = oracle.bwd_gated_vec(n(q), n(k), n(v), n(dO), n(lg))
        for name, got, ref, t in (("o", o, ro, 1e-2), ("dq", dq, rq, 1e-2), ("dk", dk, rk, 1e-2),
                                  ("dv", dv, rv, 1e-2), ("d_log_gate", dlg, rlg, 1e-3)):
            assert rel(got[:, h:h + 1], ref) < t, (h, name, rel(got[:, h:h + 1], ref))


@pytest.mark.parametrize("d,dtype,B,H,T", [(128, torch.bfloat16, 1, 2, 3000), (64, torch.float32, 2, 1, 2600),
                                           (128, torch.float32, 1, 1, 100)])
def test_gated_vec_checkpoint_equals_recompute(d, dtype, B, H, T):
    """fwd_gated_vec(ckpt=) + bwd_gated_vec(ckpt=) take the groups' entering states from the
    forward instead of recomputing them with the same kernels: every output is bitwise
    the same (T = 100: one group per sequence, the checkpoint is empty)."""
    q, k, v, dO, lg, init, D = (x.cuda() for x in case(T + 3 * d, B, H, T, d, dtype))
    ck = la.checkpoint_gated_vec(q)
    o1, f1 = la.fwd_gated_vec(q, k, v, lg, init_state=init, want_final=True)
    g1 = la.bwd_gated_vec(q, k, v, dO, lg, init_state=init, d_final=D, want_dinit=True)
    o2, f2 = la.fwd_gated_vec(q, k, v, lg, init_state=init, want_final=True, ckpt=ck)
    g2 = la.bwd_gated_vec(q, k, v, dO, lg, init_state=init, d_final=D, want_dinit=True, ckpt=ck)
    torch.cuda.synchronize()
    for name, a, b in zip(("o", "final", "dq", "dk", "dv", "d_log_gate", "d_init"), (o1, f1) + tuple(g1),
                          (o2, f2) + tuple(g2)):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("T", [1, 2, 3, 7, 8, 9, 15, 16])
@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float32)])
def test_gated_vec_short_sequences(T, d, dtype):
    """Lengths at the edges of the 8-token staging and of the two-token updates (one
    group per sequence), with an initial state and a final-state gradient."""
    B, H = 2, 2
    q, k, v, dO, lg, init, D = case(100 + T + d, B, H, T, d, dtype, lo=-0.5)
    cu = [x.cuda() for x in (q, k, v, dO, lg, init, D)]
    o, fin = la.fwd_gated_vec(cu[0], cu[1], cu[2], cu[4], init_state=cu[5], want_final=True)
    dq, dk, dv, dlg, dinit = la.bwd_gated_vec(cu[0], cu[1], cu[2], cu[3], cu[4], init_state=cu[5], d_final=cu[6],
                                              want_dinit=True)
    torch.cuda.synchronize()
    n = lambda x: x.double().numpy()
    ro, rfin = oracle.fwd_gated_vec(n(q), n(k), n(v), n(lg), init=n(init))
    rq, rk, rv, rlg, rinit = oracle.bwd_gated_vec(n(q), n(k), n(v), n(dO), n(lg), init=n(init), d_final=n(D))
    tol = 1e-4 if dtype == torch.float32 else 1e-2
    stol = 1e-4 if dtype == torch.float32 else 1e-3
    for name, got, ref, t in (("o", o, ro, tol), ("final", fin, rfin, stol), ("dq", dq, rq, tol), ("dk", dk, rk, tol),
                              ("dv", dv, rv, tol), ("d_log_gate", dlg, rlg, stol), ("d_init", dinit, rinit, stol)):
        assert rel(got, ref) < t, (name, rel(got, ref))
