"""Data-dependent gates (linattn_fwd_gated / linattn_bwd_gated) against the
fp64 oracle, through the C ABI: several chunk groups, ragged tails, initial
state and final-state gradient, mild and strong gates, and the reduction to
the per-head decay when every gate of a head is the same.  Tolerance as in
test_gpu_parity (1e-2 of max|ref| per tensor for bf16 inputs, 1e-4 for fp32).
bf16 runs on the tensor-core kernels (d = 64 as the zero-padded d = 128 problem);
fp32 inputs on the CUDA-core kernels (one sequential walk per sequence)."""
import numpy as np
import pytest
import torch

import oracle
import chunked_state_scan_causal_gb300 as la
from chunked_state_scan_causal_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 1e-2
TOLS = {torch.bfloat16: 1e-2, torch.float32: 1e-4}


def rel(got, ref):
    got = got.detach().double().cpu().numpy() if torch.is_tensor(got) else got
    return float(np.max(np.abs(got - ref))) / max(float(np.max(np.abs(ref))), 1e-30)


@pytest.fixture(scope="module", autouse=True)
def built():
    from chunked_state_scan_causal_gb300 import build
    build.build()


def case(seed, B, H, T, lo, d=128, dtype=torch.bfloat16):
    name = "bf16" if dtype == torch.bfloat16 else "f32"
    c = inputs.random_case(seed, B, H, T, d, dtype=name, sigma=1 / np.sqrt(d))
    dev = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dtype).cuda() for k, v in c.items()}
    lg = np.random.default_rng(seed + 1).uniform(lo, 0.0, (B, H, T)).astype(np.float32)
    return c, dev, lg


def f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


# lo = -4: gates down to e^-4, so a 32-token chunk of cumulative sums can span more
# than 100 (base 2) and the masks take their per-element form
@pytest.mark.parametrize("T,lo,d", [(200, -0.05, 128), (2048 + 64, -0.05, 128), (8192 + 100, -0.02, 128),
                                    (1000, -1.0, 128), (300, -4.0, 128), (200, -0.05, 64), (8192 + 100, -0.02, 64),
                                    (1000, -1.0, 64), (300, -4.0, 64)])
def test_gated_forward_and_backward(T, lo, d):
    """bf16 on the tensor-core kernels; d = 64 runs as the zero-padded d = 128 problem
    (the recorded launches are the chunked kernels and the state padding, no CUDA-core walk)."""
    B, H = 1, 3
    c, dev, lg = case(T + d, B, H, T, lo, d=d)
    r = np.random.default_rng(T + 7)
    init = (0.1 * r.standard_normal((B, H, d, d))).astype(np.float32).astype(np.float64)
    D = (0.1 * r.standard_normal((B, H, d, d))).astype(np.float32).astype(np.float64)
    ck = la.checkpoint_gated(dev["q"])
    wsf, wsb = la.workspace(dev["q"], la.OP_FWD_GATED), la.workspace(dev["q"], la.OP_BWD_GATED)
    la.linattn_timing_enable(True)
    la.linattn_timing_collect()
    o, fin = la.fwd_gated(dev["q"], dev["k"], dev["v"], f32(lg), ck, init_state=f32(init), want_final=True, ws=wsf)
    dq, dk, dv, dlg, dinit = la.bwd_gated(dev["q"], dev["k"], dev["v"], dev["dO"], f32(lg), ck, init_state=f32(init),
                                          d_final=f32(D), want_dinit=True, ws=wsb)
    torch.cuda.synchronize()
    kinds = la.linattn_timing_collect()
    la.linattn_timing_enable(False)
    assert la.device_status(wsf) == la.OK and la.device_status(wsb) == la.OK
    assert "tc_chunked_fwd" in kinds and "tc_dual_rev" in kinds, kinds
    assert "simt_fwd" not in kinds and "simt_bwd" not in kinds, kinds
    assert ("pad_d64" in kinds) == (d == 64), kinds
    lg64 = lg.astype(np.float64)
    ro, rfin = oracle.fwd_gated(c["q"], c["k"], c["v"], lg64, init=init)
    rq, rk, rv, rlg, rinit = oracle.bwd_gated(c["q"], c["k"], c["v"], c["dO"], lg64, init=init, d_final=D)
    for name, got, ref in (("o", o, ro), ("final", fin, rfin), ("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv),
                           ("d_log_gate", dlg, rlg), ("d_init", dinit, rinit)):
        assert rel(got, ref) < TOL, (name, rel(got, ref))


def test_gated_heads_of_mixed_strength_across_items():
    """32 heads of four gate kinds in one launch with more (group, sequence)
    items than SMs, so CTAs take items of different kinds in turn: mild gates,
    strong gates (cumulative log2 sums spanning about 92 over a 128-token
    block), gates with positive values (sums that rise and fall), and blocks
    spanning about 46; one head of each kind against the oracle."""
    B, H, T = 1, 32, 16384 + 100
    c = inputs.random_case(51, B, H, T, 128, dtype="bf16", sigma=1 / np.sqrt(128))
    dev = {k: torch.from_numpy(np.ascontiguousarray(v)).to(torch.bfloat16).cuda() for k, v in c.items()}
    kinds = [(-0.05, 0.0), (-1.0, 0.0), (-0.03, 0.02), (-0.5, 0.0)]
    r = np.random.default_rng(52)
    lg = np.stack([r.uniform(*kinds[h % 4], T) for h in range(H)])[None].astype(np.float32)
    ck = la.checkpoint_gated(dev["q"])
    wsf, wsb = la.workspace(dev["q"], la.OP_FWD_GATED), la.workspace(dev["q"], la.OP_BWD_GATED)
    o, _ = la.fwd_gated(dev["q"], dev["k"], dev["v"], f32(lg), ck, ws=wsf)
    dq, dk, dv, dlg, dinit = la.bwd_gated(dev["q"], dev["k"], dev["v"], dev["dO"], f32(lg), ck, want_dinit=True,
                                          ws=wsb)
    assert la.device_status(wsf) == la.OK and la.device_status(wsb) == la.OK
    lg64 = lg.astype(np.float64)
    for h in range(4):
        sl = slice(h, h + 1)
        ro, _ = oracle.fwd_gated(c["q"][:, sl], c["k"][:, sl], c["v"][:, sl], lg64[:, sl])
        rq, rk, rv, rlg, rinit = oracle.bwd_gated(c["q"][:, sl], c["k"][:, sl], c["v"][:, sl], c["dO"][:, sl],
                                                  lg64[:, sl])
        for name, got, ref in (("o", o, ro), ("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv),
                               ("d_log_gate", dlg, rlg), ("d_init", dinit, rinit)):
            assert rel(got[:, sl], ref) < TOL, (name, h, rel(got[:, sl], ref))


# the CUDA-core kernels: fp32 inputs (d = 128 and 64)
@pytest.mark.parametrize("dtype,d,T,lo", [(torch.float32, 128, 200, -0.05), (torch.float32, 64, 1000, -1.0),
                                          (torch.float32, 64, 130, -4.0)])
def test_gated_cuda_core_path(dtype, d, T, lo):
    B, H = 1, 2
    c, dev, lg = case(T + d, B, H, T, lo, d=d, dtype=dtype)
    r = np.random.default_rng(T + 11)
    init = (0.1 * r.standard_normal((B, H, d, d))).astype(np.float32).astype(np.float64)
    D = (0.1 * r.standard_normal((B, H, d, d))).astype(np.float32).astype(np.float64)
    ck = la.checkpoint_gated(dev["q"])
    o, fin = la.fwd_gated(dev["q"], dev["k"], dev["v"], f32(lg), ck, init_state=f32(init), want_final=True)
    dq, dk, dv, dlg, dinit = la.bwd_gated(dev["q"], dev["k"], dev["v"], dev["dO"], f32(lg), ck, init_state=f32(init),
                                          d_final=f32(D), want_dinit=True)
    torch.cuda.synchronize()
    lg64 = lg.astype(np.float64)
    ro, rfin = oracle.fwd_gated(c["q"], c["k"], c["v"], lg64, init=init)
    rq, rk, rv, rlg, rinit = oracle.bwd_gated(c["q"], c["k"], c["v"], c["dO"], lg64, init=init, d_final=D)
    for name, got, ref in (("o", o, ro), ("final", fin, rfin), ("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv),
                           ("d_log_gate", dlg, rlg), ("d_init", dinit, rinit)):
        assert rel(got, ref) < TOLS[dtype], (name, rel(got, ref))


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64), (torch.bfloat16, 64)])
def test_constant_gates_match_the_per_head_decay(dtype, d):
    B, H, T = 1, 2, 3000
    c, dev, _ = case(5, B, H, T, -0.1, d=d, dtype=dtype)
    lam = inputs.decay_per_head(H)
    lg = np.broadcast_to(np.log(lam.astype(np.float64))[None, :, None], (B, H, T)).astype(np.float32)
    ck = la.checkpoint_gated(dev["q"])
    o, _ = la.fwd_gated(dev["q"], dev["k"], dev["v"], f32(lg), ck)
    o2, _, _ = la.fwd(dev["q"], dev["k"], dev["v"], decay=torch.from_numpy(lam).cuda())
    dq, dk, dv, _, _ = la.bwd_gated(dev["q"], dev["k"], dev["v"], dev["dO"], f32(lg), ck)
    dq2, dk2, dv2, _ = la.bwd(dev["q"], dev["k"], dev["v"], dev["dO"], decay=torch.from_numpy(lam).cuda())
    torch.cuda.synchronize()
    for a, b in ((o, o2), (dq, dq2), (dk, dk2), (dv, dv2)):
        assert rel(a, b.double().cpu().numpy()) < TOLS[dtype]


def test_gated_empty_sequence():
    z = torch.empty((1, 2, 0, 128), dtype=torch.bfloat16, device="cuda")
    lg = torch.empty((1, 2, 0), dtype=torch.float32, device="cuda")
    D = torch.randn(1, 2, 128, 128, device="cuda")
    init = torch.randn(1, 2, 128, 128, device="cuda")
    ck = la.checkpoint_gated(z)
    _, fin = la.fwd_gated(z, z, z, lg, ck, init_state=init, want_final=True)
    _, _, _, _, dinit = la.bwd_gated(z, z, z, z, lg, ck, d_final=D, want_dinit=True)
    torch.cuda.synchronize()
    assert torch.equal(fin, init) and torch.equal(dinit, D)
