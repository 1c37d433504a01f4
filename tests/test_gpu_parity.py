"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Tolerance (max|gpu - ref| / max|ref| over each output tensor): 1e-2 for bf16
inputs, 1e-4 for fp32 inputs, 1e-5 for the fp32-only state scan.  Cases span
several 128-token tiles, several chunk groups, ragged tails (T not a multiple
of 64 or 128), decays from 0.5 to 0.99986, initial states and T = 0.
"""
import numpy as np
import pytest
import torch

import oracle
import chunked_state_scan_causal_gb300 as la
from chunked_state_scan_causal_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 1e-2, torch.float32: 1e-4}


def rel(got, ref):
    got = got.detach().double().cpu().numpy() if torch.is_tensor(got) else got
    den = max(float(np.max(np.abs(ref))), 1e-30)
    return float(np.max(np.abs(got - ref))) / den


@pytest.fixture(scope="module", autouse=True)
def built():
    from chunked_state_scan_causal_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def to_dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).cuda()


def case(seed, B, H, T, d, dtype, sigma=0.125):
    c = inputs.random_case(seed, B, H, T, d, dtype="bf16" if dtype == torch.bfloat16 else "f32", sigma=sigma)
    dev = {k: to_dev(v, dtype) for k, v in c.items()}
    return c, dev


def decays(H, kind):
    if kind is None:
        return None
    if kind == "cfg":
        lam = inputs.decay_per_head(H)
    else:
        lam = np.linspace(kind, 0.999, H).astype(np.float32)
    return lam


# ------------------------------------------------------------------ diagnostics
@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_diag_tensor_core_product(mode):
    """Every operand layout of the tensor-core MMA equals a plain fp32 matrix product."""
    g = torch.Generator().manual_seed(mode)
    A = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    D = torch.zeros(128, 128, dtype=torch.float32, device="cuda")
    st = la.linattn_diag_mma(mode, A.data_ptr(), B.data_ptr(), D.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == la.OK
    torch.cuda.synchronize()
    a, b = A.double().cpu(), B.double().cpu()
    ref = {0: a @ b.T, 1: a.T @ b, 2: a @ b, 3: a.T @ b.T, 4: a @ b}[mode].numpy()
    assert rel(D, ref) < 1e-5


# ------------------------------------------------------------------ state scan
@pytest.mark.parametrize("G", [1, 5, 32, 33, 70, 256, 257, 300, 1000])
@pytest.mark.parametrize("with_decay,with_init", [(False, False), (True, True), (True, False)])
def test_state_scan(G, with_decay, with_init):
    """Column-parallel form (G <= 256) and shuffle + decoupled look-back form (G > 256)."""
    r = np.random.default_rng(G)
    BH, dk, dv = 3, 16, 24
    U = r.standard_normal((G, BH, dk, dv)).astype(np.float32)
    a = r.uniform(0.5, 1.0, BH).astype(np.float32) if with_decay else None
    init = r.standard_normal((BH, dk, dv)).astype(np.float32) if with_init else None
    ref, ref_tot = oracle.state_scan(U, seg_decay=a, init=init)
    out, tot = la.state_scan(torch.from_numpy(U).cuda(), None if a is None else torch.from_numpy(a).cuda(),
                             None if init is None else torch.from_numpy(init).cuda(), want_total=True)
    torch.cuda.synchronize()
    assert rel(out, ref) < 1e-5
    assert rel(tot, ref_tot) < 1e-5


# ------------------------------------------------------------------ chunk_states (segment-local states)
@pytest.mark.parametrize("dtype,d,T,seg", [(torch.float32, 64, 512, 128), (torch.bfloat16, 128, 1024, 256),
                                           (torch.bfloat16, 128, 768, 384), (torch.bfloat16, 64, 512, 64),
                                           (torch.bfloat16, 64, 1280, 256)])
@pytest.mark.parametrize("dk", [None, 0.5, "cfg"])
def test_chunk_states(dtype, d, T, seg, dk):
    B, H = 2, 3
    c, dev = case(3, B, H, T, d, dtype)
    lam = decays(H, dk)
    got = la.chunk_states(dev["k"], dev["v"], seg, decay=None if lam is None else torch.from_numpy(lam).cuda())
    torch.cuda.synchronize()
    ref = oracle.segment_states(c["k"], c["v"], seg, lam=lam)
    assert rel(got, ref) < (1e-2 if dtype == torch.bfloat16 else 1e-4)


# ------------------------------------------------------------------ forward
def run_fwd(c, dev, dtype, lam, init, want_cs=False):
    dec = None if lam is None else torch.from_numpy(lam).cuda()
    init_d = None if init is None else torch.from_numpy(init.astype(np.float32)).cuda()
    ws = la.workspace(dev["q"], la.OP_FWD, dec)
    o, fin, cs = la.fwd(dev["q"], dev["k"], dev["v"], decay=dec, init_state=init_d, want_final=True,
                        want_chunk_states=want_cs, ws=ws)
    assert la.device_status(ws) == la.OK
    return o, fin, cs


def test_config1_fp32_forward_and_chunk_states():
    """The tiny fp32 workload at full size: O [1,2,1024,64] and 16 exclusive chunk states."""
    cfg = inputs.WORKLOADS[1]
    q, k, v = (inputs.make(cfg, w).cuda() for w in ("q", "k", "v"))
    o, fin, cs = la.fwd(q, k, v, want_final=True, want_chunk_states=True)
    torch.cuda.synchronize()
    ro, rcs, rfin = oracle.fwd_recurrent(q.double().cpu().numpy(), k.double().cpu().numpy(),
                                         v.double().cpu().numpy(), chunk=64)
    assert cs.shape == (1, 2, 16, 64, 64)
    assert rel(o, ro) <= 1e-4
    assert rel(cs, rcs) <= 1e-4
    assert rel(fin, rfin) <= 1e-4
    assert float(cs[:, :, 0].abs().max()) == 0.0  # exclusive: chunk 0 enters with the zero state


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("T", [64, 1000, 4096 + 64 + 40])
@pytest.mark.parametrize("dk", [None, 0.5, "cfg"])
def test_forward_chunk_states_bf16(d, T, dk):
    """bf16 inputs with the per-chunk (C = 64) exclusive states requested: the
    states entering every chunk, the outputs and the final state against the
    oracle's definition form (ragged last chunk included)."""
    B, H = 2, 3
    c, dev = case(31 + T, B, H, T, d, torch.bfloat16, sigma=1 / np.sqrt(128))
    lam = decays(H, dk)
    init = (np.random.default_rng(T + 5).standard_normal((B, H, d, d)) * 0.1).astype(np.float32).astype(np.float64)
    o, fin, cs = run_fwd(c, dev, torch.bfloat16, lam, init, want_cs=True)
    ro, rcs, rfin = oracle.fwd_recurrent(c["q"], c["k"], c["v"], lam=lam, init=init, chunk=64)
    assert cs.shape == (B, H, (T + 63) // 64, d, d)
    assert rel(cs, rcs) < 1e-2
    assert rel(o, ro) < 1e-2
    assert rel(fin, rfin) < 1e-2
    assert rel(cs[:, :, 0], init) < 1e-6   # exclusive: chunk 0 enters with the initial state


@pytest.mark.parametrize("dk", [None, "cfg"])
def test_forward_chunk_states_bf16_many_groups(dk):
    """Per-chunk states on the tensor-core path with several chunk groups per
    sequence and more (group, sequence) items than SMs (B2 H16), a ragged last
    chunk; sampled heads from both ends of the item order against the oracle."""
    B, H, T, d = 2, 16, 8192 + 200, 128
    c, dev = case(47, B, H, T, d, torch.bfloat16, sigma=1 / np.sqrt(128))
    lam = decays(H, dk)
    o, fin, cs = run_fwd(c, dev, torch.bfloat16, lam, None, want_cs=True)
    assert cs.shape == (B, H, (T + 63) // 64, d, d)
    for b, h in ((0, 0), (0, 9), (1, 15)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        ro, rcs, rfin = oracle.fwd_recurrent(c["q"][sl], c["k"][sl], c["v"][sl],
                                             lam=None if lam is None else lam[h:h + 1], chunk=64)
        assert rel(cs[sl], rcs) < 1e-2, (b, h)
        assert rel(o[sl], ro) < 1e-2, (b, h)
        assert rel(fin[sl], rfin) < 1e-2, (b, h)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 128),
                                     (torch.float32, 64)])
@pytest.mark.parametrize("T", [64, 200, 1000, 2048])
@pytest.mark.parametrize("dk", [None, 0.5, "cfg"])
def test_forward(dtype, d, T, dk):
    B, H = 1, 3
    c, dev = case(5 + T, B, H, T, d, dtype)
    lam = decays(H, dk)
    init = np.random.default_rng(T).standard_normal((B, H, d, d)) * 0.1
    init = init.astype(np.float32).astype(np.float64)
    o, fin, _ = run_fwd(c, dev, dtype, lam, init)
    ro, _, rfin = oracle.fwd_recurrent(c["q"], c["k"], c["v"], lam=lam, init=init)
    assert rel(o, ro) < TOL[dtype]
    assert rel(fin, rfin) < TOL[dtype]


def test_forward_many_groups_bf16():
    """T long enough for several chunk groups per sequence (group scan and group init exercised)."""
    B, H, T, d = 2, 2, 8192 + 128, 128
    c, dev = case(11, B, H, T, d, torch.bfloat16, sigma=1 / np.sqrt(128))
    for lam in (None, decays(H, "cfg")):
        o, fin, _ = run_fwd(c, dev, torch.bfloat16, lam, None)
        ro, _, rfin = oracle.fwd_recurrent(c["q"], c["k"], c["v"], lam=lam)
        assert rel(o, ro) < 1e-2
        assert rel(fin, rfin) < 1e-2


def test_forward_backward_lambda1_more_items_than_sms():
    """lambda = 1 with more (group, sequence) items than SMs (B2 H16, several
    groups per sequence drawn at run time), a ragged last group and an initial
    state; the checkpoint the forward writes feeds the backward."""
    B, H, T, d = 2, 16, 8192 + 200, 128
    c, dev = case(43, B, H, T, d, torch.bfloat16, sigma=1 / np.sqrt(128))
    init = (np.random.default_rng(44).standard_normal((B, H, d, d)) * 0.1).astype(np.float32)
    init_d = torch.from_numpy(init).cuda()
    ck = la.checkpoint(dev["q"])
    wsf, wsb = la.workspace(dev["q"], la.OP_FWD), la.workspace(dev["q"], la.OP_BWD)
    o, fin, _ = la.fwd(dev["q"], dev["k"], dev["v"], init_state=init_d, want_final=True, ws=wsf, ckpt=ck)
    dq, dk_, dv, dinit = la.bwd(dev["q"], dev["k"], dev["v"], dev["dO"], want_dinit=True, ws=wsb, ckpt=ck,
                                init_state=init_d)
    assert la.device_status(wsf) == la.OK and la.device_status(wsb) == la.OK
    for b, h in ((0, 0), (0, 7), (1, 8), (1, 15)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        i64 = init[sl].astype(np.float64)
        ro, _, rfin = oracle.fwd_recurrent(c["q"][sl], c["k"][sl], c["v"][sl], init=i64)
        rq, rk, rv, rinit = oracle.bwd_recurrent(c["q"][sl], c["k"][sl], c["v"][sl], c["dO"][sl], init=i64)
        for name, got, ref in (("o", o, ro), ("final", fin, rfin), ("dq", dq, rq), ("dk", dk_, rk), ("dv", dv, rv),
                               ("d_init", dinit, rinit)):
            assert rel(got[sl], ref) < 1e-2, (name, b, h)


def test_forward_empty_sequence():
    q = torch.zeros(1, 2, 0, 128, dtype=torch.bfloat16, device="cuda")
    init = torch.randn(1, 2, 128, 128, device="cuda")
    o, fin, _ = la.fwd(q, q, q, init_state=init, want_final=True)
    torch.cuda.synchronize()
    assert o.numel() == 0 and torch.equal(fin, init)


def test_forward_strided_segments_view():
    """Segments of one long sequence passed as a batch through strides (no copies)."""
    H, T, d, S = 2, 2048, 128, 4
    c, dev = case(13, 1, H, T, d, torch.bfloat16)
    seg = T // S
    view = lambda x: x[0].view(H, S, seg, d).permute(1, 0, 2, 3)   # [S, H, seg, d]
    q, k, v = (view(dev[w]) for w in ("q", "k", "v"))
    U = la.chunk_states(k, v, seg)                                   # [1, S, H, d, d]
    init, _ = la.state_scan(U[0].contiguous())                       # [S, H, d, d]
    o_seg, _, _ = la.fwd(q, k, v, init_state=init)
    o_one, _, _ = la.fwd(dev["q"], dev["k"], dev["v"])
    torch.cuda.synchronize()
    ro, _, _ = oracle.fwd_recurrent(c["q"], c["k"], c["v"])
    got = o_seg.permute(1, 0, 2, 3).reshape(1, H, T, d)
    assert rel(got, ro) < 1e-2
    assert rel(o_one, ro) < 1e-2


@pytest.mark.parametrize("width,off", [(136, 0), (144, 8)])
def test_backward_padded_rows(width, off):
    """Rows padded in memory (strides of 272 or 288 bytes; the second view also
    starts 16 bytes off a 32-byte boundary), for the inputs and the outputs: the
    dk/dv pass writes whole 32-byte sectors only where every row starts on a
    32-byte boundary, and 16-byte pieces otherwise."""
    B, H, T, d = 1, 2, 1000, 128
    c, dev = case(17, B, H, T, d, torch.bfloat16)

    def padded(x):
        buf = torch.zeros(B, H, T, width, dtype=x.dtype, device=x.device)
        view = buf[..., off:off + d]
        view.copy_(x)
        return view

    q, k, v, dO = (padded(dev[w]) for w in ("q", "k", "v", "dO"))
    outs = [padded(torch.zeros_like(dev["q"])) for _ in range(3)]
    dq, dk, dv, _ = la.bwd(q, k, v, dO, outs=outs)
    torch.cuda.synchronize()
    rq, rk, rv, _ = oracle.bwd_recurrent(c["q"], c["k"], c["v"], c["dO"])
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert rel(got, ref) < 1e-2


# ------------------------------------------------------------------ backward
@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 64)])
@pytest.mark.parametrize("T", [64, 200, 1000, 2048])
@pytest.mark.parametrize("dk", [None, 0.5, "cfg"])
def test_backward(dtype, d, T, dk):
    B, H = 1, 3
    c, dev = case(7 + T, B, H, T, d, dtype)
    lam = decays(H, dk)
    init = (np.random.default_rng(T + 1).standard_normal((B, H, d, d)) * 0.1).astype(np.float32).astype(np.float64)
    dec = None if lam is None else torch.from_numpy(lam).cuda()
    ws = la.workspace(dev["q"], la.OP_BWD, dec)
    dq, dk_, dv, dinit = la.bwd(dev["q"], dev["k"], dev["v"], dev["dO"], decay=dec,
                                init_state=torch.from_numpy(init.astype(np.float32)).cuda(), want_dinit=True, ws=ws)
    assert la.device_status(ws) == la.OK
    rq, rk, rv, rinit = oracle.bwd_recurrent(c["q"], c["k"], c["v"], c["dO"], lam=lam, init=init)
    tol = TOL[dtype]
    assert rel(dq, rq) < tol
    assert rel(dk_, rk) < tol
    assert rel(dv, rv) < tol
    assert rel(dinit, rinit) < tol


def test_forward_backward_decay_forms_mixed_across_items():
    """Per-head decays on both sides of 0.8 (at or above it the chunked kernels
    weight their operands as the tiles land and the dq pass accumulates the
    reverse aggregates; below it they weight between the products and the
    aggregate pass takes those heads) in one launch with more (group, sequence)
    items than SMs, so CTAs take items of both forms in turn; a ragged tail; a
    few heads of each form checked against the oracle."""
    B, H, T, d = 2, 16, 32768 + 200, 128  # 9 groups of 3712 tokens: 288 items
    c, dev = case(41, B, H, T, d, torch.bfloat16, sigma=1 / np.sqrt(128))
    lam = np.array([0.55, 0.97, 0.7999, 0.8, 0.99986, 0.6, 0.9, 0.75] * 2, np.float32)
    dec = torch.from_numpy(lam).cuda()
    ws = la.workspace(dev["q"], la.OP_BWD, dec)
    dq, dk_, dv, dinit = la.bwd(dev["q"], dev["k"], dev["v"], dev["dO"], decay=dec, want_dinit=True, ws=ws)
    assert la.device_status(ws) == la.OK
    wsf = la.workspace(dev["q"], la.OP_FWD, dec)
    o, fin, _ = la.fwd(dev["q"], dev["k"], dev["v"], decay=dec, want_final=True, ws=wsf)
    assert la.device_status(wsf) == la.OK
    for h in (0, 1, 2, 3):
        sl = slice(h, h + 1)
        ro, _, rfin = oracle.fwd_recurrent(c["q"][:, sl], c["k"][:, sl], c["v"][:, sl], lam=lam[sl])
        rq, rk, rv, rinit = oracle.bwd_recurrent(c["q"][:, sl], c["k"][:, sl], c["v"][:, sl], c["dO"][:, sl],
                                                 lam=lam[sl])
        for got, ref in ((o, ro), (fin, rfin), (dq, rq), (dk_, rk), (dv, rv), (dinit, rinit)):
            assert rel(got[:, sl], ref) < 1e-2, (h, float(lam[h]))


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 64)])
@pytest.mark.parametrize("T,dk", [(2048, None), (8192 + 64, "cfg"), (1000, 0.5)])
def test_checkpointed_forward_backward(dtype, d, T, dk):
    """fwd_ckpt + bwd_ckpt give the oracle's outputs (the backward reads the stored group states)."""
    B, H = 2, 2
    c, dev = case(29 + T, B, H, T, d, dtype, sigma=1 / np.sqrt(128))
    lam = decays(H, dk)
    dec = None if lam is None else torch.from_numpy(lam).cuda()
    init = (np.random.default_rng(T + 3).standard_normal((B, H, d, d)) * 0.1).astype(np.float32)
    init_d = torch.from_numpy(init).cuda()
    ck = la.checkpoint(dev["q"], dec)
    wsf, wsb = la.workspace(dev["q"], la.OP_FWD, dec), la.workspace(dev["q"], la.OP_BWD, dec)
    o, fin, _ = la.fwd(dev["q"], dev["k"], dev["v"], decay=dec, init_state=init_d, want_final=True, ws=wsf, ckpt=ck)
    dq, dk_, dv, dinit = la.bwd(dev["q"], dev["k"], dev["v"], dev["dO"], decay=dec, want_dinit=True, ws=wsb,
                                ckpt=ck, init_state=init_d)
    assert la.device_status(wsf) == la.OK and la.device_status(wsb) == la.OK
    init64 = init.astype(np.float64)
    ro, _, rfin = oracle.fwd_recurrent(c["q"], c["k"], c["v"], lam=lam, init=init64)
    rq, rk, rv, rinit = oracle.bwd_recurrent(c["q"], c["k"], c["v"], c["dO"], lam=lam, init=init64)
    tol = TOL[dtype]
    for got, ref in ((o, ro), (fin, rfin), (dq, rq), (dk_, rk), (dv, rv), (dinit, rinit)):
        assert rel(got, ref) < tol


def test_backward_many_groups_bf16():
    B, H, T, d = 1, 2, 8192 + 64, 128
    c, dev = case(17, B, H, T, d, torch.bfloat16, sigma=1 / np.sqrt(128))
    for lam in (None, decays(H, "cfg")):
        dec = None if lam is None else torch.from_numpy(lam).cuda()
        dq, dk_, dv, dinit = la.bwd(dev["q"], dev["k"], dev["v"], dev["dO"], decay=dec, want_dinit=True)
        torch.cuda.synchronize()
        rq, rk, rv, rinit = oracle.bwd_recurrent(c["q"], c["k"], c["v"], c["dO"], lam=lam)
        for got, ref in ((dq, rq), (dk_, rk), (dv, rv), (dinit, rinit)):
            assert rel(got, ref) < 1e-2


def test_device_status_clean_after_calls():
    B, H, T, d = 1, 2, 1024, 128
    c, dev = case(19, B, H, T, d, torch.bfloat16)
    ws = la.workspace(dev["q"], la.OP_BWD)
    la.bwd(dev["q"], dev["k"], dev["v"], dev["dO"], ws=ws)
    assert la.device_status(ws) == la.OK


# ------------------------------------------------------------------ recurrent decode
@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64), (torch.float32, 128)])
@pytest.mark.parametrize("T", [1, 3, 16])
@pytest.mark.parametrize("dk", [None, "cfg"])
def test_decode_steps(dtype, d, T, dk):
    """Decode of T tokens from a given state == the definition continued from that state."""
    B, H = 2, 3
    c, dev = case(23 + T, B, H, T, d, dtype)
    lam = decays(H, dk)
    init = (np.random.default_rng(T).standard_normal((B, H, d, d)) * 0.3).astype(np.float32)
    state = torch.from_numpy(init).cuda()
    o = la.decode(dev["q"], dev["k"], dev["v"], state, decay=None if lam is None else torch.from_numpy(lam).cuda())
    torch.cuda.synchronize()
    ro, _, rfin = oracle.fwd_recurrent(c["q"], c["k"], c["v"], lam=lam, init=init.astype(np.float64))
    assert rel(o, ro) < TOL[dtype]
    assert rel(state, rfin) < 1e-5


def test_bf16_d64_runs_on_the_tensor_core_kernels():
    """bf16 with d = 64 runs on the d = 128 tensor-core kernels as the zero-padded
    problem (64-column tensor maps: the tiles' other columns load as zeros; the states
    through padded copies): the recorded launches are the chunked kernels and the state
    padding, not the CUDA-core walk; many chunk groups, per-head decays, an initial
    state and a final-state gradient, every head against the oracle."""
    B, H, T, d = 1, 4, 16384 + 77, 64
    c, dev = case(61, B, H, T, d, torch.bfloat16, sigma=1 / np.sqrt(64))
    lam = np.array([1.0, 0.999, 0.9, 0.5], np.float32)
    dec = torch.from_numpy(lam).cuda()
    r = np.random.default_rng(62)
    init = (r.standard_normal((B, H, d, d)) * 0.1).astype(np.float32)
    D = (r.standard_normal((B, H, d, d)) * 0.1).astype(np.float32)
    init_d, D_d = torch.from_numpy(init).cuda(), torch.from_numpy(D).cuda()
    ck = la.checkpoint(dev["q"], dec)
    wsf, wsb = la.workspace(dev["q"], la.OP_FWD, dec), la.workspace(dev["q"], la.OP_BWD, dec)
    la.linattn_timing_enable(True)
    la.linattn_timing_collect()
    o, fin, _ = la.fwd(dev["q"], dev["k"], dev["v"], decay=dec, init_state=init_d, want_final=True, ws=wsf, ckpt=ck)
    dq, dk_, dv, dinit = la.bwd(dev["q"], dev["k"], dev["v"], dev["dO"], decay=dec, init_state=init_d, d_final=D_d,
                                want_dinit=True, ws=wsb, ckpt=ck)
    torch.cuda.synchronize()
    kinds = la.linattn_timing_collect()
    la.linattn_timing_enable(False)
    assert la.device_status(wsf) == la.OK and la.device_status(wsb) == la.OK
    assert "tc_chunked_fwd" in kinds and "tc_dual_rev" in kinds and "pad_d64" in kinds, kinds
    assert "simt_fwd" not in kinds and "simt_bwd" not in kinds, kinds
    init64, D64 = init.astype(np.float64), D.astype(np.float64)
    ro, _, rfin = oracle.fwd_recurrent(c["q"], c["k"], c["v"], lam=lam, init=init64)
    rq, rk, rv, rinit = oracle.bwd_recurrent(c["q"], c["k"], c["v"], c["dO"], lam=lam, init=init64, d_final=D64)
    for name, got, ref in (("o", o, ro), ("final", fin, rfin), ("dq", dq, rq), ("dk", dk_, rk), ("dv", dv, rv),
                           ("d_init", dinit, rinit)):
        assert rel(got, ref) < 1e-2, name
