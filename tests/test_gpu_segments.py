"""A sequence split into segments (sequence-parallel ranks) on the GPU, through
the C ABI: the gradient arriving at a segment's final state (d_final_state of
linattn_bwd / linattn_bwd_ckpt), the segment gradient states
(linattn_chunk_states_rev), and whole split forward/backward passes through
chunked_state_scan_causal_gb300.sp with ranks as threads of this process,
against the fp64 oracle.  Tolerances as in test_gpu_parity."""
import threading

import numpy as np
import pytest
import torch

import oracle
import chunked_state_scan_causal_gb300 as la
from chunked_state_scan_causal_gb300 import inputs, sp

pytestmark = pytest.mark.gpu
TOL = {torch.bfloat16: 1e-2, torch.float32: 1e-4}


def rel(got, ref):
    got = got.detach().double().cpu().numpy() if torch.is_tensor(got) else got
    return float(np.max(np.abs(got - ref))) / max(float(np.max(np.abs(ref))), 1e-30)


@pytest.fixture(scope="module", autouse=True)
def built():
    from chunked_state_scan_causal_gb300 import build
    build.build()


def case(seed, B, H, T, d, dtype, sigma=0.125):
    c = inputs.random_case(seed, B, H, T, d, dtype="bf16" if dtype == torch.bfloat16 else "f32", sigma=sigma)
    return c, {k: torch.from_numpy(np.ascontiguousarray(v)).to(dtype).cuda() for k, v in c.items()}


def lam_of(H, kind):
    return None if kind is None else inputs.decay_per_head(H)


def f32(a):
    return torch.from_numpy(a.astype(np.float32)).cuda()


@pytest.mark.parametrize("dtype,d,T", [(torch.bfloat16, 128, 2048 + 64), (torch.bfloat16, 128, 200),
                                       (torch.float32, 64, 1000), (torch.bfloat16, 64, 300)])
@pytest.mark.parametrize("kind", [None, "cfg"])
@pytest.mark.parametrize("use_ckpt", [False, True])
def test_backward_with_final_state_gradient(dtype, d, T, kind, use_ckpt):
    B, H = 1, 3
    c, dev = case(41 + T, B, H, T, d, dtype)
    lam = lam_of(H, kind)
    dec = None if lam is None else torch.from_numpy(lam).cuda()
    r = np.random.default_rng(T)
    init = (0.1 * r.standard_normal((B, H, d, d))).astype(np.float32).astype(np.float64)
    D = (0.1 * r.standard_normal((B, H, d, d))).astype(np.float32).astype(np.float64)
    ck = None
    if use_ckpt:
        ck = la.checkpoint(dev["q"], dec)
        la.fwd(dev["q"], dev["k"], dev["v"], decay=dec, init_state=f32(init), ckpt=ck)
    ws = la.workspace(dev["q"], la.OP_BWD, dec)
    dq, dk, dv, dinit = la.bwd(dev["q"], dev["k"], dev["v"], dev["dO"], decay=dec, init_state=f32(init),
                               want_dinit=True, ws=ws, ckpt=ck, d_final=f32(D))
    assert la.device_status(ws) == la.OK
    ref = oracle.bwd_recurrent(c["q"], c["k"], c["v"], c["dO"], lam=lam, init=init, d_final=D)
    for got, r_ in zip((dq, dk, dv, dinit), ref):
        assert rel(got, r_) < TOL[dtype]


def test_empty_sequence_passes_final_gradient_to_init():
    z = torch.empty((1, 2, 0, 128), dtype=torch.bfloat16, device="cuda")
    D = torch.randn(1, 2, 128, 128, device="cuda")
    _, _, _, dinit = la.bwd(z, z, z, z, want_dinit=True, d_final=D)
    torch.cuda.synchronize()
    assert torch.equal(dinit, D)


@pytest.mark.parametrize("dtype,d,T,seg", [(torch.bfloat16, 128, 1024, 256), (torch.bfloat16, 128, 768, 384),
                                           (torch.float32, 64, 512, 128), (torch.bfloat16, 128, 600, 200)])
@pytest.mark.parametrize("kind", [None, "cfg"])
def test_segment_gradient_states(dtype, d, T, seg, kind):
    B, H = 2, 3
    c, dev = case(5 + seg, B, H, T, d, dtype)
    lam = lam_of(H, kind)
    got = la.chunk_states_rev(dev["q"], dev["dO"], seg, decay=None if lam is None else torch.from_numpy(lam).cuda())
    torch.cuda.synchronize()
    assert rel(got, oracle.segment_grad_states(c["q"], c["dO"], seg, lam=lam)) < TOL[dtype]


def _split_run(dev, N, dec, init, D):
    """Forward and backward of each of N equal segments on its own thread (rank)."""
    L = dev["q"].shape[2] // N
    group = sp.ThreadExchange.Group(N, timeout=60)
    res, errs = [None] * N, []

    def rank(r):
        ex = group.rank(r)
        try:
            seg = {k: v[:, :, r * L:(r + 1) * L] for k, v in dev.items()}
            o, total, ctx = sp.forward(seg["q"], seg["k"], seg["v"], ex, decay=dec, init_state=init)
            g = sp.backward(seg["q"], seg["k"], seg["v"], seg["dO"], ctx, ex, decay=dec, d_final=D)
            res[r] = (o, total) + g
        except Exception as e:  # a failing rank releases its peers
            errs.append(e)
            ex.abort()

    th = [threading.Thread(target=rank, args=(r,)) for r in range(N)]
    for t in th:
        t.start()
    for t in th:
        t.join(timeout=300)
    torch.cuda.synchronize()
    assert not errs, errs
    return res


@pytest.mark.parametrize("dtype,d,N,L,kind", [(torch.bfloat16, 128, 4, 2048, "cfg"), (torch.bfloat16, 128, 3, 1024, None),
                                              (torch.float32, 64, 3, 500, "cfg")])
def test_split_sequence_through_the_exchange(dtype, d, N, L, kind):
    """N ranks (threads) with consecutive segments: outputs, gradients, the final
    state and the initial-state gradient equal the whole sequence's."""
    B, H = 1, 2
    c, dev = case(77 + L, B, H, N * L, d, dtype, sigma=1 / np.sqrt(128))
    lam = lam_of(H, kind)
    dec = None if lam is None else torch.from_numpy(lam).cuda()
    r = np.random.default_rng(N)
    init = (0.1 * r.standard_normal((B, H, d, d))).astype(np.float32).astype(np.float64)
    D = (0.1 * r.standard_normal((B, H, d, d))).astype(np.float32).astype(np.float64)
    res = _split_run(dev, N, dec, f32(init), f32(D))
    ro, _, rfin = oracle.fwd_recurrent(c["q"], c["k"], c["v"], lam=lam, init=init)
    rq, rk, rv, rinit = oracle.bwd_recurrent(c["q"], c["k"], c["v"], c["dO"], lam=lam, init=init, d_final=D)
    cat = lambda i: torch.cat([x[i] for x in res], dim=2)
    tol = TOL[dtype]
    assert rel(cat(0), ro) < tol
    assert rel(cat(2), rq) < tol
    assert rel(cat(3), rk) < tol
    assert rel(cat(4), rv) < tol
    for x in res:
        assert rel(x[1], rfin) < tol     # every rank holds the whole sequence's final state
        assert rel(x[5], rinit) < tol    # and the gradient of its initial state
