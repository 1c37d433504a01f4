"""Gradients of the softmax-attention segment (linattn_softmax_segment_bwd) through
the C ABI, against the fp64 oracle: dq, dk, dv of causal scaled dot-product
attention of the last Tq positions over a prefix of Tk keys and values.  The
GPU backward takes the GPU forward's o and lse, as a training step does; the
oracle differentiates the exact attention of the same bf16 inputs.

Tolerance: max|gpu - ref| / max|ref| <= 1e-2 per tensor.  The products take p
and ds rounded to bf16 (relative error 2^-9 each, fp32 accumulation), delta
comes from the bf16 o (relative 2^-9), and the outputs are rounded to bf16
(2^-9): errors of a few 2^-9 of the largest entries, well inside 1e-2.  Cases
span several 128-query and 128-key tiles, ragged tails on both sides, a prefix
longer than the segment (the diagonal inside a key tile), large scores, padded
strides with a custom scale, one query, and Tq = 0."""
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


def case(seed, B, H, Tq, Tk, sigma=1.0):
    g = torch.Generator().manual_seed(seed)
    q, k, v = (torch.randn(B, H, T, 128, generator=g) * s for T, s in ((Tq, sigma), (Tk, sigma), (Tk, 1.0)))
    dO = torch.randn(B, H, Tq, 128, generator=g)
    return tuple(x.to(torch.bfloat16) for x in (q, k, v, dO))


def run(q, k, v, dO, scale=0.0, cuda=None):
    qd, kd, vd, dOd = cuda if cuda is not None else (x.cuda() for x in (q, k, v, dO))
    o, lse = la.softmax_segment_fwd(qd, kd, vd, scale=scale, want_lse=True)
    ws = la.workspace(qd, la.OP_SOFTMAX_SEGMENT_BWD)
    dq, dk, dv = la.softmax_segment_bwd(qd, kd, vd, o, dOd, lse, scale=scale, ws=ws)
    torch.cuda.synchronize()
    assert la.device_status(ws) == la.OK
    return dq, dk, dv


def check(q, k, v, dO, scale=0.0, tol=1e-2, cuda=None):
    dq, dk, dv = run(q, k, v, dO, scale, cuda)
    n = lambda x: x.double().numpy()
    rq, rk, rv = oracle.softmax_segment_bwd(n(q), n(k), n(v), n(dO), scale=None if scale == 0.0 else scale)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        if np.max(np.abs(ref)) == 0.0:
            # one query over one key: ds = p (dO.v - dO.o) vanishes exactly; the kernel keeps
            # the rounding difference of its two fp32 dot products (dp from the product, delta
            # from the bf16 o)
            assert float(torch.max(torch.abs(got.float()))) < 1e-5, name
            continue
        assert rel(got, ref) < tol, (name, rel(got, ref))


@pytest.mark.parametrize("B,H,Tq,Tk", [(1, 2, 128, 128), (1, 2, 200, 200), (2, 3, 300, 1000), (1, 2, 640, 640),
                                       (1, 4, 64, 2048 + 17), (1, 1, 1, 1), (1, 1, 1, 777), (2, 2, 513, 1100)])
def test_softmax_segment_bwd_matches_oracle(B, H, Tq, Tk):
    check(*case(Tq * 7 + Tk + 1, B, H, Tq, Tk))


def test_softmax_segment_bwd_several_items_per_cta():
    """More items than SMs in both launches (2 x 40 sequences of 2 query and 4 key tiles),
    so CTAs go from one item's last step to the next item's first."""
    check(*case(21, 2, 40, 256, 512))


def test_softmax_segment_bwd_large_scores():
    """Scores of a few tens: sharp rows, p close to one on a few keys."""
    check(*case(3, 1, 2, 256, 700, sigma=2.5))


def test_softmax_segment_bwd_padded_strides_and_custom_scale():
    B, H, Tq, Tk = 1, 3, 250, 400
    q, k, v, dO = case(9, B, H, Tq, Tk)

    def padded(x, width=136):
        buf = torch.zeros(*x.shape[:3], width, dtype=x.dtype)
        buf[..., :128] = x
        return buf.cuda()[..., :128]

    cu = tuple(padded(x) for x in (q, k, v, dO))
    check(q, k, v, dO, scale=0.05, cuda=cu)


def test_softmax_segment_bwd_runs_the_tensor_core_kernels():
    q, k, v, dO = case(4, 1, 2, 256, 512)
    la.linattn_timing_enable(True)
    la.linattn_timing_collect()
    run(q, k, v, dO)
    kinds = la.linattn_timing_collect()
    la.linattn_timing_enable(False)
    assert {"softmax_bwd_prep", "softmax_bwd_dkdv", "softmax_bwd_dq"} <= set(kinds), kinds


def test_softmax_segment_bwd_empty_queries():
    """No queries: every key gradient is zero."""
    B, H, Tk = 1, 2, 300
    q = torch.zeros(B, H, 0, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.randn(B, H, Tk, 128, device="cuda").to(torch.bfloat16)
    lse = torch.zeros(B, H, 0, device="cuda")
    dk = torch.full_like(k, 7.0)
    dv = torch.full_like(k, 7.0)
    la.softmax_segment_bwd(q, k, k, q, q, lse, outs=(q.clone(), dk, dv))
    torch.cuda.synchronize()
    assert torch.count_nonzero(dk) == 0 and torch.count_nonzero(dv) == 0


def test_softmax_segment_bwd_full_size_sampled():
    """The benchmark's shape (B1 H16, Tq 16384 over Tk 65536), in the launch configuration
    the bench times: dq of rows spread over the segment and dk, dv of the prefix's last 64
    keys (seen by the last 64 queries only), on the first and last head, against the
    oracle; every other output finite and the status clean."""
    B, H, Tq, Tk = 1, 16, 16384, 65536
    q, k, v, dO = case(77, B, H, Tq, Tk)
    dq, dk, dv = run(q, k, v, dO)
    assert all(bool(torch.isfinite(x).all()) for x in (dq, dk, dv))
    rows = [0, 1, 127, 128, 5000, 8191, 16383]
    heads = [0, H - 1]
    n = lambda x: x[:, heads].double().numpy()
    rq, rk, rv = oracle.softmax_segment_bwd(n(q), n(k), n(v), n(dO), rows=rows, first_key=Tk - 64)
    got_q, got_k, got_v = (x[:, heads].double().cpu().numpy() for x in (dq, dk, dv))
    for name, got, ref in (("dq", got_q[:, :, rows], rq[:, :, rows]), ("dk", got_k[:, :, -64:], rk[:, :, -64:]),
                           ("dv", got_v[:, :, -64:], rv[:, :, -64:])):
        assert rel(got, ref) < 1e-2, (name, rel(got, ref))


def test_softmax_layer_split_across_thread_ranks():
    """The hybrid's softmax layers split across 4 ranks (threads of this process, one
    gather of k, v; the key and value gradients summed back to their owners), on the
    kernels: the concatenated outputs and gradients equal whole-sequence causal softmax
    attention (oracle)."""
    import threading
    from chunked_state_scan_causal_gb300 import sp
    N, L, B, H = 4, 256, 1, 2
    q, k, v, dO = case(31, B, H, N * L, N * L)
    dev = [x.cuda() for x in (q, k, v, dO)]
    group = sp.ThreadExchange.Group(N, timeout=60)
    res, errs = [None] * N, []

    def rank(r):
        ex = group.rank(r)
        try:
            seg = [x[:, :, r * L:(r + 1) * L] for x in dev]
            o, ctx = sp.softmax_forward(seg[0], seg[1], seg[2], ex)
            res[r] = (o,) + sp.softmax_backward(seg[0], seg[3], ctx, ex)
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
    n = lambda x: x.double().numpy()
    ro, _ = oracle.softmax_segment_fwd(n(q), n(k), n(v))
    rq, rk, rv = oracle.softmax_segment_bwd(n(q), n(k), n(v), n(dO))
    for i, (name, ref) in enumerate((("o", ro), ("dq", rq), ("dk", rk), ("dv", rv))):
        got = torch.cat([x[i] for x in res], dim=2)
        assert rel(got, ref) < 1e-2, (name, rel(got, ref))
