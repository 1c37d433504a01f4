"""The softmax-attention segment of the hybrid variant through the C ABI,
against the fp64 oracle (causal scaled dot-product attention of the last Tq
positions over a prefix of Tk keys and values).

Tolerance: max|gpu - ref| / max|ref| <= 1e-2 for the bf16 outputs; the
log-sum-exp (fp32, from fp32 scores and sums) within 1e-3 absolute.  Cases
span several 128-query and 128-key tiles, ragged tails, prefixes longer than
the segment (the diagonal falling inside a key tile), padded strides, large
scores (the reference maximum moving often), one query, and Tq = 0."""
import math

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
    q, k, v = (x.to(torch.bfloat16) for x in (q, k, v))
    return q, k, v


def check(q, k, v, scale=0.0, rows=None, tol=1e-2):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ws = la.workspace(qd, la.OP_SOFTMAX_SEGMENT)
    o, lse = la.softmax_segment_fwd(qd, kd, vd, scale=scale, want_lse=True, ws=ws)
    assert la.device_status(ws) == la.OK
    ro, rl = oracle.softmax_segment_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                        scale=None if scale == 0.0 else scale, rows=rows)
    if rows is not None:
        o, lse, ro, rl = o[:, :, rows], lse[:, :, rows], ro[:, :, rows], rl[:, :, rows]
    assert rel(o, ro) < tol
    assert float(np.max(np.abs(lse.double().cpu().numpy() - rl))) < 1e-3
    return o


@pytest.mark.parametrize("B,H,Tq,Tk", [(1, 2, 128, 128), (1, 2, 200, 200), (2, 3, 300, 1000), (1, 2, 1000, 1000),
                                       (1, 4, 64, 4096 + 17), (1, 1, 1, 1), (1, 1, 1, 777), (2, 2, 513, 1100)])
def test_softmax_segment_matches_oracle(B, H, Tq, Tk):
    q, k, v = case(Tq * 7 + Tk, B, H, Tq, Tk)
    check(q, k, v)


def test_softmax_segment_large_scores_move_the_reference_maximum():
    # scores of size ~ sqrt(128) * 9: the running maximum rises by far more than 8 within rows
    q, k, v = case(5, 1, 2, 384, 1024, sigma=3.0)
    check(q, k, v, scale=1.0)


def test_softmax_segment_long_prefix_sampled_rows():
    q, k, v = case(6, 1, 4, 2048, 16384 + 100)
    check(q, k, v, rows=[0, 1, 127, 128, 1000, 2047])


def test_softmax_segment_padded_strides_and_custom_scale():
    B, H, Tq, Tk = 1, 2, 300, 700
    q, k, v = case(7, B, H, Tq, Tk)

    def padded(x, width=136):
        buf = torch.zeros(*x.shape[:3], width, dtype=x.dtype)
        buf[..., :128] = x
        return buf.cuda()[..., :128]

    qd, kd, vd = padded(q), padded(k), padded(v)
    out = padded(torch.zeros_like(q))
    ws = la.workspace(qd, la.OP_SOFTMAX_SEGMENT)
    o, _ = la.softmax_segment_fwd(qd, kd, vd, scale=0.05, out=out, ws=ws)
    assert la.device_status(ws) == la.OK
    ro, _ = oracle.softmax_segment_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale=0.05)
    assert rel(o, ro) < 1e-2


def test_softmax_segment_empty_queries():
    q = torch.zeros(1, 2, 0, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.randn(1, 2, 50, 128, device="cuda").to(torch.bfloat16)
    o, lse = la.softmax_segment_fwd(q, k, k, want_lse=True)
    torch.cuda.synchronize()
    assert o.numel() == 0 and lse.numel() == 0


def test_softmax_segment_tile_sums_above_256_with_and_without_a_new_maximum():
    """Scores built along one direction: the first key tile scores near 0, the next
    tiles 3 log2-units higher (each tile's probabilities sum to ~2^10 > 2^8 while its
    maximum stays within 8 of the reference), then tiles 11 units higher (the
    reference maximum moves)."""
    g = torch.Generator().manual_seed(11)
    Tq, Tk = 256, 1024
    c = 3.0 * math.sqrt(128) / math.log2(math.e)          # score 3 (log2 units) at scale 1/sqrt(128)
    q = torch.randn(1, 1, Tq, 128, generator=g) * 0.01
    q[..., 0] = 1.0
    k = torch.randn(1, 1, Tk, 128, generator=g) * 0.01
    k[..., 128:640, 0] = c
    k[..., 640:, 0] = c * 11.0 / 3.0
    v = torch.randn(1, 1, Tk, 128, generator=g)
    check(*(x.to(torch.bfloat16) for x in (q, k, v)))
