"""fp64 reference for causal softmax attention over a gathered key/value prefix.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The hybrid variant on the LASP-2 page ("LASP-2: Rethinking Sequence
Parallelism for Linear Attention and Its Hybrid", abstract: LASP-2H carries
the one-gather exchange over to the softmax attention layers of hybrid
models) gives each
sequence-parallel rank the keys and values of every earlier position by one
gather, and the rank's queries attend causally over that prefix.  The
standard attention module is taken in its plainest form: scaled dot-product
softmax attention with scale 1/sqrt(d) and a causal mask.  For queries that
are the last Tq positions of a prefix of Tk tokens (offset = Tk - Tq):

    o_i   = sum_{j <= offset + i} softmax_j(scale * q_i . k_j) v_j
    lse_i = log sum_{j <= offset + i} exp(scale * q_i . k_j)

written row by row with numpy as the library primitive (max subtraction only
keeps exp in range; it cancels exactly in the ratio).

The backward (``softmax_segment_bwd``: the gradients of q, k, v for an output
gradient dO, which a hybrid model's training step needs of its softmax layers)
is the chain rule through the same rows: with p_ij the row's softmax weights,

    dv_j  = sum_i p_ij dO_i
    dp_ij = dO_i . v_j,   delta_i = sum_j p_ij dp_ij,   ds_ij = p_ij (dp_ij - delta_i)
    dq_i  = scale sum_j ds_ij k_j,      dk_j = scale sum_i ds_ij q_i

(the softmax Jacobian diag(p) - p p^T applied to dp), summed over the visible
pairs j <= offset + i only.
"""
from __future__ import annotations

import math

import numpy as np


def softmax_segment_fwd(q, k, v, scale=None, rows=None):
    """(o [B,H,Tq,dv], lse [B,H,Tq]) in float64; q [B,H,Tq,d], k [B,H,Tk,d], v [B,H,Tk,dv], Tk >= Tq.

    ``rows`` (optional list of query indices) limits the work to those rows;
    the other rows of the outputs are NaN."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, H, Tq, d = q.shape
    Tk = k.shape[2]
    assert k.shape[:2] == (B, H) and v.shape[:3] == (B, H, Tk) and Tk >= Tq
    off = Tk - Tq
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = np.full((B, H, Tq, v.shape[3]), np.nan)
    lse = np.full((B, H, Tq), np.nan)
    for i in (range(Tq) if rows is None else rows):
        n = off + i + 1                                         # keys 0 .. off + i
        s = sc * np.einsum("bhjd,bhd->bhj", k[:, :, :n], q[:, :, i])
        m = s.max(axis=2, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=2)
        o[:, :, i] = np.einsum("bhj,bhje->bhe", p, v[:, :, :n]) / l[..., None]
        lse[:, :, i] = m[..., 0] + np.log(l)
    return o, lse


def softmax_segment_bwd(q, k, v, dO, scale=None, rows=None, first_key=None):
    """(dq [B,H,Tq,d], dk [B,H,Tk,d], dv [B,H,Tk,dv]) in float64: the gradients of
    <o, dO> for o = softmax_segment_fwd(q, k, v, scale)[0]; Tk >= Tq.

    Sampling for long inputs: ``rows`` (a list of query indices) computes dq for those
    rows only; ``first_key`` computes dk, dv for the keys first_key .. Tk-1 only (only the
    queries that see one of them are visited, each over its whole key prefix).  The other
    entries are NaN; with either argument, only the requested outputs are formed."""
    q, k, v, dO = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dO))
    B, H, Tq, d = q.shape
    Tk = k.shape[2]
    assert k.shape[:2] == (B, H) and v.shape[:3] == (B, H, Tk) and Tk >= Tq and dO.shape == (B, H, Tq, v.shape[3])
    off = Tk - Tq
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    sampled = rows is not None or first_key is not None
    dq = np.full_like(q, np.nan) if sampled else np.zeros_like(q)
    dk = np.full_like(k, np.nan) if sampled else np.zeros_like(k)
    dv = np.full_like(v, np.nan) if sampled else np.zeros_like(v)
    if first_key is not None:
        dk[:, :, first_key:] = 0.0
        dv[:, :, first_key:] = 0.0
    if sampled:
        # query i sees key first_key once off + i >= first_key
        visit = set(rows or []) | (set(range(max(0, first_key - off), Tq)) if first_key is not None else set())
        row_list = sorted(visit)
    else:
        row_list = range(Tq)
    for i in row_list:
        n = off + i + 1                                         # keys 0 .. off + i
        s = sc * np.einsum("bhjd,bhd->bhj", k[:, :, :n], q[:, :, i])
        p = np.exp(s - s.max(axis=2, keepdims=True))
        p /= p.sum(axis=2, keepdims=True)                       # the row's softmax weights
        dp = np.einsum("bhje,bhe->bhj", v[:, :, :n], dO[:, :, i])
        delta = np.sum(p * dp, axis=2, keepdims=True)
        ds = p * (dp - delta)
        if not sampled or (rows is not None and i in rows):
            dq[:, :, i] = sc * np.einsum("bhj,bhjd->bhd", ds, k[:, :, :n])
        lo = 0 if not sampled else (first_key if first_key is not None else n)
        if lo < n:
            dv[:, :, lo:n] += p[:, :, lo:, None] * dO[:, :, i, None, :]
            dk[:, :, lo:n] += sc * ds[:, :, lo:, None] * q[:, :, i, None, :]
    return dq, dk, dv
