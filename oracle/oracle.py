"""ctypes front end of the fp64 C oracle, plus the quadratic (brute force) form.

TEST INFRASTRUCTURE ONLY -- see the package docstring.

The C file ``linattn_oracle.c`` holds the recurrent form (the definition
``S_t = lambda S_{t-1} + k_t v_t^T, o_t = S_t^T q_t``), its backward, the
chunked form (masked attention inside a chunk, query-times-state across
chunks: "Lightning Attention-2" entry on the LASP-2 page), the segment-local
states and their exclusive scan (the state each rank needs to start: ZeCO page,
abstract, All-Scan).  The quadratic form below is the masked product
``O = (Q K^T * M) V`` with ``M[t, s] = lambda^{t-s} [s <= t]``, written with
numpy matmuls as the library primitive.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "linattn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2, OpenMP, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.oracle_fwd_recurrent.argtypes = [i64, i64, i64, i64, dp, dp, dp, dp, dp, i64, dp, dp, dp]
            lib.oracle_bwd_recurrent.argtypes = [i64, i64, i64, i64, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp]
            lib.oracle_fwd_chunked.argtypes = [i64, i64, i64, i64, dp, i64, dp, dp, dp, dp, dp, dp, dp]
            lib.oracle_bwd_chunked.argtypes = [i64, i64, i64, i64, dp, i64, dp, dp, dp, dp, dp, dp, dp, dp, dp]
            lib.oracle_segment_states.argtypes = [i64, i64, i64, i64, dp, i64, dp, dp, dp]
            lib.oracle_segment_grad_states.argtypes = [i64, i64, i64, i64, dp, i64, dp, dp, dp]
            lib.oracle_fwd_gated.argtypes = [i64, i64, i64, i64, dp, dp, dp, dp, dp, dp, dp]
            lib.oracle_bwd_gated.argtypes = [i64, i64, i64, i64, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp]
            lib.oracle_fwd_gated_vec.argtypes = [i64, i64, i64, i64, dp, dp, dp, dp, dp, dp, dp]
            lib.oracle_bwd_gated_vec.argtypes = [i64, i64, i64, i64, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp]
            lib.oracle_state_scan.argtypes = [i64, i64, i64, i64, dp, dp, dp, dp, dp]
            for f in ("oracle_fwd_recurrent", "oracle_bwd_recurrent", "oracle_fwd_chunked",
                      "oracle_bwd_chunked", "oracle_segment_states", "oracle_segment_grad_states",
                      "oracle_state_scan", "oracle_fwd_gated", "oracle_bwd_gated", "oracle_fwd_gated_vec",
                      "oracle_bwd_gated_vec"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def threads_used() -> int:
    """OpenMP threads the oracle runs with (OMP_NUM_THREADS, else the CPUs we may use)."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env:
        return int(env)
    return len(os.sched_getaffinity(0))


# ----------------------------------------------------------------------------- helpers
def _f64(x):
    return None if x is None else np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _lam_bh(lam, B, H):
    """Per-(b, h) decay as a flat float64 [B*H] array, or None."""
    if lam is None:
        return None
    lam = np.asarray(lam, dtype=np.float64)
    if lam.ndim == 1:
        lam = np.broadcast_to(lam[None, :], (B, H))
    return np.ascontiguousarray(lam.reshape(B * H))


def _dims(q, k, v):
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == (B, H, T, dk) and v.shape == (B, H, T, dv)
    return B, H, T, dk, dv


# ----------------------------------------------------------------------------- recurrent
def fwd_recurrent(q, k, v, lam=None, init=None, chunk=0):
    """Definition form.  Returns (o, chunk_states or None, final_state).

    chunk_states[b, h, c] is the state entering chunk c (c * chunk tokens seen),
    so chunk_states[:, :, 0] == init (or 0).
    """
    q, k, v, init = _f64(q), _f64(k), _f64(v), _f64(init)
    B, H, T, dk, dv = _dims(q, k, v)
    o = np.empty((B, H, T, dv))
    nch = (T + chunk - 1) // chunk if chunk > 0 else 0
    cs = np.empty((B, H, nch, dk, dv)) if chunk > 0 else None
    fin = np.empty((B, H, dk, dv))
    lam_bh = _lam_bh(lam, B, H)
    _load().oracle_fwd_recurrent(B * H, T, dk, dv, _ptr(lam_bh), _ptr(q), _ptr(k), _ptr(v),
                                 _ptr(init), chunk, _ptr(o), _ptr(cs), _ptr(fin))
    return o, cs, fin


def bwd_recurrent(q, k, v, dO, lam=None, init=None, d_final=None):
    """Returns (dq, dk, dv, d_init).

    ``d_final`` [B, H, dk, dv] is the gradient arriving at the state after the
    last token (from whatever continues the sequence), or None for zero.
    """
    q, k, v, dO, init, d_final = _f64(q), _f64(k), _f64(v), _f64(dO), _f64(init), _f64(d_final)
    B, H, T, dk, dv = _dims(q, k, v)
    dq, dkk, dvv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    dinit = np.empty((B, H, dk, dv))
    lam_bh = _lam_bh(lam, B, H)
    _load().oracle_bwd_recurrent(B * H, T, dk, dv, _ptr(lam_bh), _ptr(q), _ptr(k), _ptr(v), _ptr(dO),
                                 _ptr(init), _ptr(d_final), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dinit))
    return dq, dkk, dvv, dinit


# ----------------------------------------------------------------------------- chunked
def fwd_chunked(q, k, v, chunk, lam=None, init=None):
    """Chunked form with any chunk length.  Returns (o, chunk_states, final_state)."""
    q, k, v, init = _f64(q), _f64(k), _f64(v), _f64(init)
    B, H, T, dk, dv = _dims(q, k, v)
    o = np.empty((B, H, T, dv))
    nch = (T + chunk - 1) // chunk
    cs = np.empty((B, H, nch, dk, dv))
    fin = np.empty((B, H, dk, dv))
    lam_bh = _lam_bh(lam, B, H)
    _load().oracle_fwd_chunked(B * H, T, dk, dv, _ptr(lam_bh), chunk, _ptr(q), _ptr(k), _ptr(v),
                               _ptr(init), _ptr(o), _ptr(cs), _ptr(fin))
    return o, cs, fin


def bwd_chunked(q, k, v, dO, chunk, lam=None, init=None):
    """Chunked backward with any chunk length.  Returns (dq, dk, dv, d_init)."""
    q, k, v, dO, init = _f64(q), _f64(k), _f64(v), _f64(dO), _f64(init)
    B, H, T, dk, dv = _dims(q, k, v)
    dq, dkk, dvv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    dinit = np.empty((B, H, dk, dv))
    lam_bh = _lam_bh(lam, B, H)
    _load().oracle_bwd_chunked(B * H, T, dk, dv, _ptr(lam_bh), chunk, _ptr(q), _ptr(k), _ptr(v),
                               _ptr(dO), _ptr(init), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dinit))
    return dq, dkk, dvv, dinit


# ----------------------------------------------------------------------------- segments
def segment_states(k, v, seg_len, lam=None):
    """U[g, b, h] = sum over segment g of lambda^{end_g - s} k_s v_s^T; shape [G, B, H, dk, dv]."""
    k, v = _f64(k), _f64(v)
    B, H, T, dk = k.shape
    dv = v.shape[-1]
    G = (T + seg_len - 1) // seg_len
    out = np.empty((G, B, H, dk, dv))
    lam_bh = _lam_bh(lam, B, H)
    _load().oracle_segment_states(B * H, T, dk, dv, _ptr(lam_bh), seg_len, _ptr(k), _ptr(v), _ptr(out))
    return out


def segment_grad_states(q, dO, seg_len, lam=None):
    """W[g, b, h] = sum over segment g of lambda^{s - start_g + 1} q_s dO_s^T; shape [G, B, H, dk, dv]."""
    q, dO = _f64(q), _f64(dO)
    B, H, T, dk = q.shape
    dv = dO.shape[-1]
    G = (T + seg_len - 1) // seg_len
    out = np.empty((G, B, H, dk, dv))
    lam_bh = _lam_bh(lam, B, H)
    _load().oracle_segment_grad_states(B * H, T, dk, dv, _ptr(lam_bh), seg_len, _ptr(q), _ptr(dO), _ptr(out))
    return out


def state_scan(local, seg_decay=None, init=None):
    """Exclusive scan over the leading (segment) axis of ``local`` [G, BH..., dk, dv].

    S_0 = init (or 0), S_g = a S_{g-1} + U_{g-1}; returns (S [same shape], total).
    ``seg_decay`` has the shape of the middle (BH...) axes, or is None (a = 1).
    """
    local = _f64(local)
    G = local.shape[0]
    mid = local.shape[1:-2]
    dk, dv = local.shape[-2:]
    BH = int(np.prod(mid)) if mid else 1
    a = None if seg_decay is None else np.ascontiguousarray(
        np.broadcast_to(np.asarray(seg_decay, dtype=np.float64), mid).reshape(BH))
    init = _f64(init)
    out = np.empty_like(local)
    total = np.empty(local.shape[1:])
    _load().oracle_state_scan(G, BH, dk, dv, _ptr(a), _ptr(local), _ptr(init), _ptr(out), _ptr(total))
    return out, total


# ----------------------------------------------------------------------------- quadratic
def _decay_mask(T, lam_bh):
    """M[bh, t, s] = lambda^{t-s} for s <= t, else 0."""
    t = np.arange(T)
    diff = t[:, None] - t[None, :]
    causal = diff >= 0
    if lam_bh is None:
        return causal.astype(np.float64)[None]
    m = np.where(causal[None], np.power(lam_bh[:, None, None], np.where(causal, diff, 0)[None]), 0.0)
    return m


def fwd_quadratic(q, k, v, lam=None, init=None):
    """Brute-force masked form O = (Q K^T * M) V + diag(lambda^{t+1}) Q init (small T only)."""
    q, k, v, init = _f64(q), _f64(k), _f64(v), _f64(init)
    B, H, T, dk, dv = _dims(q, k, v)
    lam_bh = _lam_bh(lam, B, H)
    M = _decay_mask(T, lam_bh).reshape(-1, T, T)
    Q, K, V = (x.reshape(B * H, T, -1) for x in (q, k, v))
    A = (Q @ K.transpose(0, 2, 1)) * M
    O = A @ V
    if init is not None:
        l = np.ones(B * H) if lam_bh is None else lam_bh
        w = np.power(l[:, None], np.arange(1, T + 1)[None, :])  # lambda^{t+1}
        O = O + w[:, :, None] * (Q @ init.reshape(B * H, dk, dv))
    return O.reshape(B, H, T, dv)


def bwd_quadratic(q, k, v, dO, lam=None, init=None):
    """Gradients of the masked form (small T only).  Returns (dq, dk, dv, d_init)."""
    q, k, v, dO, init = _f64(q), _f64(k), _f64(v), _f64(dO), _f64(init)
    B, H, T, dk, dv = _dims(q, k, v)
    lam_bh = _lam_bh(lam, B, H)
    M = _decay_mask(T, lam_bh).reshape(-1, T, T)
    Q, K, V, G = (x.reshape(B * H, T, -1) for x in (q, k, v, dO))
    dA = (G @ V.transpose(0, 2, 1)) * M          # dL/d(scores), masked
    A = (Q @ K.transpose(0, 2, 1)) * M
    dQ = dA @ K
    dK = dA.transpose(0, 2, 1) @ Q
    dV = A.transpose(0, 2, 1) @ G
    l = np.ones(B * H) if lam_bh is None else lam_bh
    w = np.power(l[:, None], np.arange(1, T + 1)[None, :])  # lambda^{t+1}
    if init is not None:
        dQ = dQ + w[:, :, None] * (G @ init.reshape(B * H, dk, dv).transpose(0, 2, 1))
    dinit = (Q * w[:, :, None]).transpose(0, 2, 1) @ G
    return (dQ.reshape(B, H, T, dk), dK.reshape(B, H, T, dk), dV.reshape(B, H, T, dv),
            dinit.reshape(B, H, dk, dv))


# ----------------------------------------------------------------------------- data-dependent gates
def fwd_gated(q, k, v, log_gate, init=None):
    """S_t = exp(log_gate_t) S_{t-1} + k_t v_t^T, o_t = S_t^T q_t.  log_gate [B, H, T].
    Returns (o, final_state)."""
    q, k, v, init, lg = _f64(q), _f64(k), _f64(v), _f64(init), _f64(log_gate)
    B, H, T, dk, dv = _dims(q, k, v)
    assert lg.shape == (B, H, T)
    o = np.empty((B, H, T, dv))
    fin = np.empty((B, H, dk, dv))
    _load().oracle_fwd_gated(B * H, T, dk, dv, _ptr(lg), _ptr(q), _ptr(k), _ptr(v), _ptr(init), _ptr(o), _ptr(fin))
    return o, fin


def bwd_gated(q, k, v, dO, log_gate, init=None, d_final=None):
    """Returns (dq, dk, dv, d_log_gate, d_init) of <dO, o> (+ <d_final, final_state>)."""
    q, k, v, dO, init, d_final, lg = (_f64(x) for x in (q, k, v, dO, init, d_final, log_gate))
    B, H, T, dk, dv = _dims(q, k, v)
    dq, dkk, dvv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    dlg = np.empty((B, H, T))
    dinit = np.empty((B, H, dk, dv))
    _load().oracle_bwd_gated(B * H, T, dk, dv, _ptr(lg), _ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(init),
                             _ptr(d_final), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dlg), _ptr(dinit))
    return dq, dkk, dvv, dlg, dinit


# ----------------------------------------------------------------------------- per-dimension gates
def fwd_gated_vec(q, k, v, log_gate, init=None):
    """S_t = diag(exp(log_gate_t)) S_{t-1} + k_t v_t^T, o_t = S_t^T q_t: one gate per token,
    head and key dimension, log_gate [B, H, T, dk].  Returns (o, final_state)."""
    q, k, v, init, lg = _f64(q), _f64(k), _f64(v), _f64(init), _f64(log_gate)
    B, H, T, dk, dv = _dims(q, k, v)
    assert lg.shape == (B, H, T, dk)
    o = np.empty((B, H, T, dv))
    fin = np.empty((B, H, dk, dv))
    _load().oracle_fwd_gated_vec(B * H, T, dk, dv, _ptr(lg), _ptr(q), _ptr(k), _ptr(v), _ptr(init), _ptr(o),
                                 _ptr(fin))
    return o, fin


def bwd_gated_vec(q, k, v, dO, log_gate, init=None, d_final=None):
    """Returns (dq, dk, dv, d_log_gate [B, H, T, dk], d_init) of <dO, o> (+ <d_final, final_state>)."""
    q, k, v, dO, init, d_final, lg = (_f64(x) for x in (q, k, v, dO, init, d_final, log_gate))
    B, H, T, dk, dv = _dims(q, k, v)
    assert lg.shape == (B, H, T, dk)
    dq, dkk, dvv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    dlg = np.empty((B, H, T, dk))
    dinit = np.empty((B, H, dk, dv))
    _load().oracle_bwd_gated_vec(B * H, T, dk, dv, _ptr(lg), _ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(init),
                                 _ptr(d_final), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dlg), _ptr(dinit))
    return dq, dkk, dvv, dlg, dinit
