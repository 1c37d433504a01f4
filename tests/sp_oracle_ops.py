"""The per-rank steps of the sequence-parallel path on the fp64 oracle, for
testing the exchange logic of ``chunked_state_scan_causal_gb300.sp`` on CPU
ranks (test infrastructure: the product path uses the CUDA kernels)."""
import numpy as np
import torch

import oracle


def _np(x):
    return None if x is None else x.detach().double().cpu().numpy()


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a))


class OracleOps:
    def chunk_states(self, k, v, seg_len, decay):
        return _t(oracle.segment_states(_np(k), _np(v), seg_len, lam=_np(decay)))

    def chunk_states_rev(self, q, dO, seg_len, decay):
        return _t(oracle.segment_grad_states(_np(q), _np(dO), seg_len, lam=_np(decay)))

    def state_scan(self, local, seg_decay, init):
        a = None if seg_decay is None else _np(seg_decay).reshape(local.shape[1:-2])
        S, total = oracle.state_scan(_np(local), seg_decay=a, init=_np(init))
        return _t(S), _t(total)

    def checkpoint(self, q, decay):
        return None

    def fwd(self, q, k, v, decay, init_state, ckpt):
        o, _, _ = oracle.fwd_recurrent(_np(q), _np(k), _np(v), lam=_np(decay), init=_np(init_state))
        return _t(o)

    def bwd(self, q, k, v, dO, decay, init_state, ckpt, d_final):
        dq, dk, dv, _ = oracle.bwd_recurrent(_np(q), _np(k), _np(v), _np(dO), lam=_np(decay),
                                             init=_np(init_state), d_final=_np(d_final))
        return _t(dq), _t(dk), _t(dv)

    def seg_decay(self, decay, B, seg_len):
        return None if decay is None else (decay.double() ** seg_len).repeat(B)

    def softmax_fwd(self, q, k, v, scale):
        o, lse = oracle.softmax_segment_fwd(_np(q), _np(k), _np(v), scale=None if scale == 0.0 else scale)
        return _t(o), _t(lse)

    def softmax_bwd(self, q, k, v, o, dO, lse, scale):
        dq, dk, dv = oracle.softmax_segment_bwd(_np(q), _np(k), _np(v), _np(dO), scale=None if scale == 0.0 else scale)
        return _t(dq), _t(dk), _t(dv)
