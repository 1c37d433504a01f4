"""The sequence-parallel exchange (chunked_state_scan_causal_gb300.sp) across CPU
processes over gloo: ranks holding consecutive segments reproduce the
whole-sequence forward and backward, and a rank that dies before the exchange
makes its peers fail within the timeout instead of hanging; the softmax layers of
the hybrid (one gather of k, v, the gradients summed back to their owners)
reproduce whole-sequence causal softmax attention.  The per-rank arithmetic is
the fp64 oracle here; on GPUs it is the library's kernels."""
import datetime
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

B, H, L, d = 1, 2, 23, 4


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(world, seed):
    r = np.random.default_rng(seed)
    T = world * L
    q, k, v, dO = (r.standard_normal((B, H, T, d)) for _ in range(4))
    init, D = r.standard_normal((B, H, d, d)), r.standard_normal((B, H, d, d))
    lam = np.array([0.9, 0.97])
    return q, k, v, dO, init, D, lam


def _init(rank, world, port):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=20))
    return dist


def _rank_split(rank, world, port, seed, out):
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from chunked_state_scan_causal_gb300 import sp
    from sp_oracle_ops import OracleOps
    import oracle
    dist = _init(rank, world, port)
    try:
        q, k, v, dO, init, D, lam = _inputs(world, seed)
        seg = slice(rank * L, (rank + 1) * L)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
        ex = sp.TorchDistExchange(timeout=20)
        ops = OracleOps()
        o, total, ctx = sp.forward(t(q[:, :, seg]), t(k[:, :, seg]), t(v[:, :, seg]), ex, decay=t(lam),
                                   init_state=t(init), ops=ops)
        dq, dk, dv, dinit = sp.backward(t(q[:, :, seg]), t(k[:, :, seg]), t(v[:, :, seg]), t(dO[:, :, seg]), ctx, ex,
                                        decay=t(lam), d_final=t(D), ops=ops)
        ro, _, rfin = oracle.fwd_recurrent(q, k, v, lam=lam, init=init)
        rq, rk, rv, rinit = oracle.bwd_recurrent(q, k, v, dO, lam=lam, init=init, d_final=D)
        err = max(float(np.abs(a.numpy() - b).max()) for a, b in (
            (o, ro[:, :, seg]), (total, rfin), (dq, rq[:, :, seg]), (dk, rk[:, :, seg]), (dv, rv[:, :, seg]),
            (dinit, rinit)))
        out.put((rank, err))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_reproduce_the_whole_sequence(world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_split, args=(r, world, port, 100 + world, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r for r, _ in res] == list(range(world))
    for r, err in res:
        assert err < 1e-10, (r, err)


def _rank_softmax(rank, world, port, seed, out):
    """LASP-2H: the rank's queries over the gathered keys and values of segments 0..rank."""
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from chunked_state_scan_causal_gb300 import sp
    from sp_oracle_ops import OracleOps
    import oracle
    dist = _init(rank, world, port)
    try:
        q, k, v, dO, _, _, _ = _inputs(world, seed)
        seg = slice(rank * L, (rank + 1) * L)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
        ex = sp.TorchDistExchange(timeout=20)
        ops = OracleOps()
        o, ctx = sp.softmax_forward(t(q[:, :, seg]), t(k[:, :, seg]), t(v[:, :, seg]), ex, scale=0.6, ops=ops)
        dq, dk, dv = sp.softmax_backward(t(q[:, :, seg]), t(dO[:, :, seg]), ctx, ex, ops=ops)
        ro, _ = oracle.softmax_segment_fwd(q, k, v, scale=0.6)
        rq, rk, rv = oracle.softmax_segment_bwd(q, k, v, dO, scale=0.6)
        err = max(float(np.abs(a.numpy() - b).max()) for a, b in (
            (o, ro[:, :, seg]), (dq, rq[:, :, seg]), (dk, rk[:, :, seg]), (dv, rv[:, :, seg])))
        out.put((rank, err))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_softmax_layer_split_reproduces_the_whole_sequence(world):
    """The softmax layers of the hybrid split across ranks (one gather of k, v; the key
    and value gradients summed back to their owners) equal causal softmax attention over
    the whole sequence, forward and backward."""
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_softmax, args=(r, world, port, 200 + world, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r for r, _ in res] == list(range(world))
    for r, err in res:
        assert err < 1e-10, (r, err)


def _rank_dies(rank, world, port, out):
    from chunked_state_scan_causal_gb300 import sp
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from sp_oracle_ops import OracleOps
    dist = _init(rank, world, port)
    if rank == 1:
        os._exit(3)  # dies before the exchange, without a goodbye
    t0 = datetime.datetime.now()
    try:
        q, k, v, dO, init, D, lam = _inputs(world, 7)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
        sp.forward(t(q[:, :, :L]), t(k[:, :, :L]), t(v[:, :, :L]), sp.TorchDistExchange(timeout=10),
                   decay=t(lam), ops=OracleOps())
        out.put(("no error", 0.0))
    except sp.SequenceParallelError:
        out.put(("SequenceParallelError", (datetime.datetime.now() - t0).total_seconds()))
    out.close()
    out.join_thread()  # flush the result before the hard exit below
    os._exit(0)  # the group cannot be torn down cleanly without the dead peer


def test_dead_rank_fails_the_exchange_within_the_timeout():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_dies, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert procs[1].exitcode == 3
    assert procs[0].exitcode == 0
    what, secs = q.get(timeout=10)
    assert what == "SequenceParallelError"
    assert secs < 60
