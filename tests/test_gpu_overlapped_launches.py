"""The chunked path's kernels start their prologue while the kernel before them on the
stream finishes (programmatic dependent launch), and each waits for it before touching
memory.  A kernel that read or wrote too early would make results depend on timing:
here whole fwd+bwd steps run back to back with no synchronisation, on two streams with
their own workspaces and checkpoints, and every output must be bitwise the output of
the same step run alone (the kernels are deterministic: an item's result does not
depend on the CTA that draws it)."""
import pytest
import torch

import chunked_state_scan_causal_gb300 as la
from chunked_state_scan_causal_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from chunked_state_scan_causal_gb300 import build
    build.build()


def _step(x, b, decay, gated, s):
    with torch.cuda.stream(s):
        if gated:
            la.fwd_gated(x["q"], x["k"], x["v"], x["lg"], b["ck"], out=b["o"], ws=b["wsf"])
            la.bwd_gated(x["q"], x["k"], x["v"], x["dO"], x["lg"], b["ck"], outs=b["g"], ws=b["wsb"],
                         dlg_out=b["dlg"])
        else:
            la.fwd(x["q"], x["k"], x["v"], decay=decay, out=b["o"], ws=b["wsf"], ckpt=b["ck"])
            la.bwd(x["q"], x["k"], x["v"], x["dO"], decay=decay, outs=b["g"], ws=b["wsb"], ckpt=b["ck"])


def _buffers(x, decay, gated):
    q = x["q"]
    b = dict(o=torch.empty_like(q), g=[torch.empty_like(q) for _ in range(3)])
    if gated:
        b.update(wsf=la.workspace(q, la.OP_FWD_GATED), wsb=la.workspace(q, la.OP_BWD_GATED),
                 ck=la.checkpoint_gated(q), dlg=torch.empty_like(x["lg"]))
    else:
        b.update(wsf=la.workspace(q, la.OP_FWD, decay), wsb=la.workspace(q, la.OP_BWD, decay),
                 ck=la.checkpoint(q, decay))
    return b


def _outs(b):
    return [b["o"]] + b["g"] + ([b["dlg"]] if "dlg" in b else [])


@pytest.mark.parametrize("workload,T", [(3, 16384), (4, 8192), (6, 8192)])
def test_back_to_back_steps_equal_an_isolated_step(workload, T):
    cfg = dict(inputs.WORKLOADS[workload])
    dev = torch.device("cuda", 0)
    x = {w: inputs.make(cfg, w, T=T).to(dev) for w in ("q", "k", "v", "dO")}
    lam = inputs.workload_decay(cfg)
    decay = None if lam is None else torch.from_numpy(lam).to(dev)
    gated = cfg.get("gates") is not None
    if gated:
        x["lg"] = inputs.make_gates(cfg, T=T, device=dev)
    ref = _buffers(x, decay, gated)
    _step(x, ref, decay, gated, torch.cuda.current_stream(dev))
    torch.cuda.synchronize()
    assert la.device_status(ref["wsf"]) == la.OK and la.device_status(ref["wsb"]) == la.OK
    s2 = torch.cuda.Stream(dev)
    bufs = [_buffers(x, decay, gated) for _ in range(2)]
    for i in range(6):
        _step(x, bufs[i % 2], decay, gated, torch.cuda.current_stream(dev) if i % 2 == 0 else s2)
    torch.cuda.synchronize()
    for b in bufs:
        assert la.device_status(b["wsf"]) == la.OK and la.device_status(b["wsb"]) == la.OK
        for got, want in zip(_outs(b), _outs(ref)):
            assert torch.equal(got, want)


def test_many_steps_at_full_size():
    """500 benchmark steps (B2 H16 T65536) back to back on one stream: the bounded waits
    never give up under the overlapped launches, and the last step's outputs are bitwise
    those of a step run alone."""
    cfg = dict(inputs.WORKLOADS[3])
    dev = torch.device("cuda", 0)
    x = {w: inputs.make(cfg, w).to(dev) for w in ("q", "k", "v", "dO")}
    s = torch.cuda.current_stream(dev)
    ref = _buffers(x, None, False)
    _step(x, ref, None, False, s)
    torch.cuda.synchronize()
    b = _buffers(x, None, False)
    for _ in range(500):
        _step(x, b, None, False, s)
    torch.cuda.synchronize()
    assert la.device_status(b["wsf"]) == la.OK and la.device_status(b["wsb"]) == la.OK
    for got, want in zip(_outs(b), _outs(ref)):
        assert torch.equal(got, want)
