"""The allocation-free state scan (linattn_state_scan_noalloc) through the C ABI,
against the fp64 oracle's exclusive scan and the workspace-taking
linattn_state_scan.

Callers that cannot allocate device memory (their host application owns all
of it, or their path must not allocate) use the allocation-free entry point,
whose scratch is a fixed array inside the library.  Two calls in a row with
different inputs check that the shared scratch is reset between calls; the
case has 300 segments (ten 32-segment tiles), long enough for the scan's
decoupled look-back, which is what goes through that scratch.  This file is
collected last on purpose.
"""
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
    oracle.build()


def _rel(a, b):
    a = a.double().cpu().numpy() if torch.is_tensor(a) else a
    b = b.double().cpu().numpy() if torch.is_tensor(b) else b
    return float(np.max(np.abs(a - b))) / max(float(np.max(np.abs(b))), 1e-30)


def test_noalloc_scan_matches_oracle_and_workspace_scan_on_two_calls():
    G, BH, dk, dv = 300, 3, 16, 24
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        g = torch.Generator().manual_seed(100 + call)
        local = torch.randn(G, BH, dk, dv, generator=g)
        decay = 0.5 + 0.5 * torch.rand(BH, generator=g)
        init = torch.randn(BH, dk, dv, generator=g)
        r_out, r_total = oracle.state_scan(local.numpy(), seg_decay=decay.numpy(), init=init.numpy())
        local_d, decay_d, init_d = local.cuda(), decay.cuda(), init.cuda()
        ref, ref_total = la.state_scan(local_d, decay_d, init_d, want_total=True)
        out = torch.full_like(local_d, float("nan"))
        total = torch.full_like(init_d, float("nan"))
        dstat = torch.full((4,), 7, dtype=torch.int32, device="cuda")
        st = la.linattn_state_scan_noalloc(G, BH, dk, dv, decay_d.data_ptr(), local_d.data_ptr(), init_d.data_ptr(),
                                           out.data_ptr(), total.data_ptr(), dstat.data_ptr(), stream)
        assert st == la.OK
        torch.cuda.synchronize()
        assert int(dstat[0]) == 0
        assert _rel(out, r_out) < 1e-5, call
        assert _rel(total, r_total) < 1e-5, call
        assert _rel(out, ref) < 1e-5, call
        assert _rel(total, ref_total) < 1e-5, call


def test_noalloc_scan_column_form_needs_no_scratch():
    """Up to 256 segments the scan runs column-parallel and touches no scratch, so a
    request far larger than the scratch's tile limit is served (16 states of 128x128)."""
    G, BH, dk, dv = 128, 16, 128, 128
    g = torch.Generator().manual_seed(7)
    local = torch.randn(G, BH, dk, dv, generator=g)
    r_out, r_total = oracle.state_scan(local.numpy())
    local_d = local.cuda()
    out = torch.full_like(local_d, float("nan"))
    total = torch.full((BH, dk, dv), float("nan"), device="cuda")
    dstat = torch.full((4,), 7, dtype=torch.int32, device="cuda")
    st = la.linattn_state_scan_noalloc(G, BH, dk, dv, None, local_d.data_ptr(), None, out.data_ptr(),
                                       total.data_ptr(), dstat[1:].data_ptr(),  # 4-byte aligned status word
                                       torch.cuda.current_stream().cuda_stream)
    assert st == la.OK
    torch.cuda.synchronize()
    assert int(dstat[1]) == 0
    assert _rel(out, r_out) < 1e-5
    assert _rel(total, r_total) < 1e-5


def test_noalloc_scan_rejects_requests_beyond_its_scratch():
    # look-back form: 300 segments -> 10 segment tiles x (16 * 128 * 128 / 8) element groups > 65536 tiles
    stream = torch.cuda.current_stream().cuda_stream
    fake = 1 << 20  # never dereferenced: the call must fail before enqueuing anything
    assert la.linattn_state_scan_noalloc(300, 16, 128, 128, None, fake, None, fake, None, None, stream) \
        == la.ERR_SCRATCH_LIMIT
