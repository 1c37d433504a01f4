"""The allocation-free state scan (linattn_state_scan_noalloc) against the
workspace-taking linattn_state_scan, through the C ABI.

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

import chunked_state_scan_causal_gb300 as la

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from chunked_state_scan_causal_gb300 import build
    build.build()


def _rel(a, b):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    return float(np.max(np.abs(a - b))) / max(float(np.max(np.abs(b))), 1e-30)


def test_noalloc_scan_matches_workspace_scan_on_two_calls():
    G, BH, dk, dv = 300, 3, 16, 24
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        g = torch.Generator().manual_seed(100 + call)
        local = torch.randn(G, BH, dk, dv, generator=g).cuda()
        decay = (0.5 + 0.5 * torch.rand(BH, generator=g)).cuda()
        init = torch.randn(BH, dk, dv, generator=g).cuda()
        ref, ref_total = la.state_scan(local, decay, init, want_total=True)
        out = torch.full_like(local, float("nan"))
        total = torch.full_like(init, float("nan"))
        dstat = torch.full((4,), 7, dtype=torch.int32, device="cuda")
        st = la.linattn_state_scan_noalloc(G, BH, dk, dv, decay.data_ptr(), local.data_ptr(), init.data_ptr(),
                                           out.data_ptr(), total.data_ptr(), dstat.data_ptr(), stream)
        assert st == la.OK
        torch.cuda.synchronize()
        assert int(dstat[0]) == 0
        assert _rel(out, ref) < 1e-5, call
        assert _rel(total, ref_total) < 1e-5, call


def test_noalloc_scan_rejects_requests_beyond_its_scratch():
    # 2 segment tiles x (16 * 128 * 128 / 8) element groups = 65536 tiles fit; 65 segments (3 tiles) do not
    stream = torch.cuda.current_stream().cuda_stream
    fake = 1 << 20  # never dereferenced: the call must fail before enqueuing anything
    assert la.linattn_state_scan_noalloc(65, 16, 128, 128, None, fake, None, fake, None, None, stream) \
        == la.ERR_SCRATCH_LIMIT
