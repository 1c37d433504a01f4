"""Bounded device waits: a look-back wait that can never be satisfied gives up,
reports LINATTN_ERR_DEVICE_TIMEOUT in the status word and lets the kernel end.

The look-back tile is kept from publishing by a diagnostic argument (set from
the host), and the wait limit is a few milliseconds; nothing faults, traps or
hangs, and the next ordinary call on the same workspace is clean.
"""
import time

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


def test_lookback_wait_gives_up_with_timeout_status():
    G, BH, dk, dv = 300, 1, 8, 8           # 10 segment tiles x 8 element groups
    ncg = BH * dk * dv // 8
    g = torch.Generator().manual_seed(11)
    local = torch.randn(G, BH, dk, dv, generator=g).cuda()
    out = torch.empty_like(local)
    st, n = la.linattn_state_scan_workspace_size(G, BH, dk, dv)
    assert st == la.OK
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    # tile (segment tile 1, element group 0) never publishes: tile 2's look-back waits 5 ms and gives up
    st = la.linattn_diag_scan_withhold(G, BH, dk, dv, local.data_ptr(), out.data_ptr(), 1 * ncg + 0, 5.0,
                                       ws.data_ptr(), ws.numel(), stream)
    assert st == la.OK
    status = la.linattn_device_status(ws.data_ptr(), stream)
    elapsed = time.perf_counter() - t0
    assert status == la.ERR_DEVICE_TIMEOUT
    assert elapsed < 0.5, elapsed
    # the columns that never meet the withheld tile are still exact
    ref, _ = oracle.state_scan(local.cpu().numpy())
    got = out.cpu().numpy().reshape(G, -1)
    refr = ref.reshape(G, -1)
    assert np.max(np.abs(got[:, 8:] - refr[:, 8:])) <= 1e-5 * np.max(np.abs(refr))
    # the next ordinary call on the same workspace is clean and exact
    out2, _ = la.state_scan(local, ws=ws)
    assert la.device_status(ws) == la.OK
    assert np.max(np.abs(out2.cpu().numpy() - ref)) <= 1e-5 * np.max(np.abs(ref))


def test_segment_decay_multipliers():
    lam = np.array([0.5, 0.9, 0.999, 1.0], dtype=np.float32)
    d = torch.from_numpy(lam).cuda()
    got = la.segment_decay(d, 3, 100).cpu().numpy()
    ref = np.tile(lam.astype(np.float64) ** 100, 3)
    assert got.shape == (12,)
    assert np.max(np.abs(got - ref) / np.maximum(ref, 1e-30)) < 1e-5
