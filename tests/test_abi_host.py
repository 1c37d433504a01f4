"""Host-side checks of the C-ABI library (no GPU needed, no kernel launched).

The library must load, export every symbol that include/linattn.h declares, and
reject malformed requests before touching the device.
"""
import ctypes
import os
import re

import pytest

import chunked_state_scan_causal_gb300 as la
from chunked_state_scan_causal_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "linattn.h")


@pytest.fixture(scope="module")
def cdll():
    build.build()
    return ctypes.CDLL(la.LIB_PATH)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(linattn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for n in ("linattn_fwd", "linattn_bwd", "linattn_chunk_states", "linattn_state_scan"):
        assert n in names


def test_every_declared_symbol_is_exported(cdll):
    missing = [n for n in declared_functions() if not hasattr(cdll, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    for n in declared_functions():
        assert hasattr(la, n), n


def test_abi_version_and_status_strings(cdll):
    assert la.linattn_abi_version() == la.ABI_VERSION == 2
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert la.status_string(code) not in ("", "unknown status")
    assert la.status_string(12345) == "unknown status"


def _shape(**kw):
    s = la.Shape()
    s.abi_version, s.B, s.H, s.T, s.dk, s.dv, s.chunk, s.dtype = la.ABI_VERSION, 1, 2, 256, 128, 128, 64, la.BF16
    s.stride_b, s.stride_h, s.stride_t = 2 * 256 * 128, 256 * 128, 128
    s.decay = None
    for k, v in kw.items():
        setattr(s, k, v)
    return s


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced (calls fail validation first)


@pytest.mark.parametrize("field,value,expected", [
    ("abi_version", 7, la.ERR_INVALID),
    ("B", 0, la.ERR_INVALID),
    ("T", -1, la.ERR_INVALID),
    ("dtype", 5, la.ERR_INVALID),
    ("stride_t", 64, la.ERR_INVALID),
    ("chunk", 32, la.ERR_UNSUPPORTED),
    ("dk", 96, la.ERR_UNSUPPORTED),
    ("dv", 64, la.ERR_UNSUPPORTED),
    ("stride_t", 129, la.ERR_ALIGN),
])
def test_fwd_rejects_bad_shapes(cdll, field, value, expected):
    s = _shape(**{field: value})
    if field == "dv":
        s.dk = 128
    st = la.linattn_fwd(s, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, 1 << 30, None)
    assert st == expected


def test_null_and_misaligned_pointers(cdll):
    s = _shape()
    assert la.linattn_fwd(s, None, FAKE, FAKE, FAKE, None, None, None, FAKE, 1 << 30, None) == la.ERR_INVALID
    assert la.linattn_fwd(s, FAKE + 2, FAKE, FAKE, FAKE, None, None, None, FAKE, 1 << 30, None) == la.ERR_ALIGN
    assert la.linattn_bwd(s, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, None, None, FAKE, 1 << 30,
                          None) == la.ERR_INVALID
    # a misaligned d_final_state is rejected before anything is enqueued
    assert la.linattn_bwd(s, FAKE, FAKE, FAKE, FAKE, None, FAKE + 4, FAKE, FAKE, FAKE, None, FAKE, 1 << 30,
                          None) == la.ERR_ALIGN
    assert la.lib().linattn_fwd(None, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, 1 << 30, None) \
        == la.ERR_INVALID


def test_workspace_checks(cdll):
    s = _shape()
    st, need = la.linattn_workspace_size(s, la.OP_FWD)
    assert st == la.OK and need >= 256
    assert la.linattn_fwd(s, FAKE, FAKE, FAKE, FAKE, None, None, None, None, 1 << 30, None) == la.ERR_WORKSPACE
    assert la.linattn_fwd(s, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE + 16, 1 << 30, None) \
        == la.ERR_WORKSPACE
    assert la.linattn_fwd(s, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, need - 1, None) == la.ERR_WORKSPACE
    assert la.linattn_workspace_size(s, 99)[0] == la.ERR_INVALID
    assert la.linattn_workspace_size(s, la.OP_CHUNK_STATES, 0)[0] == la.ERR_INVALID


def test_chunk_states_and_scan_argument_checks(cdll):
    s = _shape()
    # seg_len must divide T
    assert la.linattn_chunk_states(s, 100, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == la.ERR_UNSUPPORTED
    assert la.linattn_chunk_states(s, 0, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == la.ERR_INVALID
    assert la.linattn_chunk_states_rev(s, 100, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == la.ERR_UNSUPPORTED
    assert la.linattn_chunk_states_rev(s, 0, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == la.ERR_INVALID
    assert la.linattn_chunk_states_rev(s, 64, None, FAKE, FAKE, FAKE, 1 << 20, None) == la.ERR_INVALID
    assert la.linattn_state_scan_workspace_size(0, 1, 8, 8)[0] == la.ERR_INVALID
    assert la.linattn_state_scan_workspace_size(3, 2, 3, 3)[0] == la.ERR_UNSUPPORTED
    st, n = la.linattn_state_scan_workspace_size(64, 16, 128, 128)
    assert st == la.OK and n > 256
    assert la.linattn_state_scan(64, 16, 128, 128, None, None, None, FAKE, None, FAKE, n, None) == la.ERR_INVALID
    assert la.linattn_state_scan(64, 16, 128, 128, None, FAKE, None, FAKE, None, FAKE, n - 1, None) \
        == la.ERR_WORKSPACE
    assert la.linattn_diag_mma(9, FAKE, FAKE, FAKE, None) == la.ERR_INVALID


def test_device_status_null(cdll):
    assert la.linattn_device_status(None, None) == la.ERR_INVALID


def test_gated_entry_points_check_their_arguments(cdll):
    s = _shape()
    ck = 1 << 30  # large enough for any checkpoint size check
    # fp32 inputs take the CUDA-core path: no checkpoint, no workspace past the status header
    sh = _shape(dtype=la.F32)
    for op in (la.OP_FWD_GATED, la.OP_BWD_GATED):
        assert la.linattn_workspace_size(sh, op) == (la.OK, 256)
    assert la.linattn_workspace_size(sh, la.OP_CHECKPOINT_GATED) == (la.OK, 0)
    # bf16 with d = 64 runs as the zero-padded d = 128 problem: its checkpoint holds d = 128
    # states, and the workspace adds the padded copies of the states that cross the ABI
    sh64 = _shape(dk=64, dv=64, stride_b=2 * 256 * 64, stride_h=256 * 64, stride_t=64)
    assert la.linattn_workspace_size(sh64, la.OP_CHECKPOINT_GATED) == la.linattn_workspace_size(
        s, la.OP_CHECKPOINT_GATED)
    for op, extra in ((la.OP_FWD_GATED, 1), (la.OP_BWD_GATED, 2)):
        st, n64 = la.linattn_workspace_size(sh64, op)
        assert st == la.OK and n64 >= la.linattn_workspace_size(s, op)[1] + extra * 2 * 128 * 128 * 4
    # the per-head decay and gates exclude each other
    lam = (ctypes.c_float * 2)(0.9, 0.9)
    assert la.linattn_fwd_gated(_shape(decay=ctypes.cast(lam, ctypes.c_void_p)), FAKE, FAKE, FAKE,
                                FAKE, FAKE, None, None, FAKE, ck, FAKE, 1 << 30, None) == la.ERR_INVALID
    # a checkpoint is required, and the gates
    assert la.linattn_fwd_gated(s, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, 0, FAKE, 1 << 30,
                                None) == la.ERR_INVALID
    assert la.linattn_fwd_gated(s, FAKE, FAKE, FAKE, None, FAKE, None, None, FAKE, ck, FAKE, 1 << 30,
                                None) == la.ERR_INVALID
    assert la.linattn_bwd_gated(s, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, ck, FAKE, FAKE, FAKE, None,
                                None, FAKE, 1 << 30, None) == la.ERR_INVALID
    for op in (la.OP_FWD_GATED, la.OP_BWD_GATED, la.OP_CHECKPOINT_GATED):
        st, n = la.linattn_workspace_size(s, op)
        assert st == la.OK and n >= 256


def test_gated_vec_checkpoint_checks(cdll):
    """The per-dimension checkpoint: empty with one chunk group per sequence, otherwise
    required by the _ckpt entry points (NULL, short or misaligned: ERR_INVALID before any
    device work).  The group count follows the SM count, so the case takes one sequence
    long enough for two groups on any device (the host without a GPU counts one SM)."""
    one = _shape(H=1, T=200, stride_b=200 * 128, stride_h=200 * 128)
    assert la.linattn_workspace_size(one, la.OP_CHECKPOINT_GATED_VEC) == (la.OK, 0)
    s = _shape(H=1, T=4096, stride_b=4096 * 128, stride_h=4096 * 128)
    st, n = la.linattn_workspace_size(s, la.OP_CHECKPOINT_GATED_VEC)
    assert st == la.OK and n > 0 and n % 256 == 0
    for ck, nb in ((None, n), (FAKE, n - 256), (FAKE + 16, n)):
        assert la.linattn_fwd_gated_vec_ckpt(s, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, ck, nb, FAKE, 1 << 30,
                                             None) == la.ERR_INVALID
        assert la.linattn_bwd_gated_vec_ckpt(s, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, ck, nb, FAKE, FAKE, FAKE,
                                             FAKE, None, FAKE, 1 << 30, None) == la.ERR_INVALID
