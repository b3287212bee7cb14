"""The C-ABI library builds, loads and exports every symbol include/specverify.h
declares; host-side argument checks reject bad calls before any CUDA work
(no GPU needed: nothing here launches a kernel)."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_08_gb300 as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    sv.build()
    return sv.load()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_symbols() == sorted(sv.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_host_only_calls(lib):
    assert lib.sv_version() == 1
    assert sv.status_string(0) == "ok"
    assert "invalid" in sv.status_string(-1)
    assert "outside" in sv.status_string(1)
    # workspace: 256-byte header, then B miss flags, B cached n, B*(K+1) keys, B*nseg pairs
    n = sv.workspace_size(256, 5, 128256)
    assert n % 256 == 0 and n >= 256 + 256 * 4 * 2 + 256 * 6 * 8 + 256 * 126 * 8
    assert sv.workspace_size(0, 0, 1) == 256      # just the status header
    assert sv.workspace_size(1, 65, 10) == 0      # K > SV_MAX_K
    assert sv.workspace_size(1, 4, 0) == 0        # V < 1
    assert sv.workspace_size(1, 4, 2 ** 31) == 0  # ids must fit int32
    assert sv.workspace_size(-1, 4, 10) == 0


def test_invalid_arguments_rejected_on_host(lib):
    P = ctypes.c_void_p
    dummy = P(4096)           # never dereferenced: every call below fails its checks first
    ws = P(1 << 20)
    big = 1 << 30
    # null target / outputs, bad sizes, short strides
    assert lib.sv_verify_greedy(None, 10, dummy, 2, 3, 10, dummy, dummy, ws, big, None) == -1
    assert lib.sv_verify_greedy(dummy, 10, dummy, 2, 3, 10, None, dummy, ws, big, None) == -1
    assert lib.sv_verify_greedy(dummy, 9, dummy, 2, 3, 10, dummy, dummy, ws, big, None) == -1
    assert lib.sv_verify_greedy(dummy, 10, None, 2, 3, 10, dummy, dummy, ws, big, None) == -1
    assert lib.sv_verify_greedy(dummy, 10, dummy, 2, 65, 10, dummy, dummy, ws, big, None) == -1
    assert lib.sv_verify_greedy(dummy, 10, dummy, -1, 3, 10, dummy, dummy, ws, big, None) == -1
    # B = 0 is a no-op that touches nothing
    assert lib.sv_verify_greedy(None, 0, None, 0, 3, 10, None, None, None, 0, None) == 0
    # workspace null, misaligned, too small
    assert lib.sv_verify_greedy(dummy, 10, dummy, 2, 3, 10, dummy, dummy, None, big, None) == -2
    assert lib.sv_verify_greedy(dummy, 10, dummy, 2, 3, 10, dummy, dummy, P((1 << 20) + 8), big,
                                None) == -2
    assert lib.sv_verify_greedy(dummy, 10, dummy, 2, 3, 10, dummy, dummy, ws, 64, None) == -2
    # sampling needs q, u_accept (K > 0) and u_resample
    args = dict(p=dummy, ps=10, q=dummy, qs=10, t=dummy, ua=dummy, ur=dummy)
    def call(**kw):
        a = dict(args, **kw)
        return lib.sv_verify_sample(a["p"], a["ps"], a["q"], a["qs"], a["t"], a["ua"], a["ur"],
                                    2, 3, 10, dummy, dummy, ws, big, None)
    assert call(q=None) == -1 and call(ua=None) == -1 and call(ur=None) == -1
    assert call(qs=5) == -1
    # rounds need a mode array; committing needs lengths and max_len >= 1
    assert lib.sv_verify_round(None, dummy, 10, dummy, 10, dummy, dummy, dummy, 2, 3, 10, dummy,
                               dummy, None, None, 0, ws, big, None) == -1
    assert lib.sv_verify_round(dummy, dummy, 10, dummy, 10, dummy, dummy, dummy, 2, 3, 10, dummy,
                               dummy, dummy, None, 8, ws, big, None) == -1
    assert lib.sv_verify_round(dummy, dummy, 10, dummy, 10, dummy, dummy, dummy, 2, 3, 10, dummy,
                               dummy, dummy, dummy, 0, ws, big, None) == -1
    assert lib.sv_set_ctas_per_sm(-1) == -1
    assert lib.sv_get_status(None, None, None) == -1
