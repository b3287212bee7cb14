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


def test_alpha_logits_and_noalloc_reject_bad_arguments_on_host(lib):
    P = ctypes.c_void_p
    dummy = P(4096)           # never dereferenced: every call below fails its checks first
    ws = P(1 << 20)
    big = 1 << 30
    # acceptance-rate diagnostic: rows, strides, the alpha output and the workspace
    def alpha(p=dummy, ps=10, q=dummy, qs=10, B=2, K=3, V=10, a=dummy, e=dummy, w=ws, n=big):
        return lib.sv_alpha(p, ps, q, qs, B, K, V, a, e, w, n, None)
    assert alpha(p=None) == -1 and alpha(ps=9) == -1
    assert alpha(q=None) == -1 and alpha(qs=9) == -1 and alpha(a=None) == -1
    assert alpha(K=65) == -1 and alpha(V=0) == -1 and alpha(B=-1) == -1
    assert alpha(B=0, p=None, q=None, a=None, e=None, w=None, n=0) == 0
    assert alpha(w=None) == -2 and alpha(w=P((1 << 20) + 16)) == -2 and alpha(n=64) == -2

    # sampling from logits: the temperature must be a positive finite number
    def logits(temp=1.0, zq=dummy, ua=dummy, ur=dummy, zqs=10, K=3):
        return lib.sv_verify_sample_logits(dummy, 10, zq, zqs, dummy, ua, ur, 2, K, 10,
                                           ctypes.c_float(temp), dummy, dummy, ws, big, None)
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        assert logits(temp=bad) == -1, bad
    assert logits(zq=None) == -1 and logits(ua=None) == -1 and logits(ur=None) == -1
    assert logits(zqs=9) == -1 and logits(K=65) == -1

    # the allocation-free call refuses sizes its fixed scratch cannot hold,
    # before it looks for a device
    B, K, V = 4096, 5, 128256
    assert sv.workspace_size(B, K, V) > sv.NOALLOC_SCRATCH_BYTES
    assert lib.sv_verify_sample_noalloc(dummy, V, dummy, V, dummy, dummy, dummy, B, K, V, dummy,
                                        dummy, None) == sv.SV_ETOOLARGE
    assert lib.sv_verify_sample_noalloc(dummy, V, None, V, dummy, dummy, dummy, B, K, V, dummy,
                                        dummy, None) == -1


def test_debug_build_compiles_and_exports_every_symbol(lib, tmp_path):
    """The SV_DEBUG=1 variant (input values checked before each call's
    kernels) builds beside the regular library and offers the same calls."""
    from speculative_decoding_verification_08_gb300 import _build
    dbg = sv._declare(ctypes.CDLL(_build.build_debug(str(tmp_path / "libspecverify_debug.so"))))
    for name in declared_symbols():
        assert hasattr(dbg, name), name
    assert dbg.sv_workspace_size(256, 5, 128256) == lib.sv_workspace_size(256, 5, 128256)
    assert b"NaN" in dbg.sv_status_string(sv.STATUS_BAD_VALUE)
    assert sv.status_string(sv.STATUS_BAD_VALUE) == dbg.sv_status_string(sv.STATUS_BAD_VALUE).decode()


def test_trace_calls_refused_outside_a_trace_build(lib):
    n = ctypes.c_size_t(7)
    buf = ctypes.create_string_buffer(64)
    assert lib.sv_trace_reset(None) == -1
    assert lib.sv_trace_read(buf, 4, ctypes.byref(n), None) == -1 and n.value == 0
    assert lib.sv_trace_read(None, 4, ctypes.byref(n), None) == -1


def test_trace_build_compiles_and_exports_every_symbol(tmp_path):
    from speculative_decoding_verification_08_gb300 import _build
    tr = sv._declare(ctypes.CDLL(_build.build_trace(str(tmp_path / "libspecverify_trace.so"))))
    for name in declared_symbols():
        assert hasattr(tr, name), name
    n = ctypes.c_size_t(7)
    assert tr.sv_trace_read(None, 4, ctypes.byref(n), None) == -1 and n.value == 0


def test_trace_summary_of_known_records():
    """Two CTAs, times in ns from an arbitrary origin."""
    import numpy as np
    E = {name: i for i, name in enumerate(sv.TRACE_EVENTS)}

    def r(t, ev, cta, arg=0):
        return [t, (E[ev] << 56) | (cta << 32) | arg]

    T = 10_000_000
    recs = np.array([
        r(T, "cta_begin", 0), r(T + 500, "cta_begin", 1),
        r(T + 1000, "item_begin", 0, 3), r(T + 1800, "stage", 0, 1), r(T + 2600, "stage", 0, 2),
        r(T + 1500, "item_begin", 1, 4), r(T + 3500, "stage", 1, 1),
        r(T + 9000, "item_retired", 0, 3), r(T + 9500, "decide_begin", 0, 3),
        r(T + 12500, "decide_end", 0, 3), r(T + 11000, "item_retired", 1, 4),
        r(T + 11200, "decide_begin", 1, 4), r(T + 12200, "decide_end", 1, 4),
        r(T + 13000, "producer_end", 1),
    ], dtype=np.uint64)
    s = sv.trace_summary(recs)
    assert s["ctas"] == 2 and s["stages"] == 3
    assert s["cta_begin_spread_us"] == 0.5
    assert s["first_stage_after_begin_us"] == {"median": 2.4, "max": 3.0}
    assert s["last_stage_us"] == 3.5 and s["last_item_retired_us"] == 11.0
    assert s["last_decide_end_us"] == 12.5 and s["span_us"] == 13.0
    assert s["decide_us"] == {"median": 2.0, "max": 3.0}
    assert s["items_per_cta"] == {"median": 1.0, "max": 1.0}
    assert sv.trace_summary(np.zeros((0, 2), np.uint64)) == {}


def test_binding_constants_match_the_header():
    """Every #define of specverify.h that the binding mirrors has the same value."""
    defs = {}
    for name, expr in re.findall(r"#define\s+(SV_[A-Z0-9_]+)\s+(.+)", open(HEADER).read()):
        defs[name] = eval(re.sub(r"(\d+)u\b", r"\1", expr.split("/*")[0]), {})
    mirror = {
        "SV_OK": sv.SV_OK, "SV_EINVAL": sv.SV_EINVAL, "SV_EWORKSPACE": sv.SV_EWORKSPACE,
        "SV_ECUDA": sv.SV_ECUDA, "SV_ETOOLARGE": sv.SV_ETOOLARGE,
        "SV_NOALLOC_SCRATCH_BYTES": sv.NOALLOC_SCRATCH_BYTES, "SV_MAX_K": sv.MAX_K,
        "SV_STATUS_BAD_TOKEN": sv.STATUS_BAD_TOKEN, "SV_STATUS_ZERO_MASS": sv.STATUS_ZERO_MASS,
        "SV_STATUS_OVERFLOW": sv.STATUS_OVERFLOW, "SV_STATUS_BAD_MODE": sv.STATUS_BAD_MODE,
        "SV_STATUS_TIMEOUT": sv.STATUS_TIMEOUT, "SV_STATUS_BAD_VALUE": sv.STATUS_BAD_VALUE,
        "SV_TRACE_RECORDS": sv.TRACE_RECORDS,
    }
    for name, value in mirror.items():
        assert defs[name] == value, name


def test_trace_timeline_of_two_launches():
    """Two launches of two CTAs: each CTA's region holds launch 1's records,
    then launch 2's, each part opening with the placement record."""
    import numpy as np
    E = {name: i for i, name in enumerate(sv.TRACE_EVENTS)}

    def r(t, ev, cta, arg=0):
        return [t, (E[ev] << 56) | (cta << 32) | arg]

    T = 10_000_000
    cta0 = [r(T - 300, "cta_placed", 0), r(T, "cta_begin", 0), r(T + 1000, "stage", 0, 1),
            r(T + 5000, "cta_end", 0),
            r(T + 4000, "cta_placed", 0), r(T + 7000, "cta_begin", 0),
            r(T + 8000, "stage", 0, 1), r(T + 12000, "cta_end", 0)]
    cta1 = [r(T - 200, "cta_placed", 1), r(T + 100, "cta_begin", 1), r(T + 6000, "cta_end", 1),
            r(T + 5000, "cta_placed", 1), r(T + 7200, "cta_begin", 1),
            r(T + 13000, "cta_end", 1)]
    recs = np.array(cta0 + cta1, dtype=np.uint64)
    parts = sv.trace.split_launches(recs)
    assert [len(x) for x in parts] == [7, 7]
    tl = sv.trace_timeline(recs)
    assert len(tl["launches"]) == 2 and len(tl["between"]) == 1
    b = tl["between"][0]
    assert b["period_us"] == 7.0                      # first starts: T and T + 7000
    assert b["prev_exit_to_start_us"] == 1.0          # last exit T + 6000, next start T + 7000
    assert b["placed_before_prev_exit_us"] == 1.5     # median placement T + 4500
    l0 = tl["launches"][0]
    assert l0["cta_placed_us"] == {"median": -0.25, "max": -0.2}
    assert l0["cta_end_us"] == {"median": 5.5, "max": 6.0}
    assert l0["first_stage_after_begin_us"] == {"median": 1.0, "max": 1.0}
