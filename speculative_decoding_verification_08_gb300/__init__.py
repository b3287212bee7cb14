"""Batched speculative-decoding verification on GB300 (sm_103a).

Python binding of ``libspecverify.so`` (C ABI in ``include/specverify.h``).
This module only marshals arguments: torch CUDA tensors are checked for
dtype, device and layout and their pointers, strides and the current CUDA
stream are passed to the library, whose kernels do every step of the
verification.  There is no CPU path: if the library is missing or a tensor is
not on a CUDA device, the call raises.

The operation is the one on the "spec-verify" page (Hugging Face kernels page
phanerozoic/spec-verify), section "Usage":
``n_accepted, next_token = verify_greedy(target_probs, draft_tokens)`` -- keep
``draft_tokens[:n_accepted]`` and append ``next_token`` -- batched over B
sequences, plus the speculative-sampling rule of section "Method".
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build
from . import trace as _trace
from .trace import TRACE_EVENTS

LIBRARY = _build.LIBRARY

SV_OK = 0
SV_EINVAL = -1
SV_EWORKSPACE = -2
SV_ECUDA = -3
SV_ETOOLARGE = -4
NOALLOC_SCRATCH_BYTES = 4 << 20
STATUS_BAD_TOKEN = 1
STATUS_ZERO_MASS = 2
STATUS_OVERFLOW = 4
STATUS_BAD_MODE = 8
STATUS_TIMEOUT = 16
STATUS_BAD_VALUE = 32   # debug builds only (built with SV_DEBUG=1)
MAX_K = 64

# every symbol include/specverify.h declares
EXPORTED = (
    "sv_workspace_size", "sv_workspace_init", "sv_verify_greedy", "sv_verify_sample",
    "sv_verify_round", "sv_get_status", "sv_set_ctas_per_sm", "sv_last_grid_size",
    "sv_last_kernel_count", "sv_alpha", "sv_verify_sample_logits",
    "sv_status_string", "sv_version", "sv_verify_sample_noalloc", "sv_trace_reset",
    "sv_trace_read",
)

_lock = threading.Lock()
_lib = None


class SpecVerifyError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compiles libspecverify.so in-tree (nvcc, sm_103a)."""
    return _build.build(force=force)


def load():
    """The ctypes handle of libspecverify.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIBRARY):
            raise SpecVerifyError(
                f"{LIBRARY} is missing: build it with "
                "speculative_decoding_verification_08_gb300.build() (no CPU fallback exists)")
        _lib = _declare(ctypes.CDLL(LIBRARY))
        return _lib


def _declare(lib):
    """Sets the argument and result types of every C-ABI call on a loaded
    copy of the library (the regular build, or a debug build)."""
    P = ctypes.c_void_p
    i32, i64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.sv_workspace_size.argtypes = [i32, i32, i64]
    lib.sv_workspace_size.restype = sz
    lib.sv_workspace_init.argtypes = [P, sz, P]
    lib.sv_workspace_init.restype = ctypes.c_int
    lib.sv_verify_greedy.argtypes = [P, i64, P, i32, i32, i64, P, P, P, sz, P]
    lib.sv_verify_greedy.restype = ctypes.c_int
    lib.sv_verify_sample.argtypes = [P, i64, P, i64, P, P, P, i32, i32, i64, P, P, P, sz, P]
    lib.sv_verify_sample.restype = ctypes.c_int
    lib.sv_verify_round.argtypes = [P, P, i64, P, i64, P, P, P, i32, i32, i64, P, P,
                                    P, P, i32, P, sz, P]
    lib.sv_verify_round.restype = ctypes.c_int
    lib.sv_get_status.argtypes = [P, P, P]
    lib.sv_get_status.restype = ctypes.c_int
    lib.sv_set_ctas_per_sm.argtypes = [i32]
    lib.sv_set_ctas_per_sm.restype = ctypes.c_int
    lib.sv_last_grid_size.argtypes = []
    lib.sv_last_grid_size.restype = i64
    lib.sv_last_kernel_count.argtypes = []
    lib.sv_last_kernel_count.restype = i32
    lib.sv_alpha.argtypes = [P, i64, P, i64, i32, i32, i64, P, P, P, sz, P]
    lib.sv_alpha.restype = ctypes.c_int
    lib.sv_verify_sample_logits.argtypes = [P, i64, P, i64, P, P, P, i32, i32, i64,
                                            ctypes.c_float, P, P, P, sz, P]
    lib.sv_verify_sample_logits.restype = ctypes.c_int
    lib.sv_status_string.argtypes = [ctypes.c_int]
    lib.sv_status_string.restype = ctypes.c_char_p
    lib.sv_version.argtypes = []
    lib.sv_version.restype = ctypes.c_int
    lib.sv_verify_sample_noalloc.argtypes = [P, i64, P, i64, P, P, P, i32, i32, i64, P, P, P]
    lib.sv_verify_sample_noalloc.restype = ctypes.c_int
    lib.sv_trace_reset.argtypes = [P]
    lib.sv_trace_reset.restype = ctypes.c_int
    lib.sv_trace_read.argtypes = [P, sz, ctypes.POINTER(sz), P]
    lib.sv_trace_read.restype = ctypes.c_int
    return lib


def status_string(code: int) -> str:
    return load().sv_status_string(int(code)).decode()


def _check(rc: int, what: str):
    if rc != SV_OK:
        raise SpecVerifyError(f"{what}: {status_string(rc)} (code {rc})")


def workspace_size(B: int, K: int, V: int) -> int:
    return int(load().sv_workspace_size(B, K, V))


def set_ctas_per_sm(n: int):
    """Persistent-grid residency override (0 = as many CTAs as the SMs hold)."""
    _check(load().sv_set_ctas_per_sm(int(n)), "sv_set_ctas_per_sm")


def last_grid_size() -> int:
    return int(load().sv_last_grid_size())


def last_kernel_count() -> int:
    """Kernels the last verification call on this thread enqueued."""
    return int(load().sv_last_kernel_count())


def _torch():
    import torch
    return torch


def _stream_handle(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class Workspace:
    """Device scratch for B sequences, K drafts and vocabulary V (zeroed once)."""

    def __init__(self, B: int, K: int, V: int, device=None, stream=None):
        torch = _torch()
        nbytes = workspace_size(B, K, V)
        if nbytes == 0:
            raise SpecVerifyError(f"invalid sizes B={B} K={K} V={V}")
        dev = torch.device("cuda") if device is None else torch.device(device)
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.B, self.K, self.V, self.nbytes = B, K, V, nbytes
        _check(load().sv_workspace_init(self.ptr, nbytes, _stream_handle(stream)),
               "sv_workspace_init")

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())

    def fits(self, B, K, V) -> bool:
        return workspace_size(B, K, V) <= self.nbytes

    def status(self, stream=None) -> int:
        """Waits for the stream and returns (and clears) the device status bits."""
        out = ctypes.c_uint32(0)
        _check(load().sv_get_status(self.ptr, _stream_handle(stream), ctypes.byref(out)),
               "sv_get_status")
        return int(out.value)


_ws_cache = {}


def _workspace(ws, B, K, V, device, stream=None):
    """The caller's workspace, or one kept for these sizes and this stream.
    Calls that share a workspace must be ordered on one stream, so calls on
    different streams never share an implicit one."""
    if ws is not None:
        if not ws.fits(B, K, V):
            raise SpecVerifyError("workspace too small for these sizes")
        return ws
    key = (str(device), B, K, V, _stream_handle(stream).value)
    w = _ws_cache.get(key)
    if w is None:
        w = Workspace(B, K, V, device, stream)
        _ws_cache[key] = w
    return w


def _device_of(x):
    """The CUDA device a call on x runs on: x's own, or the current one for a
    pinned CPU tensor."""
    torch = _torch()
    return x.device if x.is_cuda else torch.device("cuda", torch.cuda.current_device())


def _usable(x) -> bool:
    """A CUDA tensor, or a CPU tensor in page-locked memory (read in place)."""
    return x.is_cuda or x.is_pinned()


def _rows3(x, rows, name, dtype):
    """(tensor viewed as [B][rows][V], B, V, row stride) with the library's layout."""
    torch = _torch()
    if not isinstance(x, torch.Tensor) or not _usable(x):
        raise SpecVerifyError(f"{name} must be a CUDA tensor or a pinned CPU tensor")
    if x.dtype != dtype:
        raise SpecVerifyError(f"{name} must be {dtype}, got {x.dtype}")
    if x.dim() == 2:
        x = x.unsqueeze(0)
    if x.dim() != 3 or x.shape[1] != rows:
        raise SpecVerifyError(f"{name}: expected [B][{rows}][V], got {tuple(x.shape)}")
    B, _, V = x.shape
    if x.stride(2) != 1:
        raise SpecVerifyError(f"{name}: the vocabulary dimension must be contiguous")
    rs = x.stride(1) if rows > 1 else (x.stride(0) if B > 1 else V)
    if rows > 1 and B > 1 and x.stride(0) != rows * rs:
        raise SpecVerifyError(f"{name}: rows of all sequences must be evenly strided")
    if rs < V:
        raise SpecVerifyError(f"{name}: row stride {rs} < V={V}")
    return x, B, V, rs


def _vec(x, n, name, dtype, device):
    torch = _torch()
    if x is None:
        return None
    if not isinstance(x, torch.Tensor) or not (x.is_pinned() or (x.is_cuda and x.device == device)):
        raise SpecVerifyError(f"{name} must be a CUDA tensor on {device} or a pinned CPU tensor")
    if x.dtype != dtype:
        raise SpecVerifyError(f"{name} must be {dtype}, got {x.dtype}")
    if not x.is_contiguous() or x.numel() != n:
        raise SpecVerifyError(f"{name}: expected {n} contiguous elements")
    return x


def _ptr(x):
    return ctypes.c_void_p(0 if x is None else x.data_ptr())


def _outputs(B, device, n_out, next_out):
    torch = _torch()
    if n_out is None:
        n_out = torch.empty(B, dtype=torch.int32, device=device)
    if next_out is None:
        next_out = torch.empty(B, dtype=torch.int32, device=device)
    _vec(n_out, B, "n_accepted", torch.int32, device)
    _vec(next_out, B, "next_token", torch.int32, device)
    return n_out, next_out


def verify_greedy(p, t, *, ws=None, n_out=None, next_out=None, stream=None):
    """Greedy verification.  p: [B][K+1][V] (or [K+1][V]) f32, t: [B][K] (or [K])
    int32 -> (n_accepted [B] int32, next_token [B] int32) on the same device."""
    torch = _torch()
    K = t.shape[-1]
    p, B, V, ps = _rows3(p, K + 1, "p", torch.float32)
    dev = _device_of(p)
    t = _vec(t, B * K, "t", torch.int32, dev)
    n_out, next_out = _outputs(B, dev, n_out, next_out)
    w = _workspace(ws, B, K, V, dev, stream)
    rc = load().sv_verify_greedy(_ptr(p), ps, _ptr(t), B, K, V, _ptr(n_out), _ptr(next_out),
                                 w.ptr, w.nbytes, _stream_handle(stream))
    _check(rc, "sv_verify_greedy")
    return n_out, next_out


def verify_sample(p, q, t, u_acc, u_res, *, ws=None, n_out=None, next_out=None, stream=None):
    """Speculative-sampling verification.  p: [B][K+1][V] f32, q: [B][K][V] f32,
    t: [B][K] int32, u_acc: [B][K] f32, u_res: [B] f64 -> (n_accepted, next_token)."""
    torch = _torch()
    K = t.shape[-1]
    p, B, V, ps = _rows3(p, K + 1, "p", torch.float32)
    dev = _device_of(p)
    q, Bq, Vq, qs = _rows3(q, K, "q", torch.float32) if K > 0 else (None, B, V, V)
    if (Bq, Vq) != (B, V):
        raise SpecVerifyError("q does not match p")
    t = _vec(t, B * K, "t", torch.int32, dev)
    u_acc = _vec(u_acc, B * K, "u_acc", torch.float32, dev)
    u_res = _vec(u_res, B, "u_res", torch.float64, dev)
    n_out, next_out = _outputs(B, dev, n_out, next_out)
    w = _workspace(ws, B, K, V, dev, stream)
    rc = load().sv_verify_sample(_ptr(p), ps, _ptr(q), qs, _ptr(t), _ptr(u_acc), _ptr(u_res),
                                 B, K, V, _ptr(n_out), _ptr(next_out), w.ptr, w.nbytes,
                                 _stream_handle(stream))
    _check(rc, "sv_verify_sample")
    return n_out, next_out


def verify_sample_noalloc(p, q, t, u_acc, u_res, *, n_out=None, next_out=None, stream=None):
    """verify_sample without a workspace, for callers that cannot allocate
    device memory while enqueueing work (framework hooks or plugin interfaces
    that forbid allocation, serving loops that must not risk a synchronising
    or failing cudaMalloc).  The scratch is a fixed 4 MiB array inside the
    library; larger sizes raise (SV_ETOOLARGE).  Calls share that array, so
    calls that overlap on the GPU race.  Pass n_out/next_out to avoid the two
    output allocations this wrapper would otherwise make."""
    torch = _torch()
    K = t.shape[-1]
    p, B, V, ps = _rows3(p, K + 1, "p", torch.float32)
    dev = _device_of(p)
    q, Bq, Vq, qs = _rows3(q, K, "q", torch.float32) if K > 0 else (None, B, V, V)
    if (Bq, Vq) != (B, V):
        raise SpecVerifyError("q does not match p")
    t = _vec(t, B * K, "t", torch.int32, dev)
    u_acc = _vec(u_acc, B * K, "u_acc", torch.float32, dev)
    u_res = _vec(u_res, B, "u_res", torch.float64, dev)
    n_out, next_out = _outputs(B, dev, n_out, next_out)
    rc = load().sv_verify_sample_noalloc(_ptr(p), ps, _ptr(q), qs, _ptr(t), _ptr(u_acc),
                                         _ptr(u_res), B, K, V, _ptr(n_out), _ptr(next_out),
                                         _stream_handle(stream))
    _check(rc, "sv_verify_sample_noalloc")
    return n_out, next_out


def verify_sample_logits(zp, zq, t, u_acc, u_res, temperature: float = 1.0, *, ws=None,
                         n_out=None, next_out=None, stream=None):
    """Sampling verification from logits: zp [B][K+1][V], zq [B][K][V] f32 (or
    [K+1][V] / [K][V]), warped by softmax(z / temperature) on the fly ->
    (n_accepted, next_token) int32 [B]."""
    torch = _torch()
    t_ = t if t.dim() == 2 else t.reshape(1, -1)
    K = t_.shape[1]
    zp, B, V, ps = _rows3(zp, K + 1, "zp", torch.float32)
    dev = _device_of(zp)
    zq, Bq, Vq, qs = _rows3(zq, K, "zq", torch.float32) if K > 0 else (None, B, V, V)
    if K > 0 and (Bq, Vq) != (B, V):
        raise SpecVerifyError("zq shape does not match zp")
    t = _vec(t, B * K, "t", torch.int32, dev)
    u_acc = _vec(u_acc, B * K, "u_acc", torch.float32, dev)
    u_res = _vec(u_res, B, "u_res", torch.float64, dev)
    n_out, next_out = _outputs(B, dev, n_out, next_out)
    w = _workspace(ws, B, K, V, dev, stream)
    _check(load().sv_verify_sample_logits(_ptr(zp), ps, _ptr(zq), qs, _ptr(t), _ptr(u_acc),
                                          _ptr(u_res), B, K, V, float(temperature), _ptr(n_out),
                                          _ptr(next_out), w.ptr, w.nbytes,
                                          _stream_handle(stream)),
           "sv_verify_sample_logits")
    return n_out, next_out


def alpha(p, q, *, ws=None, alpha_out=None, expected_out=None, stream=None):
    """Acceptance-rate diagnostic: p [B][K+1][V], q [B][K][V] f32 ->
    (alpha [B][K] f64, expected accepted length [B] f64), with
    alpha[b][i] = sum_v min(p_i / P_i, q_i / Q_i) over row totals P_i, Q_i."""
    torch = _torch()
    q3, B, V, qs = _rows3(q, q.shape[-2] if q.dim() >= 2 else 1, "q", torch.float32)
    K = q3.shape[1]
    p, Bp, Vp, ps = _rows3(p, K + 1, "p", torch.float32)
    if (Bp, Vp) != (B, V):
        raise SpecVerifyError("q shape does not match p")
    dev = _device_of(p)
    if alpha_out is None:
        alpha_out = torch.empty(B, K, dtype=torch.float64, device=dev)
    if expected_out is None:
        expected_out = torch.empty(B, dtype=torch.float64, device=dev)
    _vec(alpha_out.reshape(-1), B * K, "alpha_out", torch.float64, dev)
    _vec(expected_out, B, "expected_out", torch.float64, dev)
    w = _workspace(ws, B, K, V, dev, stream)
    _check(load().sv_alpha(_ptr(p), ps, _ptr(q3), qs, B, K, V, _ptr(alpha_out),
                           _ptr(expected_out), w.ptr, w.nbytes, _stream_handle(stream)),
           "sv_alpha")
    return alpha_out, expected_out


def verify_round(mode, p, q, t, u_acc, u_res, *, tokens=None, lengths=None, ws=None,
                 n_out=None, next_out=None, stream=None):
    """Mixed round: mode [B] uint8 (0 greedy, 1 sampling) picks each sequence's
    rule.  With tokens [B][max_len] int32 and lengths [B] int32 the round is
    committed in place (t[b][:n] then next appended)."""
    torch = _torch()
    K = t.shape[-1]
    p, B, V, ps = _rows3(p, K + 1, "p", torch.float32)
    dev = _device_of(p)
    q, Bq, Vq, qs = _rows3(q, K, "q", torch.float32) if K > 0 else (None, B, V, V)
    if (Bq, Vq) != (B, V):
        raise SpecVerifyError("q does not match p")
    mode = _vec(mode, B, "mode", torch.uint8, dev)
    t = _vec(t, B * K, "t", torch.int32, dev)
    u_acc = _vec(u_acc, B * K, "u_acc", torch.float32, dev)
    u_res = _vec(u_res, B, "u_res", torch.float64, dev)
    max_len = 0
    if tokens is not None:
        if tokens.dim() != 2 or tokens.shape[0] != B:
            raise SpecVerifyError("tokens must be [B][max_len]")
        max_len = tokens.shape[1]
        _vec(tokens, B * max_len, "tokens", torch.int32, dev)
        _vec(lengths, B, "lengths", torch.int32, dev)
    n_out, next_out = _outputs(B, dev, n_out, next_out)
    w = _workspace(ws, B, K, V, dev, stream)
    rc = load().sv_verify_round(_ptr(mode), _ptr(p), ps, _ptr(q), qs, _ptr(t), _ptr(u_acc),
                                _ptr(u_res), B, K, V, _ptr(n_out), _ptr(next_out), _ptr(tokens),
                                _ptr(lengths), max_len, w.ptr, w.nbytes, _stream_handle(stream))
    _check(rc, "sv_verify_round")
    return n_out, next_out


class HostVerifier:
    """Verification of host-resident inputs through the public calls.  Inputs
    are pinned CPU tensors; (n_accepted, next_token) come back in pinned
    memory and each call waits for them.

    mapped=True (default): the inputs are handed to the library where they
    are; the kernels read them over the host link, and only the rows the rule
    needs (the residual pair or bonus row of a sampling sequence, the rows up
    to the first miss of a greedy one) cross it.  mapped=False: every call
    first copies all inputs into device buffers."""

    def __init__(self, B: int, K: int, V: int, device=None, sampling: bool = True,
                 mapped: bool = True):
        torch = _torch()
        dev = torch.device("cuda") if device is None else torch.device(device)
        self.B, self.K, self.V, self.device, self.mapped = B, K, V, dev, mapped
        self.sampling = sampling
        if not mapped:
            self.p = torch.empty(B, K + 1, V, dtype=torch.float32, device=dev)
            self.q = torch.empty(B, K, V, dtype=torch.float32, device=dev) if sampling else None
            self.t = torch.empty(B, K, dtype=torch.int32, device=dev)
            self.u_acc = torch.empty(B, K, dtype=torch.float32, device=dev)
            self.u_res = torch.empty(B, dtype=torch.float64, device=dev)
        self.n = torch.empty(B, dtype=torch.int32, device=dev)
        self.next = torch.empty(B, dtype=torch.int32, device=dev)
        self.n_host = torch.empty(B, dtype=torch.int32, pin_memory=True)
        self.next_host = torch.empty(B, dtype=torch.int32, pin_memory=True)
        self.ws = Workspace(B, K, V, dev)

    def h2d_bytes(self) -> int:
        """Bytes of input that crossed the host link in the last call: all of
        them when copying, else what the rule read (from its n_accepted)."""
        B, K, V = self.B, self.K, self.V
        if not self.mapped:
            n = (K + 1) * V * 4 * B + K * 4 * B
            if self.sampling:
                n += K * V * 4 * B + K * 4 * B + 8 * B
            return n
        total = 0
        for n in self.n_host.tolist():
            if self.sampling:
                rows = 8 * V if n < K else 4 * V
                total += rows + 64 * min(n + 1, K) + 8 * K + 8
            else:
                total += (n + 1) * 4 * V + 4 * K + 4 * min(n + 1, K)
        return total

    def d2h_bytes(self) -> int:
        return self.B * 8

    def _pinned(self, *xs):
        for x in xs:
            if x is not None and not x.is_pinned():
                raise SpecVerifyError("HostVerifier inputs must be pinned CPU tensors")

    def sample(self, p, q, t, u_acc, u_res):
        self._pinned(p, q, t, u_acc, u_res)
        if not self.mapped:
            self.p.copy_(p, non_blocking=True)
            self.q.copy_(q, non_blocking=True)
            self.t.copy_(t, non_blocking=True)
            self.u_acc.copy_(u_acc, non_blocking=True)
            self.u_res.copy_(u_res, non_blocking=True)
            p, q, t, u_acc, u_res = self.p, self.q, self.t, self.u_acc, self.u_res
        verify_sample(p, q, t, u_acc, u_res, ws=self.ws, n_out=self.n, next_out=self.next)
        return self._finish()

    def greedy(self, p, t):
        self._pinned(p, t)
        if not self.mapped:
            self.p.copy_(p, non_blocking=True)
            self.t.copy_(t, non_blocking=True)
            p, t = self.p, self.t
        verify_greedy(p, t, ws=self.ws, n_out=self.n, next_out=self.next)
        return self._finish()

    def _finish(self):
        torch = _torch()
        self.n_host.copy_(self.n, non_blocking=True)
        self.next_host.copy_(self.next, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        return self.n_host, self.next_host


# ---------------------------------------------------------------------------
# timeline of the item kernel (a library built with SV_TRACE=1)

TRACE_RECORDS = 2048 * 1024


def trace_reset(stream=None, lib=None):
    """Clears the trace buffer on the stream (a trace build; SpecVerifyError otherwise)."""
    _check((lib or load()).sv_trace_reset(_stream_handle(stream)), "sv_trace_reset")


def trace_read(stream=None, lib=None):
    """The recorded events as a uint64 array [N][2] (time in ns, event word),
    empty slots dropped; waits for the stream."""
    import numpy as np
    buf = np.zeros((TRACE_RECORDS, 2), dtype=np.uint64)
    n = ctypes.c_size_t(0)
    _check((lib or load()).sv_trace_read(buf.ctypes.data_as(ctypes.c_void_p), TRACE_RECORDS,
                                         ctypes.byref(n), _stream_handle(stream)),
           "sv_trace_read")
    buf = buf[:n.value]
    return buf[buf[:, 0] != 0]


def trace_summary(records) -> dict:
    """Where one traced launch's time went (``trace.summary``)."""
    return _trace.summary(records)


def trace_timeline(records) -> dict:
    """Per-launch summaries of several consecutive traced launches and the
    time between them (``trace.timeline``)."""
    return _trace.timeline(records)
