"""CPU oracle for batched speculative-decoding verification (test infrastructure).

TEST INFRASTRUCTURE ONLY: the product library never imports, links or calls
anything here.  Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg use it.

The arithmetic lives in ``oracle.c`` (plain C11, fp64 masses, compiled without
fast-math or FP contraction) and follows the "spec-verify" page, section
"Method" (greedy and Leviathan/Chen sampling rules) and section "Correctness"
(unnormalised masses summed exactly).  This module only builds that file with
gcc and marshals numpy arrays to it.  Every function is pinned by
``tests/test_oracle_pins.py`` against brute-force enumeration with exact
rationals, closed forms, the analytic accepted-length law and plain greedy
decoding of a toy target; ``tests/test_oracle_mutants.py`` shows that planted
mistakes in ``oracle.c`` fail those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle_sv.so")

STATUS_BAD_TOKEN = 1
STATUS_ZERO_MASS = 2
STATUS_OVERFLOW = 4
STATUS_BAD_MODE = 8

CFLAGS = ["-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
          "-pthread", "-Wall", "-Wextra"]


def compile_source(src: str, out: str) -> str:
    """Compiles an oracle C source into a shared library at ``out``."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compiles oracle.c into liboracle_sv.so (gcc -O2, no fast-math)."""
    if (not force and os.path.exists(LIBRARY)
            and os.path.getmtime(LIBRARY) >= os.path.getmtime(SOURCE)):
        return LIBRARY
    return compile_source(SOURCE, LIBRARY)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _rows(a, rows_per_seq, name):
    """(contiguous float32 array, B, V, row stride) of a [B][rows][V] array."""
    a = _f32(a)
    if a.ndim == 2:
        a = a[None]
    if a.ndim != 3 or a.shape[1] != rows_per_seq:
        raise ValueError(f"{name}: expected [B][{rows_per_seq}][V], got {a.shape}")
    return a, a.shape[0], a.shape[2], a.shape[2]


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        i32 = ctypes.c_int
        lib.orc_argmax_lowest.argtypes = [P, i64]
        lib.orc_argmax_lowest.restype = i64
        lib.orc_icdf.argtypes = [P, i64, ctypes.c_double]
        lib.orc_icdf.restype = i64
        lib.orc_residual_cumsum.argtypes = [P, P, i64, P]
        lib.orc_residual_cumsum.restype = ctypes.c_double
        lib.orc_verify_greedy.argtypes = [P, i64, P, i32, i32, i64, P, P, P, i32]
        lib.orc_verify_greedy.restype = i32
        lib.orc_verify_sample.argtypes = [P, i64, P, i64, P, P, P, i32, i32, i64,
                                          P, P, P, i32]
        lib.orc_verify_sample.restype = i32
        lib.orc_verify_round.argtypes = [P, P, i64, P, i64, P, P, P, i32, i32, i64,
                                         P, P, P, i32]
        lib.orc_verify_round.restype = i32
        lib.orc_commit.argtypes = [P, i32, i32, P, P, P, P, i32, P]
        lib.orc_alpha.argtypes = [P, i64, P, i64, i32, i32, i64, P, P]
        lib.orc_alpha.restype = None
        lib.orc_softmax.argtypes = [P, i64, ctypes.c_double, P]
        lib.orc_softmax.restype = None
        lib.orc_verify_sample_logits.argtypes = [P, i64, P, i64, P, P, P, i32, i32, i64,
                                                 ctypes.c_double, P, P, P]
        lib.orc_verify_sample_logits.restype = ctypes.c_int
        lib.orc_commit.restype = None
        self.lib = lib
        self.path = path

    def argmax_lowest(self, row) -> int:
        row = _f32(row).ravel()
        return int(self.lib.orc_argmax_lowest(_ptr(row), row.size))

    def icdf(self, r, u: float) -> int:
        """Smallest v whose fp64 running sum of r exceeds u*sum(r); -1 if the sum is 0."""
        r = np.ascontiguousarray(r, dtype=np.float64).ravel()
        return int(self.lib.orc_icdf(_ptr(r), r.size, float(u)))

    def residual_cumsum(self, p_row, q_row=None):
        """Running fp64 sums of max(0, p - q) (of p when q is None) and their total."""
        p_row = _f32(p_row).ravel()
        q_row = None if q_row is None else _f32(q_row).ravel()
        C = np.empty(p_row.size, dtype=np.float64)
        R = self.lib.orc_residual_cumsum(_ptr(p_row), _ptr(q_row), p_row.size, _ptr(C))
        return C, float(R)

    @staticmethod
    def _outputs(B):
        return (np.empty(B, dtype=np.int32), np.empty(B, dtype=np.int32),
                np.zeros(1, dtype=np.uint32))

    def verify_greedy(self, p, t, nthreads: int = 1):
        """p [B][K+1][V] f32, t [B][K] -> (n_accepted, next_token, status bits)."""
        t = np.ascontiguousarray(t, dtype=np.int32)
        K = t.shape[-1]
        p, B, V, ps = _rows(p, K + 1, "p")
        t = t.reshape(B, K)
        n, nxt, st = self._outputs(B)
        rc = self.lib.orc_verify_greedy(_ptr(p), ps, _ptr(t), B, K, V, _ptr(n), _ptr(nxt),
                                        _ptr(st), nthreads)
        if rc != 0:
            raise MemoryError("oracle: out of host memory")
        return n, nxt, int(st[0])

    def verify_sample(self, p, q, t, u_acc, u_res, nthreads: int = 1):
        """p [B][K+1][V], q [B][K][V], t [B][K], u_acc [B][K] f32, u_res [B] f64
        -> (n_accepted, next_token, status bits)."""
        t = np.ascontiguousarray(t, dtype=np.int32)
        K = t.shape[-1]
        p, B, V, ps = _rows(p, K + 1, "p")
        q, Bq, Vq, qs = _rows(q, K, "q")
        if (Bq, Vq) != (B, V):
            raise ValueError("q shape does not match p")
        t = t.reshape(B, K)
        ua = np.ascontiguousarray(u_acc, dtype=np.float32).reshape(B, K)
        ur = np.ascontiguousarray(u_res, dtype=np.float64).reshape(B)
        n, nxt, st = self._outputs(B)
        rc = self.lib.orc_verify_sample(_ptr(p), ps, _ptr(q), qs, _ptr(t), _ptr(ua),
                                        _ptr(ur), B, K, V, _ptr(n), _ptr(nxt), _ptr(st),
                                        nthreads)
        if rc != 0:
            raise MemoryError("oracle: out of host memory")
        return n, nxt, int(st[0])

    def verify_round(self, mode, p, q, t, u_acc, u_res, nthreads: int = 1):
        """Mixed round: mode [B] u8 (0 greedy, 1 sampling) picks the rule per sequence."""
        t = np.ascontiguousarray(t, dtype=np.int32)
        K = t.shape[-1]
        p, B, V, ps = _rows(p, K + 1, "p")
        q, Bq, Vq, qs = _rows(q, K, "q")
        if (Bq, Vq) != (B, V):
            raise ValueError("q shape does not match p")
        t = t.reshape(B, K)
        md = np.ascontiguousarray(mode, dtype=np.uint8).reshape(B)
        ua = np.ascontiguousarray(u_acc, dtype=np.float32).reshape(B, K)
        ur = np.ascontiguousarray(u_res, dtype=np.float64).reshape(B)
        n, nxt, st = self._outputs(B)
        rc = self.lib.orc_verify_round(_ptr(md), _ptr(p), ps, _ptr(q), qs, _ptr(t),
                                       _ptr(ua), _ptr(ur), B, K, V, _ptr(n), _ptr(nxt),
                                       _ptr(st), nthreads)
        if rc != 0:
            raise MemoryError("oracle: out of host memory")
        return n, nxt, int(st[0])

    def alpha(self, p, q, K=None):
        """p [B][K+1][V], q [B][K][V] -> (alpha [B][K] f64, expected accepted
        length [B] f64)."""
        q = _f32(q)
        if q.ndim == 2:
            q = q[None]
        K = q.shape[1] if K is None else K
        p, B, V, ps = _rows(p, K + 1, "p")
        q, Bq, Vq, qs = _rows(q, K, "q")
        if (Bq, Vq) != (B, V):
            raise ValueError("q shape does not match p")
        a = np.empty((B, K), dtype=np.float64)
        e = np.empty(B, dtype=np.float64)
        self.lib.orc_alpha(_ptr(p), ps, _ptr(q), qs, B, K, V, _ptr(a), _ptr(e))
        return a, e

    def softmax(self, z, tau: float):
        """fp64 temperature softmax of one f32 logit row."""
        z = _f32(z).reshape(-1)
        out = np.empty(z.shape[0], dtype=np.float64)
        self.lib.orc_softmax(_ptr(z), z.shape[0], float(tau), _ptr(out))
        return out

    def verify_sample_logits(self, zp, zq, t, u_acc, u_res, tau: float):
        """Sampling verification from logits zp [B][K+1][V], zq [B][K][V] with
        temperature tau -> (n_accepted, next_token, status bits)."""
        t = np.ascontiguousarray(t, dtype=np.int32)
        K = t.shape[-1]
        zp, B, V, ps = _rows(zp, K + 1, "zp")
        zq, Bq, Vq, qs = _rows(zq, K, "zq")
        if (Bq, Vq) != (B, V):
            raise ValueError("zq shape does not match zp")
        t = t.reshape(B, K)
        ua = np.ascontiguousarray(u_acc, dtype=np.float32).reshape(B, K)
        ur = np.ascontiguousarray(u_res, dtype=np.float64).reshape(B)
        n, nxt, st = self._outputs(B)
        rc = self.lib.orc_verify_sample_logits(_ptr(zp), ps, _ptr(zq), qs, _ptr(t), _ptr(ua),
                                               _ptr(ur), B, K, V, float(tau), _ptr(n),
                                               _ptr(nxt), _ptr(st))
        if rc == -1:
            raise ValueError("temperature must be a positive finite number")
        if rc != 0:
            raise MemoryError("oracle: out of host memory")
        return n, nxt, int(st[0])

    def commit(self, t, n, nxt, tokens, lengths):
        """Appends t[b][:n[b]] and next[b] to tokens[b] in place; returns status bits."""
        t = np.ascontiguousarray(t, dtype=np.int32)
        B, K = t.shape
        n = np.ascontiguousarray(n, dtype=np.int32)
        nxt = np.ascontiguousarray(nxt, dtype=np.int32)
        if tokens.dtype != np.int32 or not tokens.flags.c_contiguous:
            raise ValueError("tokens must be a C-contiguous int32 array")
        if lengths.dtype != np.int32 or not lengths.flags.c_contiguous:
            raise ValueError("lengths must be a C-contiguous int32 array")
        st = np.zeros(1, dtype=np.uint32)
        self.lib.orc_commit(_ptr(t), B, K, _ptr(n), _ptr(nxt), _ptr(tokens), _ptr(lengths),
                            tokens.shape[1], _ptr(st))
        return int(st[0])


_lock = threading.Lock()
_default = None


def get() -> Oracle:
    """The oracle built from oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def argmax_lowest(row):
    return get().argmax_lowest(row)


def icdf(r, u):
    return get().icdf(r, u)


def residual_cumsum(p_row, q_row=None):
    return get().residual_cumsum(p_row, q_row)


def verify_greedy(p, t, nthreads=1):
    return get().verify_greedy(p, t, nthreads)


def verify_sample(p, q, t, u_acc, u_res, nthreads=1):
    return get().verify_sample(p, q, t, u_acc, u_res, nthreads)


def verify_round(mode, p, q, t, u_acc, u_res, nthreads=1):
    return get().verify_round(mode, p, q, t, u_acc, u_res, nthreads)


def commit(t, n, nxt, tokens, lengths):
    return get().commit(t, n, nxt, tokens, lengths)


def alpha(p, q, K=None):
    return get().alpha(p, q, K)


def softmax(z, tau):
    return get().softmax(z, tau)


def verify_sample_logits(zp, zq, t, u_acc, u_res, tau):
    return get().verify_sample_logits(zp, zq, t, u_acc, u_res, tau)
