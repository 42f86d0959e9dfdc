"""Python face of the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg
of the benchmark may import this module; the product path never does.  It
shares no code with the CUDA library.  All arrays are numpy float64 (exact
images of the bf16 inputs); the C side is plain single-threaded loops.

Each function follows the pages as documented in ``oracle.c``: per-head RMSNorm
then rotary embedding of q and k, cache append, causal grouped-query softmax
attention (dryft-flash-infer agent guide, "Where the wins are"), cache reset
per generate call (same guide, "What is measured").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc (no FMA contraction, plain -O2)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(
                ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-shared",
                 "-fPIC", _SRC, "-o", tmp, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


class _Geom(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
                ("D", ctypes.c_int), ("cap", ctypes.c_int),
                ("theta", ctypes.c_double), ("eps", ctypes.c_double)]


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_rmsnorm.argtypes = [ctypes.c_int, _dp, _dp, ctypes.c_double, _dp]
        lib.oracle_rmsnorm.restype = None
        lib.oracle_rope.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double, _dp, _dp]
        lib.oracle_rope.restype = None
        lib.oracle_attend.argtypes = [ctypes.c_int, ctypes.c_int, _dp, _dp, _dp, ctypes.c_long,
                                      _dp, _dp]
        lib.oracle_attend.restype = ctypes.c_int
        g = ctypes.POINTER(_Geom)
        lib.oracle_prefill_transform.argtypes = [g, _ip, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _ip]
        lib.oracle_prefill_transform.restype = ctypes.c_int
        lib.oracle_prefill_row.argtypes = [g, ctypes.c_int, ctypes.c_int, ctypes.c_int, _dp, _dp,
                                           _dp, _dp]
        lib.oracle_prefill_row.restype = ctypes.c_int
        lib.oracle_prefill.argtypes = [g, _ip, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _ip, _dp]
        lib.oracle_prefill.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [g, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _ip, _dp, _dp]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_decode_transform.argtypes = [g, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _ip, _dp]
        lib.oracle_decode_transform.restype = ctypes.c_int
        lib.oracle_reset.argtypes = [g, _ip]
        lib.oracle_reset.restype = None
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: np.ndarray):
    return a.ctypes.data_as(_dp)


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise OracleError(f"{what} failed with oracle status {rc}")


def rmsnorm(x, w, eps: float) -> np.ndarray:
    """y = w * x / sqrt(mean(x^2) + eps) for one head vector."""
    x, w = _f64(x), _f64(w)
    y = np.empty_like(x)
    _load().oracle_rmsnorm(x.size, _p(x), _p(w), eps, _p(y))
    return y


def rope(x, pos: float, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding of one head vector at position ``pos``."""
    x = _f64(x)
    y = np.empty_like(x)
    _load().oracle_rope(x.size, float(pos), float(theta), _p(x), _p(y))
    return y


def attend(q, K, V):
    """Softmax attention of q[D] over K[n][D], V[n][D]; returns (out[D], p[n])."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    n, D = K.shape
    out = np.empty(D)
    p = np.empty(n)
    _check(_load().oracle_attend(D, n, _p(q), _p(K), _p(V), D, _p(out), _p(p)), "attend")
    return out, p


@dataclass(frozen=True)
class Geometry:
    B: int
    Hq: int
    Hkv: int
    D: int
    cap: int
    theta: float = 1e6
    eps: float = 1e-6


class OracleLayer:
    """One attention layer's fp64 cache (Kc, Vc: [B][Hkv][cap][D]) and lengths."""

    def __init__(self, geom: Geometry):
        self.g = geom
        self._cg = _Geom(geom.B, geom.Hq, geom.Hkv, geom.D, geom.cap, geom.theta, geom.eps)
        self.Kc = np.zeros((geom.B, geom.Hkv, geom.cap, geom.D))
        self.Vc = np.zeros_like(self.Kc)
        self.lens = np.zeros(geom.B, dtype=np.int32)

    def reset(self) -> None:
        _load().oracle_reset(ctypes.byref(self._cg), self.lens.ctypes.data_as(_ip))

    def set_cache(self, K, V, lens) -> None:
        """Load raw cache contents (e.g. a pre-filled cache) and lengths."""
        self.Kc[...] = _f64(K)
        self.Vc[...] = _f64(V)
        self.lens[...] = np.asarray(lens, dtype=np.int32)

    def prefill_transform(self, plen, q, k, v, wq, wk) -> np.ndarray:
        g = self.g
        plen = np.ascontiguousarray(plen, dtype=np.int32)
        q, k, v, wq, wk = map(_f64, (q, k, v, wq, wk))
        qp = np.empty_like(q)
        rc = _load().oracle_prefill_transform(
            ctypes.byref(self._cg), plen.ctypes.data_as(_ip), _p(q), _p(k), _p(v), _p(wq), _p(wk),
            _p(qp), _p(self.Kc), _p(self.Vc), self.lens.ctypes.data_as(_ip))
        _check(rc, "prefill_transform")
        return qp

    def prefill_row(self, b: int, h: int, i: int, qp_row) -> np.ndarray:
        qp_row = _f64(qp_row)
        out = np.empty(self.g.D)
        rc = _load().oracle_prefill_row(ctypes.byref(self._cg), b, h, i, _p(qp_row), _p(self.Kc),
                                        _p(self.Vc), _p(out))
        _check(rc, "prefill_row")
        return out

    def prefill(self, plen, q, k, v, wq, wk):
        plen = np.ascontiguousarray(plen, dtype=np.int32)
        q, k, v, wq, wk = map(_f64, (q, k, v, wq, wk))
        qp = np.empty_like(q)
        out = np.empty_like(q)
        rc = _load().oracle_prefill(
            ctypes.byref(self._cg), plen.ctypes.data_as(_ip), _p(q), _p(k), _p(v), _p(wq), _p(wk),
            _p(qp), _p(self.Kc), _p(self.Vc), self.lens.ctypes.data_as(_ip), _p(out))
        _check(rc, "prefill")
        return qp, out

    def decode_transform(self, q, k, v, wq, wk) -> np.ndarray:
        """Norm + rotate the new tokens, append them; no attention.  Returns q'."""
        q, k, v, wq, wk = map(_f64, (q, k, v, wq, wk))
        qp = np.empty_like(q)
        rc = _load().oracle_decode_transform(
            ctypes.byref(self._cg), _p(q), _p(k), _p(v), _p(wq), _p(wk), _p(self.Kc), _p(self.Vc),
            self.lens.ctypes.data_as(_ip), _p(qp))
        _check(rc, "decode_transform")
        return qp

    def attend_cached(self, b: int, h: int, qp_row) -> np.ndarray:
        """Attention of a query of head h over all cached slots of sequence b."""
        G = self.g.Hq // self.g.Hkv
        n = int(self.lens[b])
        out, _ = attend(qp_row, self.Kc[b, h // G, :n], self.Vc[b, h // G, :n])
        return out

    def decode(self, q, k, v, wq, wk):
        q, k, v, wq, wk = map(_f64, (q, k, v, wq, wk))
        qp = np.empty_like(q)
        out = np.empty_like(q)
        rc = _load().oracle_decode(
            ctypes.byref(self._cg), _p(q), _p(k), _p(v), _p(wq), _p(wk), _p(self.Kc), _p(self.Vc),
            self.lens.ctypes.data_as(_ip), _p(qp), _p(out))
        _check(rc, "decode")
        return qp, out
