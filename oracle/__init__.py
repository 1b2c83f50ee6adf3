"""FP64 CPU oracle for chunked KDA (test infrastructure only).

This package is the yardstick the CUDA library is checked against.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``
may import it.  The product path (``linear_attention_chunked_gb300``) never imports it, and this
package imports nothing from the product.

The arithmetic lives in ``kda_oracle.c`` (plain C, double precision, token by token).  This
module only compiles it with gcc and marshals numpy arrays through ctypes.

Parity status of each function (what pins it, see tests/test_oracle_pins.py):
  * kda_fwd            -- worked examples, closed forms (pure decay, one-hot keys, exact read-back),
                          pack == per-document runs.
  * kda_bwd            -- central finite differences of L = sum(o*dO) + sum(ht*dht) on tiny inputs,
                          in g, raw, L2-norm and fast-decay forms.
  * fragment_summary   -- explicit matrix product of the per-token transitions at small d, and
                          S_out = M S_in + B against the token run; C against the token backward.
  * transfer_walk      -- associativity of the affine maps, and the walk against the unfragmented run.
  * conv1d.conv_fwd / conv1d.conv_bwd (the width-4 causal conv1d + SiLU ahead of q / k / v, plain
    numpy in FP64) -- a hand-worked example, SiLU and pure-shift closed forms, numpy.convolve,
    halo split invariance, central finite differences (tests/test_conv_pins.py; planted mistakes
    in tests/test_conv_mutants.py).
tests/test_oracle_mutants.py plants one plausible mistake at a time into a copy of kda_oracle.c
(``compile_source`` + ``using_build``) and checks that every such build fails at least one pin.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_kda.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """gcc, plain -O2, no fast-math: the one way every build of the oracle is made."""
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-std=c11", "-Wall", "-Wno-unused-result",
           "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into a shared library."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    compile_source(_SRC, tmp)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path):
    """Loads a build of kda_oracle.c and declares its entry points."""
    lib = ctypes.CDLL(path)
    i64, i32, dbl, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p
    lib.oracle_kda_fwd.argtypes = [i64, i32, i32, i32, p, p, p, p, p, p, p, p, p,
                                   ctypes.c_int, ctypes.c_int, dbl, dbl, p, p, ctypes.c_int]
    lib.oracle_kda_bwd.argtypes = [i64, i32, i32, i32, p, p, p, p, p, p, p, p, p,
                                   ctypes.c_int, ctypes.c_int, dbl, dbl, p, p,
                                   p, p, p, p, p, p, p, p, ctypes.c_int]
    lib.oracle_fragment_summary.argtypes = [i64, i32, i32, i32, p, p, p, p, p, p, p, p,
                                            ctypes.c_int, ctypes.c_int, dbl, dbl,
                                            ctypes.c_int, p, p, p, ctypes.c_int]
    lib.oracle_transfer_walk.argtypes = [i32, p, i32, i32, p, p, p, ctypes.c_int, p, p]
    for f in (lib.oracle_kda_fwd, lib.oracle_kda_bwd, lib.oracle_fragment_summary,
              lib.oracle_transfer_walk):
        f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


@contextlib.contextmanager
def using_build(path):
    """Runs the functions below on another build of kda_oracle.c (the planted-mistake tests)."""
    global _lib
    lib = _bind(path)
    with _lock:
        saved, _lib = _lib, lib
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _nthreads(n):
    return int(n) if n else (os.cpu_count() or 1)


def _f64(x, shape=None):
    if x is None:
        return None
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"oracle: expected shape {tuple(shape)}, got {a.shape}")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _cu(cu_seqlens):
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    if cu.ndim != 1 or cu.size < 1 or cu[0] != 0 or np.any(np.diff(cu) < 0):
        raise ValueError("oracle: cu_seqlens must start at 0 and be non-decreasing")
    return cu


class _Inputs:
    def __init__(self, q, k, v, beta, g_or_a, cu_seqlens, A_log, dt_bias, h0, raw):
        self.q = _f64(q)
        T, H, d = self.q.shape
        self.T, self.H, self.d = T, H, d
        self.k = _f64(k, (T, H, d))
        self.v = _f64(v, (T, H, d))
        self.beta = _f64(beta, (T, H))
        self.g = _f64(g_or_a, (T, H, d))
        self.cu = _cu(cu_seqlens)
        self.N = self.cu.size - 1
        if int(self.cu[-1]) != T:
            raise ValueError("oracle: cu_seqlens[-1] must equal T")
        self.raw = bool(raw)
        if self.raw:
            self.A_log = _f64(A_log, (H,))
            self.dt_bias = _f64(dt_bias, (H, d))
        else:
            self.A_log = None
            self.dt_bias = None
        self.h0 = _f64(h0, (self.N, H, d, d))

    def head(self):
        return (self.T, self.N, self.H, self.d, self.cu.ctypes.data_as(ctypes.c_void_p),
                _ptr(self.q), _ptr(self.k), _ptr(self.v), _ptr(self.beta), _ptr(self.g),
                _ptr(self.A_log), _ptr(self.dt_bias), _ptr(self.h0))


def kda_fwd(q, k, v, beta, g_or_a, cu_seqlens, *, raw=False, A_log=None, dt_bias=None, h0=None,
            l2norm=False, scale=1.0, eps=1e-6, nthreads=None):
    """Token-by-token forward.  Returns (o [T,H,d], ht [N,H,d,d]) as float64 numpy arrays."""
    x = _Inputs(q, k, v, beta, g_or_a, cu_seqlens, A_log, dt_bias, h0, raw)
    o = np.empty((x.T, x.H, x.d))
    ht = np.empty((x.N, x.H, x.d, x.d))
    rc = _load().oracle_kda_fwd(*x.head(), int(x.raw), int(bool(l2norm)), float(scale),
                                float(eps), _ptr(o), _ptr(ht), _nthreads(nthreads))
    if rc:
        raise RuntimeError(f"oracle_kda_fwd failed ({rc})")
    return o, ht


def kda_bwd(q, k, v, beta, g_or_a, cu_seqlens, dO, *, dht=None, raw=False, A_log=None,
            dt_bias=None, h0=None, l2norm=False, scale=1.0, eps=1e-6, nthreads=None):
    """Reverse-mode gradients of L = sum(o*dO) + sum(ht*dht).

    Returns a dict with dq, dk, dv [T,H,d], dbeta [T,H], dg (g form: dL/dg; raw form: dL/da)
    [T,H,d], dh0 [N,H,d,d], and in raw form dA_log [H] and ddt_bias [H,d]."""
    x = _Inputs(q, k, v, beta, g_or_a, cu_seqlens, A_log, dt_bias, h0, raw)
    dO = _f64(dO, (x.T, x.H, x.d))
    dht = _f64(dht, (x.N, x.H, x.d, x.d))
    out = {n: np.empty((x.T, x.H, x.d)) for n in ("dq", "dk", "dv", "dg")}
    out["dbeta"] = np.empty((x.T, x.H))
    out["dh0"] = np.empty((x.N, x.H, x.d, x.d))
    if x.raw:
        out["dA_log"] = np.empty((x.H,))
        out["ddt_bias"] = np.empty((x.H, x.d))
    rc = _load().oracle_kda_bwd(*x.head(), int(x.raw), int(bool(l2norm)), float(scale), float(eps),
                                _ptr(dO), _ptr(dht), _ptr(out["dq"]), _ptr(out["dk"]),
                                _ptr(out["dv"]), _ptr(out["dbeta"]), _ptr(out["dg"]),
                                _ptr(out.get("dA_log")), _ptr(out.get("ddt_bias")),
                                _ptr(out["dh0"]), _nthreads(nthreads))
    if rc:
        raise RuntimeError(f"oracle_kda_bwd failed ({rc})")
    return out


def fragment_summary(q, k, v, beta, g_or_a, cu_seqlens, *, mode=0, dO=None, raw=False, A_log=None,
                     dt_bias=None, l2norm=False, scale=1.0, eps=1e-6, nthreads=None):
    """Fragments are the documents of ``cu_seqlens``.

    mode 0 -> (M, B) each [F,H,d,d]; mode 1 -> C [F,H,d,d] (needs dO)."""
    x = _Inputs(q, k, v, beta, g_or_a, cu_seqlens, A_log, dt_bias, None, raw)
    F = x.N
    M = np.empty((F, x.H, x.d, x.d))
    BC = np.empty((F, x.H, x.d, x.d))
    if mode == 1:
        dO = _f64(dO, (x.T, x.H, x.d))
    head = x.head()[:-1]
    rc = _load().oracle_fragment_summary(*head, int(x.raw), int(bool(l2norm)), float(scale),
                                         float(eps), int(mode), _ptr(dO), _ptr(M), _ptr(BC),
                                         _nthreads(nthreads))
    if rc:
        raise RuntimeError(f"oracle_fragment_summary failed ({rc})")
    return (M, BC) if mode == 0 else BC


def transfer_walk(doc_frag, M, B, S0=None, *, reverse=False):
    """Returns (S_in [F,H,d,d], S_final [N,H,d,d]); see kda_oracle.c for the two directions."""
    doc_frag = _cu(doc_frag)
    M = _f64(M)
    F, H, d, _ = M.shape
    B = _f64(B, (F, H, d, d))
    N = doc_frag.size - 1
    S0 = _f64(S0, (N, H, d, d))
    S_in = np.empty((F, H, d, d))
    S_final = np.empty((N, H, d, d))
    rc = _load().oracle_transfer_walk(N, doc_frag.ctypes.data_as(ctypes.c_void_p), H, d, _ptr(M),
                                      _ptr(B), _ptr(S0), int(bool(reverse)), _ptr(S_in),
                                      _ptr(S_final))
    if rc:
        raise RuntimeError(f"oracle_transfer_walk failed ({rc})")
    return S_in, S_final
