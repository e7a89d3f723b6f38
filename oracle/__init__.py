"""FP64 CPU oracle for exact softmax attention (forward and backward).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (the CUDA library and its binding) never imports it,
and it imports nothing from the product path.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, OpenMP over
heads).  This module only compiles it, loads it with ctypes and marshals numpy
arrays.  The equations it follows are those of "Writing Speed-of-Light
Attention Backward Kernel for 5090 in CUDA", section "Mathematical
Formulation" (forward: S = QK^T/sqrt(d) + M, L = logsumexp rows, P = exp(S-L),
O = PV; backward: dV = P^T dO, dP = dO V^T, D = rowsum(dO o O),
dS = P o (dP - D), dQ = dS K/sqrt(d), dK = dS^T Q/sqrt(d)), with the caller's
``scale`` in place of 1/sqrt(d).

The sparse top-k attention with a shared latent key/value row (``dsa.py``,
numpy in double precision) is re-exported here as ``dsa_fwd`` / ``dsa_bwd``;
its pins are in ``tests/test_oracle_dsa.py``.

Parity pins: every function here is pinned by ``tests/test_oracle.py``
(finite differences of a scalar loss, the Q = 0 closed form, row-sum
invariants of P and dS, N = 1 and first-row special cases, shift and
permutation invariances, a numpy softmax cross-check and a pure-Python brute
force on tiny inputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_attn.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle C source into a shared library (gcc, OpenMP)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load_library(path: str):
    """Load an oracle shared library and declare its signatures."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lp = ctypes.POINTER(ctypes.c_long)
    L, D, I = ctypes.c_long, ctypes.c_double, ctypes.c_int
    lib.oracle_attn_fwd.argtypes = [L, L, L, D, I, dp, dp, dp, dp, dp]
    lib.oracle_attn_bwd.argtypes = [L, L, L, D, I, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp]
    lib.oracle_attn_rows.argtypes = [L, L, D, I, dp, dp, dp, dp, L, lp, dp, dp, dp]
    lib.oracle_attn_probs.argtypes = [L, L, D, I, dp, dp, dp, dp, dp, dp]
    lib.oracle_attn_bwd_rowset.argtypes = [L, L, D, I, dp, dp, dp, dp, L, lp, dp, dp, dp]
    for f in (lib.oracle_attn_fwd, lib.oracle_attn_bwd, lib.oracle_attn_rows,
              lib.oracle_attn_probs, lib.oracle_attn_bwd_rowset):
        f.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
        return _lib


def use_library(lib):
    """Swap the loaded library (tests load deliberately broken builds of the
    oracle to show that the pins catch them); returns the previous one."""
    global _lib
    with _lock:
        prev, _lib = _lib, lib
        return prev


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _heads(x: np.ndarray):
    """View [..., N, d] as [BH, N, d]."""
    if x.ndim < 2:
        raise ValueError("expected [..., N, d]")
    lead = x.shape[:-2]
    bh = int(np.prod(lead)) if lead else 1
    return x.reshape(bh, x.shape[-2], x.shape[-1]), lead


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def attn_fwd(q, k, v, scale: float, causal: bool):
    """Forward over all heads.  q, k, v: [..., N, d].  Returns (O, L)."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    qh, lead = _heads(q)
    BH, N, d = qh.shape
    o = np.empty_like(qh)
    lse = np.empty((BH, N), dtype=np.float64)
    rc = lib.oracle_attn_fwd(BH, N, d, float(scale), int(bool(causal)), _ptr(qh),
                             _ptr(_heads(k)[0]), _ptr(_heads(v)[0]), _ptr(o), _ptr(lse))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd failed ({rc})")
    return o.reshape(q.shape), lse.reshape(lead + (N,))


def attn_bwd(q, k, v, dout, scale: float, causal: bool):
    """Forward + backward over all heads.  Returns dict of dq, dk, dv, o, lse, delta."""
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    qh, lead = _heads(q)
    BH, N, d = qh.shape
    dq, dk, dv, o = (np.empty_like(qh) for _ in range(4))
    lse = np.empty((BH, N), dtype=np.float64)
    delta = np.empty((BH, N), dtype=np.float64)
    rc = lib.oracle_attn_bwd(BH, N, d, float(scale), int(bool(causal)), _ptr(qh),
                             _ptr(_heads(k)[0]), _ptr(_heads(v)[0]), _ptr(_heads(dout)[0]),
                             _ptr(dq), _ptr(dk), _ptr(dv), _ptr(o), _ptr(lse), _ptr(delta))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd failed ({rc})")
    shp = q.shape
    return dict(dq=dq.reshape(shp), dk=dk.reshape(shp), dv=dv.reshape(shp),
                o=o.reshape(shp), lse=lse.reshape(lead + (N,)),
                delta=delta.reshape(lead + (N,)))


def attn_rows(q, k, v, rows, scale: float, causal: bool, dout=None):
    """Selected query rows of ONE head (q, k, v, dout: [N, d]).

    Returns (O_rows [n, d], L_rows [n], dQ_rows [n, d] or None)."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, d = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.shape[0]
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    dq = None
    dptr = None
    if dout is not None:
        dout = _f64(dout)
        dq = np.empty((n, d), dtype=np.float64)
        dptr = dout
    rc = lib.oracle_attn_rows(N, d, float(scale), int(bool(causal)), _ptr(q), _ptr(k), _ptr(v),
                              _ptr(dptr), n, rows.ctypes.data_as(ctypes.POINTER(ctypes.c_long)),
                              _ptr(o), _ptr(lse), _ptr(dq))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_rows failed ({rc})")
    return o, lse, dq


def attn_bwd_rowset(q, k, v, dout, rows, scale: float, causal: bool):
    """Forward + backward of ONE head ([N, d] inputs) restricted to query rows
    `rows`: returns (dQ_rows [n, d], dK_part [N, d], dV_part [N, d]) where the
    parts are those rows' contributions to dK and dV.  Single-threaded."""
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    N, d = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.shape[0]
    dq = np.empty((n, d), dtype=np.float64)
    dk = np.empty((N, d), dtype=np.float64)
    dv = np.empty((N, d), dtype=np.float64)
    rc = lib.oracle_attn_bwd_rowset(N, d, float(scale), int(bool(causal)), _ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                    n, rows.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), _ptr(dq), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd_rowset failed ({rc})")
    return dq, dk, dv


def attn_probs(q, k, v, scale: float, causal: bool, dout=None):
    """P (and dS if dout is given) of ONE head, each [N, N]."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, d = q.shape
    P = np.empty((N, N), dtype=np.float64)
    dS = np.empty((N, N), dtype=np.float64) if dout is not None else None
    rc = lib.oracle_attn_probs(N, d, float(scale), int(bool(causal)), _ptr(q), _ptr(k), _ptr(v),
                               _ptr(_f64(dout) if dout is not None else None), _ptr(P), _ptr(dS))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_probs failed ({rc})")
    return P, dS


from .dsa import dsa_bwd, dsa_fwd  # noqa: E402  (numpy; no C build needed)


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
