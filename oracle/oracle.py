"""Python face of the fp64 recurrent oracle (``gdn_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg of the
benchmark may import this module; the product path never does.

The oracle follows the gated delta rule token by token (FlashQLA pages, "GDN chunked
prefill optimisation" section): decay the state by exp(g_t), read u = h^T k_t, write
beta_t (v_t - u) along k_t, emit o_t = scale h^T q_t.  Arrays are numpy fp64 in the packed
layout (tokens of all sequences back to back):

    q, k [TT, Hqk, K]   v [TT, Hv, V]   g, beta [TT, Hv]   h0, ht [N, Hv, K, V]
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
NO_ERASE = 1

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags only: it must build on x86 and Arm)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int64)
        i = ctypes.c_int
        lib.oracle_fwd.argtypes = [i, ip, i, i, i, i, dp, dp, dp, dp, dp, ctypes.c_double,
                                   dp, dp, dp, i, i]
        lib.oracle_fwd.restype = i
        lib.oracle_bwd.argtypes = [i, ip, i, i, i, i, dp, dp, dp, dp, dp, ctypes.c_double,
                                   dp, dp, dp, dp, dp, dp, dp, dp, dp, i, i]
        lib.oracle_bwd.restype = i
        lib.oracle_max_threads.restype = i
        _lib = lib
    return _lib


def _d(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # a torch tensor on the CPU
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _cu(cu_seqlens, B, T):
    if cu_seqlens is None:
        return np.arange(B + 1, dtype=np.int64) * T
    if hasattr(cu_seqlens, "detach"):
        cu_seqlens = cu_seqlens.detach().cpu().numpy()
    return np.ascontiguousarray(cu_seqlens, dtype=np.int64)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def fwd(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, flags=0, threads=None):
    """Forward recurrence.  q/k [B,T,Hqk,K], v [B,T,Hv,V], g/beta [B,T,Hv] (B=1 when
    cu_seqlens is given).  Returns (o [B,T,Hv,V], ht [N,Hv,K,V]) in fp64."""
    q, k, v, g, beta, h0 = (_f64(x) for x in (q, k, v, g, beta, h0))
    B, T, Hqk, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    cu = _cu(cu_seqlens, B, T)
    N = len(cu) - 1
    o = np.zeros((B, T, Hv, V))
    ht = np.zeros((N, Hv, K, V))
    lib = _load()
    rc = lib.oracle_fwd(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), Hqk, Hv, K, V,
                        _d(q), _d(k), _d(v), _d(g), _d(beta), float(scale), _d(h0), _d(o),
                        _d(ht), int(flags), int(threads or max_threads()))
    if rc != 0:
        raise ValueError(f"oracle_fwd rejected its arguments (rc={rc})")
    return o, ht


def bwd(q, k, v, g, beta, scale, dO, h0=None, dht=None, cu_seqlens=None, flags=0,
        threads=None):
    """Reverse mode of :func:`fwd`.  Returns dq, dk, dv, dg, dbeta, dh0 in fp64."""
    q, k, v, g, beta, h0, dO, dht = (_f64(x) for x in (q, k, v, g, beta, h0, dO, dht))
    B, T, Hqk, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    cu = _cu(cu_seqlens, B, T)
    N = len(cu) - 1
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dg = np.zeros_like(g)
    db = np.zeros_like(beta)
    dh0 = np.zeros((N, Hv, K, V))
    lib = _load()
    rc = lib.oracle_bwd(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), Hqk, Hv, K, V,
                        _d(q), _d(k), _d(v), _d(g), _d(beta), float(scale), _d(h0), _d(dO),
                        _d(dht), _d(dq), _d(dk), _d(dv), _d(dg), _d(db), _d(dh0), int(flags),
                        int(threads or max_threads()))
    if rc != 0:
        raise ValueError(f"oracle_bwd failed (rc={rc})")
    return dq, dk, dv, dg, db, dh0
