"""Test infrastructure only: fp64 CPU oracle for the gated delta rule.

Only the tests, the package's ``smoke()`` check and the benchmark's CPU
baseline leg may import this package.  The library's product path never does
and shares no code with it.

``gdn_oracle.cpp`` holds the arithmetic: the token-by-token recurrence of the
Gated DeltaNet / Kimi Delta Attention mixers (Primus hybrid-LLM pretraining
blog, section "How hybrid models are defined in Primus") in fp64 and its
reverse-mode backward.  This module compiles it with the host compiler and
wraps it with ctypes.  Every function takes arrays in the library's layout
(token tensors ``[B,T,H,D]``, states ``[B,H,dk,dv]``) and returns fp64 numpy
arrays.

Parity status of each function is recorded next to its pins in
``tests/test_oracle.py``: ``fwd`` and ``bwd`` are pinned for GDN and KDA, and
for the Mamba2 mixer (``delta=False``: the scalar-gated state without the
delta rule).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.cpp")
_LIB = os.path.join(_HERE, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gdn_oracle.cpp`` into ``libgdn_oracle.so`` (portable flags only)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.oracle_fwd.argtypes = [i] * 6 + [dp] * 8 + [i]
    lib.oracle_fwd.restype = i
    lib.oracle_bwd.argtypes = [i] * 6 + [dp] * 14 + [i]
    lib.oracle_bwd.restype = i
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _as64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (any dtype, any device)
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    if x is None:
        return None
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _dims(q, v, g, kda):
    B, T, H, dk = q.shape
    dv = v.shape[3]
    want_g = (B, T, H, dk) if kda else (B, T, H)
    if tuple(g.shape) != want_g:
        raise ValueError(f"g has shape {g.shape}, expected {want_g}")
    return B, T, H, dk, dv


def _mode(kda, delta):
    return int(bool(kda)) | (0 if delta else 2)


def fwd(q, k, v, g, beta, h0=None, kda=False, nthreads=0, _lib_override=None, delta=True):
    """Token-recurrence forward.  Returns ``(o, ht)`` as fp64 arrays.

    ``delta=False`` drops the delta rule (the state only accumulates
    ``beta k v^T``): the Mamba2 mixer of the same mixer list."""
    q, k, v, g, beta, h0 = map(_as64, (q, k, v, g, beta, h0))
    B, T, H, dk, dv = _dims(q, v, g, kda)
    o = np.zeros((B, T, H, dv))
    ht = np.zeros((B, H, dk, dv))
    rc = (_lib_override or _load()).oracle_fwd(_mode(kda, delta), B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                            _ptr(beta), _ptr(h0), _ptr(o), _ptr(ht), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_fwd failed ({rc})")
    return o, ht


def bwd(q, k, v, g, beta, h0, do, dht=None, kda=False, nthreads=0, _lib_override=None,
        delta=True):
    """Reverse-mode backward.  Returns a dict of fp64 gradients.

    Keys: ``dq, dk, dv, dg, dbeta, dh0`` (``dh0`` is the gradient with respect
    to the initial state, whether or not ``h0`` was given).
    """
    q, k, v, g, beta, h0, do, dht = map(_as64, (q, k, v, g, beta, h0, do, dht))
    B, T, H, dk, dv = _dims(q, v, g, kda)
    out = {
        "dq": np.zeros((B, T, H, dk)),
        "dk": np.zeros((B, T, H, dk)),
        "dv": np.zeros((B, T, H, dv)),
        "dg": np.zeros(g.shape),
        "dbeta": np.zeros((B, T, H)),
        "dh0": np.zeros((B, H, dk, dv)),
    }
    rc = (_lib_override or _load()).oracle_bwd(_mode(kda, delta), B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                            _ptr(beta), _ptr(h0), _ptr(do), _ptr(dht), _ptr(out["dq"]),
                            _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]),
                            _ptr(out["dbeta"]), _ptr(out["dh0"]), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_bwd failed ({rc})")
    return out


class Variant:
    """The same wrappers bound to another build of the oracle source.

    Used by the mutation test, which compiles copies of ``gdn_oracle.cpp``
    with a planted mistake and checks that the pins reject each of them."""

    def __init__(self, so_path):
        self._lib = _bind(so_path)

    def fwd(self, *a, **kw):
        return fwd(*a, _lib_override=self._lib, **kw)

    def bwd(self, *a, **kw):
        return bwd(*a, _lib_override=self._lib, **kw)
