"""float64 CPU oracle for Kimi Delta Attention (KDA).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never calls it and shares no code with it.

The arithmetic lives in ``kda_oracle.c`` (plain C, float64, OpenMP over heads);
this module compiles it with gcc on first use (or from ``build()``) and wraps
it for numpy arrays.  Sources for every function are cited in the C file:
"KDA 训练 → 推理 手写实现" (K3 README) tables 实现路线表 (rows L1, L2, L6) and
关键约束 / 风险点, and the "KDA CUDA Trainer" README section on the mixing module.

Parity of every function here is pinned by ``tests/test_oracle_*.py`` against
closed forms, invariants and finite differences (nothing is "parity unpinned").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (OpenMP if available)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, d, p = ctypes.c_int, ctypes.c_double, _D
            lib.kda_oracle_fwd_recurrent.argtypes = [i] * 6 + [d] + [p] * 8
            lib.kda_oracle_bwd_recurrent.argtypes = [i] * 6 + [d] + [p] * 14
            lib.kda_oracle_fwd_chunked.argtypes = [i] * 6 + [d, i] + [p] * 8
            lib.kda_oracle_l2norm.argtypes = [ctypes.c_long, i, p, p]
            lib.kda_oracle_l2norm_bwd.argtypes = [ctypes.c_long, i, p, p, p]
            lib.kda_oracle_chunk_wy.argtypes = [i] * 3 + [p] * 11
            lib.kda_oracle_step.argtypes = [i] * 5 + [d] + [p] * 7
            lib.kda_oracle_num_threads.restype = i
            for f in ("kda_oracle_fwd_recurrent", "kda_oracle_bwd_recurrent",
                      "kda_oracle_fwd_chunked", "kda_oracle_chunk_wy",
                      "kda_oracle_step", "kda_oracle_l2norm", "kda_oracle_l2norm_bwd"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().kda_oracle_num_threads())


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    if x is None:
        return None
    return x.ctypes.data_as(_D)


def _dims(q, v, g):
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    assert g.shape == (B, T, HV, K) and HV % H == 0
    return B, T, H, HV, K, V


def fwd_recurrent(q, k, v, g, beta, scale=None, h0=None):
    """Token-by-token forward.  Returns (o [B,T,HV,V], ht [B,HV,K,V])."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    B, T, H, HV, K, V = _dims(q, v, g)
    scale = K ** -0.5 if scale is None else float(scale)
    h0 = None if h0 is None else _f64(h0)
    o = np.zeros((B, T, HV, V))
    ht = np.zeros((B, HV, K, V))
    _load().kda_oracle_fwd_recurrent(B, T, H, HV, K, V, scale, _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(ht))
    return o, ht


def bwd_recurrent(q, k, v, g, beta, do, scale=None, h0=None, dht=None):
    """Reverse-time backward.  Returns dict dq, dk (at H), dv, dg, dbeta, dh0."""
    q, k, v, g, beta, do = map(_f64, (q, k, v, g, beta, do))
    B, T, H, HV, K, V = _dims(q, v, g)
    scale = K ** -0.5 if scale is None else float(scale)
    h0 = None if h0 is None else _f64(h0)
    dht = None if dht is None else _f64(dht)
    out = dict(dq=np.zeros((B, T, H, K)), dk=np.zeros((B, T, H, K)),
               dv=np.zeros((B, T, HV, V)), dg=np.zeros((B, T, HV, K)),
               dbeta=np.zeros((B, T, HV)), dh0=np.zeros((B, HV, K, V)))
    _load().kda_oracle_bwd_recurrent(
        B, T, H, HV, K, V, scale, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
        _ptr(do), _ptr(dht), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
        _ptr(out["dg"]), _ptr(out["dbeta"]), _ptr(out["dh0"]))
    return out


def fwd_chunked(q, k, v, g, beta, chunk, scale=None, h0=None):
    """Chunk-form forward (any chunk size >= 1).  Returns (o, ht)."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    B, T, H, HV, K, V = _dims(q, v, g)
    scale = K ** -0.5 if scale is None else float(scale)
    h0 = None if h0 is None else _f64(h0)
    o = np.zeros((B, T, HV, V))
    ht = np.zeros((B, HV, K, V))
    _load().kda_oracle_fwd_chunked(B, T, H, HV, K, V, scale, int(chunk), _ptr(q), _ptr(k),
                                   _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(ht))
    return o, ht


def chunk_wy(qs, k, v, g, beta):
    """The step (1)-(3) quantities of one chunk of one head.

    qs (n,K) is the already-scaled query.  Returns dict G, A, T, W, U, Aqk.
    """
    qs, k, v, g, beta = map(_f64, (qs, k, v, g, beta))
    n, K = k.shape
    V = v.shape[1]
    out = dict(G=np.zeros((n, K)), A=np.zeros((n, n)), T=np.zeros((n, n)),
               W=np.zeros((n, K)), U=np.zeros((n, V)), Aqk=np.zeros((n, n)))
    _load().kda_oracle_chunk_wy(n, K, V, _ptr(qs), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                _ptr(out["G"]), _ptr(out["A"]), _ptr(out["T"]),
                                _ptr(out["W"]), _ptr(out["U"]), _ptr(out["Aqk"]))
    return out


def step(q, k, v, g, beta, state, scale=None):
    """One decode token.  q,k [B,H,K]; v [B,HV,V]; g [B,HV,K]; beta [B,HV].

    ``state`` [B,HV,K,V] float64 is updated IN PLACE; returns o [B,HV,V].
    """
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    assert state.dtype == np.float64 and state.flags["C_CONTIGUOUS"]
    B, H, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    scale = K ** -0.5 if scale is None else float(scale)
    o = np.zeros((B, HV, V))
    _load().kda_oracle_step(B, H, HV, K, V, scale, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                            _ptr(beta), _ptr(state), _ptr(o))
    return o


def l2norm(x):
    """x / max(||x||_2, 1e-12) over the last axis (float64)."""
    x = _f64(x)
    y = np.zeros_like(x)
    K = x.shape[-1]
    _load().kda_oracle_l2norm(x.size // K if K else 0, K, _ptr(x), _ptr(y))
    return y


def l2norm_bwd(x, dy):
    """Gradient with respect to x of <dy, l2norm(x)> (last axis, float64)."""
    x, dy = _f64(x), _f64(dy)
    dx = np.zeros_like(x)
    K = x.shape[-1]
    _load().kda_oracle_l2norm_bwd(x.size // K if K else 0, K, _ptr(x), _ptr(dy), _ptr(dx))
    return dx


def head_slice(x, b, head, kind):
    """Slice one head out of a full tensor, keeping 4-D [1,T,1,X] shape.

    kind: 'tok' for [B,T,H*,X] tensors, 'beta' for [B,T,HV], 'state' for
    [B,HV,K,V].  Used to run the oracle on sampled heads of large workloads.
    """
    x = np.asarray(x)
    if kind == "tok":
        return x[b:b + 1, :, head:head + 1, :]
    if kind == "beta":
        return x[b:b + 1, :, head:head + 1]
    if kind == "state":
        return x[b:b + 1, head:head + 1]
    raise ValueError(kind)
