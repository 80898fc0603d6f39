"""Thin ctypes binding of libkda.so (C ABI declared in include/kda.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  torch provides device memory and the current stream.  If the
library is missing the first call raises ``KdaError``; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libkda.so")

KDA_F32, KDA_BF16 = 0, 1
IMPLS = {"auto": 0, "simt": 1, "tcgen05": 2}
_STATUS = {0: "ok", 1: "invalid argument", 2: "invalid shape", 3: "unsupported",
           4: "alignment", 5: "workspace", 6: "cuda error", 7: "timeout"}


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: kda status {status} ({_STATUS.get(status, '?')})")
        self.status = status


class KdaDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("HV", ctypes.c_int), ("K", ctypes.c_int), ("V", ctypes.c_int),
                ("chunk_size", ctypes.c_int), ("scale", ctypes.c_float),
                ("dtype", ctypes.c_int), ("impl", ctypes.c_int), ("qk_l2norm", ctypes.c_int)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libkda.so (built by ``gated_delta_rule_41_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise KdaError(-1, f"libkda.so not built ({_LIB_PATH}); run "
                               "`python -m gated_delta_rule_41_gb300.build`")
        lib = ctypes.CDLL(_LIB_PATH)
        P, D, I, S = ctypes.c_void_p, ctypes.POINTER(KdaDims), ctypes.c_int, ctypes.c_size_t
        lib.kda_chunk_workspace_bytes.argtypes = [D, I]
        lib.kda_chunk_workspace_bytes.restype = S
        for name in ("kda_chunk_fwd", "kda_chunk_fwd_save"):
            getattr(lib, name).argtypes = [D, P, P, P, P, P, P, P, I, P, P, S, P]
            getattr(lib, name).restype = I
        for name in ("kda_chunk_bwd", "kda_chunk_bwd_saved"):
            getattr(lib, name).argtypes = [D] + [P] * 15 + [S, P]
            getattr(lib, name).restype = I
        lib.kda_chunk_workspace_bytes_varlen.argtypes = [D, I, I]
        lib.kda_chunk_workspace_bytes_varlen.restype = S
        for name in ("kda_chunk_fwd_varlen", "kda_chunk_fwd_varlen_save"):
            getattr(lib, name).argtypes = [D, P, I, P, P, P, P, P, P, P, I, P, P, S, P]
            getattr(lib, name).restype = I
        for name in ("kda_chunk_bwd_varlen", "kda_chunk_bwd_varlen_saved"):
            getattr(lib, name).argtypes = [D, P, I] + [P] * 15 + [S, P]
            getattr(lib, name).restype = I
        lib.kda_recurrent_step.argtypes = [D] + [P] * 8
        lib.kda_recurrent_step.restype = I
        lib.kda_check.argtypes = [P]
        lib.kda_check.restype = I
        lib.kda_status_str.argtypes = [I]
        lib.kda_status_str.restype = ctypes.c_char_p
        lib.kda_version.restype = I
        lib.kda_timing_enable.argtypes = [I]
        lib.kda_timing_enable.restype = None
        lib.kda_timing_count.restype = I
        lib.kda_timing_entry.argtypes = [I, ctypes.c_char_p, I, ctypes.POINTER(ctypes.c_double),
                                         ctypes.POINTER(ctypes.c_long)]
        lib.kda_timing_entry.restype = I
        lib.kda_selftest_mma.argtypes = [P, P, P, I, I, P, P]
        lib.kda_selftest_mma.restype = I
        lib.kda_selftest_wait_timeout.argtypes = [ctypes.c_longlong, P]
        lib.kda_selftest_wait_timeout.restype = I
        _lib = lib
        return lib


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return KDA_BF16
    if t == torch.float32:
        return KDA_F32
    raise KdaError(3, f"dtype {t} (bf16 or fp32 only)")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check_dev(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise KdaError(1, "tensors must be contiguous CUDA tensors")


def make_dims(q, v, chunk_size=64, scale=None, impl="auto", qk_l2norm=False) -> KdaDims:
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    return KdaDims(B, T, H, HV, K, V, chunk_size,
                   float(K ** -0.5 if scale is None else scale), _dtype_code(q.dtype),
                   IMPLS[impl], int(bool(qk_l2norm)))


def workspace_bytes(dims: KdaDims, for_bwd: bool) -> int:
    return int(load_library().kda_chunk_workspace_bytes(ctypes.byref(dims), int(for_bwd)))


def _workspace(dims, for_bwd, device, workspace):
    need = workspace_bytes(dims, for_bwd)
    if need == 0:
        return None, 0
    if workspace is not None and workspace.numel() * workspace.element_size() >= need:
        return workspace, need
    return torch.empty(need, dtype=torch.uint8, device=device), need


def _raise(st, what):
    if st != 0:
        raise KdaError(st, what)


class SavedForward:
    """Workspace filled by ``chunk_kda_fwd(..., save_for_backward=True)``.

    Pass it as ``saved=`` to ``chunk_kda_bwd`` with the same inputs, before
    any other call writes the workspace."""

    def __init__(self, workspace, nbytes, dims):
        self.workspace, self.nbytes, self.dims = workspace, nbytes, dims


def chunk_kda_fwd(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=False,
                  chunk_size=64, impl="auto", workspace=None, out=None, final_state=None,
                  stream=None, save_for_backward=False, use_qk_l2norm_in_kernel=False):
    """Chunked KDA forward.  Returns (o, final_state or None), plus a
    ``SavedForward`` when ``save_for_backward`` is set.  With
    ``use_qk_l2norm_in_kernel`` the kernels L2-normalise q and k themselves."""
    lib = load_library()
    _check_dev(q, k, v, g, beta, initial_state)
    dims = make_dims(q, v, chunk_size, scale, impl, use_qk_l2norm_in_kernel)
    o = torch.empty_like(v) if out is None else out
    ht = None
    if output_final_state:
        ht = (torch.empty(dims.B, dims.HV, dims.K, dims.V, dtype=torch.float32, device=q.device)
              if final_state is None else final_state)
    ws, nws = _workspace(dims, save_for_backward, q.device, workspace)
    fn = lib.kda_chunk_fwd_save if save_for_backward else lib.kda_chunk_fwd
    st = fn(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
            _ptr(initial_state), _ptr(o), int(output_final_state), _ptr(ht), _ptr(ws), nws,
            _stream(stream))
    _raise(st, "kda_chunk_fwd_save" if save_for_backward else "kda_chunk_fwd")
    if save_for_backward:
        return o, ht, SavedForward(ws, nws, dims)
    return o, ht


def chunk_kda_bwd(q, k, v, g, beta, do, dht=None, scale=None, initial_state=None,
                  chunk_size=64, impl="auto", workspace=None, grads=None, stream=None,
                  saved=None, use_qk_l2norm_in_kernel=False):
    """Backward of chunk_kda_fwd.  Returns dict dq, dk, dv, dg, dbeta, dh0.
    With ``saved`` (from a saving forward on the same inputs) the tensor-core
    kernels start from the saved intermediates instead of recomputing them.
    With ``use_qk_l2norm_in_kernel``, dq and dk are the gradients with respect
    to the raw (unnormalised) q and k."""
    lib = load_library()
    _check_dev(q, k, v, g, beta, do, dht, initial_state)
    dims = make_dims(q, v, chunk_size, scale, impl, use_qk_l2norm_in_kernel)
    if grads is None:
        grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                     dg=torch.empty_like(g), dbeta=torch.empty_like(beta),
                     dh0=(torch.empty(dims.B, dims.HV, dims.K, dims.V, dtype=torch.float32,
                                      device=q.device) if initial_state is not None else None))
    if saved is not None:
        if (saved.dims.B, saved.dims.T, saved.dims.H, saved.dims.HV, saved.dims.K, saved.dims.V,
                saved.dims.chunk_size, saved.dims.impl, saved.dims.qk_l2norm) != (
                    dims.B, dims.T, dims.H, dims.HV, dims.K, dims.V, dims.chunk_size, dims.impl,
                    dims.qk_l2norm):
            raise KdaError(1, "chunk_kda_bwd: saved forward has other dims")
        ws, nws, fn, what = saved.workspace, saved.nbytes, lib.kda_chunk_bwd_saved, \
            "kda_chunk_bwd_saved"
    else:
        ws, nws = _workspace(dims, True, q.device, workspace)
        fn, what = lib.kda_chunk_bwd, "kda_chunk_bwd"
    st = fn(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
            _ptr(initial_state), _ptr(do), _ptr(dht), _ptr(grads["dq"]), _ptr(grads["dk"]),
            _ptr(grads["dv"]), _ptr(grads["dg"]), _ptr(grads["dbeta"]), _ptr(grads.get("dh0")),
            _ptr(ws), nws, _stream(stream))
    _raise(st, what)
    return grads


def _check_cu(cu_seqlens):
    if (cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1
            or not cu_seqlens.is_contiguous()):
        raise KdaError(1, "cu_seqlens must be a contiguous 1-D int32 CUDA tensor")
    return cu_seqlens.numel() - 1


def chunk_kda_fwd_varlen(q, k, v, g, beta, cu_seqlens, scale=None, initial_state=None,
                         output_final_state=False, chunk_size=64, impl="auto", workspace=None,
                         out=None, final_state=None, stream=None, use_qk_l2norm_in_kernel=False,
                         save_for_backward=False):
    """Forward over sequences packed along T: q, k [1,T,H,K]; v [1,T,HV,V];
    g [1,T,HV,K]; beta [1,T,HV]; ``cu_seqlens`` int32 [N+1] on the device.
    ``initial_state`` / the final state are [N,HV,K,V].  Returns (o, ht), or
    (o, ht, saved) with ``save_for_backward`` (pass ``saved`` to
    ``chunk_kda_bwd_varlen`` with the same inputs and cu_seqlens)."""
    lib = load_library()
    _check_dev(q, k, v, g, beta, initial_state)
    nseq = _check_cu(cu_seqlens)
    dims = make_dims(q, v, chunk_size, scale, impl, use_qk_l2norm_in_kernel)
    o = torch.empty_like(v) if out is None else out
    ht = None
    if output_final_state:
        ht = (torch.empty(nseq, dims.HV, dims.K, dims.V, dtype=torch.float32, device=q.device)
              if final_state is None else final_state)
    need = int(lib.kda_chunk_workspace_bytes_varlen(ctypes.byref(dims), nseq,
                                                   int(save_for_backward)))
    ws = workspace if (workspace is not None and workspace.numel() >= need) else \
        torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    fn = lib.kda_chunk_fwd_varlen_save if save_for_backward else lib.kda_chunk_fwd_varlen
    st = fn(ctypes.byref(dims), _ptr(cu_seqlens), nseq, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
            _ptr(beta), _ptr(initial_state), _ptr(o), int(output_final_state), _ptr(ht), _ptr(ws),
            need, _stream(stream))
    _raise(st, "kda_chunk_fwd_varlen")
    if save_for_backward:
        return o, ht, SavedForward(ws, need, dims)
    return o, ht


def chunk_kda_bwd_varlen(q, k, v, g, beta, do, cu_seqlens, dht=None, scale=None,
                         initial_state=None, chunk_size=64, impl="auto", workspace=None,
                         grads=None, stream=None, use_qk_l2norm_in_kernel=False, saved=None):
    """Backward of chunk_kda_fwd_varlen.  Returns dict dq, dk, dv, dg, dbeta,
    dh0 (dh0 [N,HV,K,V] when ``initial_state`` is given).  With ``saved``
    (from a saving forward on the same inputs and cu_seqlens) the tensor-core
    kernels start from the saved intermediates."""
    lib = load_library()
    _check_dev(q, k, v, g, beta, do, dht, initial_state)
    nseq = _check_cu(cu_seqlens)
    dims = make_dims(q, v, chunk_size, scale, impl, use_qk_l2norm_in_kernel)
    if grads is None:
        grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                     dg=torch.empty_like(g), dbeta=torch.empty_like(beta),
                     dh0=(torch.empty(nseq, dims.HV, dims.K, dims.V, dtype=torch.float32,
                                      device=q.device) if initial_state is not None else None))
    if saved is not None:
        if (saved.dims.T, saved.dims.H, saved.dims.HV, saved.dims.K, saved.dims.V,
                saved.dims.chunk_size, saved.dims.impl, saved.dims.qk_l2norm) != (
                    dims.T, dims.H, dims.HV, dims.K, dims.V, dims.chunk_size, dims.impl,
                    dims.qk_l2norm):
            raise KdaError(1, "chunk_kda_bwd_varlen: saved forward has other dims")
        ws, need, fn = saved.workspace, saved.nbytes, lib.kda_chunk_bwd_varlen_saved
    else:
        need = int(lib.kda_chunk_workspace_bytes_varlen(ctypes.byref(dims), nseq, 1))
        ws = workspace if (workspace is not None and workspace.numel() >= need) else \
            torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        fn = lib.kda_chunk_bwd_varlen
    st = fn(ctypes.byref(dims), _ptr(cu_seqlens), nseq, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
            _ptr(beta), _ptr(initial_state), _ptr(do), _ptr(dht), _ptr(grads["dq"]),
            _ptr(grads["dk"]), _ptr(grads["dv"]), _ptr(grads["dg"]), _ptr(grads["dbeta"]),
            _ptr(grads.get("dh0")), _ptr(ws), need, _stream(stream))
    _raise(st, "kda_chunk_bwd_varlen")
    return grads


def recurrent_step(q, k, v, g, beta, state, scale=None, out=None, stream=None,
                   use_qk_l2norm_in_kernel=False):
    """One decode token: q,k [B,H,K]; v [B,HV,V]; g [B,HV,K]; beta [B,HV];
    ``state`` [B,HV,K,V] float32 updated in place.  Returns o [B,HV,V]."""
    lib = load_library()
    _check_dev(q, k, v, g, beta, state)
    B, H, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    dims = KdaDims(B, 1, H, HV, K, V, 64, float(K ** -0.5 if scale is None else scale),
                   _dtype_code(q.dtype), 0, int(bool(use_qk_l2norm_in_kernel)))
    o = torch.empty_like(v) if out is None else out
    st = lib.kda_recurrent_step(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                _ptr(beta), _ptr(state), _ptr(o), _stream(stream))
    _raise(st, "kda_recurrent_step")
    return o


def check(stream=None):
    """Synchronise the stream and raise on any error a kernel recorded."""
    _raise(load_library().kda_check(_stream(stream)), "kda_check")


def timing_enable(on: bool):
    """Start (clear) or stop per-kernel device timing inside the library."""
    load_library().kda_timing_enable(int(on))


def timing_read() -> dict:
    """{kernel name: (total device ms, launches)} since timing_enable(True)."""
    lib = load_library()
    out = {}
    for i in range(lib.kda_timing_count()):
        name = ctypes.create_string_buffer(64)
        ms, n = ctypes.c_double(), ctypes.c_long()
        if lib.kda_timing_entry(i, name, 64, ctypes.byref(ms), ctypes.byref(n)) == 0:
            out[name.value.decode()] = (ms.value, n.value)
    return out


def selftest_mma(A, B, use_tma=True, a_mn=False, b_mn=False, stream=None):
    """D = A @ B^T through one tcgen05 MMA chain.  A [128,64] and B [N,64] bf16
    (K-major), or, with a_mn / b_mn, A^T [64,128] / B^T [64,N] (MN-major)."""
    lib = load_library()
    _check_dev(A, B)
    N = B.shape[1] if b_mn else B.shape[0]
    flags = int(use_tma) | (int(a_mn) << 1) | (int(b_mn) << 2)
    D = torch.zeros(128, N, dtype=torch.float32, device=A.device)
    status = torch.zeros(1, dtype=torch.int32, device=A.device)
    st = lib.kda_selftest_mma(_ptr(A), _ptr(B), _ptr(D), N, flags, _ptr(status),
                              _stream(stream))
    _raise(st, "kda_selftest_mma")
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise KdaError(7, "kda_selftest_mma")
    return D
