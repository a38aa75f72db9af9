"""GB300 (sm_103a) Gated DeltaNet / Kimi Delta Attention token mixer.

Thin ctypes binding over the C ABI in ``include/gdn.h`` (``libgdn.so``).  The
functions here only marshal arguments: they check dtypes and devices, allocate
the outputs and the backward workspace with PyTorch, and pass raw device
pointers and the current CUDA stream to the library.  Every step of the
computation runs in the library's CUDA kernels; there is no other path.  If
the library has not been built, every call raises.

Names follow the ABI: ``gdn_fwd``, ``gdn_bwd``, ``kda_fwd``, ``kda_bwd`` and
``mamba2_fwd``, ``mamba2_bwd`` (the scalar-gated state without the delta rule);
the training pair with a saved context ``gdn_fwd_save`` / ``gdn_bwd_saved``
(and the KDA and Mamba2 pairs), whose forward keeps what the backward would
recompute; and the token-recurrent ``gdn_decode`` / ``kda_decode`` for a few
tokens per sequence.  The mixer's fused neighbours: ``short_conv_fwd`` /
``short_conv_bwd`` (causal depthwise convolution + SiLU, with the per-head
L2 norm for q and k) and ``gated_rmsnorm_fwd`` / ``gated_rmsnorm_bwd``.
Token tensors are ``[B, T, H, D]`` (fp32 or bf16, all the same dtype), ``g``
is ``[B, T, H]`` (GDN) or ``[B, T, H, dk]`` (KDA) fp32, ``beta`` ``[B, T, H]``
fp32, states ``[B, H, dk, dv]`` fp32.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")

GDN_F32, GDN_BF16, GDN_BF16_G16 = 0, 1, 2
_DTYPES = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16}


class GdnShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("chunk", ctypes.c_int),
                ("dtype", ctypes.c_int)]


class ConvShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("D", ctypes.c_int), ("W", ctypes.c_int), ("dtype", ctypes.c_int)]


class NormShape(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_longlong), ("D", ctypes.c_int), ("dtype", ctypes.c_int)]


class GdnError(RuntimeError):
    pass


_lock = threading.Lock()
_lib = None
EXPORTS = ("gdn_fwd", "gdn_bwd", "kda_fwd", "kda_bwd", "gdn_fwd_workspace", "kda_fwd_workspace",
           "gdn_bwd_workspace", "kda_bwd_workspace", "gdn_ctx_bytes", "kda_ctx_bytes",
           "gdn_fwd_save", "kda_fwd_save", "gdn_bwd_saved", "kda_bwd_saved",
           "mamba2_fwd", "mamba2_bwd", "mamba2_fwd_save", "mamba2_bwd_saved",
           "mamba2_fwd_workspace", "mamba2_bwd_workspace", "mamba2_ctx_bytes",
           "gdn_decode", "kda_decode",
           "gdn_status_str", "gdn_last_cuda_error", "gdn_device_status", "gdn_uses_tensor_cores",
           "gdn_wait_selftest", "kda_uses_tensor_cores",
           "gdn_varlen_workspace", "kda_varlen_workspace", "mamba2_varlen_workspace",
           "gdn_fwd_varlen", "gdn_bwd_varlen", "kda_fwd_varlen", "kda_bwd_varlen",
           "mamba2_fwd_varlen", "mamba2_bwd_varlen",
           "gdn_short_conv_fwd", "gdn_short_conv_bwd", "gdn_short_conv_bwd_workspace",
           "gdn_gated_rmsnorm_fwd", "gdn_gated_rmsnorm_bwd", "gdn_gated_rmsnorm_bwd_workspace",
           "gdn_profile_begin", "gdn_profile_end", "gdn_profile_read", "gdn_kernel_name")


def lib():
    """The loaded ``libgdn.so``; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise GdnError(f"{LIB_PATH} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            vp, sz, fp = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p
            sp = ctypes.POINTER(GdnShape)
            for name in ("gdn_fwd_workspace", "kda_fwd_workspace", "gdn_bwd_workspace",
                         "kda_bwd_workspace", "gdn_ctx_bytes", "kda_ctx_bytes",
                         "mamba2_fwd_workspace", "mamba2_bwd_workspace", "mamba2_ctx_bytes"):
                getattr(L, name).argtypes = [sp]
                getattr(L, name).restype = sz
            for name in ("gdn_fwd", "kda_fwd", "gdn_fwd_save", "kda_fwd_save", "mamba2_fwd",
                         "mamba2_fwd_save"):
                getattr(L, name).argtypes = [sp] + [vp] * 8 + [vp, sz, vp]
                getattr(L, name).restype = ctypes.c_int
            for name in ("gdn_bwd", "kda_bwd", "gdn_bwd_saved", "kda_bwd_saved", "mamba2_bwd",
                         "mamba2_bwd_saved"):
                getattr(L, name).argtypes = [sp] + [vp] * 14 + [vp, sz, vp]
                getattr(L, name).restype = ctypes.c_int
            for name in ("gdn_decode", "kda_decode"):
                getattr(L, name).argtypes = [sp] + [vp] * 8 + [vp]
                getattr(L, name).restype = ctypes.c_int
            L.gdn_status_str.argtypes = [ctypes.c_int]
            L.gdn_status_str.restype = ctypes.c_char_p
            L.gdn_last_cuda_error.argtypes = []
            L.gdn_last_cuda_error.restype = ctypes.c_int
            L.gdn_device_status.argtypes = []
            L.gdn_device_status.restype = ctypes.c_int
            for name in ("gdn_varlen_workspace", "kda_varlen_workspace", "mamba2_varlen_workspace"):
                getattr(L, name).argtypes = [sp, ctypes.c_int, ctypes.c_int]
                getattr(L, name).restype = sz
            for name in ("gdn_fwd_varlen", "kda_fwd_varlen", "mamba2_fwd_varlen"):
                getattr(L, name).argtypes = [sp, vp, ctypes.c_int] + [vp] * 8 + [vp, sz, vp]
                getattr(L, name).restype = ctypes.c_int
            for name in ("gdn_bwd_varlen", "kda_bwd_varlen", "mamba2_bwd_varlen"):
                getattr(L, name).argtypes = [sp, vp, ctypes.c_int] + [vp] * 14 + [vp, sz, vp]
                getattr(L, name).restype = ctypes.c_int
            L.gdn_wait_selftest.argtypes = [ctypes.c_int, vp]
            L.gdn_wait_selftest.restype = ctypes.c_int
            for name in ("gdn_uses_tensor_cores", "kda_uses_tensor_cores"):
                getattr(L, name).argtypes = [sp]
                getattr(L, name).restype = ctypes.c_int
            cs, ns, f32, i32 = (ctypes.POINTER(ConvShape), ctypes.POINTER(NormShape),
                                ctypes.c_float, ctypes.c_int)
            L.gdn_short_conv_fwd.argtypes = [cs, vp, vp, vp, i32, f32, f32, vp, i32, vp]
            L.gdn_short_conv_fwd.restype = ctypes.c_int
            L.gdn_short_conv_bwd_workspace.argtypes = [cs]
            L.gdn_short_conv_bwd_workspace.restype = sz
            L.gdn_short_conv_bwd.argtypes = [cs, vp, vp, vp, vp, vp, i32, f32, f32, vp, i32, vp, sz,
                                             vp]
            L.gdn_short_conv_bwd.restype = ctypes.c_int
            L.gdn_gated_rmsnorm_fwd.argtypes = [ns, vp, vp, vp, vp, f32, vp]
            L.gdn_gated_rmsnorm_fwd.restype = ctypes.c_int
            L.gdn_gated_rmsnorm_bwd_workspace.argtypes = [ns]
            L.gdn_gated_rmsnorm_bwd_workspace.restype = sz
            L.gdn_gated_rmsnorm_bwd.argtypes = [ns, vp, vp, vp, vp, vp, vp, vp, f32, vp, sz, vp]
            L.gdn_gated_rmsnorm_bwd.restype = ctypes.c_int
            L.gdn_profile_begin.argtypes = [ctypes.c_int]
            L.gdn_profile_begin.restype = ctypes.c_int
            L.gdn_profile_end.argtypes = []
            L.gdn_profile_end.restype = ctypes.c_int
            L.gdn_profile_read.argtypes = [ctypes.POINTER(ctypes.c_int),
                                           ctypes.POINTER(ctypes.c_float), ctypes.c_int]
            L.gdn_profile_read.restype = ctypes.c_int
            L.gdn_kernel_name.argtypes = [ctypes.c_int]
            L.gdn_kernel_name.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _ptr(x):
    return None if x is None else ctypes.c_void_p(x.data_ptr())


def _check(rc):
    if rc != 0:
        L = lib()
        msg = L.gdn_status_str(rc).decode()
        if rc == -6:
            msg += f" (cudaError {L.gdn_last_cuda_error()})"
        raise GdnError(msg)


def make_shape(q, v, chunk, g=None) -> GdnShape:
    """The ABI shape of a call; a bf16 ``g`` (KDA) selects GDN_BF16_G16."""
    B, T, H, dk = q.shape
    dt = _DTYPES[q.dtype]
    if g is not None and g.dtype == torch.bfloat16:
        dt = GDN_BF16_G16
    return GdnShape(B, T, H, dk, v.shape[3], chunk, dt)


def _validate(q, k, v, g, beta, kda, extra=()):
    if q.dtype not in _DTYPES:
        raise GdnError(f"unsupported dtype {q.dtype}")
    dev = q.device
    if dev.type != "cuda":
        raise GdnError("inputs must be CUDA tensors (the library has no CPU path)")
    B, T, H, dk = q.shape
    dv = v.shape[3]
    want = {"k": (k, (B, T, H, dk), q.dtype), "v": (v, (B, T, H, dv), q.dtype),
            "g": (g, (B, T, H, dk) if kda else (B, T, H),
                  torch.bfloat16 if (kda and g is not None and g.dtype == torch.bfloat16
                                     and q.dtype == torch.bfloat16) else torch.float32),
            "beta": (beta, (B, T, H), torch.float32)}
    for name, (x, shape, dt) in list(want.items()) + list(extra):
        if x is None:
            continue
        if tuple(x.shape) != tuple(shape) or x.dtype != dt or x.device != dev:
            raise GdnError(f"{name}: expected {tuple(shape)} {dt} on {dev}, got "
                           f"{tuple(x.shape)} {x.dtype} on {x.device}")
        if not x.is_contiguous():
            raise GdnError(f"{name} must be contiguous")


def _stream(dev):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _mixer(kda, delta):
    if kda and not delta:
        raise GdnError("the per-key-dimension gate is only offered with the delta rule (KDA)")
    return "kda" if kda else ("gdn" if delta else "mamba2")


def _entry(kda, delta, name):
    """The ABI function ``<mixer>_<name>``."""
    return getattr(lib(), f"{_mixer(kda, delta)}_{name}")


def fwd_workspace_bytes(q, v, chunk=64, kda=False, delta=True) -> int:
    s = make_shape(q, v, chunk)
    return int(_entry(kda, delta, "fwd_workspace")(ctypes.byref(s)))


def bwd_workspace_bytes(q, v, chunk=64, kda=False, delta=True) -> int:
    s = make_shape(q, v, chunk)
    return int(_entry(kda, delta, "bwd_workspace")(ctypes.byref(s)))


def ctx_bytes(q, v, chunk=64, kda=False, delta=True) -> int:
    """Bytes of the saved context of ``*_fwd_save`` / ``*_bwd_saved``."""
    s = make_shape(q, v, chunk)
    return int(_entry(kda, delta, "ctx_bytes")(ctypes.byref(s)))


def _workspace(need, given, device):
    if given is not None and given.numel() >= need:
        return given
    return torch.empty(max(need, 16), dtype=torch.uint8, device=device)


def uses_tensor_cores(q, v, chunk=64, kda=False) -> bool:
    s = make_shape(q, v, chunk)
    fn = lib().kda_uses_tensor_cores if kda else lib().gdn_uses_tensor_cores
    return bool(fn(ctypes.byref(s)))


def _fwd(kda, q, k, v, g, beta, h0=None, chunk=64, output_final_state=True, out=None,
         workspace=None, ctx=None, delta=True):
    B, T, H, dk = q.shape
    dv = v.shape[3]
    _validate(q, k, v, g, beta, kda, [("h0", (h0, (B, H, dk, dv), torch.float32))])
    o = out if out is not None else torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    ht = (torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
          if output_final_state else None)
    if ctx is not None:
        _check_ctx(ctx, ctx_bytes(q, v, chunk, kda, delta), q.device)
        ws = ctx
        fn = _entry(kda, delta, "fwd_save")
    else:
        ws = _workspace(fwd_workspace_bytes(q, v, chunk, kda, delta), workspace, q.device)
        fn = _entry(kda, delta, "fwd")
    s = make_shape(q, v, chunk, g)
    _check(fn(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o),
              _ptr(ht), _ptr(ws), ws.numel(), _stream(q.device)))
    return o, ht


def _check_ctx(ctx, need, device):
    if (not isinstance(ctx, torch.Tensor) or ctx.dtype != torch.uint8 or ctx.device != device
            or not ctx.is_contiguous() or ctx.numel() < need):
        raise GdnError(f"ctx must be a contiguous uint8 tensor of at least {need} bytes "
                       f"on {device} (see new_ctx)")


def _bwd(kda, q, k, v, g, beta, h0, do, dht=None, chunk=64, want_dh0=True, workspace=None,
         ctx=None, delta=True):
    B, T, H, dk = q.shape
    dv = v.shape[3]
    _validate(q, k, v, g, beta, kda, [("h0", (h0, (B, H, dk, dv), torch.float32)),
                                      ("do", (do, (B, T, H, dv), q.dtype)),
                                      ("dht", (dht, (B, H, dk, dv), torch.float32))])
    e = lambda x: torch.empty_like(x)
    dq, dk_, dv_, dg, dbeta = e(q), e(k), e(v), e(g), e(beta)
    dh0 = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device) if want_dh0 else None
    if ctx is not None:
        _check_ctx(ctx, ctx_bytes(q, v, chunk, kda, delta), q.device)
        ws = ctx
        fn = _entry(kda, delta, "bwd_saved")
    else:
        ws = _workspace(bwd_workspace_bytes(q, v, chunk, kda, delta), workspace, q.device)
        fn = _entry(kda, delta, "bwd")
    s = make_shape(q, v, chunk, g)
    _check(fn(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(do),
              _ptr(dht), _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dg), _ptr(dbeta), _ptr(dh0),
              _ptr(ws), ws.numel(), _stream(q.device)))
    return {"dq": dq, "dk": dk_, "dv": dv_, "dg": dg, "dbeta": dbeta, "dh0": dh0}


def gdn_fwd(q, k, v, g, beta, h0=None, chunk=64, output_final_state=True, workspace=None):
    """GDN forward.  Returns ``(o, ht)`` (``ht`` None if not requested).  ``workspace``
    (uint8 CUDA tensor) is used when it holds ``fwd_workspace_bytes`` bytes, else one
    is allocated."""
    return _fwd(False, q, k, v, g, beta, h0, chunk, output_final_state, workspace=workspace)


def kda_fwd(q, k, v, g, beta, h0=None, chunk=64, output_final_state=True, workspace=None):
    """KDA forward (``g`` is ``[B,T,H,dk]``).  Returns ``(o, ht)``."""
    return _fwd(True, q, k, v, g, beta, h0, chunk, output_final_state, workspace=workspace)


def gdn_bwd(q, k, v, g, beta, h0, do, dht=None, chunk=64, want_dh0=True, workspace=None):
    """GDN backward.  Returns a dict ``dq, dk, dv, dg, dbeta, dh0``."""
    return _bwd(False, q, k, v, g, beta, h0, do, dht, chunk, want_dh0, workspace)


def kda_bwd(q, k, v, g, beta, h0, do, dht=None, chunk=64, want_dh0=True, workspace=None):
    """KDA backward.  Returns a dict ``dq, dk, dv, dg, dbeta, dh0``."""
    return _bwd(True, q, k, v, g, beta, h0, do, dht, chunk, want_dh0, workspace)


def new_ctx(q, v, chunk=64, kda=False, delta=True):
    """An uninitialised saved-context buffer for ``q``/``v``'s shape."""
    return torch.empty(max(16, ctx_bytes(q, v, chunk, kda, delta)), dtype=torch.uint8,
                       device=q.device)


def gdn_fwd_save(q, k, v, g, beta, h0=None, chunk=64, output_final_state=True, ctx=None):
    """GDN forward that also leaves the saved context for ``gdn_bwd_saved``.
    Returns ``(o, ht, ctx)``; ``ctx`` (from ``new_ctx``) is allocated if not given."""
    ctx = new_ctx(q, v, chunk) if ctx is None else ctx
    o, ht = _fwd(False, q, k, v, g, beta, h0, chunk, output_final_state, ctx=ctx)
    return o, ht, ctx


def kda_fwd_save(q, k, v, g, beta, h0=None, chunk=64, output_final_state=True, ctx=None):
    """KDA forward that also leaves the saved context for ``kda_bwd_saved``."""
    ctx = new_ctx(q, v, chunk, True) if ctx is None else ctx
    o, ht = _fwd(True, q, k, v, g, beta, h0, chunk, output_final_state, ctx=ctx)
    return o, ht, ctx


def gdn_bwd_saved(q, k, v, g, beta, h0, do, ctx, dht=None, chunk=64, want_dh0=True):
    """GDN backward reading the context ``gdn_fwd_save`` left in ``ctx`` (the same
    q, k, v, g, beta, h0 must be passed).  Returns the dict of ``gdn_bwd``."""
    return _bwd(False, q, k, v, g, beta, h0, do, dht, chunk, want_dh0, ctx=ctx)


def kda_bwd_saved(q, k, v, g, beta, h0, do, ctx, dht=None, chunk=64, want_dh0=True):
    """KDA backward reading the context ``kda_fwd_save`` left in ``ctx``."""
    return _bwd(True, q, k, v, g, beta, h0, do, dht, chunk, want_dh0, ctx=ctx)


def mamba2_fwd(q, k, v, g, beta, h0=None, chunk=64, output_final_state=True, workspace=None):
    """Mamba2 forward (``g`` is ``[B,T,H]``): the scalar-gated state without the
    delta rule, ``H_t = exp(g_t) H_{t-1} + beta_t k_t v_t^T``.  Returns ``(o, ht)``."""
    return _fwd(False, q, k, v, g, beta, h0, chunk, output_final_state, workspace=workspace,
                delta=False)


def mamba2_bwd(q, k, v, g, beta, h0, do, dht=None, chunk=64, want_dh0=True, workspace=None):
    """Mamba2 backward.  Returns a dict ``dq, dk, dv, dg, dbeta, dh0``."""
    return _bwd(False, q, k, v, g, beta, h0, do, dht, chunk, want_dh0, workspace, delta=False)


def mamba2_fwd_save(q, k, v, g, beta, h0=None, chunk=64, output_final_state=True, ctx=None):
    """Mamba2 forward that also leaves the saved context for ``mamba2_bwd_saved``."""
    ctx = new_ctx(q, v, chunk, delta=False) if ctx is None else ctx
    o, ht = _fwd(False, q, k, v, g, beta, h0, chunk, output_final_state, ctx=ctx, delta=False)
    return o, ht, ctx


def mamba2_bwd_saved(q, k, v, g, beta, h0, do, ctx, dht=None, chunk=64, want_dh0=True):
    """Mamba2 backward reading the context ``mamba2_fwd_save`` left in ``ctx``."""
    return _bwd(False, q, k, v, g, beta, h0, do, dht, chunk, want_dh0, ctx=ctx, delta=False)


# ------------------------------------------------------------------ packed sequences

def varlen_workspace_bytes(q, v, nseq, chunk=64, kda=False, delta=True, backward=False) -> int:
    """Workspace bytes of a packed-sequence call (``*_varlen_workspace``)."""
    s = make_shape(q, v, chunk)
    return int(_entry(kda, delta, "varlen_workspace")(ctypes.byref(s), int(nseq), int(backward)))


def _check_cu(cu_seqlens, q):
    if (not isinstance(cu_seqlens, torch.Tensor) or cu_seqlens.dtype != torch.int32
            or cu_seqlens.device != q.device or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1
            or not cu_seqlens.is_contiguous()):
        raise GdnError("cu_seqlens must be a contiguous 1-D int32 tensor on the inputs' device")
    if q.shape[0] != 1:
        raise GdnError("packed sequences: the token tensors must be [1, T, H, D]")
    return cu_seqlens.numel() - 1


def _fwd_varlen(kda, delta, q, k, v, g, beta, cu_seqlens, h0, chunk, workspace):
    nseq = _check_cu(cu_seqlens, q)
    _, T, H, dk = q.shape
    dv = v.shape[3]
    _validate(q, k, v, g, beta, kda, [("h0", (h0, (nseq, H, dk, dv), torch.float32))])
    o = torch.empty((1, T, H, dv), dtype=q.dtype, device=q.device)
    ht = torch.empty((nseq, H, dk, dv), dtype=torch.float32, device=q.device)
    ws = _workspace(varlen_workspace_bytes(q, v, nseq, chunk, kda, delta), workspace, q.device)
    s = make_shape(q, v, chunk, g)
    _check(_entry(kda, delta, "fwd_varlen")(ctypes.byref(s), _ptr(cu_seqlens), nseq, _ptr(q), _ptr(k),
                                            _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(ht),
                                            _ptr(ws), ws.numel(), _stream(q.device)))
    return o, ht


def _bwd_varlen(kda, delta, q, k, v, g, beta, cu_seqlens, h0, do, dht, chunk, workspace):
    nseq = _check_cu(cu_seqlens, q)
    _, T, H, dk = q.shape
    dv = v.shape[3]
    _validate(q, k, v, g, beta, kda, [("h0", (h0, (nseq, H, dk, dv), torch.float32)),
                                      ("do", (do, (1, T, H, dv), q.dtype)),
                                      ("dht", (dht, (nseq, H, dk, dv), torch.float32))])
    e = lambda x: torch.empty_like(x)
    dq, dk_, dv_, dg, dbeta = e(q), e(k), e(v), e(g), e(beta)
    dh0 = torch.empty((nseq, H, dk, dv), dtype=torch.float32, device=q.device)
    ws = _workspace(varlen_workspace_bytes(q, v, nseq, chunk, kda, delta, True), workspace, q.device)
    s = make_shape(q, v, chunk, g)
    _check(_entry(kda, delta, "bwd_varlen")(ctypes.byref(s), _ptr(cu_seqlens), nseq, _ptr(q), _ptr(k),
                                            _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(do), _ptr(dht),
                                            _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dg), _ptr(dbeta),
                                            _ptr(dh0), _ptr(ws), ws.numel(), _stream(q.device)))
    return {"dq": dq, "dk": dk_, "dv": dv_, "dg": dg, "dbeta": dbeta, "dh0": dh0}


def gdn_fwd_varlen(q, k, v, g, beta, cu_seqlens, h0=None, chunk=64, workspace=None):
    """GDN forward over packed sequences: token tensors ``[1, T, H, D]``,
    ``cu_seqlens`` an int32 device tensor of ``nseq + 1`` offsets, ``h0`` and the
    returned ``ht`` ``[nseq, H, dk, dv]``.  Returns ``(o, ht)``."""
    return _fwd_varlen(False, True, q, k, v, g, beta, cu_seqlens, h0, chunk, workspace)


def gdn_bwd_varlen(q, k, v, g, beta, cu_seqlens, h0, do, dht=None, chunk=64, workspace=None):
    """GDN backward over packed sequences; returns the dict of ``gdn_bwd``."""
    return _bwd_varlen(False, True, q, k, v, g, beta, cu_seqlens, h0, do, dht, chunk, workspace)


def kda_fwd_varlen(q, k, v, g, beta, cu_seqlens, h0=None, chunk=64, workspace=None):
    """KDA forward over packed sequences (``g`` is ``[1, T, H, dk]``)."""
    return _fwd_varlen(True, True, q, k, v, g, beta, cu_seqlens, h0, chunk, workspace)


def kda_bwd_varlen(q, k, v, g, beta, cu_seqlens, h0, do, dht=None, chunk=64, workspace=None):
    """KDA backward over packed sequences."""
    return _bwd_varlen(True, True, q, k, v, g, beta, cu_seqlens, h0, do, dht, chunk, workspace)


def mamba2_fwd_varlen(q, k, v, g, beta, cu_seqlens, h0=None, chunk=64, workspace=None):
    """Mamba2 forward over packed sequences."""
    return _fwd_varlen(False, False, q, k, v, g, beta, cu_seqlens, h0, chunk, workspace)


def mamba2_bwd_varlen(q, k, v, g, beta, cu_seqlens, h0, do, dht=None, chunk=64, workspace=None):
    """Mamba2 backward over packed sequences."""
    return _bwd_varlen(False, False, q, k, v, g, beta, cu_seqlens, h0, do, dht, chunk, workspace)


# ---------------------------------------------------------------- neighbours
NORM_EPS = 1e-6  # the recipe's normalisation epsilon


def _nb_check(name, x, dtype=None, device=None, shape=None):
    if not isinstance(x, torch.Tensor):
        raise GdnError(f"{name} must be a tensor")
    if x.device.type != "cuda":
        raise GdnError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if dtype is not None and x.dtype != dtype:
        raise GdnError(f"{name}: expected {dtype}, got {x.dtype}")
    if device is not None and x.device != device:
        raise GdnError(f"{name}: expected device {device}, got {x.device}")
    if shape is not None and tuple(x.shape) != tuple(shape):
        raise GdnError(f"{name}: expected shape {tuple(shape)}, got {tuple(x.shape)}")
    if not x.is_contiguous():
        raise GdnError(f"{name} must be contiguous")


def _conv_args(x, w, H, cu_seqlens):
    _nb_check("x", x)
    if x.dtype not in _DTYPES or x.dim() != 3:
        raise GdnError("x must be [B, T, H*D] fp32 or bf16")
    B, T, CH = x.shape
    if H <= 0 or CH % H:
        raise GdnError(f"H={H} does not divide the {CH} channels of x")
    _nb_check("w", w, torch.float32, x.device)
    if w.dim() != 2 or w.shape[0] != CH:
        raise GdnError(f"w must be [{CH}, W] fp32")
    nseq = 0
    if cu_seqlens is not None:
        if (cu_seqlens.dtype != torch.int32 or cu_seqlens.device != x.device
                or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1 or not cu_seqlens.is_contiguous()):
            raise GdnError("cu_seqlens must be a contiguous 1-D int32 tensor on x's device")
        nseq = cu_seqlens.numel() - 1
    return ConvShape(B, T, H, CH // H, w.shape[1], _DTYPES[x.dtype]), nseq


def short_conv_fwd(x, w, H, l2norm=False, scale=1.0, eps=NORM_EPS, cu_seqlens=None):
    """Causal depthwise short convolution + SiLU over ``x [B, T, H*D]`` with
    ``w [H*D, W]`` fp32; with ``l2norm`` each head's D outputs of a token are
    scaled to ``scale * y / sqrt(|y|^2 + eps)`` (the q and k inputs of the
    mixer).  ``cu_seqlens`` (int32, B = 1) restarts the convolution at every
    packed sequence.  Returns ``z`` (layout and dtype of x)."""
    s, nseq = _conv_args(x, w, H, cu_seqlens)
    z = torch.empty_like(x)
    _check(lib().gdn_short_conv_fwd(ctypes.byref(s), _ptr(x), _ptr(w), _ptr(z), int(bool(l2norm)),
                                    float(scale), float(eps), _ptr(cu_seqlens), nseq,
                                    _stream(x.device)))
    return z


def short_conv_bwd(x, w, dz, H, l2norm=False, scale=1.0, eps=NORM_EPS, cu_seqlens=None,
                   workspace=None):
    """Gradients of ``short_conv_fwd``: returns ``(dx, dw)`` (dw fp32, a
    reproducible sum over the tokens)."""
    s, nseq = _conv_args(x, w, H, cu_seqlens)
    _nb_check("dz", dz, x.dtype, x.device, x.shape)
    dx = torch.empty_like(x)
    dw = torch.empty_like(w)
    need = int(lib().gdn_short_conv_bwd_workspace(ctypes.byref(s)))
    ws = _workspace(need, workspace, x.device)
    _check(lib().gdn_short_conv_bwd(ctypes.byref(s), _ptr(x), _ptr(w), _ptr(dz), _ptr(dx), _ptr(dw),
                                    int(bool(l2norm)), float(scale), float(eps), _ptr(cu_seqlens),
                                    nseq, _ptr(ws), ws.numel(), _stream(x.device)))
    return dx, dw


def _norm_args(o, gate, weight):
    _nb_check("o", o)
    if o.dtype not in _DTYPES or o.dim() < 1:
        raise GdnError("o must be [..., D] fp32 or bf16")
    _nb_check("gate", gate, o.dtype, o.device, o.shape)
    D = o.shape[-1]
    _nb_check("weight", weight, torch.float32, o.device, (D,))
    return NormShape(o.numel() // D if D else 0, D, _DTYPES[o.dtype])


def gated_rmsnorm_fwd(o, gate, weight, eps=NORM_EPS):
    """``o / sqrt(mean(o^2) + eps) * weight * SiLU(gate)`` over the last
    dimension of ``o`` (e.g. the mixer output ``[B, T, H, dv]``); ``weight``
    ``[D]`` fp32.  Returns ``out`` (layout and dtype of o)."""
    s = _norm_args(o, gate, weight)
    out = torch.empty_like(o)
    _check(lib().gdn_gated_rmsnorm_fwd(ctypes.byref(s), _ptr(o), _ptr(gate), _ptr(weight), _ptr(out),
                                       float(eps), _stream(o.device)))
    return out


def gated_rmsnorm_bwd(o, gate, weight, dout, eps=NORM_EPS, workspace=None):
    """Gradients of ``gated_rmsnorm_fwd``: returns ``(do, dgate, dweight)``."""
    s = _norm_args(o, gate, weight)
    _nb_check("dout", dout, o.dtype, o.device, o.shape)
    d_o, dgate = torch.empty_like(o), torch.empty_like(gate)
    dweight = torch.empty_like(weight)
    need = int(lib().gdn_gated_rmsnorm_bwd_workspace(ctypes.byref(s)))
    ws = _workspace(need, workspace, o.device)
    _check(lib().gdn_gated_rmsnorm_bwd(ctypes.byref(s), _ptr(o), _ptr(gate), _ptr(weight), _ptr(dout),
                                       _ptr(d_o), _ptr(dgate), _ptr(dweight), float(eps), _ptr(ws),
                                       ws.numel(), _stream(o.device)))
    return d_o, dgate, dweight


def _decode(kda, q, k, v, g, beta, state=None, inplace=True, chunk=64):
    B, T, H, dk = q.shape
    dv = v.shape[3]
    _validate(q, k, v, g, beta, kda, [("state", (state, (B, H, dk, dv), torch.float32))])
    o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    ht = state if (inplace and state is not None) else torch.empty(
        (B, H, dk, dv), dtype=torch.float32, device=q.device)
    s = make_shape(q, v, chunk, g)
    fn = lib().kda_decode if kda else lib().gdn_decode
    _check(fn(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
              _ptr(o), _ptr(ht), _stream(q.device)))
    return o, ht


def gdn_decode(q, k, v, g, beta, state=None, inplace=True):
    """GDN forward run token by token (decode; a few tokens per sequence).
    Returns ``(o, ht)``; with ``inplace`` (and a ``state``) the state tensor is
    updated in place and returned as ``ht``.  ``state`` None is the zero state."""
    return _decode(False, q, k, v, g, beta, state, inplace)


def kda_decode(q, k, v, g, beta, state=None, inplace=True):
    """KDA forward run token by token (``g`` is ``[B,T,H,dk]``); see ``gdn_decode``."""
    return _decode(True, q, k, v, g, beta, state, inplace)


def wait_selftest(max_tries=5):
    """Runs the device-side timeout path once (see gdn_wait_selftest in gdn.h)."""
    _check(lib().gdn_wait_selftest(max_tries, _stream(torch.device("cuda", torch.cuda.current_device()))))


def device_status() -> int:
    """Reads and clears the device status word (0 = OK, -7 = a wait timed out)."""
    return int(lib().gdn_device_status())


class KernelTimer:
    """Times every kernel the library launches from this thread with CUDA
    events recorded on the launch stream (the ABI's gdn_profile_* hook).

    ``with KernelTimer(cap) as t: ...`` then ``t.records()`` gives a list of
    ``(kernel_name, ms)`` in launch order and ``t.launches`` the launch count."""

    def __init__(self, cap=4096):
        self.cap = cap
        self.launches = 0

    def __enter__(self):
        _check(lib().gdn_profile_begin(self.cap))
        return self

    def __exit__(self, *exc):
        self.launches = int(lib().gdn_profile_end())
        return False

    def records(self):
        ids = (ctypes.c_int * self.cap)()
        ms = (ctypes.c_float * self.cap)()
        n = lib().gdn_profile_read(ids, ms, self.cap)
        if n < 0:
            _check(n)
        return [(lib().gdn_kernel_name(ids[i]).decode(), float(ms[i])) for i in range(n)]


class GatedDeltaRule(torch.autograd.Function):
    """Autograd wrapper: forward via ``*_fwd`` (``*_fwd_save`` with
    ``save_context``), backward via ``*_bwd`` (``*_bwd_saved``).  The inputs
    are saved; with ``save_context`` the forward also keeps the per-chunk
    entry states and solve results (``ctx_bytes``) instead of the backward
    recomputing them."""

    @staticmethod
    def forward(ctx, q, k, v, g, beta, h0, chunk, kda, save_context, delta=True):
        saved = new_ctx(q, v, chunk, kda, delta) if save_context else None
        o, ht = _fwd(kda, q, k, v, g, beta, h0, chunk, True, ctx=saved, delta=delta)
        ctx.save_for_backward(q, k, v, g, beta, h0)
        ctx.chunk, ctx.kda, ctx.saved, ctx.delta = chunk, kda, saved, delta
        return o, ht

    @staticmethod
    def backward(ctx, do, dht):
        q, k, v, g, beta, h0 = ctx.saved_tensors
        gr = _bwd(ctx.kda, q, k, v, g, beta, h0, do.contiguous(),
                  None if dht is None else dht.contiguous(), ctx.chunk, h0 is not None,
                  ctx=ctx.saved, delta=ctx.delta)
        ctx.saved = None
        return (gr["dq"], gr["dk"], gr["dv"], gr["dg"], gr["dbeta"], gr["dh0"], None, None,
                None, None)


def gated_delta_rule(q, k, v, g, beta, h0=None, chunk=64, kda=False, save_context=True,
                     delta=True):
    """Differentiable mixer: returns ``(o, final_state)``.  ``save_context``
    trades ``ctx_bytes`` of device memory per call for a faster backward;
    ``delta=False`` selects the Mamba2 mixer (no delta rule, scalar gate)."""
    _mixer(kda, delta)
    return GatedDeltaRule.apply(q, k, v, g, beta, h0, chunk, kda, save_context, delta)
