"""C-ABI library: loads, exports every declared symbol, validates on the host.

These run without a GPU: every call here returns from host-side argument
validation before anything is enqueued (or has no work: B = 0).
"""
import ctypes
import os
import re

import pytest

import gated_delta_rule_bwd_gb300 as gdn
from gated_delta_rule_bwd_gb300 import build as gbuild

HEADER = os.path.join(gbuild.INCLUDE, "gdn.h")

GDN_OK, GDN_ERR_ARG, GDN_ERR_SHAPE, GDN_ERR_DTYPE, GDN_ERR_ALIGN, GDN_ERR_WORKSPACE = 0, -1, -2, -3, -4, -5


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return gdn.lib()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"GDN_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_abi():
    names = set(declared_symbols())
    assert {"gdn_fwd", "gdn_bwd", "kda_fwd", "kda_bwd", "gdn_bwd_workspace",
            "kda_bwd_workspace", "gdn_status_str"} <= names


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name


def test_only_the_abi_is_exported(L):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", gdn.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(declared_symbols())


def shape(B=1, T=64, H=2, dk=16, dv=16, chunk=16, dtype=0):
    return gdn.GdnShape(B, T, H, dk, dv, chunk, dtype)


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails or B = 0 first


def call_fwd(L, s, kda=False, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, h0=None, o=FAKE, ht=None)
    args.update(over)
    fn = L.kda_fwd if kda else L.gdn_fwd
    return fn(ctypes.byref(s), args["q"], args["k"], args["v"], args["g"], args["beta"],
              args["h0"], args["o"], args["ht"], None, 0, None)


def call_bwd(L, s, ws=None, ws_bytes=0, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, h0=None, do=FAKE, dht=None, dq=FAKE,
             dk=FAKE, dv=FAKE, dg=FAKE, dbeta=FAKE, dh0=None)
    a.update(over)
    return L.gdn_bwd(ctypes.byref(s), a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], a["do"],
                     a["dht"], a["dq"], a["dk"], a["dv"], a["dg"], a["dbeta"], a["dh0"], ws,
                     ws_bytes, None)


def test_shape_validation(L):
    assert call_fwd(L, shape(chunk=17)) == GDN_ERR_SHAPE
    assert call_fwd(L, shape(chunk=128)) == GDN_ERR_SHAPE
    assert call_fwd(L, shape(dk=0)) == GDN_ERR_SHAPE
    assert call_fwd(L, shape(dv=129)) == GDN_ERR_SHAPE
    assert call_fwd(L, shape(T=-1)) == GDN_ERR_SHAPE
    assert call_fwd(L, shape(dtype=7)) == GDN_ERR_DTYPE
    assert L.gdn_fwd(None, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, None, 0, None) == GDN_ERR_ARG


def test_null_and_alignment_checks(L):
    assert call_fwd(L, shape(), q=None) == GDN_ERR_ARG
    assert call_fwd(L, shape(), o=None) == GDN_ERR_ARG
    assert call_fwd(L, shape(), kda=True, beta=None) == GDN_ERR_ARG
    assert call_fwd(L, shape(), v=ctypes.c_void_p(0x10008)) == GDN_ERR_ALIGN
    assert call_bwd(L, shape(), dg=ctypes.c_void_p(0x10004)) == GDN_ERR_ALIGN
    assert call_bwd(L, shape(), do=None) == GDN_ERR_ARG


def test_workspace_query_and_check(L):
    s = shape()
    need = L.gdn_bwd_workspace(ctypes.byref(s))
    assert need > 0
    assert L.gdn_bwd_workspace(ctypes.byref(shape(chunk=3))) == 0
    assert call_bwd(L, s) == GDN_ERR_WORKSPACE
    assert call_bwd(L, s, ws=FAKE, ws_bytes=need - 1) == GDN_ERR_WORKSPACE
    # chunk-entry states of the recompute pass: B*H*N*dk*dv values at least
    # (bf16 on the tensor-core path, fp32 on the CUDA-core path)
    big = shape(B=2, T=2048, H=4, dk=128, dv=128, chunk=64, dtype=1)
    assert L.gdn_bwd_workspace(ctypes.byref(big)) >= 2 * 4 * 32 * 128 * 128 * 2
    assert L.kda_bwd_workspace(ctypes.byref(big)) >= 2 * 4 * 32 * 128 * 128 * 4
    f32 = shape(B=2, T=2048, H=4, dk=128, dv=128, chunk=64, dtype=0)
    assert L.gdn_bwd_workspace(ctypes.byref(f32)) >= 2 * 4 * 32 * 128 * 128 * 4
    # the tensor-core path also keeps T = (I + A)^-1 of every chunk (bf16 64 x 64)
    assert L.gdn_bwd_workspace(ctypes.byref(big)) >= 2 * 4 * 32 * (128 * 128 + 64 * 64) * 2


def test_forward_workspace_query_and_check(L):
    big = shape(B=2, T=2048, H=4, dk=128, dv=128, chunk=64, dtype=1)
    need = L.gdn_fwd_workspace(ctypes.byref(big))
    assert need >= 2 * 4 * 32 * 64 * 64 * 2      # T of every chunk, bf16
    assert need <= L.gdn_bwd_workspace(ctypes.byref(big))
    assert call_fwd(L, big) == GDN_ERR_WORKSPACE
    fn = L.gdn_fwd
    args = (ctypes.byref(big), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None)
    assert fn(*args, FAKE, need - 1, None) == GDN_ERR_WORKSPACE
    assert fn(*args, ctypes.c_void_p(0x10008), need, None) == GDN_ERR_ALIGN
    # few sequences with many chunks: the forward runs in segments and also
    # keeps three fp32 dk x dv states per segment
    long = shape(B=1, T=64 * 1024, H=2, dk=128, dv=128, chunk=64, dtype=1)
    assert L.gdn_fwd_workspace(ctypes.byref(long)) > 2 * 1024 * 64 * 64 * 2 + 3 * 2 * 128 * 128 * 4
    # the CUDA-core paths (fp32) need none
    f32 = shape(B=2, T=2048, H=4, dk=128, dv=128, chunk=64, dtype=0)
    assert L.gdn_fwd_workspace(ctypes.byref(f32)) == 0
    assert L.kda_fwd_workspace(ctypes.byref(f32)) == 0
    assert L.gdn_fwd_workspace(ctypes.byref(shape(chunk=3))) == 0
    # the KDA tensor-core forward keeps each chunk's scaled Kp|Qp, Km and T
    # tiles (56 KB) and its factor vectors, plus a flag per sequence
    kda_need = L.kda_fwd_workspace(ctypes.byref(big))
    assert kda_need >= 2 * 4 * 32 * (32768 + 16384 + 8192)
    assert kda_need <= L.kda_bwd_workspace(ctypes.byref(big))
    fn = L.kda_fwd
    assert fn(*args, FAKE, kda_need - 1, None) == GDN_ERR_WORKSPACE


def test_saved_context_size_and_check(L):
    big = shape(B=2, T=2048, H=4, dk=128, dv=128, chunk=64, dtype=1)
    need = L.gdn_ctx_bytes(ctypes.byref(big))
    # the backward's workspace (entry states + T tiles) as the forward leaves it
    assert need >= L.gdn_bwd_workspace(ctypes.byref(big))
    assert need >= L.gdn_fwd_workspace(ctypes.byref(big))
    long = shape(B=1, T=64 * 1024, H=2, dk=128, dv=128, chunk=64, dtype=1)
    assert L.gdn_ctx_bytes(ctypes.byref(long)) >= max(L.gdn_fwd_workspace(ctypes.byref(long)),
                                                      L.gdn_bwd_workspace(ctypes.byref(long)))
    # CUDA-core path: the context is the backward's workspace
    f32 = shape(B=2, T=2048, H=4, dk=128, dv=128, chunk=64, dtype=0)
    assert L.gdn_ctx_bytes(ctypes.byref(f32)) == L.gdn_bwd_workspace(ctypes.byref(f32))
    assert L.kda_ctx_bytes(ctypes.byref(big)) == L.kda_bwd_workspace(ctypes.byref(big))
    assert L.gdn_ctx_bytes(ctypes.byref(shape(B=0))) == 0
    assert L.gdn_ctx_bytes(ctypes.byref(shape(chunk=3))) == 0
    fwd_args = (ctypes.byref(big), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None)
    bwd_args = (ctypes.byref(big),) + (FAKE,) * 5 + (None, FAKE, None) + (FAKE,) * 5 + (None,)
    for fn, args in ((L.gdn_fwd_save, fwd_args), (L.gdn_bwd_saved, bwd_args)):
        assert fn(*args, None, 0, None) == GDN_ERR_WORKSPACE
        # a buffer big enough for the plain pass is still too small for the context
        assert fn(*args, FAKE, need - 1, None) == GDN_ERR_WORKSPACE
        assert fn(*args, ctypes.c_void_p(0x10008), need, None) == GDN_ERR_ALIGN
    assert L.gdn_fwd_save(ctypes.byref(shape(B=0)), *fwd_args[1:], None, 0, None) == GDN_OK
    assert L.kda_bwd_saved(ctypes.byref(shape(H=0)), *bwd_args[1:], None, 0, None) == GDN_OK


def test_decode_validation(L):
    def dec(s, kda=False, **over):
        a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, h0=None, o=FAKE, ht=None)
        a.update(over)
        fn = L.kda_decode if kda else L.gdn_decode
        return fn(ctypes.byref(s), a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], a["o"],
                  a["ht"], None)
    assert dec(shape(chunk=17)) == GDN_ERR_SHAPE
    assert dec(shape(dk=129)) == GDN_ERR_SHAPE
    assert dec(shape(dtype=5)) == GDN_ERR_DTYPE
    assert dec(shape(), q=None) == GDN_ERR_ARG
    assert dec(shape(), kda=True, beta=None) == GDN_ERR_ARG
    assert dec(shape(), o=ctypes.c_void_p(0x10004)) == GDN_ERR_ALIGN
    assert dec(shape(), ht=ctypes.c_void_p(0x10008)) == GDN_ERR_ALIGN
    assert dec(shape(B=0)) == GDN_OK
    # no tokens, state updated in place: nothing to do (nothing is launched)
    assert dec(shape(T=0), q=None, k=None, v=None, g=None, beta=None, o=None, h0=FAKE,
               ht=FAKE) == GDN_OK


def test_empty_batch_is_a_no_op(L):
    assert call_fwd(L, shape(B=0)) == GDN_OK
    assert call_fwd(L, shape(H=0), q=None) == GDN_OK
    assert call_bwd(L, shape(B=0)) == GDN_OK


def test_status_strings(L):
    for code in range(-7, 1):
        assert L.gdn_status_str(code).startswith(b"GDN_")
    assert b"unknown" in L.gdn_status_str(5)


def test_tensor_core_selection_rule(L):
    # only bf16, dk = dv = 128, chunk 64 takes the tensor-core kernels
    for s in (shape(dtype=0, dk=128, dv=128, chunk=64), shape(dtype=1, dk=64, dv=128, chunk=64),
              shape(dtype=1, dk=128, dv=128, chunk=32)):
        assert L.gdn_uses_tensor_cores(ctypes.byref(s)) == 0
    assert L.gdn_uses_tensor_cores(ctypes.byref(shape(dtype=1, dk=128, dv=128, chunk=64))) == 1
    for s in (shape(dtype=0, dk=128, dv=128, chunk=64), shape(dtype=1, dk=128, dv=64, chunk=64)):
        assert L.kda_uses_tensor_cores(ctypes.byref(s)) == 0
    assert L.kda_uses_tensor_cores(ctypes.byref(shape(dtype=1, dk=128, dv=128, chunk=64))) == 1


def test_binding_refuses_cpu_tensors(L):
    import torch
    x = torch.zeros(1, 4, 1, 16)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_fwd(x, x, x, torch.zeros(1, 4, 1), torch.zeros(1, 4, 1), chunk=16)


def test_wait_selftest_validates_its_argument(L):
    assert L.gdn_wait_selftest(0, None) == GDN_ERR_ARG
    assert L.gdn_wait_selftest(1001, None) == GDN_ERR_ARG


def test_varlen_validation(L):
    s1 = shape(B=1, T=100, H=2, dk=128, dv=128, chunk=64, dtype=1)
    need = L.gdn_varlen_workspace(ctypes.byref(s1), 3, 0)
    # the chunk offsets come first, then the forward's T tiles for up to
    # ceil(T / 64) + nseq chunks per head
    assert need >= 2 * (2 + 3) * 64 * 64 * 2
    assert L.gdn_varlen_workspace(ctypes.byref(s1), 3, 1) > need
    assert L.gdn_varlen_workspace(ctypes.byref(shape(B=2)), 3, 0) == 0   # B must be 1
    cu = FAKE
    args = (FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None)
    fn = L.gdn_fwd_varlen
    assert fn(ctypes.byref(shape(B=2, T=100)), cu, 3, *args, FAKE, 1 << 30, None) == GDN_ERR_SHAPE
    assert fn(ctypes.byref(s1), None, 3, *args, FAKE, 1 << 30, None) == GDN_ERR_ARG
    assert fn(ctypes.byref(s1), ctypes.c_void_p(0x10002), 3, *args, FAKE, 1 << 30, None) == GDN_ERR_ALIGN
    assert fn(ctypes.byref(s1), cu, -1, *args, FAKE, 1 << 30, None) == GDN_ERR_SHAPE
    assert fn(ctypes.byref(s1), cu, 3, *args, FAKE, need - 1, None) == GDN_ERR_WORKSPACE
    assert fn(ctypes.byref(s1), cu, 0, *args, None, 0, None) == GDN_OK  # no sequences: nothing to do
    assert L.gdn_status_str(-8).decode().startswith("GDN_ERR_SEQLENS")


def conv_shape(B=1, T=64, H=2, D=128, W=4, dtype=1):
    return gdn.ConvShape(B, T, H, D, W, dtype)


def call_conv_fwd(L, s, x=FAKE, w=FAKE, z=FAKE, eps=1e-6, cu=None, nseq=0):
    return L.gdn_short_conv_fwd(ctypes.byref(s), x, w, z, 1, 1.0, eps, cu, nseq, None)


def call_conv_bwd(L, s, ws=FAKE, ws_bytes=1 << 30, **over):
    a = dict(x=FAKE, w=FAKE, dz=FAKE, dx=FAKE, dw=FAKE)
    a.update(over)
    return L.gdn_short_conv_bwd(ctypes.byref(s), a["x"], a["w"], a["dz"], a["dx"], a["dw"], 1, 1.0,
                                1e-6, None, 0, ws, ws_bytes, None)


def test_short_conv_validation(L):
    for bad in (conv_shape(D=16), conv_shape(D=96), conv_shape(W=0), conv_shape(W=5),
                conv_shape(T=-1), conv_shape(B=1 << 16, T=1 << 15)):
        assert call_conv_fwd(L, bad) == GDN_ERR_SHAPE
    assert call_conv_fwd(L, conv_shape(dtype=3)) == GDN_ERR_DTYPE
    assert call_conv_fwd(L, conv_shape(), eps=-1.0) == GDN_ERR_ARG
    assert call_conv_fwd(L, conv_shape(), eps=float("nan")) == GDN_ERR_ARG
    assert call_conv_fwd(L, conv_shape(), x=None) == GDN_ERR_ARG
    assert call_conv_fwd(L, conv_shape(), z=ctypes.c_void_p(0x10008)) == GDN_ERR_ALIGN
    assert L.gdn_short_conv_fwd(None, FAKE, FAKE, FAKE, 0, 1.0, 1e-6, None, 0, None) == GDN_ERR_ARG
    # packed: B must be 1, nseq >= 0, cu_seqlens 4-byte aligned
    assert call_conv_fwd(L, conv_shape(B=2), cu=FAKE, nseq=2) == GDN_ERR_SHAPE
    assert call_conv_fwd(L, conv_shape(), cu=FAKE, nseq=-1) == GDN_ERR_SHAPE
    assert call_conv_fwd(L, conv_shape(), cu=ctypes.c_void_p(0x10002), nseq=2) == GDN_ERR_ALIGN
    # no token: nothing to do
    assert call_conv_fwd(L, conv_shape(B=0), x=None, z=None) == GDN_OK
    assert call_conv_fwd(L, conv_shape(H=0), x=None, z=None) == GDN_OK


def test_short_conv_workspace(L):
    s = conv_shape(B=16, T=2048, H=8, D=128, W=4)
    need = L.gdn_short_conv_bwd_workspace(ctypes.byref(s))
    # fp32 partial sums of dw [H*D, W]: one row per CTA (one CTA per SM)
    assert 8 * 128 * 4 * 4 <= need <= 4 << 20
    assert L.gdn_short_conv_bwd_workspace(ctypes.byref(conv_shape(D=48))) == 0
    assert call_conv_bwd(L, conv_shape(), ws=None, ws_bytes=0) == GDN_ERR_WORKSPACE
    small = L.gdn_short_conv_bwd_workspace(ctypes.byref(conv_shape()))
    assert call_conv_bwd(L, conv_shape(), ws_bytes=small - 1) == GDN_ERR_WORKSPACE
    assert call_conv_bwd(L, conv_shape(), dw=None) == GDN_ERR_ARG
    assert call_conv_bwd(L, conv_shape(), dx=ctypes.c_void_p(0x10004)) == GDN_ERR_ALIGN


def test_gated_rmsnorm_validation(L):
    def fwd(s, **over):
        a = dict(o=FAKE, gate=FAKE, weight=FAKE, out=FAKE, eps=1e-6)
        a.update(over)
        return L.gdn_gated_rmsnorm_fwd(ctypes.byref(s), a["o"], a["gate"], a["weight"], a["out"],
                                       a["eps"], None)
    ok = gdn.NormShape(1000, 128, 1)
    assert fwd(gdn.NormShape(1000, 100, 1)) == GDN_ERR_SHAPE
    assert fwd(gdn.NormShape(-1, 128, 1)) == GDN_ERR_SHAPE
    assert fwd(gdn.NormShape(1000, 128, 2)) == GDN_ERR_DTYPE
    assert fwd(ok, weight=None) == GDN_ERR_ARG
    assert fwd(ok, eps=-1e-6) == GDN_ERR_ARG
    assert fwd(ok, gate=ctypes.c_void_p(0x10002)) == GDN_ERR_ALIGN
    assert fwd(gdn.NormShape(0, 128, 1), o=None, out=None) == GDN_OK
    need = L.gdn_gated_rmsnorm_bwd_workspace(ctypes.byref(ok))
    assert 128 * 4 <= need <= 600 * 128 * 4
    r = L.gdn_gated_rmsnorm_bwd(ctypes.byref(ok), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6,
                                FAKE, need - 1, None)
    assert r == GDN_ERR_WORKSPACE


def test_neighbour_binding_refuses_cpu_tensors(L):
    import torch
    x = torch.zeros(1, 8, 256, dtype=torch.bfloat16)
    with pytest.raises(gdn.GdnError):
        gdn.short_conv_fwd(x, torch.zeros(256, 4), H=2)
    with pytest.raises(gdn.GdnError):
        gdn.gated_rmsnorm_fwd(x, x, torch.ones(256))


def test_bf16_gate_dtype_is_kda_only(L):
    s = shape(B=1, T=64, H=2, dk=128, dv=128, chunk=64, dtype=2)
    assert call_fwd(L, s) == GDN_ERR_DTYPE                      # GDN
    assert call_fwd(L, s, kda=True, o=None) == GDN_ERR_ARG       # KDA: accepted, then NULL o
    assert L.mamba2_fwd(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, None, 0,
                        None) == GDN_ERR_DTYPE
    assert L.kda_uses_tensor_cores(ctypes.byref(s)) == 1
    assert L.kda_bwd_workspace(ctypes.byref(s)) == L.kda_bwd_workspace(
        ctypes.byref(shape(B=1, T=64, H=2, dk=128, dv=128, chunk=64, dtype=1)))
