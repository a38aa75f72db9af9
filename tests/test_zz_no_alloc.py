"""gdn_bwd_noalloc: the backward pass for callers that cannot allocate.

Some callers cannot call cudaMalloc: an allocator hook that must not re-enter
the allocator, a thread inside a framework that owns all device memory, a
path that forbids allocation once running.  gdn_bwd needs a workspace they
could not provide, so the library offers gdn_bwd_noalloc, which takes its
scratch from a fixed device array built into the library.

This file checks, through the C ABI, that it returns the same gradients as
gdn_bwd, bit for bit (both run the same deterministic kernels on the same
inputs), on two calls in a row -- the second call finds the scratch array as
the first one left it -- for a tensor-core shape and a CUDA-core fp32 shape
(whose workspace is laid out differently inside the array), and that shapes
needing more scratch than the array holds are refused before anything runs.
It is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import gated_delta_rule_bwd_gb300 as gdn
from gated_delta_rule_bwd_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

BF16_REL = 2e-2
GDN_ERR_WORKSPACE = -5


def _noalloc_fn():
    L = gdn.lib()
    fn = L.gdn_bwd_noalloc
    fn.argtypes = [ctypes.POINTER(gdn.GdnShape)] + [ctypes.c_void_p] * 15
    fn.restype = ctypes.c_int
    return fn


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(x, chunk=64):
    """Outputs are allocated here, by the caller; the entry point allocates nothing."""
    out = {"dq": torch.empty_like(x.q), "dk": torch.empty_like(x.k), "dv": torch.empty_like(x.v),
           "dg": torch.empty_like(x.g), "dbeta": torch.empty_like(x.beta),
           "dh0": torch.empty_like(x.h0)}
    s = gdn.make_shape(x.q, x.v, chunk)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = _noalloc_fn()(ctypes.byref(s), _p(x.q), _p(x.k), _p(x.v), _p(x.g), _p(x.beta), _p(x.h0),
                       _p(x.do), _p(x.dht), _p(out["dq"]), _p(out["dk"]), _p(out["dv"]),
                       _p(out["dg"]), _p(out["dbeta"]), _p(out["dh0"]), stream)
    assert rc == 0, gdn.lib().gdn_status_str(rc)
    torch.cuda.synchronize()
    return out


def _rel_l2(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


# B, T, H, dk, dv, chunk, dtype: the tensor-core path, then the CUDA-core fp32 path
SHAPES = [(2, 200, 2, 128, 128, 64, "bf16"), (2, 100, 3, 32, 48, 32, "f32")]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda c: "x".join(map(str, c)))
def test_noalloc_matches_gdn_bwd_on_two_calls_in_a_row(shape):
    B, T, H, dk, dv, chunk, dtype = shape
    for seed in (11, 12):
        x = make_inputs(B, T, H, dk, dv, dtype=dtype, h0_std=0.1, with_dht=True,
                        seed=seed).to("cuda")
        got = _call_noalloc(x, chunk)
        ref = gdn.gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, x.do, x.dht, chunk=chunk)
        torch.cuda.synchronize()
        for name, r in ref.items():
            assert torch.isfinite(got[name].float()).all(), name
            assert _rel_l2(got[name], r) <= BF16_REL, (seed, name)
            assert torch.equal(got[name], r), (seed, name)


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # the 300M pre-training shape needs far more than the built-in scratch
    s = gdn.GdnShape(16, 2048, 8, 128, 128, 64, gdn.GDN_BF16)
    assert gdn.lib().gdn_bwd_workspace(ctypes.byref(s)) > (32 << 20)
    fake = ctypes.c_void_p(0x10000)  # refused on the host before anything is launched
    rc = _noalloc_fn()(ctypes.byref(s), *([fake] * 14), None)
    assert rc == GDN_ERR_WORKSPACE
