"""GPU kernels of the fused neighbours against the fp64 oracle, element by element.

Short convolution (+ SiLU, + the per-head L2 norm) and gated RMS norm,
forward and backward, through the C ABI.  The oracle sees the same bytes
(bf16 values upcast to fp64).  Tolerances, from the arithmetic: the kernels
compute in fp32 and round each output once, so
* bf16 outputs: |x - ref| <= 2^-8 |ref| + 1e-4 rms(ref) elementwise (one
  rounding to 8 significant bits, plus the fp32 arithmetic);
* fp32 outputs (fp32 inputs, and dw / dweight always):
  |x - ref| <= 2e-5 |ref| + 2e-5 rms(ref) elementwise (fp32 sums over a few
  terms; the fast exponential, reciprocal and reciprocal square root are
  within a few ulp), and dw / dweight (sums over every token) within a
  relative L2 error of 1e-5.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_bwd_gb300 as gdn
from gated_delta_rule_bwd_gb300.inputs import make_neighbour_inputs
from oracle import neighbours as nb

pytestmark = pytest.mark.gpu

EPS = 1e-6


def np64(t):
    return t.detach().double().cpu().numpy()


def check(name, got, ref, bf16_out):
    got = np64(got) if torch.is_tensor(got) else got
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    if ref.size == 0:
        return
    rms = np.sqrt(np.mean(ref * ref))
    rel, ab = (2.0 ** -8, 1e-4) if bf16_out else (2e-5, 2e-5)
    err = np.abs(got - ref)
    bound = rel * np.abs(ref) + ab * rms
    i = np.argmax(err - bound)
    assert np.all(err <= bound), (f"{name}: |err| {err.flat[i]:.3e} > bound {bound.flat[i]:.3e} "
                                  f"at {np.unravel_index(i, ref.shape)} (ref {ref.flat[i]:.4e})")


def check_sum(name, got, ref):
    check(name, got, ref, False)
    got = np64(got)
    r = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert r <= 1e-5, f"{name}: rel-L2 {r:.3e}"


def conv_ref(x, w, dz, H, l2norm, scale, cu=None):
    """Oracle over each sequence (packed: one call per sequence)."""
    xs, ws, dzs = np64(x), np64(w), np64(dz)
    if cu is None:
        z, _ = nb.short_conv_fwd(xs, ws, H, l2norm, scale, EPS)
        dx, dw = nb.short_conv_bwd(xs, ws, dzs, H, l2norm, scale, EPS)
        return z, dx, dw
    z, dx = np.zeros_like(xs), np.zeros_like(xs)
    dw = np.zeros_like(ws)
    for a, b in zip(cu[:-1], cu[1:]):
        if b > a:
            z[:, a:b], _ = nb.short_conv_fwd(xs[:, a:b], ws, H, l2norm, scale, EPS)
            dxs, dws = nb.short_conv_bwd(xs[:, a:b], ws, dzs[:, a:b], H, l2norm, scale, EPS)
            dx[:, a:b] = dxs
            dw += dws
    return z, dx, dw


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("l2norm", [False, True])
def test_short_conv_matches_oracle(dtype, D, W, l2norm):
    # T = 77: two full 32-token runs and a ragged one per row; B * T also
    # leaves runs that cross from one row into the next
    H = 2
    x = make_neighbour_inputs(2, 77, H, D, W, dtype=dtype, seed=D + W).to("cuda")
    scale = D ** -0.5 if l2norm else 1.0
    z = gdn.short_conv_fwd(x.x, x.w, H, l2norm, scale)
    dx, dw = gdn.short_conv_bwd(x.x, x.w, x.dz, H, l2norm, scale)
    torch.cuda.synchronize()
    z_ref, dx_ref, dw_ref = conv_ref(x.x, x.w, x.dz, H, l2norm, scale)
    bf = dtype == "bf16"
    check("z", z, z_ref, bf)
    check("dx", dx, dx_ref, bf)
    check_sum("dw", dw, dw_ref)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("l2norm", [False, True])
def test_short_conv_packed_sequences(dtype, l2norm):
    # empty sequences, sequences shorter than the filter, one that spans
    # several 32-token runs, a boundary inside a run
    cu = [0, 0, 2, 3, 40, 40, 105, 106, 150]
    H, D, W = 3, 64, 4
    x = make_neighbour_inputs(1, cu[-1], H, D, W, dtype=dtype, seed=5).to("cuda")
    cut = torch.tensor(cu, dtype=torch.int32, device="cuda")
    z = gdn.short_conv_fwd(x.x, x.w, H, l2norm, 0.5, cu_seqlens=cut)
    dx, dw = gdn.short_conv_bwd(x.x, x.w, x.dz, H, l2norm, 0.5, cu_seqlens=cut)
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    z_ref, dx_ref, dw_ref = conv_ref(x.x, x.w, x.dz, H, l2norm, 0.5, cu)
    bf = dtype == "bf16"
    check("z", z, z_ref, bf)
    check("dx", dx, dx_ref, bf)
    check_sum("dw", dw, dw_ref)


def test_short_conv_invalid_offsets_are_reported():
    """Offsets that do not partition [0, T) set GDN_ERR_SEQLENS; the kernels
    clamp every sequence to the token range, so nothing is read or written
    outside the arrays."""
    H, D = 2, 32
    x = make_neighbour_inputs(1, 64, H, D, 4, seed=1).to("cuda")
    for cu in ([0, 50, 30, 64], [0, 10, 70], [3, 20, 64]):
        cut = torch.tensor(cu, dtype=torch.int32, device="cuda")
        gdn.short_conv_fwd(x.x, x.w, H, True, 1.0, cu_seqlens=cut)
        torch.cuda.synchronize()
        assert gdn.device_status() == -8, cu
        gdn.short_conv_bwd(x.x, x.w, x.dz, H, True, 1.0, cu_seqlens=cut)
        torch.cuda.synchronize()
        assert gdn.device_status() == -8, cu
    assert gdn.device_status() == 0


def test_short_conv_empty_and_deterministic():
    x = make_neighbour_inputs(0, 5, 2, 128, 4).to("cuda")
    z = gdn.short_conv_fwd(x.x, x.w, 2)
    dx, dw = gdn.short_conv_bwd(x.x, x.w, x.dz, 2)
    torch.cuda.synchronize()
    assert z.numel() == 0 and dx.numel() == 0 and torch.all(dw == 0)
    x = make_neighbour_inputs(4, 300, 4, 128, 4, seed=3).to("cuda")
    a = gdn.short_conv_bwd(x.x, x.w, x.dz, 4, True, 0.1)
    b = gdn.short_conv_bwd(x.x, x.w, x.dz, 4, True, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_short_conv_full_size():
    """The 300M pre-training shape (B16 T2048, H8 x D128 = 1024 channels per
    projection, width 4): z and dx on two sampled rows, dw over every row."""
    B, T, H, D = 16, 2048, 8, 128
    x = make_neighbour_inputs(B, T, H, D, 4, seed=11).to("cuda")
    z = gdn.short_conv_fwd(x.x, x.w, H, True, D ** -0.5)
    dx, dw = gdn.short_conv_bwd(x.x, x.w, x.dz, H, True, D ** -0.5)
    torch.cuda.synchronize()
    for b in (0, B - 1):
        sl = slice(b, b + 1)
        zr, dxr, _ = conv_ref(x.x[sl], x.w, x.dz[sl], H, True, D ** -0.5)
        check(f"z[{b}]", z[sl], zr, True)
        check(f"dx[{b}]", dx[sl], dxr, True)
    xs, ws, dzs = np64(x.x), np64(x.w), np64(x.dz)
    _, dw_ref = nb.short_conv_bwd(xs, ws, dzs, H, True, D ** -0.5, EPS)
    check_sum("dw", dw, dw_ref)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("D", [32, 64, 128])
def test_gated_rmsnorm_matches_oracle(dtype, D):
    # 2 x 37 x 3 = 222 rows: not a multiple of a CTA's rows
    x = make_neighbour_inputs(2, 37, 3, D, dtype=dtype, seed=D).to("cuda")
    out = gdn.gated_rmsnorm_fwd(x.o, x.gate, x.weight)
    do, dgate, dweight = gdn.gated_rmsnorm_bwd(x.o, x.gate, x.weight, x.dout)
    torch.cuda.synchronize()
    o, g, w, dout = np64(x.o), np64(x.gate), np64(x.weight), np64(x.dout)
    bf = dtype == "bf16"
    check("out", out, nb.gated_rmsnorm_fwd(o, g, w, EPS), bf)
    ref = nb.gated_rmsnorm_bwd(o, g, w, dout, EPS)
    check("do", do, ref[0], bf)
    check("dgate", dgate, ref[1], bf)
    check_sum("dweight", dweight, ref[2])


def test_gated_rmsnorm_zero_rows_and_full_size():
    # an all-zero row of o gives out = 0 and finite gradients (eps > 0)
    x = make_neighbour_inputs(1, 8, 2, 128, seed=2).to("cuda")
    x.o[0, 3] = 0
    out = gdn.gated_rmsnorm_fwd(x.o, x.gate, x.weight)
    grads = gdn.gated_rmsnorm_bwd(x.o, x.gate, x.weight, x.dout)
    torch.cuda.synchronize()
    assert torch.all(out[0, 3] == 0) and all(torch.isfinite(t).all() for t in grads)
    # the 300M shape: mixer output [16, 2048, 8, 128]
    x = make_neighbour_inputs(16, 2048, 8, 128, seed=13).to("cuda")
    out = gdn.gated_rmsnorm_fwd(x.o, x.gate, x.weight)
    do, dgate, dweight = gdn.gated_rmsnorm_bwd(x.o, x.gate, x.weight, x.dout)
    torch.cuda.synchronize()
    o, g, w, dout = np64(x.o), np64(x.gate), np64(x.weight), np64(x.dout)
    rows = (slice(0, 1), slice(15, 16))
    for sl in rows:
        check("out", out[sl], nb.gated_rmsnorm_fwd(o[sl], g[sl], w, EPS), True)
        ref = nb.gated_rmsnorm_bwd(o[sl], g[sl], w, dout[sl], EPS)
        check("do", do[sl], ref[0], True)
        check("dgate", dgate[sl], ref[1], True)
    check_sum("dweight", dweight, nb.gated_rmsnorm_bwd(o, g, w, dout, EPS)[2])
