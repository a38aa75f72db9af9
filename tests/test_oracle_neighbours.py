"""Pins of the fused-neighbour oracle (CPU only).

The short convolution and the gated norm are checked against what fixes them
independently of the oracle's loops: numpy's convolution routine and torch's
depthwise conv1d / rms_norm / SiLU in fp64 (with torch's own autograd for the
gradients), central finite differences, causality, the unit norm of the
normalised q/k rows (up to the epsilon under the root), and a closed form of the gated norm's RMS.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import neighbours as nb


def conv_inputs(B=2, T=11, H=2, D=3, W=4, seed=0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((B, T, H * D)), rng.standard_normal((H * D, W)) * 0.5


def test_conv_matches_numpy_convolve():
    x, w = conv_inputs()
    _, s = nb.short_conv_fwd(x, w, H=2)
    for b in range(x.shape[0]):
        for c in range(x.shape[2]):
            ref = np.convolve(x[b, :, c], w[c, ::-1])[: x.shape[1]]
            np.testing.assert_allclose(s[b, :, c], ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("l2norm", [False, True])
def test_conv_matches_torch_depthwise_conv_and_autograd(l2norm):
    B, T, H, D, W = 2, 9, 2, 4, 4
    x, w = conv_inputs(B, T, H, D, W, seed=1)
    dz = np.random.default_rng(2).standard_normal(x.shape)
    scale = 0.5 if l2norm else 1.0
    xt = torch.tensor(x, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    s = F.conv1d(xt.transpose(1, 2), wt[:, None, :], padding=W - 1, groups=H * D)[..., :T]
    y = F.silu(s).transpose(1, 2)
    if l2norm:
        y4 = y.reshape(B, T, H, D)
        y = (scale * y4 / torch.sqrt((y4 * y4).sum(-1, keepdim=True) + 1e-6)).reshape(B, T, H * D)
    (y * torch.tensor(dz)).sum().backward()
    z, _ = nb.short_conv_fwd(x, w, H, l2norm, scale)
    np.testing.assert_allclose(z, y.detach().numpy(), rtol=1e-12, atol=1e-12)
    dx, dw = nb.short_conv_bwd(x, w, dz, H, l2norm, scale)
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_conv_is_causal_and_normalised():
    x, w = conv_inputs(B=1, T=12, H=2, D=5)
    z, _ = nb.short_conv_fwd(x, w, H=2, l2norm=True, scale=0.25)
    x2 = x.copy()
    x2[0, 7] += 1.0
    z2, _ = nb.short_conv_fwd(x2, w, H=2, l2norm=True, scale=0.25)
    np.testing.assert_array_equal(z[0, :7], z2[0, :7])
    assert np.max(np.abs(z[0, 7] - z2[0, 7])) > 1e-3
    _, s = nb.short_conv_fwd(x, w, H=2)
    y = (s / (1 + np.exp(-s))).reshape(1, 12, 2, 5)
    ss = np.sum(y * y, axis=-1)
    norms = np.linalg.norm(z.reshape(1, 12, 2, 5), axis=-1)
    np.testing.assert_allclose(norms, 0.25 * np.sqrt(ss / (ss + 1e-6)), rtol=1e-13)
    # an all-zero input row gives a zero (finite) output row
    z0, _ = nb.short_conv_fwd(np.zeros((1, 3, 10)), w, H=2, l2norm=True)
    assert np.all(z0 == 0)


def _fd(f, x, eps=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + eps
        a = f()
        x[i] = old - eps
        b = f()
        x[i] = old
        g[i] = (a - b) / (2 * eps)
    return g


def test_conv_gradients_match_finite_differences():
    x, w = conv_inputs(B=1, T=6, H=2, D=2, W=3, seed=4)
    dz = np.random.default_rng(5).standard_normal(x.shape)
    loss = lambda: float(np.sum(nb.short_conv_fwd(x, w, 2, True, 0.7)[0] * dz))
    dx, dw = nb.short_conv_bwd(x, w, dz, 2, True, 0.7)
    np.testing.assert_allclose(dx, _fd(loss, x), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dw, _fd(loss, w), rtol=1e-6, atol=1e-7)


def norm_inputs(seed=0, shape=(2, 5, 3, 8)):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(shape), rng.standard_normal(shape),
            1.0 + 0.1 * rng.standard_normal(shape[-1]))


def test_gated_norm_matches_torch_and_autograd():
    o, gate, weight = norm_inputs(1)
    dout = np.random.default_rng(2).standard_normal(o.shape)
    ot, gt, wt = (torch.tensor(a, requires_grad=True) for a in (o, gate, weight))
    ref = F.rms_norm(ot, (o.shape[-1],), wt, eps=1e-6) * F.silu(gt)
    (ref * torch.tensor(dout)).sum().backward()
    np.testing.assert_allclose(nb.gated_rmsnorm_fwd(o, gate, weight), ref.detach().numpy(),
                               rtol=1e-12, atol=1e-12)
    do, dg, dw = nb.gated_rmsnorm_bwd(o, gate, weight, dout)
    np.testing.assert_allclose(do, ot.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dg, gt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_gated_norm_closed_form_rms_and_finite_differences():
    o, gate, weight = norm_inputs(3, (1, 3, 2, 6))
    out = nb.gated_rmsnorm_fwd(o, gate, weight, eps=1e-6)
    base = out / (weight * gate / (1 + np.exp(-gate)))
    ms = np.mean(o * o, axis=-1)
    np.testing.assert_allclose(np.sqrt(np.mean(base * base, axis=-1)), np.sqrt(ms / (ms + 1e-6)),
                               rtol=1e-12)
    dout = np.random.default_rng(4).standard_normal(o.shape)
    loss = lambda: float(np.sum(nb.gated_rmsnorm_fwd(o, gate, weight) * dout))
    do, dg, dw = nb.gated_rmsnorm_bwd(o, gate, weight, dout)
    np.testing.assert_allclose(do, _fd(loss, o), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dg, _fd(loss, gate), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dw, _fd(loss, weight), rtol=1e-6, atol=1e-7)
