"""The chunk forward with every decay folded into element-scaled operands
(CPU only): the form a tensor-core KDA kernel takes, since the per-dimension
decays cannot be applied as row scalings of a product the way the scalar GDN
gate is.  Pinned to the chunk form and the oracle, and checked at bf16
operand precision against the bf16 bar (rel-L2 <= 2e-2) for the workloads'
gate distribution and for gates that decay ten times faster.
"""
import os
import sys

import numpy as np
import pytest

import oracle

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import chunk_reference as cr  # noqa: E402


def inputs(T, H, dk, dv, kda, g_mean, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, T, H, dk))
    k = rng.standard_normal((1, T, H, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True) * np.sqrt(dk)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, T, H, dv))
    gshape = (1, T, H, dk) if kda else (1, T, H)
    g = -np.log1p(np.exp(-rng.normal(g_mean, 1.0, gshape)))  # logsigmoid
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((1, T, H))))
    h0 = rng.standard_normal((1, H, dk, dv)) * 0.3
    return q, k, v, g, beta, h0


def rel(x, ref):
    return np.linalg.norm(x - ref) / np.linalg.norm(ref)


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("chunk,T", [(16, 40), (64, 150)])
def test_factored_form_equals_chunk_form(kda, chunk, T):
    x = inputs(T, 2, 24, 16, kda, 2.0, seed=1)
    o_ref, h_ref = cr.forward(*x, chunk, kda)
    o, h, ok = cr.forward_factored(*x, chunk, kda)
    assert ok
    assert rel(o, o_ref) < 1e-12 and rel(h, h_ref) < 1e-12


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("g_mean", [2.0, -1.0])
def test_bf16_operands_meet_the_bf16_bar(kda, g_mean):
    # g_mean 2: the workloads' gates (about -0.13 a token); -1: about -1.3 a
    # token, a 64-token range near 80 in each dimension
    x = inputs(256, 2, 128, 128, kda, g_mean, seed=2)
    o_ref, h_ref = oracle.fwd(*x, kda=kda)
    o, h, ok = cr.forward_factored(*x, 64, kda, operand=cr.bf16_round)
    assert ok
    assert rel(o, o_ref) < 2e-2, rel(o, o_ref)
    assert rel(h, h_ref) < 2e-2, rel(h, h_ref)


def test_ranges_beyond_the_factor_limit_are_flagged():
    # about -6 a token: a 64-token range of ~380, past what the factors can hold
    x = inputs(64, 1, 16, 16, True, -6.0, seed=3)
    _, _, ok = cr.forward_factored(*x, 64, True)
    assert not ok


def grads_inputs(T, H, dk, dv, kda, g_mean, seed):
    x = inputs(T, H, dk, dv, kda, g_mean, seed)
    rng = np.random.default_rng(seed + 100)
    do = rng.standard_normal((1, T, H, dv))
    dht = rng.standard_normal((1, H, dk, dv)) * 0.1
    return x, do, dht


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("chunk,T", [(16, 40), (64, 150)])
def test_factored_backward_equals_chunk_backward(kda, chunk, T):
    x, do, dht = grads_inputs(T, 2, 24, 16, kda, 2.0, seed=4)
    ref = cr.backward(*x, do, dht, chunk, kda)
    got = cr.backward_factored(*x, do, dht, chunk, kda)
    for n in ref:
        assert rel(got[n], ref[n]) < 1e-10, n


def tf32_round(x):
    """Round to 10 explicit mantissa bits (the TF32 operand format), ties to even."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0xFFF + ((u >> 13) & 1)) & 0xFFFFE000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("g_mean", [2.0, -1.0])
def test_factored_backward_with_bf16_operands(kda, g_mean):
    """With the three scaled tiles K exp(+-(gamma - lam)) and Q exp(gamma - lam)
    at TF32 precision and every other operand in bf16, every gradient meets
    the bf16 bar, for the workloads' gates and for gates that decay ten times
    faster.  (With those tiles in bf16 as well, dg at the faster gates is a
    difference of nearly equal decayed sums whose rounding no longer cancels;
    the other gradients are unaffected, which is checked too.)"""
    x, do, dht = grads_inputs(192, 1, 128, 128, kda, g_mean, seed=5)
    ref = oracle.bwd(*x, do, dht, kda=kda)
    mixed = cr.backward_factored(*x, do, dht, 64, kda, operand=cr.bf16_round,
                                 scaled_operand=tf32_round)
    for n in ref:
        assert rel(mixed[n], ref[n]) < 1e-2, (n, rel(mixed[n], ref[n]))
    got = cr.backward_factored(*x, do, dht, 64, kda, operand=cr.bf16_round)
    for n in ref:
        if n != "dg":
            assert rel(got[n], ref[n]) < 2e-2, (n, rel(got[n], ref[n]))

