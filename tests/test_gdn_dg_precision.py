"""Precision of the tensor-core GDN backward's log-gate gradient (CPU only).

A numpy model of one reverse-scan chunk of the tensor-core backward, with
bf16 rounding at the places the kernel rounds (every MMA operand tile: the T
tile, the entry state, P, beta R, dU, U and U f, dZ, e dR, M, dP o Gam, e dO;
sums and TMEM values in full precision), computes dg the way the kernel does:
from the term decomposition of the chunk's cumulative-log-gate gradient,
whose terms are all full-precision chunk matrices --
  q . (the state term of dQ, a separate accumulator) = e dO . (Q H_in),
  + rowsum - colsum of Z = dP o P and of dA o A,
  - e dR . (K H_in), - s_j with s_j = f_j u_j . (dH^T k_j),
plus the chunk-end state terms, reverse-summed inside the chunk.

The pin: on the inputs of the GPU test of fast-decaying gates
(logsigmoid(N(mu, 1)) gates, mu from the workloads' 2 down to -5, 64-token
gate ranges up to about 320) this form stays within 5e-3 of the oracle's dg.
The scalar gate's rescaling identity dg = revcumsum(q . dq - v . dv) + carry,
which an earlier kernel used, is a difference of two large, nearly equal
sums there; the test also checks that the model reproduces that failure
(so that it does model the rounding that matters).
"""
import os
import sys

import numpy as np
import pytest

import oracle

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import chunk_reference as cr  # noqa: E402

rnd = cr.bf16_round


def chunk_bwd_model(Q, K, V, g, beta, H, dO, dH):
    """One chunk (n = 64 rows) of the tensor-core backward at its rounding
    points; H is the bf16 entry state (dk x dv), dH the fp32 gradient of the
    exit state.  Returns (dH_in, dg_kernel, dg_identity)."""
    n = Q.shape[0]
    gam = np.cumsum(g)
    e, eC, f = np.exp(gam), np.exp(gam[-1]), np.exp(gam[-1] - gam)
    low = np.tril(np.ones((n, n)))
    strict = np.tril(np.ones((n, n)), -1)
    Gam = np.exp(np.where(low > 0, gam[:, None] - gam[None, :], 0.0)) * low
    KK, QK = K @ K.T, Q @ K.T
    A = beta[:, None] * KK * Gam * strict
    T = rnd(np.linalg.inv(np.eye(n) + A))            # the solve kernel's bf16 tile
    P = QK * Gam
    KH = K @ H
    R = V - e[:, None] * KH
    dHb = rnd(dH)                                     # bf16 copy of dG
    dU = f[:, None] * (K @ dHb) + rnd(P).T @ dO
    U = T @ rnd(beta[:, None] * R)
    Ub = rnd(U)
    dZ = T.T @ rnd(dU)
    dR = beta[:, None] * dZ
    edRb = rnd(e[:, None] * dR)
    dA = -(rnd(dZ) @ Ub.T) * strict
    dP = (dO @ Ub.T) * low
    dPG = rnd(dP * Gam)
    edO = rnd(e[:, None] * dO)
    dH_in = eC * dH + Q.T @ edO - K.T @ edRb
    dq1 = edO @ H.T                                   # state term of dQ (own accumulator)
    dq = dq1 + dPG @ K
    s = f * np.sum(U * (K @ dHb), axis=1)             # s_j = f_j u_j . (dG K^T)_j
    carry = eC * np.sum(dH * H) + s.sum()
    Z = dP * P
    Ga = dA * A
    dgam = (np.sum(Q * dq1, axis=1) + Z.sum(1) - Z.sum(0) + Ga.sum(1) - Ga.sum(0)
            - e * np.sum(dR * KH, axis=1) - s)
    dg_kernel = np.cumsum(dgam[::-1])[::-1] + carry
    dlc = np.sum(Q * dq, axis=1) - np.sum(V * dR, axis=1)
    dg_identity = np.cumsum(dlc[::-1])[::-1] + carry
    return dH_in, dg_kernel, dg_identity


def model_backward(q, k, v, g, beta, h0, do, dht):
    """One sequence (T a multiple of 64): entry states from the fp64 chunk
    forward, stored in bf16 (as the saved context holds them)."""
    T = q.shape[0]
    S = h0.astype(np.float64)
    states = []
    for c0 in range(0, T, 64):
        states.append(S)
        _, S = cr.chunk_forward(q[c0:c0 + 64], k[c0:c0 + 64], v[c0:c0 + 64], g[c0:c0 + 64],
                                beta[c0:c0 + 64], S, False)
    dH = dht.astype(np.float64)
    dg_k, dg_id = np.zeros(T), np.zeros(T)
    for ci in reversed(range(T // 64)):
        sl = slice(64 * ci, 64 * ci + 64)
        dH, a, b = chunk_bwd_model(q[sl], k[sl], v[sl], g[sl], beta[sl], rnd(states[ci]),
                                   do[sl], dH)
        dg_k[sl], dg_id[sl] = a, b
    return dg_k, dg_id


def case(mu, h):
    """Head h of the inputs the GPU test of fast-decaying gates uses."""
    from gated_delta_rule_bwd_gb300.inputs import make_inputs
    x = make_inputs(1, 256, 2, 128, 128, dtype="bf16", g_mean=mu, h0_std=0.3, with_dht=True,
                    seed=21)
    tok = lambda t: t[0, :, h].double().numpy()
    return (x, tok(x.q), tok(x.k), tok(x.v), x.g[0, :, h].double().numpy(),
            x.beta[0, :, h].double().numpy(), x.h0[0, h].double().numpy(), tok(x.do),
            x.dht[0, h].double().numpy())


def rel(x, ref):
    return np.linalg.norm(x - ref) / np.linalg.norm(ref)


@pytest.mark.parametrize("mu", [2.0, 0.0, -1.0, -3.0, -5.0])
def test_kernel_dg_form_stays_accurate(mu):
    kern, ident, refs = [], [], []
    for h in range(2):
        x, *args = case(mu, h)
        if h == 0:
            ref = oracle.bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, x.do, x.dht)
        a, b = model_backward(*args)
        kern.append(a)
        ident.append(b)
        refs.append(ref["dg"][0, :, h])
    kern, ident, refs = map(np.concatenate, (kern, ident, refs))
    r_kern, r_id = rel(kern, refs), rel(ident, refs)
    assert r_kern < 5e-3, (r_kern, r_id)
    if mu <= -3:  # the rounding this models does break the rescaling identity here
        assert r_id > 2e-2, (r_kern, r_id)
