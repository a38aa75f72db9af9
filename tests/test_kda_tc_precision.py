"""Precision of the KDA tensor-core kernels' formulation (CPU only).

A numpy model of the KDA tensor-core forward and reverse scan at their
rounding points: the prep kernel's scaled bf16 tiles Kp = K o Ep, Km = K o Em,
Qp = Q o Ep (Ep = exp(gamma - lam), Em = exp(lam - gamma), lam the middle of
each key dimension's gamma range in the chunk), the bf16 T tile, the state
kept in the chunk's reference frame and rounded to bf16 as an operand, bf16
copies of every other product operand, fp32 (here fp64) sums.  The backward
follows the kernel: U = beta R + (T - I) beta R and dZ = dU + (T - I)^T dU
with the identity part in full precision, the four dq / dk accumulators, dP's
diagonal kept out of the products, Ep / Em formed in full precision in the
last epilogue, and dg from the scaled tiles.

Pins: every output within 1.5e-2 of the fp64 oracle (the bar is 2e-2) for
the workloads' gates and for per-dimension gates decaying up to about ten
times faster (mu = 0, -1; chunk gate ranges up to about 107, past the
kernels' range limit of 80, which the model does not apply).  dbeta is the
output closest to the bar there; taking T's identity part in full precision
is what keeps it well inside (checked by the ablation below).
"""
import os
import sys

import numpy as np
import pytest

import oracle

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import chunk_reference as cr  # noqa: E402

rnd = cr.bf16_round
C = 64


def prep(K, Q, g):
    gam = np.cumsum(g, axis=0)
    lam = 0.5 * (gam.max(0) + gam.min(0))
    Ep, Em = np.exp(gam - lam), np.exp(lam - gam)
    return dict(Kp=rnd(K * Ep), Km=rnd(K * Em), Qp=rnd(Q * Ep), Ep=Ep, Em=Em, elam=np.exp(lam),
                cf=np.exp(gam[-1] - lam))


def model(q, k, v, g, beta, h0, do, dht, identity_fp32=True, diag_apart=True):
    """One sequence (T a multiple of 64); returns (o, ht, grads)."""
    T, dk = k.shape
    N = T // C
    low, strict = np.tril(np.ones((C, C))), np.tril(np.ones((C, C)), -1)
    pps = [prep(k[C * c:C * c + C], q[C * c:C * c + C], g[C * c:C * c + C]) for c in range(N)]
    # forward, state in each chunk's frame
    Gt = pps[0]["elam"][:, None] * h0
    states, Ts, o = [], [], np.zeros((T, v.shape[1]))
    for c in range(N):
        sl = slice(C * c, C * c + C)
        pp, V, bt = pps[c], v[sl], beta[sl]
        KK = np.tril(pp["Kp"] @ pp["Km"].T, -1)
        Tt = rnd(np.linalg.inv(np.eye(C) + bt[:, None] * KK))
        Gb = rnd(Gt)
        T2 = rnd(Tt * bt[None, :])
        U = T2 @ V - rnd(T2 @ pp["Kp"]) @ Gb
        Ub = rnd(U)
        o[sl] = pp["Qp"] @ Gb + rnd(np.tril(pp["Qp"] @ pp["Km"].T)) @ Ub
        X = Gt + pp["Km"].T @ Ub
        nxt = pps[c + 1]["elam"] if c + 1 < N else np.ones(dk)
        Gt = (pp["cf"] * nxt)[:, None] * X
        states.append(Gb)
        Ts.append(Tt)
    ht = Gt
    # reverse scan
    gr = {n: np.zeros_like(x) for n, x in (("dq", q), ("dk", k), ("dv", v), ("dg", g))}
    gr["dbeta"] = np.zeros(T)
    dGh = pps[N - 1]["cf"][:, None] * dht
    for c in reversed(range(N)):
        sl = slice(C * c, C * c + C)
        pp, V, dO, bt, Gb, Tt = pps[c], v[sl], do[sl], beta[sl], states[c], Ts[c]
        Kp, Km, Qp = pp["Kp"], pp["Km"], pp["Qp"]
        KK = (Kp @ Km.T) * strict
        P = (Qp @ Km.T) * low
        R = V - Kp @ Gb
        TI = Tt - np.eye(C)
        bR = bt[:, None] * R
        U = bR + TI @ rnd(bR) if identity_fp32 else Tt @ rnd(bR)
        Ub = rnd(U)
        dGb = rnd(dGh)
        dU = Km @ dGb + rnd(P).T @ dO
        dZ = dU + TI.T @ rnd(dU) if identity_fp32 else Tt.T @ rnd(dU)
        dR = bt[:, None] * dZ
        dRb = rnd(dR)
        dA = -(rnd(dZ) @ Ub.T) * strict
        dPf = (dO @ Ub.T) * low
        dPd = np.diag(dPf).copy() if diag_apart else np.zeros(C)
        Po = rnd(dPf * strict) if diag_apart else rnd(dPf)
        M = rnd(bt[:, None] * dA)
        aQ = dO @ Gb.T + Po @ Km
        aP = -dRb @ Gb.T + M @ Km
        aF = Ub @ dGb.T
        aM = Po.T @ Qp + M.T @ Kp
        Ep, Em = pp["Ep"], pp["Em"]
        gr["dq"][sl] = Ep * aQ + dPd[:, None] * (Kp * Em)
        gr["dk"][sl] = Ep * aP + Em * (aF + aM) + dPd[:, None] * (Qp * Em)
        gr["dv"][sl] = dR
        gr["dbeta"][sl] = np.sum(dZ * R, 1) + np.sum(dA * KK, 1)
        dgam = Qp * aQ + Kp * aP - Km * (aM + aF)
        carry = np.sum(dGh * Gb, axis=1) + np.sum(Km * aF, axis=0)
        gr["dg"][sl] = np.cumsum(dgam[::-1], 0)[::-1] + carry[None, :]
        dGin = pp["elam"][:, None] * (dGh + Qp.T @ dO - Kp.T @ dRb)
        dGh = pps[c - 1]["cf"][:, None] * dGin if c > 0 else dGin
    gr["dh0"] = dGh
    return o, ht, gr


def errors(mu, **kw):
    from gated_delta_rule_bwd_gb300.inputs import make_inputs
    x = make_inputs(1, 256, 2, 128, 128, kda=True, dtype="bf16", g_mean=mu, h0_std=0.3,
                    with_dht=True, seed=21)
    o_ref, ht_ref = oracle.fwd(x.q, x.k, x.v, x.g, x.beta, x.h0, kda=True)
    ref = oracle.bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, x.do, x.dht, kda=True)
    got = {n: [] for n in ("o", "ht", "dq", "dk", "dv", "dg", "dbeta", "dh0")}
    want = {n: [] for n in got}
    for h in range(2):
        t = lambda a: a[0, :, h].double().numpy()
        o, ht, gr = model(t(x.q), t(x.k), t(x.v), t(x.g), x.beta[0, :, h].double().numpy(),
                          x.h0[0, h].double().numpy(), t(x.do), x.dht[0, h].double().numpy(), **kw)
        got["o"].append(o)
        want["o"].append(o_ref[0, :, h])
        got["ht"].append(ht)
        want["ht"].append(ht_ref[0, h])
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            got[n].append(gr[n])
            want[n].append(ref[n][0, :, h])
        got["dh0"].append(gr["dh0"])
        want["dh0"].append(ref["dh0"][0, h])
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    return {n: rel(np.concatenate([a.ravel() for a in got[n]]),
                   np.concatenate([b.ravel() for b in want[n]])) for n in got}


@pytest.mark.parametrize("mu", [2.0, 0.0, -1.0])
def test_kda_kernel_form_within_the_bf16_bar(mu):
    e = errors(mu)
    assert max(e.values()) < 1.5e-2, e


def test_fp32_identity_part_of_T_reduces_the_dbeta_error():
    base, ablated = errors(-1.0)["dbeta"], errors(-1.0, identity_fp32=False)["dbeta"]
    assert ablated > 1.3 * base, (base, ablated)


def test_dP_diagonal_apart_is_exact():
    """Taking dP's diagonal out of the products and adding it to dq and dk
    changes nothing but rounding: every output agrees to 1e-3 either way."""
    a, b = errors(0.0), errors(0.0, diag_apart=False)
    for n in a:
        assert abs(a[n] - b[n]) < 1e-3, (n, a[n], b[n])
