"""Chunkwise form of the gated delta rule in numpy fp64 (test-side restatement).

This is the chunk algorithm the CUDA kernels implement, written as plainly as
possible so that the tests can pin it against the token-by-token oracle:
forward for every chunk size (including a ragged tail), and the reverse chunk
scan for the backward pass.  It does not import the oracle or the library.

Per sequence and chunk of n tokens, with gamma = within-chunk cumulative sum
of the log gate (per key dimension for KDA, broadcast over it for GDN) and
Gam[r,j,d] = exp(gamma[r,d] - gamma[j,d]) for j <= r (0 above the diagonal):

    A = strict_lower( beta_r * sum_d k_rd k_jd Gam[r,j,d] )
    R = V - (K * E) H_in,           E = exp(gamma)
    U = (I + A)^-1 diag(beta) R     (the WY / UT transform)
    P = lower_incl( sum_d q_rd k_jd Gam[r,j,d] )
    O = (Q * E) H_in + P U
    H_out = diag(exp(gamma_last)) H_in + (K * exp(gamma_last - gamma))^T U

The backward pass walks the chunks in reverse, given dO and the gradient of
H_out, and returns the gradient of H_in for the previous chunk.  Log-gate
gradients are accumulated per position as d(gamma) and turned into d(g) by a
reverse cumulative sum inside the chunk.
"""
from __future__ import annotations

import numpy as np


def _chunk_gates(g_chunk, dk, kda):
    gam = np.cumsum(g_chunk, axis=0)
    if not kda:
        gam = np.repeat(gam[:, None], dk, axis=1)
    n = gam.shape[0]
    diff = gam[:, None, :] - gam[None, :, :]          # [r, j, d]
    mask = np.tril(np.ones((n, n), dtype=bool))
    Gam = np.where(mask[:, :, None], np.exp(np.where(mask[:, :, None], diff, 0.0)), 0.0)
    return gam, Gam, mask


def chunk_forward(Q, K, V, g, beta, H_in, kda, delta=True):
    """One chunk's output and exit state.  ``delta=False`` drops the delta
    rule (the Mamba2 mixer): A = 0 and R = V, so U = diag(beta) V."""
    dk = K.shape[1]
    n = K.shape[0]
    gam, Gam, mask = _chunk_gates(g, dk, kda)
    E = np.exp(gam)
    F = np.exp(gam[-1][None, :] - gam)
    KKg = np.einsum("rd,jd,rjd->rj", K, K, Gam)
    A = np.tril(beta[:, None] * KKg, -1) if delta else np.zeros((n, n))
    L = np.eye(n) + A
    R = V - (K * E) @ H_in if delta else V
    U = np.linalg.solve(L, beta[:, None] * R)
    P = np.einsum("rd,jd,rjd->rj", Q, K, Gam) * mask
    O = (Q * E) @ H_in + P @ U
    H_out = np.exp(gam[-1])[:, None] * H_in + (K * F).T @ U
    return O, H_out


def forward(q, k, v, g, beta, h0, chunk, kda=False, delta=True):
    """Chunked forward over [B,T,H,*] inputs; returns (o, ht)."""
    B, T, H, dk = q.shape
    dv = v.shape[3]
    o = np.zeros((B, T, H, dv))
    ht = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if h0 is None else h0[b, h].astype(np.float64)
            for c0 in range(0, T, chunk):
                c1 = min(T, c0 + chunk)
                o[b, c0:c1, h], S = chunk_forward(q[b, c0:c1, h], k[b, c0:c1, h], v[b, c0:c1, h],
                                                  g[b, c0:c1, h], beta[b, c0:c1, h], S, kda, delta)
            ht[b, h] = S
    return o, ht


def chunk_backward(Q, K, V, g, beta, H_in, dO, dH_out, kda, delta=True):
    """Gradients of one chunk; returns (dQ, dK, dV, dg, dbeta, dH_in)."""
    dk = K.shape[1]
    n = K.shape[0]
    gam, Gam, mask = _chunk_gates(g, dk, kda)
    E = np.exp(gam)
    eC = np.exp(gam[-1])
    F = np.exp(gam[-1][None, :] - gam)
    KKg = np.einsum("rd,jd,rjd->rj", K, K, Gam)
    A = np.tril(beta[:, None] * KKg, -1) if delta else np.zeros((n, n))
    L = np.eye(n) + A
    R = V - (K * E) @ H_in if delta else V
    U = np.linalg.solve(L, beta[:, None] * R)
    P = np.einsum("rd,jd,rjd->rj", Q, K, Gam) * mask

    dgam = np.zeros((n, dk))
    # H_out = diag(eC) H_in + (K*F)^T U
    dH_in = eC[:, None] * dH_out
    dgam[-1] += eC * np.sum(dH_out * H_in, axis=1)
    UdH = U @ dH_out.T                                   # [n, dk]
    dK = F * UdH
    dF = K * UdH
    dgam[-1] += np.sum(dF * F, axis=0)
    dgam -= dF * F
    dU = (K * F) @ dH_out
    # O = (Q*E) H_in + P U
    dQE = dO @ H_in.T
    dQ = E * dQE
    dgam += Q * E * dQE
    dH_in += (Q * E).T @ dO
    dP = (dO @ U.T) * mask
    dU += P.T @ dO
    # P[r,j] = sum_d q_rd k_jd Gam[r,j,d]
    dQP = np.einsum("rj,jd,rjd->rd", dP, K, Gam)
    dKP = np.einsum("rj,rd,rjd->jd", dP, Q, Gam)
    dQ += dQP
    dK += dKP
    dgam += Q * dQP - K * dKP
    # U = L^-1 diag(beta) R
    dZ = np.linalg.solve(L.T, dU)
    dA = np.tril(-dZ @ U.T, -1) if delta else np.zeros((n, n))
    dbeta = np.sum(dZ * R, axis=1) + np.sum(dA * KKg, axis=1)
    dR = beta[:, None] * dZ
    # R = V - (K*E) H_in
    dV = dR
    if delta:
        dKE = -dR @ H_in.T
        dK += E * dKE
        dgam += K * E * dKE
        dH_in -= (K * E).T @ dR
    # A[r,j] = beta_r sum_d k_rd k_jd Gam[r,j,d]   (j < r)
    dAt = dA * beta[:, None]
    X = np.einsum("rj,jd,rjd->rd", dAt, K, Gam)
    Y = np.einsum("rj,rd,rjd->jd", dAt, K, Gam)
    dK += X + Y
    dgam += K * X - K * Y
    # gamma = cumsum(g)
    dg = np.cumsum(dgam[::-1], axis=0)[::-1]
    if not kda:
        dg = dg.sum(axis=1)
    return dQ, dK, dV, dg, dbeta, dH_in


def backward(q, k, v, g, beta, h0, do, dht, chunk, kda=False, delta=True):
    """Chunked backward (state recompute, then reverse chunk scan)."""
    B, T, H, dk = q.shape
    dv = v.shape[3]
    out = {n: np.zeros(x.shape) for n, x in (("dq", q), ("dk", k), ("dv", v), ("dg", g),
                                               ("dbeta", beta))}
    out["dh0"] = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if h0 is None else h0[b, h].astype(np.float64)
            starts = list(range(0, T, chunk))
            states = []
            for c0 in starts:
                c1 = min(T, c0 + chunk)
                states.append(S)
                _, S = chunk_forward(q[b, c0:c1, h], k[b, c0:c1, h], v[b, c0:c1, h],
                                     g[b, c0:c1, h], beta[b, c0:c1, h], S, kda, delta)
            dS = np.zeros((dk, dv)) if dht is None else dht[b, h].astype(np.float64)
            for ci in reversed(range(len(starts))):
                c0 = starts[ci]
                c1 = min(T, c0 + chunk)
                sl = slice(c0, c1)
                dQ, dK, dV, dg, db, dS = chunk_backward(q[b, sl, h], k[b, sl, h], v[b, sl, h],
                                                        g[b, sl, h], beta[b, sl, h], states[ci],
                                                        do[b, sl, h], dS, kda, delta)
                out["dq"][b, sl, h] = dQ
                out["dk"][b, sl, h] = dK
                out["dv"][b, sl, h] = dV
                out["dg"][b, sl, h] = dg
                out["dbeta"][b, sl, h] = db
            out["dh0"][b, h] = dS
    return out


# ---------------------------------------------------------------- factored operands
#
# The same chunk forward written the way a tensor-core kernel forms it: every
# decay folded into element-scaled operand tiles, so that each intra-chunk
# product is one plain matrix product.  Around a per-key-dimension reference
# lam_d (the midpoint of the chunk's gamma range in that dimension),
#     exp(gamma_rd - gamma_jd) = exp(gamma_rd - lam_d) * exp(lam_d - gamma_jd),
# each factor at most exp(half the range); the form is usable while that stays
# below the fp32 / bf16 exponent range (FACTOR_LIMIT).

FACTOR_LIMIT = 80.0


def bf16_round(x):
    """Round to the nearest bfloat16 (ties to even), returned as float64."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def chunk_forward_factored(Q, K, V, g, beta, H_in, kda, operand=None):
    """One chunk's forward from element-scaled operands; returns (O, H_out, ok).

    ``operand`` (e.g. ``bf16_round``) is applied to every matrix that enters a
    product as an operand -- the scaled K and Q tiles, T, the bf16 copy of the
    state and U -- while sums stay fp64, as tensor cores accumulate in fp32.
    ``ok`` is False when a dimension's gamma range exceeds 2 * FACTOR_LIMIT
    (the kernel then needs its exact per-element path)."""
    rnd = operand if operand is not None else (lambda x: x)
    dk = K.shape[1]
    n = K.shape[0]
    gam = np.cumsum(g, axis=0)
    if not kda:
        gam = np.repeat(gam[:, None], dk, axis=1)
    lam = 0.5 * (gam.max(axis=0) + gam.min(axis=0))
    ok = bool(np.all(gam.max(axis=0) - gam.min(axis=0) <= 2 * FACTOR_LIMIT))
    Kp = rnd(K * np.exp(gam - lam))
    Km = rnd(K * np.exp(lam - gam))
    Qp = rnd(Q * np.exp(gam - lam))
    KE = rnd(K * np.exp(gam))
    QE = rnd(Q * np.exp(gam))
    KF = rnd(K * np.exp(gam[-1][None, :] - gam))
    A = np.tril(beta[:, None] * (Kp @ Km.T), -1)
    P = np.tril(Qp @ Km.T)
    T = rnd(np.linalg.inv(np.eye(n) + A))
    G = rnd(H_in)                                   # the state as an operand
    U = T @ (beta[:, None] * (rnd(V) - KE @ G))
    Ur = rnd(U)
    O = QE @ G + rnd(P) @ Ur
    H_out = np.exp(gam[-1])[:, None] * H_in + KF.T @ Ur
    return O, H_out, ok


def forward_factored(q, k, v, g, beta, h0, chunk, kda=False, operand=None):
    """Chunked forward through ``chunk_forward_factored``; returns (o, ht, ok)."""
    B, T, H, dk = q.shape
    dv = v.shape[3]
    o = np.zeros((B, T, H, dv))
    ht = np.zeros((B, H, dk, dv))
    ok = True
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if h0 is None else h0[b, h].astype(np.float64)
            for c0 in range(0, T, chunk):
                c1 = min(T, c0 + chunk)
                o[b, c0:c1, h], S, fine = chunk_forward_factored(
                    q[b, c0:c1, h], k[b, c0:c1, h], v[b, c0:c1, h], g[b, c0:c1, h],
                    beta[b, c0:c1, h], S, kda, operand)
                ok = ok and fine
            ht[b, h] = S
    return o, ht, ok


def chunk_backward_factored(Q, K, V, g, beta, H_in, dO, dH_out, kda, operand=None,
                            scaled_operand=None):
    """``chunk_backward`` from element-scaled operands; returns
    (dQ, dK, dV, dg, dbeta, dH_in).  Each decayed sum over a row or column of
    a chunk matrix is one product with a scaled tile and a row scaling:
        sum_j M[r,j] K[j,d] Gam[r,j,d] = exp(gamma_rd - lam_d) (M Km)[r,d]
        sum_r M[r,j] X[r,d] Gam[r,j,d] = exp(lam_d - gamma_jd) (M^T Xp)[j,d]
    with Km = K exp(lam - gamma), Xp = X exp(gamma - lam).  ``operand`` rounds
    every product operand, as in ``chunk_forward_factored``; ``scaled_operand``,
    if given, rounds the three scaled tiles Kp, Km, Qp instead."""
    rnd = operand if operand is not None else (lambda x: x)
    srnd = scaled_operand if scaled_operand is not None else rnd
    dk = K.shape[1]
    n = K.shape[0]
    gam = np.cumsum(g, axis=0)
    if not kda:
        gam = np.repeat(gam[:, None], dk, axis=1)
    lam = 0.5 * (gam.max(axis=0) + gam.min(axis=0))
    Ep, Em = np.exp(gam - lam), np.exp(lam - gam)
    E, eC, F = np.exp(gam), np.exp(gam[-1]), np.exp(gam[-1][None, :] - gam)
    mask = np.tril(np.ones((n, n), dtype=bool))
    Kp, Km, Qp = srnd(K * Ep), srnd(K * Em), srnd(Q * Ep)
    KE, QE, KF = rnd(K * E), rnd(Q * E), rnd(K * F)
    KKs = np.tril(Kp @ Km.T, -1)                    # strictly lower decayed K K^T
    L = np.eye(n) + beta[:, None] * KKs
    T = rnd(np.linalg.inv(L))
    G = rnd(H_in)
    R = V - KE @ G
    U = T @ (beta[:, None] * rnd(R))
    Ur = rnd(U)
    P = np.tril(Qp @ Km.T)
    dOr, dHr = rnd(dO), rnd(dH_out)

    dgam = np.zeros((n, dk))
    dH_in = eC[:, None] * dH_out
    dgam[-1] += eC * np.sum(dH_out * H_in, axis=1)
    UdH = U @ dH_out.T
    dK = F * UdH
    dF = K * UdH
    dgam[-1] += np.sum(dF * F, axis=0)
    dgam -= dF * F
    dU = KF @ dHr + rnd(P).T @ dOr
    dQE = dOr @ G.T
    dQ = E * dQE
    dgam += Q * E * dQE
    dH_in += QE.T @ dOr
    dP = rnd((dOr @ Ur.T) * mask)
    dQP = Ep * (dP @ Km)
    dKP = Em * (dP.T @ Qp)
    dQ += dQP
    dK += dKP
    dgam += Q * dQP - K * dKP
    dZ = T.T @ dU
    dA = np.tril(-rnd(dZ) @ Ur.T, -1)
    dbeta = np.sum(dZ * R, axis=1) + np.sum(dA * KKs, axis=1)
    dR = beta[:, None] * dZ
    dRr = rnd(dR)
    dV = dR
    dKE = -dRr @ G.T
    dK += E * dKE
    dgam += K * E * dKE
    dH_in -= KE.T @ dRr
    dAt = rnd(dA * beta[:, None])
    X = Ep * (dAt @ Km)
    Y = Em * (dAt.T @ Kp)
    dK += X + Y
    dgam += K * X - K * Y
    dg = np.cumsum(dgam[::-1], axis=0)[::-1]
    if not kda:
        dg = dg.sum(axis=1)
    return dQ, dK, dV, dg, dbeta, dH_in


def backward_factored(q, k, v, g, beta, h0, do, dht, chunk, kda=False, operand=None,
                      scaled_operand=None):
    """``backward`` through the factored chunk forms (entry states from the
    factored forward at the same operand precision)."""
    B, T, H, dk = q.shape
    dv = v.shape[3]
    out = {n: np.zeros(x.shape) for n, x in (("dq", q), ("dk", k), ("dv", v), ("dg", g),
                                               ("dbeta", beta))}
    out["dh0"] = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if h0 is None else h0[b, h].astype(np.float64)
            starts = list(range(0, T, chunk))
            states = []
            for c0 in starts:
                c1 = min(T, c0 + chunk)
                states.append(S)
                _, S, _ = chunk_forward_factored(q[b, c0:c1, h], k[b, c0:c1, h], v[b, c0:c1, h],
                                                 g[b, c0:c1, h], beta[b, c0:c1, h], S, kda,
                                                 operand)
            dS = np.zeros((dk, dv)) if dht is None else dht[b, h].astype(np.float64)
            for ci in reversed(range(len(starts))):
                c0 = starts[ci]
                sl = slice(c0, min(T, c0 + chunk))
                dQ, dK, dV, dg, db, dS = chunk_backward_factored(
                    q[b, sl, h], k[b, sl, h], v[b, sl, h], g[b, sl, h], beta[b, sl, h],
                    states[ci], do[b, sl, h], dS, kda, operand, scaled_operand)
                out["dq"][b, sl, h] = dQ
                out["dk"][b, sl, h] = dK
                out["dv"][b, sl, h] = dV
                out["dg"][b, sl, h] = dg
                out["dbeta"][b, sl, h] = db
            out["dh0"][b, h] = dS
    return out

