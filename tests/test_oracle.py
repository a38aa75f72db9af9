"""Pins for the fp64 oracle (CPU only).

The mixer definition (Primus hybrid-LLM pretraining blog, section "How hybrid
models are defined in Primus": GDN = delta rule + one scalar forget gate per
head; KDA = one gate per key dimension) fixes the following facts, each of
which the oracle must reproduce.  Each is computed here without the oracle:

* exact rational brute force of the state-matrix form S_t = a S (I - b k k^T)
  + b v k^T (tiny sizes, fractions.Fraction);
* beta = 0: closed form H_t = exp(sum g) H0 (no write, pure decay);
* mutually orthogonal keys and zero initial state: the delta correction
  vanishes and the output is the quadratic gated-linear-attention form;
* g = 0, beta = 1, orthonormal keys: every stored value is retrieved exactly,
  a repeated key keeps only its latest value;
* small-beta limit: o(eps*beta)/eps -> gated linear attention;
* gradients against central finite differences;
* KDA with a gate broadcast over the key dimension equals GDN;
* running [0, tau) then [tau, T) with the state handed over equals one run,
  forward and backward;
* contraction: with ||k|| = 1, beta in [0,1], g <= 0,
  ||H_t||_2 <= ||H_{t-1}||_2 + beta_t ||v_t||.
"""
import os
import sys
from fractions import Fraction

import numpy as np
import pytest

import oracle

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import chunk_reference  # noqa: E402

RNG = np.random.default_rng(1234)


def rand_inputs(B, T, H, dk, dv, kda=False, h0=True, rng=None, gscale=0.3):
    rng = rng or np.random.default_rng(0)
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    g = -np.abs(rng.standard_normal((B, T, H, dk) if kda else (B, T, H))) * gscale
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    hh = rng.standard_normal((B, H, dk, dv)) * 0.5 if h0 else None
    return q, k, v, g, beta, hh


# ---------------------------------------------------------------- brute force

def _frac_mat(x):
    return [[Fraction(e) for e in row] for row in x]


def _mm(a, b):
    return [[sum(a[i][l] * b[l][j] for l in range(len(b))) for j in range(len(b[0]))]
            for i in range(len(a))]


@pytest.mark.parametrize("kda", [False, True])
def test_exact_state_matrix_form(kda):
    """S-form recurrence in exact rationals; gates a = 1/2, 3/4 (g = log a)."""
    dk, dv, T = 2, 3, 4
    rng = np.random.default_rng(7)
    qi = rng.integers(-3, 4, (T, dk))
    ki = rng.integers(-2, 3, (T, dk))
    vi = rng.integers(-3, 4, (T, dv))
    bets = [Fraction(1, 2), Fraction(1, 3), Fraction(3, 4), Fraction(1)]
    if kda:
        gates = [[Fraction(1, 2), Fraction(3, 4)], [Fraction(1), Fraction(1, 2)],
                 [Fraction(3, 4), Fraction(3, 4)], [Fraction(1, 2), Fraction(1)]]
    else:
        gates = [Fraction(1, 2), Fraction(3, 4), Fraction(1), Fraction(1, 2)]
    S = [[Fraction(0)] * dk for _ in range(dv)]
    o_exact = []
    for t in range(T):
        k = [[Fraction(int(x))] for x in ki[t]]
        v = [[Fraction(int(x))] for x in vi[t]]
        kt = [[Fraction(int(x)) for x in ki[t]]]
        b = bets[t]
        I_bkk = [[(Fraction(1) if i == j else Fraction(0)) - b * k[i][0] * k[j][0]
                  for j in range(dk)] for i in range(dk)]
        if kda:
            Dg = [[gates[t][i] if i == j else Fraction(0) for j in range(dk)] for i in range(dk)]
            left = _mm(S, Dg)
        else:
            left = [[gates[t] * e for e in row] for row in S]
        S = _mm(left, I_bkk)
        vk = _mm(v, kt)
        S = [[S[i][j] + b * vk[i][j] for j in range(dk)] for i in range(dv)]
        q = [[Fraction(int(x))] for x in qi[t]]
        o_exact.append([float(r[0]) for r in _mm(S, q)])
    gf = np.log(np.array([[float(x) for x in row] for row in gates]) if kda
                else np.array([float(x) for x in gates]))
    q = qi.astype(float)[None, :, None, :]
    k = ki.astype(float)[None, :, None, :]
    v = vi.astype(float)[None, :, None, :]
    g = gf[None, :, None, :] if kda else gf[None, :, None]
    beta = np.array([float(x) for x in bets])[None, :, None]
    o, ht = oracle.fwd(q, k, v, g, beta, kda=kda)
    np.testing.assert_allclose(o[0, :, 0], np.array(o_exact), rtol=1e-12, atol=1e-12)
    S_f = np.array([[float(e) for e in row] for row in S])
    np.testing.assert_allclose(ht[0, 0], S_f.T, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- P1: beta = 0

@pytest.mark.parametrize("kda", [False, True])
def test_beta_zero_is_pure_decay(kda):
    q, k, v, g, beta, h0 = rand_inputs(2, 9, 2, 5, 3, kda=kda)
    beta[:] = 0.0
    o, ht = oracle.fwd(q, k, v, g, beta, h0, kda=kda)
    gam = np.cumsum(g, axis=1)
    for b in range(2):
        for h in range(2):
            for t in range(9):
                dec = np.exp(gam[b, t, h])
                Ht = (dec[:, None] if kda else dec) * h0[b, h]
                np.testing.assert_allclose(o[b, t, h], Ht.T @ q[b, t, h], rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(ht[b, h], Ht, rtol=1e-13, atol=1e-14)
    o0, ht0 = oracle.fwd(q, k, v, g, beta, None, kda=kda)
    assert np.all(o0 == 0.0) and np.all(ht0 == 0.0)


# ------------------------------------------------- P2: reduction to gated linear attention

def gla_quadratic(q, k, v, g, beta, kda):
    """o_t = sum_{j<=t} sum_d q_td k_jd exp(gam_td - gam_jd) beta_j v_j (per sequence)."""
    B, T, H, dk = q.shape
    gam = np.cumsum(g, axis=1)
    o = np.zeros(v.shape)
    for b in range(B):
        for h in range(H):
            for t in range(T):
                for j in range(t + 1):
                    if kda:
                        w = np.sum(q[b, t, h] * k[b, j, h] * np.exp(gam[b, t, h] - gam[b, j, h]))
                    else:
                        w = np.exp(gam[b, t, h] - gam[b, j, h]) * (q[b, t, h] @ k[b, j, h])
                    o[b, t, h] += w * beta[b, j, h] * v[b, j, h]
    return o


def test_orthogonal_keys_reduce_to_gla_gdn():
    T, dk, dv = 6, 8, 4
    rng = np.random.default_rng(3)
    q, _, v, g, beta, _ = rand_inputs(1, T, 1, dk, dv, rng=rng, h0=False)
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm[:, :T].T.copy()[None, :, None, :]
    o, _ = oracle.fwd(q, k, v, g, beta)
    np.testing.assert_allclose(o, gla_quadratic(q, k, v, g, beta, False), rtol=1e-12, atol=1e-13)


def test_one_hot_keys_reduce_to_gla_kda():
    # distinct one-hot keys stay orthogonal after any per-dimension decay
    T, dk, dv = 5, 7, 3
    rng = np.random.default_rng(4)
    q, _, v, g, beta, _ = rand_inputs(1, T, 1, dk, dv, kda=True, rng=rng, h0=False)
    perm = rng.permutation(dk)[:T]
    k = np.zeros((1, T, 1, dk))
    for t in range(T):
        k[0, t, 0, perm[t]] = 1.0
    o, _ = oracle.fwd(q, k, v, g, beta, kda=True)
    np.testing.assert_allclose(o, gla_quadratic(q, k, v, g, beta, True), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("kda", [False, True])
def test_small_beta_limit_is_gla(kda):
    q, k, v, g, beta, _ = rand_inputs(1, 10, 2, 4, 3, kda=kda, h0=False)
    ref = gla_quadratic(q, k, v, g, beta, kda)
    errs = []
    for eps in (1e-3, 1e-4):
        o, _ = oracle.fwd(q, k, v, g, eps * beta, kda=kda)
        errs.append(np.max(np.abs(o / eps - ref)))
    assert errs[0] < 1e-2 * np.max(np.abs(ref))
    assert 5 < errs[0] / errs[1] < 20  # O(eps) convergence


# ------------------------------------------------- P3: exact retrieval

def test_orthonormal_keys_retrieve_values():
    T, dk, dv = 6, 8, 5
    rng = np.random.default_rng(5)
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm[:, :T].T.copy()
    keys[4] = keys[1]  # key 1 is rewritten at t=4
    k = keys[None, :, None, :]
    v = rng.standard_normal((1, T, 1, dv))
    q = rng.standard_normal((1, T, 1, dk))
    g = np.zeros((1, T, 1))
    beta = np.ones((1, T, 1))
    _, ht = oracle.fwd(q, k, v, g, beta)
    for j in range(T):
        want = v[0, 4, 0] if j == 1 else v[0, j, 0]
        np.testing.assert_allclose(ht[0, 0].T @ keys[j], want, rtol=1e-12, atol=1e-12)


# ------------------------------------------------- P5: finite differences

@pytest.mark.parametrize("kda", [False, True])
def test_gradients_match_finite_differences(kda):
    B, T, H, dk, dv = 1, 7, 1, 3, 2
    rng = np.random.default_rng(11 + kda)
    q, k, v, g, beta, h0 = rand_inputs(B, T, H, dk, dv, kda=kda, rng=rng)
    do = rng.standard_normal((B, T, H, dv))
    dht = rng.standard_normal((B, H, dk, dv))
    args = dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0)

    def loss(a):
        o, ht = oracle.fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], kda=kda)
        return float(np.sum(o * do) + np.sum(ht * dht))

    grads = oracle.bwd(q, k, v, g, beta, h0, do, dht, kda=kda)
    names = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "h0": "dh0"}
    eps = 1e-6
    for name, gname in names.items():
        x = args[name]
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + eps
            lp = loss(args)
            x[idx] = old - eps
            lm = loss(args)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        scale = max(1.0, np.max(np.abs(fd)))
        err = np.max(np.abs(grads[gname] - fd)) / scale
        assert err < 1e-6, (name, err)


# ------------------------------------------------- P6: KDA with broadcast gate = GDN

def test_kda_broadcast_gate_equals_gdn():
    B, T, H, dk, dv = 2, 11, 2, 6, 5
    q, k, v, g, beta, h0 = rand_inputs(B, T, H, dk, dv)
    gk = np.repeat(g[..., None], dk, axis=-1)
    do = RNG.standard_normal((B, T, H, dv))
    dht = RNG.standard_normal((B, H, dk, dv))
    o1, h1 = oracle.fwd(q, k, v, g, beta, h0)
    o2, h2 = oracle.fwd(q, k, v, gk, beta, h0, kda=True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(h1, h2)
    g1 = oracle.bwd(q, k, v, g, beta, h0, do, dht)
    g2 = oracle.bwd(q, k, v, gk, beta, h0, do, dht, kda=True)
    for n in ("dq", "dk", "dv", "dbeta", "dh0"):
        np.testing.assert_allclose(g1[n], g2[n], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g1["dg"], g2["dg"].sum(-1), rtol=1e-11, atol=1e-12)


# ------------------------------------------------- P7: split sequence

@pytest.mark.parametrize("kda", [False, True])
def test_split_sequence_hands_over_state(kda):
    B, T, H, dk, dv, tau = 1, 13, 2, 4, 3, 5
    q, k, v, g, beta, h0 = rand_inputs(B, T, H, dk, dv, kda=kda)
    do = RNG.standard_normal((B, T, H, dv))
    dht = RNG.standard_normal((B, H, dk, dv))
    o, ht = oracle.fwd(q, k, v, g, beta, h0, kda=kda)
    sl = lambda x, a, b: x[:, a:b]
    oa, ha = oracle.fwd(*(sl(x, 0, tau) for x in (q, k, v, g, beta)), h0, kda=kda)
    ob, hb = oracle.fwd(*(sl(x, tau, T) for x in (q, k, v, g, beta)), ha, kda=kda)
    np.testing.assert_allclose(np.concatenate([oa, ob], 1), o, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(hb, ht, rtol=1e-13, atol=1e-13)
    full = oracle.bwd(q, k, v, g, beta, h0, do, dht, kda=kda)
    gb = oracle.bwd(*(sl(x, tau, T) for x in (q, k, v, g, beta)), ha, sl(do, tau, T), dht, kda=kda)
    ga = oracle.bwd(*(sl(x, 0, tau) for x in (q, k, v, g, beta)), h0, sl(do, 0, tau), gb["dh0"],
                    kda=kda)
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        np.testing.assert_allclose(np.concatenate([ga[n], gb[n]], 1), full[n], rtol=1e-12,
                                   atol=1e-12)
    np.testing.assert_allclose(ga["dh0"], full["dh0"], rtol=1e-12, atol=1e-12)


# ------------------------------------------------- P8: contraction bound

@pytest.mark.parametrize("kda", [False, True])
def test_state_norm_contraction_bound(kda):
    T, dk, dv = 40, 6, 4
    q, k, v, g, beta, h0 = rand_inputs(1, T, 1, dk, dv, kda=kda)
    H = h0
    for t in range(T):
        sl = lambda x: x[:, t:t + 1]
        _, Hn = oracle.fwd(sl(q), sl(k), sl(v), sl(g), sl(beta), H, kda=kda)
        lhs = np.linalg.norm(Hn[0, 0], 2)
        rhs = np.linalg.norm(H[0, 0], 2) + beta[0, t, 0] * np.linalg.norm(v[0, t, 0])
        assert lhs <= rhs * (1 + 1e-12)
        H = Hn


def test_empty_and_zero_length():
    q, k, v, g, beta, h0 = rand_inputs(1, 0, 1, 4, 3)
    o, ht = oracle.fwd(q, k, v, g, beta, h0)
    assert o.shape == (1, 0, 1, 3)
    np.testing.assert_array_equal(ht, h0)
    gr = oracle.bwd(q, k, v, g, beta, h0, np.zeros((1, 0, 1, 3)), np.ones((1, 1, 4, 3)))
    np.testing.assert_array_equal(gr["dh0"], np.ones((1, 1, 4, 3)))


# ------------------------------------------------- P4: chunked form = token form


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("chunk,T", [(1, 7), (2, 9), (4, 13), (16, 37), (16, 48)])
def test_chunked_form_equals_token_form(kda, chunk, T):
    B, H, dk, dv = 1, 2, 5, 4
    rng = np.random.default_rng(100 + chunk)
    q, k, v, g, beta, h0 = rand_inputs(B, T, H, dk, dv, kda=kda, rng=rng)
    do = rng.standard_normal((B, T, H, dv))
    dht = rng.standard_normal((B, H, dk, dv))
    o_ref, ht_ref = oracle.fwd(q, k, v, g, beta, h0, kda=kda)
    o, ht = chunk_reference.forward(q, k, v, g, beta, h0, chunk, kda)
    np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ht, ht_ref, rtol=1e-11, atol=1e-12)
    gr = oracle.bwd(q, k, v, g, beta, h0, do, dht, kda=kda)
    gc = chunk_reference.backward(q, k, v, g, beta, h0, do, dht, chunk, kda)
    for n in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        np.testing.assert_allclose(gc[n], gr[n], rtol=1e-10, atol=1e-11, err_msg=n)


# ------------------------------------------------- scaling identity of the scalar gate

def test_gdn_gate_gradient_scaling_identity():
    """With one scalar gate per head, H_t = c_t Hhat_t (c_t = prod of the gates)
    turns the gates into a rescaling of q (by c_t) and v (by 1/c_t), so
    dL/dlog c_t = q_t.dq_t - v_t.dv_t (+ <dht, ht> at the last token) and
    dg is its reverse cumulative sum over the sequence."""
    T = 21
    q, k, v, g, beta, h0 = rand_inputs(2, T, 3, 5, 4, rng=np.random.default_rng(21))
    rng = np.random.default_rng(22)
    do = rng.standard_normal((2, T, 3, 4))
    dht = rng.standard_normal((2, 3, 5, 4))
    _, ht = oracle.fwd(q, k, v, g, beta, h0)
    gr = oracle.bwd(q, k, v, g, beta, h0, do, dht)
    dlogc = (q * gr["dq"]).sum(-1) - (v * gr["dv"]).sum(-1)
    dlogc[:, -1] += (dht * ht).sum((-1, -2))
    want = np.cumsum(dlogc[:, ::-1], axis=1)[:, ::-1]
    np.testing.assert_allclose(gr["dg"], want, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- worked examples

def _golden_cases():
    """Parses tests/golden/worked_examples.txt (hand-derived values)."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "worked_examples.txt")
    cases, cur = {}, None
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        if line.startswith("["):
            cur = cases.setdefault(line.strip("[]"), {})
            continue
        key, val = (x.strip() for x in line.split("=", 1))

        def num(tok):
            if tok.startswith("ln(") and tok.endswith(")"):
                return float(np.log(float(Fraction(tok[3:-1]))))
            return float(Fraction(tok))
        cur[key] = [[num(t) for t in part.split()] for part in val.split("|")]
    return cases


@pytest.mark.parametrize("name", ["gdn", "kda"])
def test_hand_worked_examples(name):
    c = _golden_cases()[name]
    T = int(c["T"][0][0])
    kda = name == "kda"
    tok = lambda key: np.array(c[key], dtype=np.float64).reshape(1, T, 1, -1)
    g = np.array(c["g"], dtype=np.float64).reshape(1, T, 1, -1)
    g = g if kda else g.reshape(1, T, 1)
    beta = np.array(c["beta"], dtype=np.float64).reshape(1, T, 1)
    h0 = np.array(c["h0"], dtype=np.float64).reshape(1, 1, 2, 2)
    o, ht = oracle.fwd(tok("q"), tok("k"), tok("v"), g, beta, h0, kda=kda)
    np.testing.assert_allclose(o.reshape(T, 2), np.array(c["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(ht.reshape(2, 2), np.array(c["ht"]), rtol=0, atol=1e-12)



# ------------------------------------------------- the Mamba2 mixer (no delta rule)
#
# The same mixer list describes Mamba2 as the scalar-gated state that GDN
# extends with the delta rule; without it the state only accumulates,
# H_t = a_t H_{t-1} + beta_t k_t v_t^T, which unrolls into gated linear
# attention for any keys (not only orthogonal ones).

def _decayed_h0_term(q, g, h0, kda):
    """exp(gamma_t) applied to h0, read out by q_t (per sequence, per token)."""
    gam = np.cumsum(g, axis=1)
    B, T, H, dk = q.shape
    out = np.zeros((B, T, H, h0.shape[-1]))
    for b in range(B):
        for h in range(H):
            for t in range(T):
                a = np.exp(gam[b, t, h]) if kda else np.full(dk, np.exp(gam[b, t, h]))
                out[b, t, h] = (a * q[b, t, h]) @ h0[b, h]
    return out


@pytest.mark.parametrize("kda", [False, True])
def test_no_delta_is_gated_linear_attention(kda):
    q, k, v, g, beta, h0 = rand_inputs(2, 9, 2, 5, 3, kda=kda, rng=np.random.default_rng(31))
    o, ht = oracle.fwd(q, k, v, g, beta, h0, kda=kda, delta=False)
    ref = gla_quadratic(q, k, v, g, beta, kda) + _decayed_h0_term(q, g, h0, kda)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)
    # final state in closed form: sum_j exp(gam_T - gam_j) beta_j k_j v_j^T + exp(gam_T) h0
    gam = np.cumsum(g, axis=1)
    for b in range(2):
        for h in range(2):
            last = gam[b, -1, h]
            want = (np.exp(last) if kda else np.exp(last) * np.ones(5))[:, None] * h0[b, h]
            for j in range(9):
                dec = np.exp(last - gam[b, j, h]) if kda else np.exp(last - gam[b, j, h]) * np.ones(5)
                want = want + np.outer(dec * k[b, j, h], beta[b, j, h] * v[b, j, h])
            np.testing.assert_allclose(ht[b, h], want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("kda", [False, True])
def test_no_delta_gradients_match_finite_differences(kda):
    B, T, H, dk, dv = 1, 6, 1, 3, 2
    rng = np.random.default_rng(41 + kda)
    q, k, v, g, beta, h0 = rand_inputs(B, T, H, dk, dv, kda=kda, rng=rng)
    do = rng.standard_normal((B, T, H, dv))
    dht = rng.standard_normal((B, H, dk, dv))
    args = dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0)

    def loss(a):
        o, ht = oracle.fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], kda=kda, delta=False)
        return float(np.sum(o * do) + np.sum(ht * dht))

    grads = oracle.bwd(q, k, v, g, beta, h0, do, dht, kda=kda, delta=False)
    names = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "h0": "dh0"}
    eps = 1e-6
    for name, gname in names.items():
        x = args[name]
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + eps
            lp = loss(args)
            x[idx] = old - eps
            lm = loss(args)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        scale = max(1.0, np.max(np.abs(fd)))
        assert np.max(np.abs(grads[gname] - fd)) / scale < 1e-6, name


@pytest.mark.parametrize("chunk,T", [(4, 13), (16, 40)])
def test_no_delta_chunked_form_equals_token_form(chunk, T):
    q, k, v, g, beta, h0 = rand_inputs(2, T, 2, 6, 5, rng=np.random.default_rng(51))
    do = np.random.default_rng(52).standard_normal(v.shape)
    dht = np.random.default_rng(53).standard_normal(h0.shape)
    o, ht = oracle.fwd(q, k, v, g, beta, h0, delta=False)
    oc, htc = chunk_reference.forward(q, k, v, g, beta, h0, chunk, delta=False)
    np.testing.assert_allclose(oc, o, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(htc, ht, rtol=1e-11, atol=1e-12)
    ref = oracle.bwd(q, k, v, g, beta, h0, do, dht, delta=False)
    got = chunk_reference.backward(q, k, v, g, beta, h0, do, dht, chunk, delta=False)
    for n in ref:
        np.testing.assert_allclose(got[n], ref[n], rtol=1e-10, atol=1e-11, err_msg=n)
