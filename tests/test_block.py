"""The mixer with its fused neighbours (block_fwd / block_bwd) against the
oracle's composition.

The oracle runs the same chain in fp64: short convolutions (q and k
L2-normalised, q scaled by D^-1/2), the mixer's token recurrence, the gated
norm, and the backward in reverse order.  Where the library stores a tensor
between two calls in bf16 (q, k, v, o; do, dq, dk, dv), the oracle rounds
the same tensor to bf16 at the same point, so that both sides feed every op
the same values; inside each op the oracle stays in fp64.  Tolerance: the
mixer's bf16 bar, relative L2 error <= 2e-2 per output tensor.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_bwd_gb300 as gdn
import oracle
from gated_delta_rule_bwd_gb300.block import block_bwd, block_fwd
from gated_delta_rule_bwd_gb300.inputs import make_block_inputs
from oracle import neighbours as nb

pytestmark = pytest.mark.gpu

EPS = 1e-6
BAR = 2e-2


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()


def np64(t):
    return None if t is None else t.detach().double().cpu().numpy()


def oracle_block(x, kda, cu=None):
    B, T, CH = x.xq.shape
    H = x.g.shape[2]
    D = CH // H
    xq, xk, xv, wq, wk, wv = map(np64, (x.xq, x.xk, x.xv, x.wq, x.wk, x.wv))
    g, beta, gate, weight, dout = map(np64, (x.g, x.beta, x.gate, x.weight, x.dout))
    segs = [(0, T)] if cu is None else list(zip(cu[:-1], cu[1:]))

    def conv_f(xx, w, l2, sc):
        z = np.zeros_like(xx)
        for a, b in segs:
            if b > a:
                z[:, a:b] = nb.short_conv_fwd(xx[:, a:b], w, H, l2, sc, EPS)[0]
        return z

    def conv_b(xx, w, dz, l2, sc):
        dx, dw = np.zeros_like(xx), np.zeros_like(w)
        for a, b in segs:
            if b > a:
                d1, d2 = nb.short_conv_bwd(xx[:, a:b], w, dz[:, a:b], H, l2, sc, EPS)
                dx[:, a:b] = d1
                dw += d2
        return dx, dw

    shp = (B, T, H, D)
    q = bf16(conv_f(xq, wq, True, D ** -0.5)).reshape(shp)
    k = bf16(conv_f(xk, wk, True, 1.0)).reshape(shp)
    v = bf16(conv_f(xv, wv, False, 1.0)).reshape(shp)
    o = np.zeros(shp)
    gr = {n: np.zeros(shp) for n in ("dq", "dk", "dv")}
    gr["dg"], gr["dbeta"] = np.zeros_like(g), np.zeros_like(beta)
    hts = []
    o_parts = []
    for a, b in segs:
        sl = slice(a, b)
        oo, ht = oracle.fwd(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], None, kda=kda)
        o[:, sl] = oo
        hts.append(ht)
        o_parts.append((sl, oo))
    ob = bf16(o)
    out = nb.gated_rmsnorm_fwd(ob, gate, weight, EPS)
    do, dgate, dweight = nb.gated_rmsnorm_bwd(ob, gate, weight, dout, EPS)
    do = bf16(do)
    for a, b in segs:
        if b <= a:
            continue
        sl = slice(a, b)
        r = oracle.bwd(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], None, do[:, sl], None,
                       kda=kda)
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            gr[n][:, sl] = r[n]
    flat = lambda t: bf16(t).reshape(B, T, CH)
    dxq, dwq = conv_b(xq, wq, flat(gr["dq"]), True, D ** -0.5)
    dxk, dwk = conv_b(xk, wk, flat(gr["dk"]), True, 1.0)
    dxv, dwv = conv_b(xv, wv, flat(gr["dv"]), False, 1.0)
    return {"out": out, "ht": np.concatenate(hts, 0), "dxq": dxq, "dxk": dxk, "dxv": dxv,
            "dwq": dwq, "dwk": dwk, "dwv": dwv, "dg": gr["dg"], "dbeta": gr["dbeta"],
            "dgate": dgate, "dweight": dweight}


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


@pytest.mark.parametrize("kda", [False, True])
def test_block_matches_oracle_composition(kda):
    x = make_block_inputs(2, 160, 2, 128, 4, kda=kda, seed=3)
    d = x.to("cuda")
    out, ht, saved = block_fwd(d.xq, d.xk, d.xv, d.wq, d.wk, d.wv, d.g, d.beta, d.gate, d.weight,
                               kda=kda)
    gr = block_bwd(saved, d.dout)
    torch.cuda.synchronize()
    ref = oracle_block(x, kda)
    got = {"out": out, "ht": ht, **gr}
    errs = {n: rel(np64(got[n]), ref[n]) for n in ref}
    bad = {n: e for n, e in errs.items() if not e <= BAR}
    assert not bad, errs
    assert gdn.device_status() == 0


def test_block_packed_sequences():
    cu = [0, 37, 37, 100, 228]
    x = make_block_inputs(1, cu[-1], 2, 128, 4, seed=4)
    d = x.to("cuda")
    cut = torch.tensor(cu, dtype=torch.int32, device="cuda")
    out, ht, saved = block_fwd(d.xq, d.xk, d.xv, d.wq, d.wk, d.wv, d.g, d.beta, d.gate, d.weight,
                               cu_seqlens=cut)
    gr = block_bwd(saved, d.dout)
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    ref = oracle_block(x, False, cu)
    got = {"out": out, "ht": ht, **gr}
    errs = {n: rel(np64(got[n]), ref[n]) for n in ref}
    bad = {n: e for n, e in errs.items() if not e <= BAR}
    assert not bad, errs
