"""GPU kernels against the fp64 oracle, element by element, through the C ABI.

Tolerances (per output tensor: o, final state, dq, dk, dv, dg, dbeta, dh0):
* fp32 inputs: relative L2 error <= 1e-5 and max |x - ref| <= 1e-4 * rms(ref);
* bf16 inputs (fp32 state and accumulation): relative L2 error <= 2e-2.
The oracle sees exactly the bytes the GPU sees (bf16 values upcast to fp64).
Full-size workloads are checked on sampled (b, h) sequences, which are
independent problems the oracle solves one by one.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_bwd_gb300 as gdn
import oracle
from gated_delta_rule_bwd_gb300 import workloads as W
from gated_delta_rule_bwd_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

FP32_REL, FP32_MAXABS, BF16_REL = 1e-5, 1e-4, 2e-2


def rel_l2(x, ref):
    ref = np.asarray(ref, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    den = np.linalg.norm(ref)
    return np.linalg.norm(x - ref) / den if den > 0 else np.linalg.norm(x)


def check(name, got, ref, fp32):
    got = got.detach().double().cpu().numpy() if torch.is_tensor(got) else got
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    r = rel_l2(got, ref)
    if fp32:
        rms = np.sqrt(np.mean(np.square(ref))) if ref.size else 0.0
        m = np.max(np.abs(got - ref)) if ref.size else 0.0
        assert r <= FP32_REL, f"{name}: rel-L2 {r:.3e} > {FP32_REL}"
        assert m <= FP32_MAXABS * rms, f"{name}: max-abs {m:.3e} > {FP32_MAXABS} * rms {rms:.3e}"
    else:
        assert r <= BF16_REL, f"{name}: rel-L2 {r:.3e} > {BF16_REL}"
    return r


def run_gpu(x, chunk, fwd_only=False, delta=True):
    d = x.to("cuda")
    fwd = gdn.kda_fwd if x.kda else (gdn.gdn_fwd if delta else gdn.mamba2_fwd)
    bwd = gdn.kda_bwd if x.kda else (gdn.gdn_bwd if delta else gdn.mamba2_bwd)
    o, ht = fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, chunk=chunk)
    gr = None
    if not fwd_only:
        gr = bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.do, d.dht, chunk=chunk)
    torch.cuda.synchronize()
    return o, ht, gr


def compare(x, o, ht, gr, fp32, pairs=None, delta=True):
    """Compare GPU results for the sequences in ``pairs`` (default: all)."""
    if pairs is not None:
        sub = x.select(pairs)
        pick_tok = lambda t: torch.stack([t[b, :, h] for b, h in pairs], 0).unsqueeze(2)
        pick_st = lambda t: torch.stack([t[b, h] for b, h in pairs], 0).unsqueeze(1)
    else:
        sub = x
        pick_tok = pick_st = lambda t: t
    o_ref, ht_ref = oracle.fwd(sub.q, sub.k, sub.v, sub.g, sub.beta, sub.h0, kda=x.kda, delta=delta)
    errs = {"o": check("o", pick_tok(o.cpu()), o_ref, fp32),
            "ht": check("ht", pick_st(ht.cpu()), ht_ref, fp32)}
    if gr is not None:
        ref = oracle.bwd(sub.q, sub.k, sub.v, sub.g, sub.beta, sub.h0, sub.do, sub.dht, kda=x.kda,
                         delta=delta)
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            errs[n] = check(n, pick_tok(gr[n].cpu()), ref[n], fp32)
        errs["dh0"] = check("dh0", pick_st(gr["dh0"].cpu()), ref["dh0"], fp32)
    return errs


# ----------------------------------------------------------- small cases, every output

SMALL = [
    # B, T, H, dk, dv, chunk, dtype, kda, h0, dht
    (1, 64, 2, 16, 16, 16, "f32", False, False, False),   # the tiny fp32 workload
    (1, 64, 2, 16, 16, 16, "f32", True, False, False),
    (2, 100, 3, 32, 48, 32, "f32", False, True, True),     # ragged tail, dk != dv
    (2, 100, 3, 32, 48, 16, "f32", True, True, True),
    (1, 37, 2, 24, 40, 64, "f32", False, True, True),      # T < chunk, odd sizes
    (1, 1, 1, 8, 8, 16, "f32", True, True, True),          # one token
    (2, 200, 2, 64, 64, 64, "bf16", False, True, True),
    (2, 200, 2, 64, 64, 64, "bf16", True, True, True),
    (1, 300, 2, 128, 128, 64, "f32", False, True, True),   # full head dims on CUDA cores
    (1, 300, 2, 128, 128, 64, "f32", True, True, True),
    (2, 192, 2, 128, 128, 32, "bf16", False, True, False),
    (2, 200, 2, 128, 128, 64, "bf16", False, True, True),  # tensor-core path, 8-token tail
    (1, 37, 3, 128, 128, 64, "bf16", False, True, True),   # tensor-core path, T < chunk
    (2, 200, 2, 128, 128, 64, "bf16", True, True, True),   # KDA tensor-core path, 8-token tail
    (1, 37, 3, 128, 128, 64, "bf16", True, True, True),    # KDA tensor-core path, T < chunk
    (1, 64, 2, 128, 128, 64, "bf16", True, False, True),   # KDA tensor-core path, one full chunk
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "x".join(map(str, c)))
def test_small_cases_match_oracle(case):
    B, T, H, dk, dv, chunk, dtype, kda, h0, dht = case
    x = make_inputs(B, T, H, dk, dv, kda=kda, dtype=dtype, h0_std=0.3 if h0 else None,
                    with_dht=dht, seed=1)
    o, ht, gr = run_gpu(x, chunk)
    compare(x, o, ht, gr, fp32=dtype == "f32")


def test_tiny_fp32_workload():
    w = W.GDN_TINY_FP32
    x = w.make()
    o, ht, gr = run_gpu(x, w.chunk)
    compare(x, o, ht, gr, fp32=True)


@pytest.mark.parametrize("w", [W.GDN_300M_BF16, W.KDA_300M_BF16, W.GDN_1B_BF16_H0],
                         ids=lambda w: w.name)
def test_training_workloads_sampled(w):
    x = w.make()
    o, ht, gr = run_gpu(x, w.chunk)
    rng = np.random.default_rng(0)
    pairs = [(0, 0), (w.B - 1, w.H - 1)] + [(int(rng.integers(w.B)), int(rng.integers(w.H)))
                                              for _ in range(2)]
    compare(x, o, ht, gr, fp32=False, pairs=pairs)


def test_long_context_forward_sampled():
    """1M-token forward: final state and outputs of four heads (the first, two
    middle ones, the last) vs the oracle."""
    w = W.GDN_1M_FWD_BF16
    x = w.make(device="cuda")
    fwd = gdn.gdn_fwd
    o, ht = fwd(x.q, x.k, x.v, x.g, x.beta, x.h0, chunk=w.chunk)
    torch.cuda.synchronize()
    heads = [0, w.H // 3, 2 * w.H // 3, w.H - 1]
    pairs = [(0, h) for h in heads]
    sub = x.select(pairs).to("cpu")
    o_ref, ht_ref = oracle.fwd(sub.q, sub.k, sub.v, sub.g, sub.beta, None)
    got_o = torch.stack([o[0, :, h] for h in heads], 0).unsqueeze(2).cpu()
    got_ht = torch.stack([ht[0, h] for h in heads], 0).unsqueeze(1).cpu()
    check("ht", got_ht, ht_ref, fp32=False)
    check("o", got_o, o_ref, fp32=False)


def test_segmented_forward_matches_oracle():
    """Few sequences, many chunks: the forward splits each sequence into
    segments (here five; transition and local-state passes, an fp32 combine,
    then the output pass).  Output and final state against the oracle, with an initial
    state and a ragged tail; the combine kernel must have run."""
    x = make_inputs(1, 64 * 160 + 17, 2, 128, 128, dtype="bf16", h0_std=0.3, seed=12)
    d = x.to("cuda")
    with gdn.KernelTimer() as t:
        o, ht = gdn.gdn_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0)
        torch.cuda.synchronize()
    names = [n for n, _ in t.records()]
    assert "tc_combine" in names and names.count("tc_fwd_segment") == 2, names
    compare(x, o, ht, None, fp32=False)


def test_many_segments_forward_matches_oracle():
    """One long sequence: the forward takes as many segments as the minimum
    segment length allows (63 of 33 chunks here), so the combine chains 63
    segment maps and its column blocks.  Output and final state against the
    oracle, with an initial state and a ragged tail."""
    x = make_inputs(1, 64 * 2048 + 5, 1, 128, 128, dtype="bf16", h0_std=0.3, seed=15)
    d = x.to("cuda")
    with gdn.KernelTimer() as t:
        o, ht = gdn.gdn_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0)
        torch.cuda.synchronize()
    names = [n for n, _ in t.records()]
    assert "tc_combine" in names and names.count("tc_fwd_segment") == 2, names
    compare(x, o, ht, None, fp32=False)


# ----------------------------------------------------------- fast-decaying gates

# The workloads' gates are logsigmoid(N(2, 1)), about -0.13 a token.  These
# decay 5-40 times faster: 64-token ranges of about 48, 86, 191 and 320, the
# last three past the tensor-core kernels' factor limit, so their decays take
# the exact per-element path.  dg is the output this stresses: its terms are
# large and nearly cancel when the state forgets quickly.
FAST = [0.0, -1.0, -3.0, -5.0]


@pytest.mark.parametrize("g_mean", FAST)
def test_fast_decaying_gates_match_oracle(g_mean):
    x = make_inputs(1, 256, 2, 128, 128, dtype="bf16", g_mean=g_mean, h0_std=0.3,
                    with_dht=True, seed=21)
    o, ht, gr = run_gpu(x, 64)
    ref = oracle.bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, x.do, x.dht)
    o_ref, ht_ref = oracle.fwd(x.q, x.k, x.v, x.g, x.beta, x.h0)
    check("o", o.cpu(), o_ref, fp32=False)
    check("ht", ht.cpu(), ht_ref, fp32=False)
    for n in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        check(n, gr[n].cpu(), ref[n], fp32=False)


# KDA: per-key-dimension gates logsigmoid(N(mu, 1)).  The tensor-core kernels
# take a sequence while every 64-token chunk's cumulative log gate spans at
# most 80 in each dimension (mu = 0: largest span about 65); wider spans send
# the sequence to the CUDA-core kernels inside the same call (mu = -1, -3).
KDA_FAST = [0.0, -1.0, -3.0]


@pytest.mark.parametrize("g_mean", KDA_FAST)
def test_kda_fast_decaying_gates_match_oracle(g_mean):
    x = make_inputs(1, 256, 2, 128, 128, kda=True, dtype="bf16", g_mean=g_mean, h0_std=0.3,
                    with_dht=True, seed=21)
    o, ht, gr = run_gpu(x, 64)
    compare(x, o, ht, gr, fp32=False)


def test_kda_mixed_paths_in_one_call():
    """One call whose sequences split between the paths: batch row 0 has the
    workloads' slowly decaying gates (tensor cores), row 1 gates so fast that
    its chunks exceed the factor range (CUDA cores); both match the oracle,
    with the saved context and without."""
    x = make_inputs(2, 200, 2, 128, 128, kda=True, dtype="bf16", h0_std=0.3, with_dht=True, seed=22)
    fast = make_inputs(2, 200, 2, 128, 128, kda=True, dtype="bf16", g_mean=-3.0, h0_std=0.3,
                       with_dht=True, seed=22)
    x.g[1] = fast.g[1]
    o, ht, gr = run_gpu(x, 64)
    compare(x, o, ht, gr, fp32=False)
    d = x.to("cuda")
    o2, ht2, ctx = gdn.kda_fwd_save(d.q, d.k, d.v, d.g, d.beta, d.h0)
    gr2 = gdn.kda_bwd_saved(d.q, d.k, d.v, d.g, d.beta, d.h0, d.do, ctx, d.dht)
    torch.cuda.synchronize()
    assert torch.equal(o2, o) and torch.equal(ht2, ht)
    for n in gr:
        assert torch.equal(gr2[n], gr[n]), n


# ----------------------------------------------------------- Mamba2 (no delta rule)

MAMBA2 = [
    # B, T, H, dk, dv, chunk, dtype
    (1, 64, 2, 16, 16, 16, "f32"),        # CUDA-core path
    (2, 100, 3, 32, 48, 32, "f32"),       # ragged tail, dk != dv
    (2, 200, 2, 128, 128, 64, "bf16"),    # tensor-core path, 8-token tail
    (1, 37, 3, 128, 128, 64, "bf16"),     # tensor-core path, T < chunk
]


@pytest.mark.parametrize("case", MAMBA2, ids=lambda c: "x".join(map(str, c)))
def test_mamba2_matches_oracle(case):
    B, T, H, dk, dv, chunk, dtype = case
    x = make_inputs(B, T, H, dk, dv, dtype=dtype, h0_std=0.3, with_dht=True, seed=23)
    o, ht, gr = run_gpu(x, chunk, delta=False)
    compare(x, o, ht, gr, fp32=dtype == "f32", delta=False)


@pytest.mark.parametrize("g_mean", [2.0, -1.0, -3.0])
def test_mamba2_training_shape_and_fast_gates(g_mean):
    """The 300M training shape (sampled sequences) at the workloads' gates, and
    a short case at fast-decaying gates; the saved-context pair gives the same
    bits as the recomputing one."""
    if g_mean == 2.0:
        x = make_inputs(16, 2048, 8, 128, 128, dtype="bf16", seed=24)
        pairs = [(0, 0), (15, 7), (5, 3)]
    else:
        x = make_inputs(1, 256, 2, 128, 128, dtype="bf16", g_mean=g_mean, h0_std=0.3,
                        with_dht=True, seed=25)
        pairs = None
    o, ht, gr = run_gpu(x, 64, delta=False)
    compare(x, o, ht, gr, fp32=False, pairs=pairs, delta=False)
    d = x.to("cuda")
    o2, ht2, ctx = gdn.mamba2_fwd_save(d.q, d.k, d.v, d.g, d.beta, d.h0)
    gr2 = gdn.mamba2_bwd_saved(d.q, d.k, d.v, d.g, d.beta, d.h0, d.do, ctx, d.dht)
    torch.cuda.synchronize()
    assert torch.equal(o2, o) and torch.equal(ht2, ht)
    for n in gr:
        assert torch.equal(gr2[n], gr[n]), n


def test_mamba2_autograd_and_no_solve():
    """The differentiable wrapper with delta=False, and the tensor-core
    Mamba2 step launches no triangular solve."""
    x = make_inputs(1, 128, 2, 128, 128, dtype="bf16", h0_std=0.1, seed=26).to("cuda")
    with gdn.KernelTimer() as t:
        gdn.mamba2_fwd(x.q, x.k, x.v, x.g, x.beta, x.h0)
        gdn.mamba2_bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, x.do)
        torch.cuda.synchronize()
    names = [n for n, _ in t.records()]
    assert names == ["tc_fwd", "tc_states", "tc_bwd"], names
    q, k, v = (t.clone().requires_grad_() for t in (x.q, x.k, x.v))
    o, ht = gdn.gated_delta_rule(q, k, v, x.g, x.beta, x.h0, delta=False)
    (o.float() * x.do.float()).sum().backward()
    ref = gdn.mamba2_bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, x.do)
    assert torch.equal(q.grad, ref["dq"]) and torch.equal(v.grad, ref["dv"])


# ----------------------------------------------------------- saved context

SAVED = [
    # B, T, H, dk, dv, chunk, dtype, kda
    (2, 200, 2, 128, 128, 64, "bf16", False),   # tensor-core path, 8-token tail
    (1, 37, 3, 128, 128, 64, "bf16", False),    # tensor-core path, T < chunk
    (2, 100, 3, 32, 48, 32, "f32", False),      # CUDA-core path: fp32 entry states
    (2, 200, 2, 64, 64, 64, "bf16", True),      # KDA, CUDA-core path
    (2, 200, 2, 128, 128, 64, "bf16", True),    # KDA tensor-core path
]


@pytest.mark.parametrize("case", SAVED, ids=lambda c: "x".join(map(str, c)))
def test_saved_context_matches_oracle_and_recompute(case):
    """*_fwd_save then *_bwd_saved against the oracle, and bit-equal to the
    recomputing *_fwd / *_bwd.  The context buffer starts out as garbage, so
    every byte the backward reads must have been written by the forward; the
    backward launches neither the solve nor the states pass."""
    B, T, H, dk, dv, chunk, dtype, kda = case
    x = make_inputs(B, T, H, dk, dv, kda=kda, dtype=dtype, h0_std=0.3, with_dht=True, seed=13)
    d = x.to("cuda")
    fwd_s = gdn.kda_fwd_save if kda else gdn.gdn_fwd_save
    bwd_s = gdn.kda_bwd_saved if kda else gdn.gdn_bwd_saved
    ctx = gdn.new_ctx(d.q, d.v, chunk, kda).fill_(0xAB)
    o, ht, ctx = fwd_s(d.q, d.k, d.v, d.g, d.beta, d.h0, chunk=chunk, ctx=ctx)
    with gdn.KernelTimer() as t:
        gr = bwd_s(d.q, d.k, d.v, d.g, d.beta, d.h0, d.do, ctx, d.dht, chunk=chunk)
        torch.cuda.synchronize()
    names = [n for n, _ in t.records()]
    if gdn.uses_tensor_cores(d.q, d.v, chunk, kda):
        # KDA: the CUDA-core kernels run too, for the sequences flagged (none here)
        assert names == (["kda_tc_bwd", "simt_bwd", "simt_bwd_reduce"] if kda else ["tc_bwd"]), names
    else:
        assert names == ["simt_bwd", "simt_bwd_reduce"], names
    compare(x, o, ht, gr, fp32=dtype == "f32")
    ro, rht, rgr = run_gpu(x, chunk)
    assert torch.equal(o, ro) and torch.equal(ht, rht)
    for n in rgr:
        assert torch.equal(gr[n], rgr[n]), n


def test_saved_context_from_segmented_forward():
    """The context left by a segmented forward (five segments; entry states
    of later segments come from the fp32 combine).  dO is zero from token tau
    on and there is no final-state gradient, so the gradients of the first
    tau tokens are those of the prefix problem alone (which the oracle
    solves) and the rest are zero.  Over the whole sequence the result
    matches the recomputing backward up to the rounding of the segment entry
    states."""
    T, tau = 64 * 160 + 17, 4000
    x = make_inputs(1, T, 2, 128, 128, dtype="bf16", h0_std=0.3, seed=14)
    x.do[:, tau:] = 0
    d = x.to("cuda")
    ctx = gdn.new_ctx(d.q, d.v).fill_(0xAB)
    with gdn.KernelTimer() as t:
        o, ht, ctx = gdn.gdn_fwd_save(d.q, d.k, d.v, d.g, d.beta, d.h0, ctx=ctx)
        gr = gdn.gdn_bwd_saved(d.q, d.k, d.v, d.g, d.beta, d.h0, d.do, ctx)
        torch.cuda.synchronize()
    names = [n for n, _ in t.records()]
    assert "tc_combine" in names and names.count("tc_solve") == 1, names
    assert "tc_states" not in names, names
    po, pht = gdn.gdn_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0)
    assert torch.equal(o, po) and torch.equal(ht, pht)
    pre = lambda t: t[:, :tau].contiguous()
    ref = oracle.bwd(pre(x.q), pre(x.k), pre(x.v), pre(x.g), pre(x.beta), x.h0, pre(x.do), None)
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        full = np.zeros(gr[n].shape)
        full[:, :tau] = ref[n]
        check(n, gr[n].cpu(), full, fp32=False)
    check("dh0", gr["dh0"].cpu(), ref["dh0"], fp32=False)
    rg = gdn.gdn_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.do)
    for n in rg:
        assert rel_l2(gr[n].float().cpu(), rg[n].float().cpu()) < 5e-3, n


def test_saved_context_step_replays_in_a_cuda_graph():
    """The training step (forward with saved context, then backward) captured
    in a CUDA graph, whose kernels keep their overlapped-launch edges: each
    replay reads the inputs' current contents and gives the bits of eager
    calls on them."""
    x = make_inputs(2, 200, 2, 128, 128, dtype="bf16", h0_std=0.1, with_dht=True, seed=15)
    y = make_inputs(2, 200, 2, 128, 128, dtype="bf16", h0_std=0.1, with_dht=True, seed=16)
    d = x.to("cuda")
    ctx = gdn.new_ctx(d.q, d.v)

    def step():
        o, ht, _ = gdn.gdn_fwd_save(d.q, d.k, d.v, d.g, d.beta, d.h0, ctx=ctx)
        gr = gdn.gdn_bwd_saved(d.q, d.k, d.v, d.g, d.beta, d.h0, d.do, ctx, d.dht)
        return [o, ht] + [gr[n] for n in sorted(gr)]

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up off the capture stream
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = step()
    for src in (x, y, x):
        for n in ("q", "k", "v", "g", "beta", "h0", "do", "dht"):
            getattr(d, n).copy_(getattr(src, n))
        ref = [t.clone() for t in step()]
        for t in out:
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for a, b in zip(out, ref):
            assert torch.equal(a, b)


# ----------------------------------------------------------- decode

DECODE = [
    # B, T, H, dk, dv, dtype, kda
    (3, 1, 2, 128, 128, "bf16", False),   # single-token step, full head dims
    (3, 1, 2, 128, 128, "bf16", True),
    (2, 3, 3, 40, 24, "f32", False),      # a few tokens, odd sizes (a partial column slice)
    (2, 3, 3, 40, 24, "f32", True),
    (1, 5, 2, 128, 96, "f32", False),
]


@pytest.mark.parametrize("case", DECODE, ids=lambda c: "x".join(map(str, c)))
def test_decode_matches_oracle(case):
    """Token-by-token decode against the oracle's forward (outputs and final
    state), updating the state in place and into a new tensor."""
    B, T, H, dk, dv, dtype, kda = case
    x = make_inputs(B, T, H, dk, dv, kda=kda, dtype=dtype, h0_std=0.3, seed=17)
    d = x.to("cuda")
    dec = gdn.kda_decode if kda else gdn.gdn_decode
    o1, ht1 = dec(d.q, d.k, d.v, d.g, d.beta, d.h0, inplace=False)
    st = d.h0.clone()
    o2, ht2 = dec(d.q, d.k, d.v, d.g, d.beta, st, inplace=True)
    torch.cuda.synchronize()
    assert ht2.data_ptr() == st.data_ptr()
    assert torch.equal(o1, o2) and torch.equal(ht1, ht2)
    compare(x, o1, ht1, None, fp32=dtype == "f32")


def test_decode_steps_chain_like_one_call():
    """Three single-token calls on an in-place state equal one three-token
    call, and both match the chunkwise tensor-core forward."""
    x = make_inputs(2, 3, 4, 128, 128, dtype="bf16", h0_std=0.2, seed=18)
    d = x.to("cuda")
    st = d.h0.clone()
    outs = []
    for t in range(3):
        sl = lambda u: u[:, t:t + 1].contiguous()
        o, _ = gdn.gdn_decode(sl(d.q), sl(d.k), sl(d.v), sl(d.g), sl(d.beta), st)
        outs.append(o)
    o3, h3 = gdn.gdn_decode(d.q, d.k, d.v, d.g, d.beta, d.h0, inplace=False)
    of, hf = gdn.gdn_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(outs, 1), o3) and torch.equal(st, h3)
    assert rel_l2(o3.float().cpu(), of.float().cpu()) < BF16_REL
    assert rel_l2(h3.cpu(), hf.cpu()) < BF16_REL


# ----------------------------------------------------------- invariants on the GPU

def test_kda_with_broadcast_gate_equals_gdn():
    """KDA with one gate value repeated over the key dimension against GDN
    (both on their tensor-core kernels): equal within the bf16 tolerance; dg
    of GDN is the sum of KDA's over the key dimension."""
    x = make_inputs(2, 130, 2, 128, 128, dtype="bf16", h0_std=0.1, with_dht=True, seed=3)
    d = x.to("cuda")
    gk = d.g[..., None].expand(*d.g.shape, 128).contiguous()
    o1, h1 = gdn.gdn_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0)
    o2, h2 = gdn.kda_fwd(d.q, d.k, d.v, gk, d.beta, d.h0)
    g1 = gdn.gdn_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.do, d.dht)
    g2 = gdn.kda_bwd(d.q, d.k, d.v, gk, d.beta, d.h0, d.do, d.dht)
    assert rel_l2(o2.float().cpu(), o1.float().cpu()) < BF16_REL
    assert rel_l2(h2.cpu(), h1.cpu()) < BF16_REL
    for n in ("dq", "dk", "dv", "dbeta", "dh0"):
        assert rel_l2(g2[n].float().cpu(), g1[n].float().cpu()) < BF16_REL, n
    assert rel_l2(g2["dg"].sum(-1).cpu(), g1["dg"].cpu()) < BF16_REL


@pytest.mark.parametrize("kda", [False, True])
def test_split_sequence_hands_over_state(kda):
    T, tau = 256, 128
    x = make_inputs(2, T, 2, 128, 128, kda=kda, dtype="bf16", h0_std=0.1, with_dht=True, seed=4)
    d = x.to("cuda")
    fwd = gdn.kda_fwd if kda else gdn.gdn_fwd
    bwd = gdn.kda_bwd if kda else gdn.gdn_bwd
    sl = lambda t, a, b: t[:, a:b].contiguous()
    o, ht = fwd(d.q, d.k, d.v, d.g, d.beta, d.h0)
    oa, ha = fwd(*(sl(t, 0, tau) for t in (d.q, d.k, d.v, d.g, d.beta)), d.h0)
    ob, hb = fwd(*(sl(t, tau, T) for t in (d.q, d.k, d.v, d.g, d.beta)), ha)
    assert rel_l2(torch.cat([oa, ob], 1).float().cpu(), o.float().cpu()) < 1e-2
    assert rel_l2(hb.cpu(), ht.cpu()) < 1e-3
    full = bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.do, d.dht)
    gb = bwd(*(sl(t, tau, T) for t in (d.q, d.k, d.v, d.g, d.beta)), ha, sl(d.do, tau, T), d.dht)
    ga = bwd(*(sl(t, 0, tau) for t in (d.q, d.k, d.v, d.g, d.beta)), d.h0, sl(d.do, 0, tau),
             gb["dh0"])
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        assert rel_l2(torch.cat([ga[n], gb[n]], 1).float().cpu(), full[n].float().cpu()) < 1e-2, n
    assert rel_l2(ga["dh0"].cpu(), full["dh0"].cpu()) < 1e-2


@pytest.mark.parametrize("kda", [False, True])
def test_results_are_deterministic(kda):
    x = make_inputs(2, 200, 2, 128, 128, kda=kda, dtype="bf16", h0_std=0.1, with_dht=True, seed=5)
    r1 = run_gpu(x, 64)
    r2 = run_gpu(x, 64)
    assert torch.equal(r1[0], r2[0]) and torch.equal(r1[1], r2[1])
    for n in r1[2]:
        assert torch.equal(r1[2][n], r2[2][n]), n


def test_shared_workspace_across_calls():
    """One caller-provided workspace reused by the forward and the backward
    call, twice in a row (as a training loop does): every result bit-equal to
    calls that each allocate their own workspace."""
    x = make_inputs(2, 200, 2, 128, 128, dtype="bf16", h0_std=0.1, with_dht=True, seed=11)
    d = x.to("cuda")
    need = max(gdn.fwd_workspace_bytes(d.q, d.v), gdn.bwd_workspace_bytes(d.q, d.v))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ref_o, ref_ht = gdn.gdn_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0)
    ref_g = gdn.gdn_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.do, d.dht)
    for _ in range(2):
        o, ht = gdn.gdn_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, workspace=ws)
        gr = gdn.gdn_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.do, d.dht, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(ht, ref_ht)
        for n in ref_g:
            assert torch.equal(gr[n], ref_g[n]), n


def test_beta_zero_gives_pure_decay_on_gpu():
    x = make_inputs(1, 96, 2, 128, 128, dtype="bf16", h0_std=0.5, seed=6)
    x.beta.zero_()
    d = x.to("cuda")
    o, ht = gdn.gdn_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0)
    gam = torch.cumsum(x.g.double(), 1)                       # [B,T,H]
    ht_ref = torch.exp(gam[:, -1])[..., None, None] * x.h0.double()
    assert rel_l2(ht.cpu(), ht_ref) < 1e-5


def test_empty_sequence_copies_state():
    x = make_inputs(2, 0, 2, 16, 16, dtype="f32", h0_std=1.0, with_dht=True, seed=7)
    d = x.to("cuda")
    o, ht = gdn.gdn_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, chunk=16)
    gr = gdn.gdn_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.do, d.dht, chunk=16)
    torch.cuda.synchronize()
    assert o.shape[1] == 0
    assert torch.equal(ht, d.h0) and torch.equal(gr["dh0"], d.dht)


@pytest.mark.parametrize("save_context", [True, False])
def test_autograd_wrapper_matches_direct_calls(save_context):
    x = make_inputs(1, 128, 2, 128, 128, dtype="bf16", h0_std=0.1, seed=8).to("cuda")
    q, k, v = (t.clone().requires_grad_() for t in (x.q, x.k, x.v))
    o, ht = gdn.gated_delta_rule(q, k, v, x.g, x.beta, x.h0, save_context=save_context)
    (o.float() * x.do.float()).sum().backward()
    ref = gdn.gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, x.do)
    assert torch.equal(q.grad, ref["dq"]) and torch.equal(v.grad, ref["dv"])


# ----------------------------------------------------------- bounded waits

def test_bounded_wait_timeout_is_reported_and_context_survives():
    """A device-side wait that nothing completes (no copy or tensor-core
    operation in flight) runs out after its bounded polls; the kernel records
    GDN_ERR_DEVICE_TIMEOUT, frees its tensor memory and returns.  The status
    word reports it once, and the next library calls run normally."""
    assert gdn.device_status() == 0
    gdn.wait_selftest(5)
    torch.cuda.synchronize()
    assert gdn.device_status() == -7
    assert gdn.device_status() == 0  # read and cleared
    x = make_inputs(1, 130, 2, 128, 128, dtype="bf16", h0_std=0.1, with_dht=True, seed=19)
    o, ht, gr = run_gpu(x, 64)
    compare(x, o, ht, gr, fp32=False)
    assert gdn.device_status() == 0


# ----------------------------------------------------------- packed variable-length sequences

def _pack(seqs):
    """Concatenate per-sequence MixerInputs (B = 1 each) along the tokens."""
    cat = lambda n: torch.cat([getattr(x, n) for x in seqs], 1)
    st = lambda n: None if getattr(seqs[0], n) is None else torch.cat([getattr(x, n) for x in seqs], 0)
    lens = [x.q.shape[1] for x in seqs]
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    return {n: cat(n) for n in ("q", "k", "v", "g", "beta", "do")} | {"h0": st("h0"), "dht": st("dht")}, cu


# lengths: a one-token sequence, chunk boundaries inside and at the end of a
# 64-token chunk, an empty sequence, a sequence longer than two chunks
VARLEN = [
    # lengths, dk, dv, chunk, dtype, mixer
    ([1, 64, 100, 37, 0, 130], 128, 128, 64, "bf16", "gdn"),
    ([1, 64, 100, 37, 0, 130], 128, 128, 64, "bf16", "kda"),
    ([1, 64, 100, 37, 0, 130], 128, 128, 64, "bf16", "mamba2"),
    ([5, 16, 33, 0, 50], 32, 48, 16, "f32", "gdn"),
    ([5, 16, 33, 0, 50], 32, 48, 32, "f32", "kda"),
    ([5, 16, 33, 0, 50], 32, 48, 16, "f32", "mamba2"),
]


@pytest.mark.parametrize("case", VARLEN, ids=lambda c: f"{c[5]}-{c[4]}-d{c[1]}x{c[2]}-C{c[3]}")
def test_varlen_matches_oracle_per_sequence(case):
    """Packed sequences against the oracle run on each sequence alone (its own
    initial state and final-state gradient), every output."""
    lens, dk, dv, chunk, dtype, mixer = case
    kda, delta = mixer == "kda", mixer != "mamba2"
    seqs = [make_inputs(1, L, 2, dk, dv, kda=kda, dtype=dtype, h0_std=0.3, with_dht=True,
                        seed=100 + i) for i, L in enumerate(lens)]
    x, cu = _pack(seqs)
    d = {n: (t.to("cuda") if t is not None else None) for n, t in x.items()}
    cu_d = cu.to("cuda")
    fwd = getattr(gdn, f"{mixer}_fwd_varlen")
    bwd = getattr(gdn, f"{mixer}_bwd_varlen")
    o, ht = fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_d, d["h0"], chunk=chunk)
    gr = bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_d, d["h0"], d["do"], d["dht"], chunk=chunk)
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    fp32 = dtype == "f32"
    for i, sq in enumerate(seqs):
        a, b = int(cu[i]), int(cu[i + 1])
        o_ref, ht_ref = oracle.fwd(sq.q, sq.k, sq.v, sq.g, sq.beta, sq.h0, kda=kda, delta=delta)
        check(f"ht[{i}]", ht[i:i + 1].cpu(), ht_ref, fp32)
        if b == a:
            assert torch.equal(gr["dh0"][i:i + 1].cpu(), sq.dht), "empty sequence: dh0 = dht"
            continue
        ref = oracle.bwd(sq.q, sq.k, sq.v, sq.g, sq.beta, sq.h0, sq.do, sq.dht, kda=kda, delta=delta)
        check(f"o[{i}]", o[:, a:b].cpu(), o_ref, fp32)
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            check(f"{n}[{i}]", gr[n][:, a:b].cpu(), ref[n], fp32)
        check(f"dh0[{i}]", gr["dh0"][i:i + 1].cpu(), ref["dh0"], fp32)


def test_varlen_equal_lengths_match_the_batch_call():
    """Packed sequences of equal length give the bits of the batched call on the
    same data (the same kernels, addressed differently)."""
    x = make_inputs(3, 200, 2, 128, 128, dtype="bf16", h0_std=0.3, with_dht=True, seed=27)
    d = x.to("cuda")
    flat = lambda t: t.reshape(1, -1, *t.shape[2:]).contiguous()
    cu = torch.tensor([0, 200, 400, 600], dtype=torch.int32, device="cuda")
    o, ht = gdn.gdn_fwd_varlen(flat(d.q), flat(d.k), flat(d.v), flat(d.g), flat(d.beta), cu, d.h0)
    gr = gdn.gdn_bwd_varlen(flat(d.q), flat(d.k), flat(d.v), flat(d.g), flat(d.beta), cu, d.h0,
                            flat(d.do), d.dht)
    ro, rht = gdn.gdn_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0)
    rg = gdn.gdn_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.do, d.dht)
    torch.cuda.synchronize()
    assert torch.equal(o, flat(ro)) and torch.equal(ht, rht)
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.equal(gr[n], flat(rg[n])), n
    assert torch.equal(gr["dh0"], rg["dh0"])


def test_varlen_invalid_offsets_are_reported():
    """Offsets that decrease are found on the device: nothing is computed, the
    status word says GDN_ERR_SEQLENS, and the next call runs normally."""
    x = make_inputs(1, 100, 2, 128, 128, dtype="bf16", seed=28).to("cuda")
    cu = torch.tensor([0, 60, 40, 100], dtype=torch.int32, device="cuda")
    gdn.gdn_fwd_varlen(x.q, x.k, x.v, x.g, x.beta, cu)
    torch.cuda.synchronize()
    assert gdn.device_status() == -8
    assert gdn.device_status() == 0
    good = torch.tensor([0, 60, 100], dtype=torch.int32, device="cuda")
    o, ht = gdn.gdn_fwd_varlen(x.q, x.k, x.v, x.g, x.beta, good)
    torch.cuda.synchronize()
    assert gdn.device_status() == 0 and torch.isfinite(o.float()).all()


# ----------------------------------------------------------- KDA with a bf16 gate

def _as_f32_gate(x):
    """The same inputs with the bf16 gate widened to fp32 (identical values)."""
    import copy
    y = copy.copy(x)
    y.g = x.g.float()
    return y


BF16_GATE = [
    # B, T, H, dk, dv, chunk, g_mean: path
    (2, 200, 2, 128, 128, 64, 2.0),    # tensor cores, 8-token tail
    (1, 37, 3, 128, 128, 64, 2.0),     # tensor cores, T < chunk
    (1, 256, 2, 128, 128, 64, -3.0),   # gates past the factor range: CUDA-core fallback
    (2, 100, 3, 64, 64, 32, 2.0),      # CUDA cores
]


@pytest.mark.parametrize("case", BF16_GATE, ids=lambda c: "x".join(map(str, c)))
def test_kda_bf16_gate_matches_oracle_and_fp32_gate(case):
    """KDA with g and dg in bf16 (GDN_BF16_G16): against the oracle on the
    bf16 gate's values, and bit for bit against the fp32-gate call on the same
    values (every output but dg equal; dg equal to the fp32 call's dg rounded
    to bf16), with the saved-context pair equal to the recomputing one."""
    B, T, H, dk, dv, chunk, g_mean = case
    x = make_inputs(B, T, H, dk, dv, kda=True, dtype="bf16", g_mean=g_mean, h0_std=0.3,
                    with_dht=True, seed=31, g_dtype="bf16")
    assert x.g.dtype == torch.bfloat16
    o, ht, gr = run_gpu(x, chunk)
    assert gr["dg"].dtype == torch.bfloat16
    compare(x, o, ht, gr, fp32=False)
    o32, ht32, gr32 = run_gpu(_as_f32_gate(x), chunk)
    assert torch.equal(o, o32) and torch.equal(ht, ht32)
    for n in ("dq", "dk", "dv", "dbeta", "dh0"):
        assert torch.equal(gr[n], gr32[n]), n
    assert torch.equal(gr["dg"], gr32["dg"].to(torch.bfloat16))
    d = x.to("cuda")
    o2, ht2, ctx = gdn.kda_fwd_save(d.q, d.k, d.v, d.g, d.beta, d.h0, chunk=chunk)
    gr2 = gdn.kda_bwd_saved(d.q, d.k, d.v, d.g, d.beta, d.h0, d.do, ctx, d.dht, chunk=chunk)
    torch.cuda.synchronize()
    assert torch.equal(o2, o) and torch.equal(ht2, ht)
    for n in gr:
        assert torch.equal(gr2[n], gr[n]), n


def test_kda_bf16_gate_varlen_and_decode():
    """The bf16 gate through the packed-sequence calls and the decode step."""
    lens = [1, 64, 100, 0, 77]
    seqs = [make_inputs(1, L, 2, 128, 128, kda=True, dtype="bf16", h0_std=0.3, with_dht=True,
                        seed=200 + i, g_dtype="bf16") for i, L in enumerate(lens)]
    x, cu = _pack(seqs)
    d = {n: (t.to("cuda") if t is not None else None) for n, t in x.items()}
    cu_d = cu.to("cuda")
    o, ht = gdn.kda_fwd_varlen(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_d, d["h0"])
    gr = gdn.kda_bwd_varlen(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_d, d["h0"], d["do"],
                            d["dht"])
    torch.cuda.synchronize()
    assert gdn.device_status() == 0 and gr["dg"].dtype == torch.bfloat16
    for i, sq in enumerate(seqs):
        a, b = int(cu[i]), int(cu[i + 1])
        o_ref, ht_ref = oracle.fwd(sq.q, sq.k, sq.v, sq.g, sq.beta, sq.h0, kda=True)
        check(f"ht[{i}]", ht[i:i + 1].cpu(), ht_ref, False)
        if b == a:
            continue
        ref = oracle.bwd(sq.q, sq.k, sq.v, sq.g, sq.beta, sq.h0, sq.do, sq.dht, kda=True)
        check(f"o[{i}]", o[:, a:b].cpu(), o_ref, False)
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            check(f"{n}[{i}]", gr[n][:, a:b].cpu(), ref[n], False)
    # decode: four tokens of 16 sequences, state updated in place
    y = make_inputs(16, 4, 2, 128, 128, kda=True, dtype="bf16", h0_std=0.3, seed=7, g_dtype="bf16")
    dy = y.to("cuda")
    state = dy.h0.clone()
    od, _ = gdn.kda_decode(dy.q, dy.k, dy.v, dy.g, dy.beta, state)
    torch.cuda.synchronize()
    o_ref, ht_ref = oracle.fwd(y.q, y.k, y.v, y.g, y.beta, y.h0, kda=True)
    check("decode o", od.cpu(), o_ref, False)
    check("decode ht", state.cpu(), ht_ref, False)
