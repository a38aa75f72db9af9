"""Host-side logic of bench.py (CPU only): the algorithmic work it divides by,
the clock record it attaches, and the ncu traffic it reads from profiles/."""
import datetime
import json
import os

import pytest

import bench
from gated_delta_rule_bwd_gb300 import workloads as W


def test_algorithmic_work_of_the_300m_shape():
    # per token-head at dk = dv = 128, C = 64: forward 2C(3dk + 2dv) + 6 dk dv + C^2/3,
    # backward 2C(7dk + 5dv) + 14 dk dv + C^2/3; bf16 bytes 1032 + 1808
    a = bench.algorithmic(W.GDN_300M_BF16)
    assert a["fwd_flops"] == pytest.approx(181589.33, abs=0.01)
    assert a["bwd_flops"] == pytest.approx(427349.33, abs=0.01)
    assert (a["fwd_bytes"], a["bwd_bytes"]) == (1032, 1808)
    k = bench.algorithmic(W.KDA_300M_BF16)  # the gate is dk fp32 values per token-head
    assert (k["fwd_bytes"], k["bwd_bytes"]) == (1540, 2824)


def test_kernel_work_assigns_the_op_to_its_main_kernel():
    w = W.GDN_300M_BF16
    th, seqs = w.B * w.T * w.H, w.B * w.H
    nb, nf = bench.kernel_work(w, "tc_bwd")
    assert nb == 1808 * th + 4 * 128 * 128 * seqs  # + dh0 write
    assert bench.kernel_work(w, "tc_solve") == (0.0, 0.0)
    assert bench.kernel_work(w, "tc_fwd")[0] == 1032 * th + 4 * 128 * 128 * seqs


def test_decode_bytes():
    # fp32 state read and written, bf16 q, k, v, o, fp32 g and beta
    assert bench.decode_bytes(W.GDN_DECODE_BF16) == 2 * 4 * 128 * 128 + 2 * 512 + 8
    assert bench.decode_bytes(W.KDA_DECODE_BF16) == 2 * 4 * 128 * 128 + 2 * 512 + 4 * 128 + 4


def _clock_rows(path, rows):
    with open(path, "w") as f:
        for ts, mhz, reason in rows:
            stamp = datetime.datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
            f.write(f"{stamp}, 0, {mhz}, 2070, 400.5, 0x0, Not Active, Not Active, Not Active, "
                    f"{reason}\n")


def test_clock_record_keeps_the_samples_of_the_timed_region(tmp_path):
    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "clocks.csv")
    t = 1_800_000_000.0
    _clock_rows(cs.path, [(t - 1.0, 1000, "Not Active"), (t + 0.1, 2070, "Not Active"),
                          (t + 0.2, 2060, "Active"), (t + 5.0, 900, "Not Active")])
    s = cs.summary(t, t + 1.0)
    assert s["samples"] == 2 and s["samples_in_timed_region"]
    assert s["sm_mhz"] == pytest.approx(2065.0)
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_record_without_samples_in_the_region_says_so(tmp_path):
    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "clocks.csv")
    t = 1_800_000_000.0
    _clock_rows(cs.path, [(t - 1.0, 2070, "Not Active")])
    s = cs.summary(t, t + 0.01)
    assert s["samples"] == 1 and not s["samples_in_timed_region"]


def test_recorded_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    import hashlib
    csrc = tmp_path / "gated_delta_rule_bwd_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "gdn_tc.cu"
    src.write_text("// kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles" / "tc_bwd_gdn_300m_bf16.md").write_text(
        f"# title\n\nkernel_source_sha256_16: {sha}   (note)\ntraffic_bytes_per_launch: 1234\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("tc_bwd", "gdn_300m") == 1234.0
    assert bench.recorded_traffic("tc_fwd", "gdn_300m") is None  # no summary for it
    src.write_text("// kernel v2\n")  # the kernel changed since the capture
    assert bench.recorded_traffic("tc_bwd", "gdn_300m") is None


def test_committed_profiles_parse():
    # every committed kernel summary names a source hash and a traffic figure;
    # the bench record holds one parseable JSON line per workload
    root = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles")
    names = [n for n in os.listdir(root) if n.endswith(".md")]
    assert names
    for n in names:
        text = open(os.path.join(root, n)).read()
        if n.startswith("bench_"):
            lines = [json.loads(l) for l in text.splitlines() if l.startswith("{")]
            assert lines and all("roofline" in d and "clocks" in d for d in lines), n
            continue
        assert "kernel_source_sha256_16:" in text and "traffic_bytes_per_launch:" in text, n


def test_default_step_counts(monkeypatch):
    seen = {}
    monkeypatch.setattr(bench, "run_ours", lambda a: seen.setdefault("ours", (a.steps, a.warmup)))
    monkeypatch.setattr(bench, "run_decode", lambda a: seen.setdefault("dec", (a.steps, a.warmup)))
    monkeypatch.setattr(bench, "run_reference", lambda a: seen.setdefault("ref", (a.steps, a.warmup)))
    monkeypatch.setattr(bench, "run_forward", lambda a: seen.setdefault("fwd", (a.steps, a.warmup)))
    for argv in (["bench.py"], ["bench.py", "--workload", "gdn_decode"],
                 ["bench.py", "--workload", "gdn_1m"],
                 ["bench.py", "--impl", "reference"], ["bench.py", "--steps", "7", "--warmup", "1"]):
        monkeypatch.setattr("sys.argv", argv)
        seen.clear()
        bench.main()
        (key, (steps, warmup)), = seen.items()
        if argv == ["bench.py"]:
            assert key == "ours" and steps == 1000 and warmup >= 3
        elif "gdn_decode" in argv:
            assert key == "dec" and steps == 5000
        elif "gdn_1m" in argv:
            assert key == "fwd" and steps == 40 and warmup == 3
        elif "reference" in argv:
            assert key == "ref" and steps == 20
        else:
            assert (steps, warmup) == (7, 3)  # at least three warm-up steps
