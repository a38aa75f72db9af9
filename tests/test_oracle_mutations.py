"""The pins must reject a wrong oracle (CPU only).

Each case compiles a copy of the oracle source with one plausible mistake
planted in it (a dropped term, a wrong sign, a wrong index, a stale operand)
and runs the pin suite of ``test_oracle.py`` against that copy.  At least one
pin must fail for every mutant; the real oracle passes them all.
"""
import inspect
import os
import subprocess

import pytest

import oracle
import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.cpp")

# (name, exact source text, replacement).  Each text occurs exactly once.
MUTANTS = [
    ("output_reads_previous_state",
     "ot[j] += Hs[(size_t)i * dv + j] * qt[i];",
     "ot[j] += Hn[(size_t)i * dv + j] * qt[i];"),
    ("erase_term_sign",
     "const double u = bt * (vt[j] - vp[j]);\n      Hnext",
     "const double u = bt * (vt[j] + vp[j]);\n      Hnext"),
    ("prediction_skips_decay",
     "    for (int j = 0; j < dv; ++j) vp[j] += Pbuf[(size_t)i * dv + j] * kt[i];",
     "    for (int j = 0; j < dv; ++j) vp[j] += Hprev[(size_t)i * dv + j] * kt[i];"),
    ("kda_gate_wrong_index",
     "const double a = std::exp(d.kda ? gt[i] : gt[0]);\n    for (int j = 0; j < dv; ++j) Pbuf",
     "const double a = std::exp(d.kda ? gt[0] : gt[0]);\n    for (int j = 0; j < dv; ++j) Pbuf"),
    ("dg_uses_undecayed_state",
     "s += dP[e] * P[e];",
     "s += dP[e] * Hprev[e];"),
    ("dk_drops_prediction_term",
     "        dkt[i] += s;\n      }\n      // P = a H_{t-1}",
     "        dkt[i] += 0.0 * s;\n      }\n      // P = a H_{t-1}"),
    ("dbeta_wrong_sign",
     "db += du[j] * (vt[j] - vp[j]);",
     "db -= du[j] * (vt[j] - vp[j]);"),
    ("state_grad_not_decayed",
     "dH[e] = a * dP[e];",
     "dH[e] = dP[e];"),
    ("no_delta_still_predicts",
     "  if (!d.no_delta)\n    for (int i = 0; i < dk; ++i)\n      for (int j = 0; j < dv; ++j) vp[j] += Pbuf",
     "  if (true)\n    for (int i = 0; i < dk; ++i)\n      for (int j = 0; j < dv; ++j) vp[j] += Pbuf"),
    ("no_delta_backward_keeps_prediction_grad",
     "dvp[j] = d.no_delta ? 0.0 : -bt * du[j];",
     "dvp[j] = -bt * du[j];"),
    ("kda_state_grad_drops_gate",
     "dH[(size_t)i * dv + j] = a * dP[(size_t)i * dv + j];",
     "dH[(size_t)i * dv + j] = dP[(size_t)i * dv + j];"),
]


def _pin_calls():
    """Every test function of the pin suite with each of its parameter sets."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        grids = [m.args for m in marks if m.name == "parametrize"]
        combos = [{}]
        for argnames, values in grids:
            names = [a.strip() for a in argnames.split(",")]
            new = []
            for c in combos:
                for v in values:
                    vv = v if len(names) > 1 else (v,)
                    new.append({**c, **dict(zip(names, vv))})
            combos = new
        for c in combos:
            calls.append((name, fn, c))
    return calls


def _caught(variant):
    saved = pins.oracle
    pins.oracle = variant
    try:
        for name, fn, kw in _pin_calls():
            try:
                fn(**kw)
            except Exception:
                return name
    finally:
        pins.oracle = saved
    return None


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutated = tmp_path / "mutant.cpp"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-fPIC", "-shared", "-pthread", str(mutated),
                    "-o", str(so)], check=True)
    assert _caught(oracle.Variant(str(so))) is not None, f"no pin rejects mutant {name}"


def test_real_oracle_passes_every_pin():
    assert _caught(oracle) is None
