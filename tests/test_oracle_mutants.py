"""The oracle's pins must catch plausible mistakes.

Each mutant below is a one-token edit of gdn_ref.c of the kind the pins are
meant to rule out (a dropped term, a wrong sign, a wrong index, a swapped or
transposed operand, read-before-write). The mutant is compiled to a temporary
library, swapped in for the double-precision oracle, and every pin of
tests/test_oracle.py is run against it: at least one must fail. Host-only.
"""
import inspect
import itertools
import os
import subprocess

import pytest

import oracle
from oracle import build as obuild

from . import test_oracle as pins

MUTANTS = [
    ("softplus guard moved", "if (v > (gdn_real)20) return v;", "if (v > (gdn_real)2) return v;"),
    ("silu sign", "gdn_ref_silu(gdn_real x) { return x / ((gdn_real)1 + R_EXP(-x)); }",
     "gdn_ref_silu(gdn_real x) { return x / ((gdn_real)1 + R_EXP(x)); }"),
    ("sigmoid sign", "R_EXP(-b[i])", "R_EXP(b[i])"),
    ("gate dt sign", "alpha[idx] + dt[h]", "alpha[idx] - dt[h]"),
    ("gate a index", "g[idx] = a[h] *", "g[idx] = a[0] *"),
    ("conv taps reversed", "pre += hist[u] * wc[u];", "pre += hist[u] * wc[taps - 1 - u];"),
    ("conv current tap", "gdn_real pre = x * wc[K - 1];", "gdn_real pre = x * wc[0];"),
    ("conv rolls the convolved value", "hist[taps - 1] = x;", "hist[taps - 1] = pre;"),
    ("conv drops current input", "gdn_real pre = x * wc[K - 1];", "gdn_real pre = 0 * wc[K - 1];"),
    ("l2 norm without sqrt", "R_FMAX(R_SQRT(ss), eps)", "R_FMAX(ss, eps)"),
    ("decay dropped", "row[i] = row[i] * decay;", "row[i] = row[i];"),
    ("delta sign", "(vv[j] - pred) * b", "(vv[j] + pred) * b"),
    ("beta dropped", "(vv[j] - pred) * b", "(vv[j] - pred)"),
    ("pred against q", "pred += row[i] * kv[i];", "pred += row[i] * qv[i];"),
    ("rank-1 write with v", "row[i] = row[i] + kv[i] * delta;", "row[i] = row[i] + vv[i] * delta;"),
    ("read before write", "acc += row[i] * qv[i];", "acc += (row[i] - kv[i] * delta) * qv[i];"),
    ("blocked GQA mapping", "const int kh = vh % Hk;", "const int kh = vh / (H / Hk);"),
    ("scale dropped", "yv[j] = scale * acc;", "yv[j] = acc;"),
    ("v index by i", "const gdn_real delta = (vv[j] - pred) * b;",
     "const gdn_real delta = (vv[S - 1 - j] - pred) * b;"),
    ("rms uses the sum", "R_SQRT(ss / (gdn_real)head_dim + eps)", "R_SQRT(ss + eps)"),
    ("norm weight per row", "yr[d] * inv_rms * w[d] *", "yr[d] * inv_rms * w[0] *"),
    ("gate not applied in norm", "* gdn_ref_silu(zr[d]);", "* zr[d];"),
    ("k normed from q slice", "gdn_ref_l2norm(conv_out + key_dim, kn, Hk, S, l2_eps);",
     "gdn_ref_l2norm(conv_out, kn, Hk, S, l2_eps);"),
    ("beta from alpha", "gdn_ref_sigmoid(b + (size_t)n * H, bt, H);",
     "gdn_ref_sigmoid(alpha + (size_t)n * H, bt, H);"),
    ("slots ignored", "return slots ? (int)slots[n] : n;", "return n;"),
]


def _pin_calls():
    """(name, fn, kwargs) for every pin in test_oracle, double precision only."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_") or name == "test_oracle_precisions_agree":
            continue
        grids = [([m.args[0]] if isinstance(m.args[0], str) else m.args[0], m.args[1])
                 for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        axes = []
        for argnames, values in grids:
            names = [a.strip() for a in (argnames[0].split(",") if len(argnames) == 1 else argnames)]
            if names == ["prec"]:
                values = ["f64"]
            axes.append([dict(zip(names, v if len(names) > 1 else (v,))) for v in values])
        for combo in itertools.product(*axes) if axes else [()]:
            kw = {}
            for part in combo:
                kw.update(part)
            calls.append((name, fn, kw))
    return calls


def _fails(calls):
    failed = []
    for name, fn, kw in calls:
        try:
            fn(**kw)
        except (AssertionError, FloatingPointError, ValueError) as exc:  # noqa: PERF203
            failed.append(f"{name}{kw}: {type(exc).__name__}")
    return failed


@pytest.fixture(scope="module")
def source():
    with open(obuild.SRC) as f:
        return f.read()


def test_unmutated_copy_passes_every_pin(tmp_path, source):
    lib = _compile(tmp_path, "clean", source)
    prev = oracle._swap_library("f64", lib)
    try:
        assert _fails(_pin_calls()) == []
    finally:
        oracle._restore_library("f64", prev)


def _compile(tmp_path, tag, text):
    src = tmp_path / f"{tag}.c"
    src.write_text(text)
    hdr = tmp_path / "gdn_ref.h"
    if not hdr.exists():
        hdr.write_text(open(os.path.join(obuild.HERE, "gdn_ref.h")).read())
    lib = tmp_path / f"lib_{tag}.so"
    subprocess.run([os.environ.get("CC", "gcc"), *obuild.CFLAGS, "-DGDN_REF_DOUBLE", str(src),
                    "-o", str(lib), "-lm"], check=True, capture_output=True)
    return str(lib)


@pytest.mark.parametrize("label,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, label, old, new):
    assert source.count(old) == 1, f"mutation site for '{label}' not unique in gdn_ref.c"
    lib = _compile(tmp_path, "mutant", source.replace(old, new))
    prev = oracle._swap_library("f64", lib)
    try:
        failed = _fails(_pin_calls())
    finally:
        oracle._restore_library("f64", prev)
    assert failed, f"no pin caught the mutant '{label}'"
