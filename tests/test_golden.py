"""Golden fixtures: closed-form constants and the oracle regression fixture."""
import os

import numpy as np
import pytest

import oracle

from .golden import make_golden

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read(name):
    vals = {}
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, *nums = line.split()
                vals[key] = np.array([float(x) for x in nums])
    return vals


def test_closed_forms():
    cf = _read("closed_forms.txt")
    for prec, tol in (("f64", 1e-15), ("f32", 3e-7)):
        assert oracle.softplus(0.0, prec) == pytest.approx(cf["softplus_at_0"][0], rel=tol)
        assert oracle.silu(1.0, prec) == pytest.approx(cf["silu_at_1"][0], rel=tol)
        assert oracle.sigmoid(np.zeros(1), prec)[0] == cf["sigmoid_at_0"][0]
        g = oracle.decay_gate(np.zeros((1, 1)), np.zeros(1), -np.ones(1), prec)
        assert g[0, 0] == pytest.approx(cf["gate_a_minus1_dt0_alpha0"][0], rel=tol)
    assert oracle.softplus(20.0, "f64") - 20.0 == pytest.approx(
        cf["softplus_at_20_minus_20"][0], rel=1e-3)


def test_oracle_regression_fixture():
    want = _read("tiny_oracle_f64.txt")
    got = make_golden.compute()
    assert set(want) == set(got)
    for key in want:
        np.testing.assert_allclose(got[key], want[key], rtol=1e-12, atol=1e-12, err_msg=key)
