"""Oracle against hand-derived fixtures in tests/golden/ (format definitions
and closed forms; each file states its source)."""
import math
import os

import numpy as np

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_e4m3_codes_golden():
    for code, val in _rows("e4m3fn_codes.txt"):
        got = O.e4m3_decode(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))
            assert O.e4m3_round(float(val)) == float(val)


def test_e2m1_codes_and_rounding_golden():
    for kind, a, b in [r[:3] for r in _rows("e2m1_cases.txt")]:
        if kind == "code":
            got = O.e2m1_decode(int(a, 16))
            assert got == float(b) and math.copysign(1, got) == math.copysign(1, float(b)), (a, b)
        else:
            assert O.e2m1_round(float(a)) == float(b), (a, b)


def test_bf16_cases_golden():
    for inp, out in _rows("bf16_rne_cases.txt"):
        assert O.bf16_round(float(inp)) == float(out), (inp, out)


def test_closed_forms_golden():
    for row in _rows("closed_forms.txt"):
        name = row[0]
        if name.startswith("silu("):
            z = float(name[5:-1])
            assert O.silu(z) == np.float64(row[1]) or abs(O.silu(z) - float(row[1])) < 1e-16
        elif name.startswith("rms_norm_const"):
            args = dict(kv.split("=") for kv in name[len("rms_norm_const("):-1].split(","))
            c, eps = float(args["c"]), float(args["eps"])
            y = O.rms_norm(np.full((1, 32), c), np.ones(32), eps)
            assert np.all(y == float(row[1])), (name, y[0, 0])
        elif name.startswith("topk2_logits"):
            ids, w = O.topk_renorm(np.array([[0.0, math.log(3.0), 0.0, 0.0]]), 2)
            assert ids.tolist() == [[1, 0]]
            np.testing.assert_allclose(w, [[0.75, 0.25]], rtol=1e-15)


def test_tiny_workload_regression_fixture():
    """The oracle's tiny-workload output, written by tests/golden/make_tiny_oracle.py
    (which calls only oracle/).  Guards the oracle against silent changes."""
    import workloads
    from tests.golden.make_tiny_oracle import compute, parse
    ref = parse(os.path.join(GOLD, "tiny_oracle.txt"))
    got = compute(workloads.make_inputs("c1_tiny", "cpu"))
    np.testing.assert_array_equal(got["ids"], ref["ids"])
    np.testing.assert_allclose(got["topk_w"], ref["topk_w"], rtol=1e-15)
    np.testing.assert_array_equal(got["out"], ref["out"])
