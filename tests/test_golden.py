"""The 8 x 32 fp32 fixture: generator determinism and oracle regression.

The fixture's expected values were written by ``tests/golden/make_tiny_golden.py``
from the CPU oracle alone; the oracle itself is pinned in ``test_oracle_pins``.
"""
import json
import os

import numpy as np
import torch

import oracle
from distillation_ce_tvd_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_bt8_v32_f32.json")


def load_tiny():
    with open(GOLDEN) as f:
        return json.load(f)


def test_generator_reproduces_fixture_inputs():
    d = load_tiny()
    w = workloads.make("tiny_bt8_v32_f32", "cpu")
    assert torch.equal(w.student, torch.tensor(d["student"], dtype=torch.float32))
    assert torch.equal(w.teacher, torch.tensor(d["teacher"], dtype=torch.float32))
    assert w.target.tolist() == d["target"]
    # the recipe's structure: row 3 ties exactly, row 5 is ignored
    assert torch.equal(w.student[3], w.teacher[3]) and w.target[5] == -100


def test_oracle_reproduces_fixture():
    d = load_tiny()
    s = np.array(d["student"], np.float32)
    t = np.array(d["teacher"], np.float32)
    fwd = oracle.fused_ce_tvd_forward(s, t, d["target"], d["ignore_index"], threads=1)
    for k, v in d["forward"].items():
        np.testing.assert_allclose(fwd[k], v, rtol=0, atol=1e-15)
    g, _ = oracle.fused_ce_tvd_backward(s, t, d["target"], d["grad_ce"], d["grad_tvd"],
                                        d["ignore_index"], threads=1)
    np.testing.assert_allclose(g, d["grad_student"], rtol=0, atol=1e-15)
    assert d["forward"]["tvd"][3] == 0.0 and d["forward"]["sigma"][3] == 0.0
