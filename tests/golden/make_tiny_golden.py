"""Writes tests/golden/tiny_bt8_v32_f32.json: the 8 x 32 fp32 workload's inputs
and the CPU oracle's outputs for them.  Calls only the oracle and the seeded
input generator; run from the repository root:

    python tests/golden/make_tiny_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from distillation_ce_tvd_gb300 import workloads  # noqa: E402


def main():
    w = workloads.make("tiny_bt8_v32_f32", "cpu")
    fwd = oracle.fused_ce_tvd_forward(w.student, w.teacher, w.target, w.ignore_index, threads=1)
    grad, st = oracle.fused_ce_tvd_backward(w.student, w.teacher, w.target, w.grad_ce,
                                            w.grad_tvd, w.ignore_index, threads=1)
    ce_fwd = oracle.ce_forward(w.student, w.target, w.ignore_index, threads=1)
    ce_grad, _ = oracle.ce_backward(w.student, w.target, w.grad_ce, w.ignore_index, threads=1)
    doc = {
        "about": "8 x 32 fp32 workload (seed 0): inputs from the seeded generator and "
                 "outputs of the CPU fp64 oracle. Written by tests/golden/make_tiny_golden.py.",
        "ignore_index": w.ignore_index,
        "student": w.student.tolist(),
        "teacher": w.teacher.tolist(),
        "target": w.target.tolist(),
        "grad_ce": w.grad_ce.tolist(),
        "grad_tvd": w.grad_tvd.tolist(),
        "forward": {k: fwd[k].tolist() for k in ("ce", "tvd", "student_lse", "teacher_lse", "sigma")},
        "status": fwd["status"] | st,
        "grad_student": grad.tolist(),
        "ce_only": {"ce": ce_fwd["ce"].tolist(), "lse": ce_fwd["lse"].tolist(),
                    "grad": ce_grad.tolist()},
    }
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_bt8_v32_f32.json")
    with open(out, "w") as f:
        json.dump(doc, f, indent=1)
    print("wrote", out)


if __name__ == "__main__":
    main()
