"""CPU fp64 oracle for the fused CE + TVD distillation loss.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path never
imports this package, and this package imports nothing from the product
package.

The arithmetic lives in ``fused_ce_tvd_oracle.c`` (plain C, fp64, two exact
passes per row; see its header for the passages of the PR #1384 analysis it
follows).  This module only compiles it with gcc, loads it with ctypes and
marshals numpy / torch-CPU arrays into it.

Every function here is pinned by ``tests/test_oracle_pins.py`` against values
the mathematics fixes (closed forms, invariants, finite differences, a
hand-worked example and fp64 PyTorch autograd).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fused_ce_tvd_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libfct_oracle.so")

F32, BF16, F64 = 0, 1, 2
TARGET_OUT_OF_RANGE = 0x1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into a shared library (gcc, OpenMP if present)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-fno-fast-math", _SRC]
    try:
        subprocess.run(base + ["-fopenmp", "-o", tmp, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        # No OpenMP runtime: the pragmas are ignored and rows run serially.
        subprocess.run(base + ["-o", tmp, "-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.oracle_fused_ce_tvd_forward.argtypes = [
                vp, i64, vp, i64, i32, vp, i64, i64, i64, vp, vp, vp, vp, vp, i32]
            lib.oracle_fused_ce_tvd_forward.restype = i32
            lib.oracle_fused_ce_tvd_backward.argtypes = [
                vp, i64, vp, i64, i32, vp, i64, i64, i64, vp, vp, i64, vp, i32]
            lib.oracle_fused_ce_tvd_backward.restype = i32
            lib.oracle_ce_forward.argtypes = [vp, i64, i32, vp, i64, i64, i64, vp, vp, i32]
            lib.oracle_ce_forward.restype = i32
            lib.oracle_ce_backward.argtypes = [vp, i64, i32, vp, i64, i64, i64, vp, i64, vp, i32]
            lib.oracle_ce_backward.restype = i32
            lib.oracle_row_probs.argtypes = [vp, i64, vp, i64, i32, i64, i64, vp, vp]
            lib.oracle_row_probs.restype = None
            dbl = ctypes.c_double
            lib.oracle_mean_loss.argtypes = [vp, vp, vp, i64, i64, dbl, dbl, vp, vp, vp]
            lib.oracle_mean_loss.restype = i64
            _lib = lib
    return _lib


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def _logits(x):
    """(array, dtype code, ld) for a 2-D logit matrix on the host.

    Accepts numpy float32/float64 arrays and torch CPU tensors of float32,
    bfloat16 or float64.  bf16 is handed over as its raw 16-bit patterns.
    The array must have unit stride along V; rows may be padded (ld >= V).
    """
    if hasattr(x, "detach"):  # torch tensor, CPU
        import torch
        x = x.detach()
        if x.device.type != "cpu":
            raise ValueError("oracle inputs must live on the host")
        if x.dtype == torch.bfloat16:
            a = x.view(torch.int16).numpy().view(np.uint16)
            code = BF16
        elif x.dtype == torch.float32:
            a, code = x.numpy(), F32
        elif x.dtype == torch.float64:
            a, code = x.numpy(), F64
        else:
            raise TypeError(f"unsupported logit dtype {x.dtype}")
    else:
        a = np.asarray(x)
        code = {np.dtype(np.float32): F32, np.dtype(np.float64): F64,
                np.dtype(np.uint16): BF16}[a.dtype]
    if a.ndim != 2:
        raise ValueError("logits must be 2-D (BT, V)")
    if a.strides[1] != a.itemsize or a.strides[0] % a.itemsize:
        a = np.ascontiguousarray(a)
    ld = a.strides[0] // a.itemsize if a.shape[0] > 1 else a.shape[1]
    return a, code, ld


def _i64(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _f64(x, n):
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64).reshape(-1))
    if a.size not in (1, n):
        raise ValueError("upstream gradient must hold 1 or BT values")
    return a, (0 if a.size == 1 else 1)


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def fused_ce_tvd_forward(student, teacher, target, ignore_index=-100, threads=None):
    """Per-row ce, tvd, student_lse, teacher_lse, sigma (fp64) and status."""
    s, code, ld_s = _logits(student)
    t, code_t, ld_t = _logits(teacher)
    if code != code_t or s.shape != t.shape:
        raise ValueError("student and teacher must share dtype and shape")
    tg = _i64(target)
    BT, V = s.shape
    out = {k: np.empty(BT, np.float64) for k in ("ce", "tvd", "student_lse", "teacher_lse", "sigma")}
    st = _load().oracle_fused_ce_tvd_forward(
        _ptr(s), ld_s, _ptr(t), ld_t, code, _ptr(tg), BT, V, int(ignore_index),
        _ptr(out["ce"]), _ptr(out["tvd"]), _ptr(out["student_lse"]),
        _ptr(out["teacher_lse"]), _ptr(out["sigma"]), _threads(threads))
    out["status"] = int(st)
    return out


def fused_ce_tvd_backward(student, teacher, target, grad_ce, grad_tvd,
                          ignore_index=-100, threads=None):
    """fp64 gradient of grad_ce.ce + grad_tvd.tvd w.r.t. the student logits."""
    s, code, ld_s = _logits(student)
    t, code_t, ld_t = _logits(teacher)
    if code != code_t or s.shape != t.shape:
        raise ValueError("student and teacher must share dtype and shape")
    tg = _i64(target)
    BT, V = s.shape
    gce, stride_ce = _f64(grad_ce, BT)
    gtvd, stride_tvd = _f64(grad_tvd, BT)
    if stride_ce != stride_tvd:
        gce = np.broadcast_to(gce, (BT,)).copy()
        gtvd = np.broadcast_to(gtvd, (BT,)).copy()
        stride_ce = 1
    grad = np.empty((BT, V), np.float64)
    st = _load().oracle_fused_ce_tvd_backward(
        _ptr(s), ld_s, _ptr(t), ld_t, code, _ptr(tg), BT, V, int(ignore_index),
        _ptr(gce), _ptr(gtvd), stride_ce, _ptr(grad), _threads(threads))
    return grad, int(st)


def ce_forward(logits, target, ignore_index=-100, threads=None):
    """Per-row ce and lse (fp64) and status."""
    x, code, ld = _logits(logits)
    tg = _i64(target)
    BT, V = x.shape
    ce = np.empty(BT, np.float64)
    lse = np.empty(BT, np.float64)
    st = _load().oracle_ce_forward(_ptr(x), ld, code, _ptr(tg), BT, V,
                                   int(ignore_index), _ptr(ce), _ptr(lse),
                                   _threads(threads))
    return {"ce": ce, "lse": lse, "status": int(st)}


def ce_backward(logits, target, grad_ce, ignore_index=-100, threads=None):
    """fp64 gradient of grad_ce.ce w.r.t. the logits, and status."""
    x, code, ld = _logits(logits)
    tg = _i64(target)
    BT, V = x.shape
    gce, stride = _f64(grad_ce, BT)
    grad = np.empty((BT, V), np.float64)
    st = _load().oracle_ce_backward(_ptr(x), ld, code, _ptr(tg), BT, V,
                                    int(ignore_index), _ptr(gce), stride,
                                    _ptr(grad), _threads(threads))
    return grad, int(st)


def row_probs(student, teacher, row):
    """fp64 softmax rows p (student) and q (teacher) of one row."""
    s, code, ld_s = _logits(student)
    t, _, ld_t = _logits(teacher)
    V = s.shape[1]
    p = np.empty(V, np.float64)
    q = np.empty(V, np.float64)
    _load().oracle_row_probs(_ptr(s), ld_s, _ptr(t), ld_t, code, int(row), V,
                             _ptr(p), _ptr(q))
    return p, q


def mean_loss(ce, tvd, target, ignore_index=-100, alpha=1.0, beta=1.0):
    """(loss, grad_ce, grad_tvd, n) of the mean over non-ignored rows."""
    ce = np.ascontiguousarray(np.asarray(ce, np.float64))
    tvd = np.ascontiguousarray(np.asarray(tvd, np.float64))
    tg = _i64(target)
    out = np.zeros(3, np.float64)
    n = _load().oracle_mean_loss(_ptr(ce), _ptr(tvd), _ptr(tg), tg.size, int(ignore_index),
                                 float(alpha), float(beta), ctypes.c_void_p(out.ctypes.data),
                                 ctypes.c_void_p(out.ctypes.data + 8),
                                 ctypes.c_void_p(out.ctypes.data + 16))
    return float(out[0]), float(out[1]), float(out[2]), int(n)
