"""ctypes binding of libfused_ce_tvd.so (declared in include/fused_ce_tvd.h).

Argument marshalling only: tensors become device pointers, row strides and
dtype codes; outputs are allocated with torch when the caller passes none;
the work is launched on the current torch CUDA stream.  Every step of the
computation runs in the library's CUDA kernels.  There is no fallback: if
the library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import _build

FCT_F32, FCT_BF16 = 0, 1
FCT_DEV_TARGET_OUT_OF_RANGE = 0x1
IGNORE_INDEX = -100

_lock = threading.Lock()
_lib = None

EXPORTS = ("fused_ce_tvd_forward", "fused_ce_tvd_forward_ex", "fused_ce_tvd_backward",
           "fused_ce_tvd_forward_backward", "fused_ce_tvd_forward_backward_ex",
           "fused_ce_tvd_host_workspace_size", "fused_ce_tvd_forward_backward_host",
           "fused_ce_tvd_signs_row_bytes", "fused_ce_tvd_forward_signs",
           "fused_ce_tvd_forward_signs_ex", "fused_ce_tvd_backward_signs",
           "ce_forward", "ce_forward_ex", "ce_backward", "ce_forward_backward",
           "ce_forward_backward_ex", "fused_ce_tvd_mean_upstream", "fused_ce_tvd_mean_loss",
           "fused_linear_ce_tvd_workspace_size", "fused_linear_ce_tvd_forward_backward",
           "fused_linear_ce_tvd_forward_backward_noalloc", "fct_gemm_bf16",
           "fct_gemm_bf16_workspace_size",
           "fused_ce_tvd_vp_lse", "fused_ce_tvd_vp_merge_lse", "fused_ce_tvd_vp_tvd",
           "fused_ce_tvd_vp_merge_tvd", "fused_ce_tvd_vp_backward",
           "fct_status_string", "fct_version")


class Options(ctypes.Structure):
    """fct_options: launch options of one call (see include/fused_ce_tvd.h)."""
    _fields_ = [("ctas_per_row", ctypes.c_int32), ("l2_keep", ctypes.c_int32),
                ("stagger", ctypes.c_float), ("ring", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 4)]


RING_AUTO, RING_CP_ASYNC, RING_TMA = 0, 1, 2


def options(ctas_per_row: int = 0, l2_keep: int = 0, stagger: float = 0.0,
            ring: int = RING_AUTO) -> Options | None:
    """An fct_options value, or None when every field is automatic."""
    if ctas_per_row == 0 and l2_keep == 0 and stagger == 0.0 and ring == RING_AUTO:
        return None
    return Options(int(ctas_per_row), int(l2_keep), float(stagger), int(ring))


class FctError(RuntimeError):
    """A non-zero fct_status returned by the library."""

    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the shared library and declare its ABI."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        lib = ctypes.CDLL(path or _build.build())
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        op = ctypes.POINTER(Options)
        lib.fused_ce_tvd_forward.argtypes = [vp, i64, vp, i64, i32, vp, i64, i64, i64,
                                             vp, vp, vp, vp, vp, vp, vp]
        lib.fused_ce_tvd_forward_ex.argtypes = [vp, i64, vp, i64, i32, vp, i64, i64, i64,
                                                vp, vp, vp, vp, vp, op, vp, vp]
        lib.fused_ce_tvd_forward_ex.restype = i32
        lib.fused_ce_tvd_backward.argtypes = [vp, i64, vp, i64, i32, vp, i64, i64, i64,
                                              vp, vp, vp, vp, vp, i64, vp, i64, vp, vp]
        lib.fused_ce_tvd_forward_backward.argtypes = [vp, i64, vp, i64, i32, vp, i64, i64, i64,
                                                      vp, vp, i64, vp, vp, vp, vp, vp, vp, i64,
                                                      vp, vp]
        lib.fused_ce_tvd_forward_backward_ex.argtypes = [vp, i64, vp, i64, i32, vp, i64, i64,
                                                         i64, vp, vp, i64, vp, vp, vp, vp, vp,
                                                         vp, i64, op, vp, vp]
        lib.fused_ce_tvd_forward_backward_ex.restype = i32
        lib.fused_ce_tvd_host_workspace_size.argtypes = [i64, i32, i64]
        lib.fused_ce_tvd_host_workspace_size.restype = ctypes.c_size_t
        lib.fused_ce_tvd_forward_backward_host.argtypes = [
            vp, i64, vp, i64, i32, vp, i64, i64, i64, vp, vp, i64, vp, vp, vp, vp, vp, vp, i64,
            vp, ctypes.c_size_t, i64, vp, vp]
        lib.fused_ce_tvd_forward_backward_host.restype = i32
        lib.fused_ce_tvd_signs_row_bytes.argtypes = [i64, i32]
        lib.fused_ce_tvd_signs_row_bytes.restype = i64
        lib.fused_ce_tvd_forward_signs.argtypes = [vp, i64, vp, i64, i32, vp, i64, i64, i64,
                                                   vp, vp, vp, vp, vp, vp, i64, vp, vp]
        lib.fused_ce_tvd_forward_signs.restype = i32
        lib.fused_ce_tvd_forward_signs_ex.argtypes = [vp, i64, vp, i64, i32, vp, i64, i64, i64,
                                                      vp, vp, vp, vp, vp, vp, i64, op, vp, vp]
        lib.fused_ce_tvd_forward_signs_ex.restype = i32
        lib.fused_ce_tvd_backward_signs.argtypes = [vp, i64, vp, i64, i32, vp, i64, i64, i64,
                                                    vp, vp, vp, vp, i64, vp, vp, i64, vp, i64,
                                                    vp, vp]
        lib.fused_ce_tvd_backward_signs.restype = i32
        lib.ce_forward.argtypes = [vp, i64, i32, vp, i64, i64, i64, vp, vp, vp, vp]
        lib.ce_forward_ex.argtypes = [vp, i64, i32, vp, i64, i64, i64, vp, vp, op, vp, vp]
        lib.ce_forward_ex.restype = i32
        lib.ce_backward.argtypes = [vp, i64, i32, vp, i64, i64, i64, vp, vp, i64, vp, i64, vp, vp]
        lib.ce_forward_backward.argtypes = [vp, i64, i32, vp, i64, i64, i64, vp, i64, vp, vp, vp,
                                            i64, vp, vp]
        lib.ce_forward_backward.restype = i32
        lib.ce_forward_backward_ex.argtypes = [vp, i64, i32, vp, i64, i64, i64, vp, i64, vp, vp,
                                               vp, i64, op, vp, vp]
        lib.ce_forward_backward_ex.restype = i32
        dbl = ctypes.c_double
        lib.fused_linear_ce_tvd_workspace_size.argtypes = [i64, i64, i32]
        lib.fused_linear_ce_tvd_workspace_size.restype = ctypes.c_size_t
        lib.fused_linear_ce_tvd_forward_backward.argtypes = [
            vp, i64, vp, i64, i64, vp, i64, vp, i64, i64, vp, i64, i64, i64, vp, vp, i64,
            vp, vp, vp, vp, vp, vp, i64, vp, i64, i32, vp, ctypes.c_size_t, i64, vp, vp]
        lib.fused_linear_ce_tvd_forward_backward.restype = i32
        lib.fused_linear_ce_tvd_forward_backward_noalloc.argtypes = [
            vp, i64, vp, i64, i64, vp, i64, vp, i64, i64, vp, i64, i64, i64, vp, vp, i64,
            vp, vp, vp, vp, vp, vp, i64, vp, i64, vp, vp]
        lib.fused_linear_ce_tvd_forward_backward_noalloc.restype = i32
        lib.fct_gemm_bf16.argtypes = [vp, i64, i32, vp, i64, i32, vp, i64, i32, i64, i64, i64,
                                      vp, ctypes.c_size_t, vp, vp]
        lib.fct_gemm_bf16.restype = i32
        lib.fct_gemm_bf16_workspace_size.argtypes = [i64, i64]
        lib.fct_gemm_bf16_workspace_size.restype = ctypes.c_size_t
        lib.fused_ce_tvd_mean_upstream.argtypes = [vp, i64, i64, dbl, dbl, vp, vp, vp, vp]
        lib.fused_ce_tvd_mean_loss.argtypes = [vp, vp, vp, i64, i64, dbl, dbl, vp, vp]
        for f in ("fused_ce_tvd_forward", "fused_ce_tvd_backward", "fused_ce_tvd_forward_backward",
                  "ce_forward", "ce_backward", "fused_ce_tvd_mean_upstream",
                  "fused_ce_tvd_mean_loss"):
            getattr(lib, f).restype = i32
        lib.fused_ce_tvd_vp_lse.argtypes = [vp, i64, vp, i64, i32, vp, i64, i64, i64, i64, vp, vp]
        lib.fused_ce_tvd_vp_merge_lse.argtypes = [vp, i64, vp, i64, i64, i64, vp, vp, vp, vp, vp]
        lib.fused_ce_tvd_vp_tvd.argtypes = [vp, i64, vp, i64, i32, vp, i64, i64, i64, vp, vp, vp, vp]
        lib.fused_ce_tvd_vp_merge_tvd.argtypes = [vp, i64, vp, i64, i64, vp, vp, vp]
        lib.fused_ce_tvd_vp_backward.argtypes = [vp, i64, vp, i64, i32, vp, i64, i64, i64, i64, i64,
                                                 vp, vp, vp, vp, vp, i64, vp, i64, vp, vp]
        for f in ("fused_ce_tvd_vp_lse", "fused_ce_tvd_vp_merge_lse", "fused_ce_tvd_vp_tvd",
                  "fused_ce_tvd_vp_merge_tvd", "fused_ce_tvd_vp_backward"):
            getattr(lib, f).restype = i32
        lib.fct_status_string.argtypes = [i32]
        lib.fct_status_string.restype = ctypes.c_char_p
        lib.fct_version.argtypes = []
        lib.fct_version.restype = i32
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().fct_status_string(int(status)).decode()


def version() -> int:
    return load().fct_version()


# ------------------------------------------------------------------ marshalling

def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr() if t is not None else None)


def _logits(x: torch.Tensor, name: str):
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if x.dim() != 2 or (x.shape[1] > 1 and x.stride(1) != 1):
        raise ValueError(f"{name} must be (BT, V) with unit stride along V")
    code = {torch.float32: FCT_F32, torch.bfloat16: FCT_BF16}.get(x.dtype)
    if code is None:
        raise TypeError(f"{name}: dtype {x.dtype} is not float32 or bfloat16")
    ld = x.stride(0) if x.shape[0] > 1 else x.shape[1]
    return code, max(int(ld), int(x.shape[1]))


def _rows(x: torch.Tensor, n: int, name: str, dtype=torch.float32) -> torch.Tensor:
    if not x.is_cuda or x.dtype != dtype or x.dim() != 1 or x.numel() != n or (n > 1 and x.stride(0) != 1):
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} vector of {n} values")
    return x


def _upstream(g, BT: int, device, name: str):
    """(tensor, grad_stride): a per-row fp32 vector, or one value broadcast."""
    if not torch.is_tensor(g):
        g = torch.tensor([float(g)], device=device, dtype=torch.float32)
    if g.numel() == 1:
        g = g.reshape(1).to(device=device, dtype=torch.float32)
        return g, 0
    return _rows(g, BT, name), 1


def _opts(opts):
    """(suffix, extra ctypes args): the plain entry point for None, else its _ex form."""
    if opts is None:
        return "", ()
    if not isinstance(opts, Options):
        raise TypeError("options must be a binding.Options (see binding.options())")
    return "_ex", (ctypes.byref(opts),)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int, what: str):
    if rc != 0:
        raise FctError(rc, what)


def _out(x, n, device, name):
    if x is None:
        return torch.empty(n, device=device, dtype=torch.float32)
    return _rows(x, n, name)


# ------------------------------------------------------------------ entry points

def fused_ce_tvd_forward(student, teacher, target, ignore_index=IGNORE_INDEX, *, ce=None,
                         tvd=None, student_lse=None, teacher_lse=None, sigma=None,
                         dev_status=None, stream=None, options=None):
    """Per-row (ce, tvd, student_lse, teacher_lse, sigma), all fp32 (BT,)."""
    code, ld_s = _logits(student, "student")
    code_t, ld_t = _logits(teacher, "teacher")
    if code != code_t or student.shape != teacher.shape:
        raise ValueError("student and teacher must share shape and dtype")
    BT, V = student.shape
    dev = student.device
    _rows(target, BT, "target", torch.int64)
    outs = [_out(x, BT, dev, n) for x, n in ((ce, "ce"), (tvd, "tvd"), (student_lse, "student_lse"),
                                             (teacher_lse, "teacher_lse"), (sigma, "sigma"))]
    sfx, extra = _opts(options)
    rc = getattr(load(), "fused_ce_tvd_forward" + sfx)(
        _ptr(student), ld_s, _ptr(teacher), ld_t, code, _ptr(target), BT, V, int(ignore_index),
        *map(_ptr, outs), *extra, _ptr(dev_status), _stream(stream))
    _check(rc, "fused_ce_tvd_forward")
    return tuple(outs)


def fused_ce_tvd_backward(student, teacher, target, student_lse, teacher_lse, sigma,
                          grad_ce, grad_tvd, ignore_index=IGNORE_INDEX, *, grad_student=None,
                          inplace=False, dev_status=None, stream=None):
    """Gradient of sum_r grad_ce[r]*ce[r] + grad_tvd[r]*tvd[r] w.r.t. the student.

    ``inplace=True`` writes it over ``student`` and returns ``student``.
    """
    code, ld_s = _logits(student, "student")
    code_t, ld_t = _logits(teacher, "teacher")
    if code != code_t or student.shape != teacher.shape:
        raise ValueError("student and teacher must share shape and dtype")
    BT, V = student.shape
    dev = student.device
    _rows(target, BT, "target", torch.int64)
    for x, n in ((student_lse, "student_lse"), (teacher_lse, "teacher_lse"), (sigma, "sigma")):
        _rows(x, BT, n)
    gce, stride_ce = _upstream(grad_ce, BT, dev, "grad_ce")
    gtvd, stride_tvd = _upstream(grad_tvd, BT, dev, "grad_tvd")
    if stride_ce != stride_tvd:
        gce, gtvd = gce.expand(BT).contiguous(), gtvd.expand(BT).contiguous()
    stride = max(stride_ce, stride_tvd)
    if inplace:
        grad_student = student
    elif grad_student is None:
        grad_student = torch.empty_like(student)
    code_g, ld_g = _logits(grad_student, "grad_student")
    if code_g != code or grad_student.shape != student.shape:
        raise ValueError("grad_student must match the student's shape and dtype")
    rc = load().fused_ce_tvd_backward(_ptr(student), ld_s, _ptr(teacher), ld_t, code,
                                      _ptr(target), BT, V, int(ignore_index), _ptr(student_lse),
                                      _ptr(teacher_lse), _ptr(sigma), _ptr(gce), _ptr(gtvd),
                                      stride, _ptr(grad_student), ld_g, _ptr(dev_status),
                                      _stream(stream))
    _check(rc, "fused_ce_tvd_backward")
    return grad_student


def fused_ce_tvd_forward_backward(student, teacher, target, grad_ce, grad_tvd,
                                  ignore_index=IGNORE_INDEX, *, ce=None, tvd=None,
                                  student_lse=None, teacher_lse=None, sigma=None,
                                  grad_student=None, inplace=False, dev_status=None,
                                  stream=None, options=None):
    """Forward and backward in one launch, given the upstream gradients.

    Returns (ce, tvd, student_lse, teacher_lse, sigma, grad_student); the
    results equal fused_ce_tvd_forward followed by fused_ce_tvd_backward.
    """
    code, ld_s = _logits(student, "student")
    code_t, ld_t = _logits(teacher, "teacher")
    if code != code_t or student.shape != teacher.shape:
        raise ValueError("student and teacher must share shape and dtype")
    BT, V = student.shape
    dev = student.device
    _rows(target, BT, "target", torch.int64)
    gce, stride_ce = _upstream(grad_ce, BT, dev, "grad_ce")
    gtvd, stride_tvd = _upstream(grad_tvd, BT, dev, "grad_tvd")
    if stride_ce != stride_tvd:
        gce, gtvd = gce.expand(BT).contiguous(), gtvd.expand(BT).contiguous()
    stride = max(stride_ce, stride_tvd)
    outs = [_out(x, BT, dev, n) for x, n in ((ce, "ce"), (tvd, "tvd"), (student_lse, "student_lse"),
                                             (teacher_lse, "teacher_lse"), (sigma, "sigma"))]
    if inplace:
        grad_student = student
    elif grad_student is None:
        grad_student = torch.empty_like(student)
    code_g, ld_g = _logits(grad_student, "grad_student")
    if code_g != code or grad_student.shape != student.shape:
        raise ValueError("grad_student must match the student's shape and dtype")
    sfx, extra = _opts(options)
    rc = getattr(load(), "fused_ce_tvd_forward_backward" + sfx)(
        _ptr(student), ld_s, _ptr(teacher), ld_t, code, _ptr(target), BT, V, int(ignore_index),
        _ptr(gce), _ptr(gtvd), stride, *map(_ptr, outs), _ptr(grad_student), ld_g,
        *extra, _ptr(dev_status), _stream(stream))
    _check(rc, "fused_ce_tvd_forward_backward")
    return (*outs, grad_student)


def fused_ce_tvd_signs_row_bytes(V: int, dtype) -> int:
    """Minimum row stride, in bytes, of the sign words for V logits of ``dtype``."""
    code = {torch.float32: FCT_F32, torch.bfloat16: FCT_BF16}[dtype]
    return int(load().fused_ce_tvd_signs_row_bytes(int(V), code))


def _signs(x, BT, V, dtype, device):
    if x is None:
        return torch.empty(BT, fused_ce_tvd_signs_row_bytes(V, dtype), device=device,
                           dtype=torch.uint8)
    if not x.is_cuda or x.dtype != torch.uint8 or x.dim() != 2 or x.shape[0] != BT or \
            (BT > 1 and x.stride(1) != 1):
        raise ValueError(f"signs must be a (BT, >= row bytes) uint8 CUDA tensor with unit "
                         f"column stride")
    return x


def fused_ce_tvd_forward_signs(student, teacher, target, ignore_index=IGNORE_INDEX, *, ce=None,
                               tvd=None, student_lse=None, teacher_lse=None, sigma=None,
                               signs=None, dev_status=None, stream=None, options=None):
    """fused_ce_tvd_forward that also stores the sign words its backward reads
    instead of the teacher.  Returns (ce, tvd, student_lse, teacher_lse, sigma,
    signs), signs a (BT, row bytes) uint8 tensor."""
    code, ld_s = _logits(student, "student")
    code_t, ld_t = _logits(teacher, "teacher")
    if code != code_t or student.shape != teacher.shape:
        raise ValueError("student and teacher must share shape and dtype")
    BT, V = student.shape
    dev = student.device
    _rows(target, BT, "target", torch.int64)
    outs = [_out(x, BT, dev, n) for x, n in ((ce, "ce"), (tvd, "tvd"), (student_lse, "student_lse"),
                                             (teacher_lse, "teacher_lse"), (sigma, "sigma"))]
    signs = _signs(signs, BT, V, student.dtype, dev)
    ld_b = int(signs.stride(0)) if BT > 1 else int(signs.shape[1])
    sfx, extra = _opts(options)
    rc = getattr(load(), "fused_ce_tvd_forward_signs" + sfx)(
        _ptr(student), ld_s, _ptr(teacher), ld_t, code, _ptr(target), BT, V, int(ignore_index),
        *map(_ptr, outs), _ptr(signs), ld_b, *extra, _ptr(dev_status), _stream(stream))
    _check(rc, "fused_ce_tvd_forward_signs")
    return (*outs, signs)


def fused_ce_tvd_backward_signs(student, teacher, target, student_lse, teacher_lse, sigma, signs,
                                grad_ce, grad_tvd, ignore_index=IGNORE_INDEX, *,
                                grad_student=None, inplace=False, dev_status=None, stream=None):
    """fused_ce_tvd_backward reading the forward's sign words instead of the
    teacher (which rows with a tie still need); bit-identical gradient."""
    code, ld_s = _logits(student, "student")
    code_t, ld_t = _logits(teacher, "teacher")
    if code != code_t or student.shape != teacher.shape:
        raise ValueError("student and teacher must share shape and dtype")
    BT, V = student.shape
    dev = student.device
    _rows(target, BT, "target", torch.int64)
    for x, n in ((student_lse, "student_lse"), (teacher_lse, "teacher_lse"), (sigma, "sigma")):
        _rows(x, BT, n)
    signs = _signs(signs, BT, V, student.dtype, dev)
    ld_b = int(signs.stride(0)) if BT > 1 else int(signs.shape[1])
    gce, stride_ce = _upstream(grad_ce, BT, dev, "grad_ce")
    gtvd, stride_tvd = _upstream(grad_tvd, BT, dev, "grad_tvd")
    if stride_ce != stride_tvd:
        gce, gtvd = gce.expand(BT).contiguous(), gtvd.expand(BT).contiguous()
    stride = max(stride_ce, stride_tvd)
    if inplace:
        grad_student = student
    elif grad_student is None:
        grad_student = torch.empty_like(student)
    code_g, ld_g = _logits(grad_student, "grad_student")
    if code_g != code or grad_student.shape != student.shape:
        raise ValueError("grad_student must match the student's shape and dtype")
    rc = load().fused_ce_tvd_backward_signs(
        _ptr(student), ld_s, _ptr(teacher), ld_t, code, _ptr(target), BT, V, int(ignore_index),
        _ptr(student_lse), _ptr(teacher_lse), _ptr(sigma), _ptr(signs), ld_b, _ptr(gce),
        _ptr(gtvd), stride, _ptr(grad_student), ld_g, _ptr(dev_status), _stream(stream))
    _check(rc, "fused_ce_tvd_backward_signs")
    return grad_student


def ce_forward(logits, target, ignore_index=IGNORE_INDEX, *, ce=None, lse=None,
               dev_status=None, stream=None, options=None):
    """Per-row (ce, lse) of plain cross-entropy, fp32 (BT,)."""
    code, ld = _logits(logits, "logits")
    BT, V = logits.shape
    _rows(target, BT, "target", torch.int64)
    ce = _out(ce, BT, logits.device, "ce")
    lse = _out(lse, BT, logits.device, "lse")
    sfx, extra = _opts(options)
    rc = getattr(load(), "ce_forward" + sfx)(_ptr(logits), ld, code, _ptr(target), BT, V,
                                             int(ignore_index), _ptr(ce), _ptr(lse), *extra,
                                             _ptr(dev_status), _stream(stream))
    _check(rc, "ce_forward")
    return ce, lse


def ce_backward(logits, target, lse, grad_ce, ignore_index=IGNORE_INDEX, *, grad_logits=None,
                inplace=False, dev_status=None, stream=None):
    """Gradient of sum_r grad_ce[r]*ce[r] w.r.t. the logits."""
    code, ld = _logits(logits, "logits")
    BT, V = logits.shape
    _rows(target, BT, "target", torch.int64)
    _rows(lse, BT, "lse")
    gce, stride = _upstream(grad_ce, BT, logits.device, "grad_ce")
    if inplace:
        grad_logits = logits
    elif grad_logits is None:
        grad_logits = torch.empty_like(logits)
    code_g, ld_g = _logits(grad_logits, "grad_logits")
    if code_g != code or grad_logits.shape != logits.shape:
        raise ValueError("grad_logits must match the logits' shape and dtype")
    rc = load().ce_backward(_ptr(logits), ld, code, _ptr(target), BT, V, int(ignore_index),
                            _ptr(lse), _ptr(gce), stride, _ptr(grad_logits), ld_g,
                            _ptr(dev_status), _stream(stream))
    _check(rc, "ce_backward")
    return grad_logits


def ce_forward_backward(logits, target, grad_ce, ignore_index=IGNORE_INDEX, *, ce=None, lse=None,
                        grad_logits=None, inplace=False, dev_status=None, stream=None,
                        options=None):
    """Cross-entropy forward and backward in one launch: (ce, lse, grad_logits),
    bit-identical to ce_forward followed by ce_backward."""
    code, ld = _logits(logits, "logits")
    BT, V = logits.shape
    dev = logits.device
    _rows(target, BT, "target", torch.int64)
    gce, stride = _upstream(grad_ce, BT, dev, "grad_ce")
    ce = _out(ce, BT, dev, "ce")
    lse = _out(lse, BT, dev, "lse")
    if inplace:
        grad_logits = logits
    elif grad_logits is None:
        grad_logits = torch.empty_like(logits)
    code_g, ld_g = _logits(grad_logits, "grad_logits")
    if code_g != code or grad_logits.shape != logits.shape:
        raise ValueError("grad_logits must match the logits' shape and dtype")
    sfx, extra = _opts(options)
    rc = getattr(load(), "ce_forward_backward" + sfx)(
        _ptr(logits), ld, code, _ptr(target), BT, V, int(ignore_index), _ptr(gce), stride,
        _ptr(ce), _ptr(lse), _ptr(grad_logits), ld_g, *extra, _ptr(dev_status), _stream(stream))
    _check(rc, "ce_forward_backward")
    return ce, lse, grad_logits


def fused_ce_tvd_mean_upstream(target, ignore_index=IGNORE_INDEX, alpha=1.0, beta=1.0, *,
                               grad_ce=None, grad_tvd=None, count=None, stream=None):
    """Upstream gradients (alpha/n, beta/n) of the mean over the n kept rows,
    as 1-element device tensors, and n (1-element int64)."""
    if not target.is_cuda or target.dtype != torch.int64 or target.dim() != 1:
        raise ValueError("target must be a CUDA int64 vector")
    dev = target.device
    gce = grad_ce if grad_ce is not None else torch.empty(1, device=dev, dtype=torch.float32)
    gtvd = grad_tvd if grad_tvd is not None else torch.empty(1, device=dev, dtype=torch.float32)
    cnt = count if count is not None else torch.empty(1, device=dev, dtype=torch.int64)
    rc = load().fused_ce_tvd_mean_upstream(_ptr(target), target.numel(), int(ignore_index),
                                           float(alpha), float(beta), _ptr(gce), _ptr(gtvd),
                                           _ptr(cnt), _stream(stream))
    _check(rc, "fused_ce_tvd_mean_upstream")
    return gce, gtvd, cnt


def fused_ce_tvd_mean_loss(ce, tvd, target, ignore_index=IGNORE_INDEX, alpha=1.0, beta=1.0, *,
                           loss=None, stream=None):
    """(alpha * sum ce + beta * sum tvd) / n over the kept rows, as a 1-element tensor."""
    BT = target.numel()
    _rows(ce, BT, "ce")
    _rows(tvd, BT, "tvd")
    _rows(target, BT, "target", torch.int64)
    out = loss if loss is not None else torch.empty(1, device=ce.device, dtype=torch.float32)
    rc = load().fused_ce_tvd_mean_loss(_ptr(ce), _ptr(tvd), _ptr(target), BT, int(ignore_index),
                                       float(alpha), float(beta), _ptr(out), _stream(stream))
    _check(rc, "fused_ce_tvd_mean_loss")
    return out


def fused_ce_tvd_host_workspace_size(V: int, dtype, block_rows: int) -> int:
    """Bytes of device workspace fused_ce_tvd_forward_backward_host needs."""
    code = {torch.float32: FCT_F32, torch.bfloat16: FCT_BF16}[dtype]
    return int(load().fused_ce_tvd_host_workspace_size(int(V), code, int(block_rows)))


def _host(x, name, dtype=None, dims=None):
    if x.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if dtype is not None and x.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    if dims is not None and x.dim() != dims:
        raise ValueError(f"{name} must have {dims} dimension(s)")
    if x.dim() == 1 and x.numel() > 1 and x.stride(0) != 1:
        raise ValueError(f"{name} must be contiguous")
    if x.dim() == 2 and x.shape[1] > 1 and x.stride(1) != 1:
        raise ValueError(f"{name} must have unit stride along V")
    return x


def fused_ce_tvd_forward_backward_host(student, teacher, target, grad_ce, grad_tvd,
                                       ignore_index=IGNORE_INDEX, *, ce=None, tvd=None,
                                       student_lse=None, teacher_lse=None, sigma=None,
                                       grad_student=None, want_grad=True, block_rows=512,
                                       workspace=None, status=None, device=None, stream=None):
    """Single-launch forward + backward with every input and output in host memory.

    ``student``/``teacher`` (BT, V), ``target`` (BT,) int64 and the upstream
    gradients (BT values or one) are CPU tensors, page-locked for the copies
    to overlap the compute (``tensor.pin_memory()``).  The library copies row
    blocks of ``block_rows`` rows through a device ``workspace`` (allocated
    here when not given), computes them, and copies the gradient and the five
    per-row outputs back into CPU tensors (allocated pinned when not given).
    Returns (ce, tvd, student_lse, teacher_lse, sigma, grad_student); read them
    after synchronising ``stream``.  ``status`` (a 1-element int32 CPU tensor)
    receives the device status bits.
    """
    _host(student, "student", dims=2)
    _host(teacher, "teacher", dims=2)
    if student.dtype != teacher.dtype or student.shape != teacher.shape:
        raise ValueError("student and teacher must share shape and dtype")
    code = {torch.float32: FCT_F32, torch.bfloat16: FCT_BF16}.get(student.dtype)
    if code is None:
        raise TypeError(f"dtype {student.dtype} is not float32 or bfloat16")
    BT, V = student.shape
    ld_s = max(int(student.stride(0)) if BT > 1 else V, V)
    ld_t = max(int(teacher.stride(0)) if BT > 1 else V, V)
    _host(target, "target", torch.int64, 1)
    if target.numel() != BT:
        raise ValueError("target must hold BT values")
    ups = []
    for g, name in ((grad_ce, "grad_ce"), (grad_tvd, "grad_tvd")):
        if not torch.is_tensor(g):
            g = torch.tensor([float(g)], dtype=torch.float32)
        _host(g, name, torch.float32)
        g = g.reshape(-1) if g.dim() != 1 else g
        if g.numel() not in (1, BT) or (g.numel() > 1 and g.stride(0) != 1):
            raise ValueError(f"{name} must be a contiguous float32 vector of {BT} values or one")
        ups.append(g)
    stride_ce, stride_tvd = int(ups[0].numel() != 1 or BT == 1), int(ups[1].numel() != 1 or BT == 1)
    if stride_ce != stride_tvd:
        ups = [u.expand(BT).contiguous() if u.numel() == 1 else u for u in ups]
    stride = max(stride_ce, stride_tvd)
    pin = student.is_pinned()
    outs = []
    for x, n in ((ce, "ce"), (tvd, "tvd"), (student_lse, "student_lse"),
                 (teacher_lse, "teacher_lse"), (sigma, "sigma")):
        if x is None:
            x = torch.empty(BT, dtype=torch.float32, pin_memory=pin)
        _host(x, n, torch.float32, 1)
        if x.numel() != BT:
            raise ValueError(f"{n} must hold BT values")
        outs.append(x)
    if grad_student is None and want_grad:
        grad_student = torch.empty(BT, V, dtype=student.dtype, pin_memory=pin)
    ld_g = V
    if grad_student is not None:
        _host(grad_student, "grad_student", student.dtype, 2)
        if grad_student.shape != student.shape:
            raise ValueError("grad_student must match the student's shape")
        ld_g = max(int(grad_student.stride(0)) if BT > 1 else V, V)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    rows = max(1, min(int(block_rows), max(BT, 1)))
    need = fused_ce_tvd_host_workspace_size(V, student.dtype, rows)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=dev, dtype=torch.uint8)
    if not workspace.is_cuda:
        raise ValueError("workspace must be device memory")
    if status is not None:
        _host(status, "status", torch.int32, 1)
    with torch.cuda.device(dev):
        rc = load().fused_ce_tvd_forward_backward_host(
            _ptr(student), ld_s, _ptr(teacher), ld_t, code, _ptr(target), BT, V,
            int(ignore_index), _ptr(ups[0]), _ptr(ups[1]), stride, *map(_ptr, outs),
            _ptr(grad_student), ld_g, _ptr(workspace),
            workspace.numel() * workspace.element_size(), rows, _ptr(status), _stream(stream))
    _check(rc, "fused_ce_tvd_forward_backward_host")
    return (*outs, grad_student)


# ------------------------------------------------------------------ vocabulary shards

def _pair(student, teacher):
    code, ld_s = _logits(student, "student")
    code_t, ld_t = _logits(teacher, "teacher")
    if code != code_t or student.shape != teacher.shape:
        raise ValueError("student and teacher shards must share shape and dtype")
    return code, ld_s, ld_t


def _parts(x, k, name):
    if not x.is_cuda or x.dtype != torch.float32 or x.dim() != 3 or x.shape[2] != k or \
            not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous (n_shards, BT, {k}) float32 CUDA tensor")
    return x


def fused_ce_tvd_vp_lse(student, teacher, target, v_begin, ignore_index=IGNORE_INDEX, *,
                        part=None, stream=None):
    """Pass 1 on one vocabulary shard: (BT, 3) float32 of the shard's student
    lse, teacher lse and the student logit at the target when the shard holds
    it.  ``student``/``teacher`` are the shard's (BT, V_shard) columns;
    ``v_begin`` their first column in the full vocabulary."""
    code, ld_s, ld_t = _pair(student, teacher)
    BT, Vs = student.shape
    _rows(target, BT, "target", torch.int64)
    if part is None:
        part = torch.empty(BT, 3, device=student.device, dtype=torch.float32)
    rc = load().fused_ce_tvd_vp_lse(_ptr(student), ld_s, _ptr(teacher), ld_t, code, _ptr(target),
                                    BT, Vs, int(v_begin), int(ignore_index), _ptr(part),
                                    _stream(stream))
    _check(rc, "fused_ce_tvd_vp_lse")
    return part


def fused_ce_tvd_vp_merge_lse(parts, target, V, ignore_index=IGNORE_INDEX, *, ce=None,
                              student_lse=None, teacher_lse=None, dev_status=None, stream=None):
    """Merge of pass 1 over the shards (``parts``: (n_shards, BT, 3), shard
    order): (ce, student_lse, teacher_lse)."""
    _parts(parts, 3, "parts")
    n, BT = parts.shape[0], parts.shape[1]
    _rows(target, BT, "target", torch.int64)
    dev = parts.device
    outs = [_out(x, BT, dev, nm) for x, nm in ((ce, "ce"), (student_lse, "student_lse"),
                                               (teacher_lse, "teacher_lse"))]
    rc = load().fused_ce_tvd_vp_merge_lse(_ptr(parts), n, _ptr(target), BT, int(V),
                                          int(ignore_index), *map(_ptr, outs), _ptr(dev_status),
                                          _stream(stream))
    _check(rc, "fused_ce_tvd_vp_merge_lse")
    return tuple(outs)


def fused_ce_tvd_vp_tvd(student, teacher, target, student_lse, teacher_lse,
                        ignore_index=IGNORE_INDEX, *, part=None, stream=None):
    """Pass 2 on one shard: (BT, 2) float32 of the shard's sum of p*sign(p - q)
    and q*sign(p - q), p and q from the merged lse values."""
    code, ld_s, ld_t = _pair(student, teacher)
    BT, Vs = student.shape
    _rows(target, BT, "target", torch.int64)
    _rows(student_lse, BT, "student_lse")
    _rows(teacher_lse, BT, "teacher_lse")
    if part is None:
        part = torch.empty(BT, 2, device=student.device, dtype=torch.float32)
    rc = load().fused_ce_tvd_vp_tvd(_ptr(student), ld_s, _ptr(teacher), ld_t, code, _ptr(target), BT,
                                    Vs, int(ignore_index), _ptr(student_lse), _ptr(teacher_lse),
                                    _ptr(part), _stream(stream))
    _check(rc, "fused_ce_tvd_vp_tvd")
    return part


def fused_ce_tvd_vp_merge_tvd(parts, target, ignore_index=IGNORE_INDEX, *, tvd=None, sigma=None,
                              stream=None):
    """Merge of pass 2 over the shards (``parts``: (n_shards, BT, 2)): (tvd, sigma)."""
    _parts(parts, 2, "parts")
    n, BT = parts.shape[0], parts.shape[1]
    _rows(target, BT, "target", torch.int64)
    dev = parts.device
    outs = [_out(x, BT, dev, nm) for x, nm in ((tvd, "tvd"), (sigma, "sigma"))]
    rc = load().fused_ce_tvd_vp_merge_tvd(_ptr(parts), n, _ptr(target), BT, int(ignore_index),
                                          *map(_ptr, outs), _stream(stream))
    _check(rc, "fused_ce_tvd_vp_merge_tvd")
    return tuple(outs)


def fused_ce_tvd_vp_backward(student, teacher, target, v_begin, V, student_lse, teacher_lse, sigma,
                             grad_ce, grad_tvd, ignore_index=IGNORE_INDEX, *, grad_student=None,
                             inplace=False, dev_status=None, stream=None):
    """Pass 3 on one shard: the gradient of the shard's columns."""
    code, ld_s, ld_t = _pair(student, teacher)
    BT, Vs = student.shape
    dev = student.device
    _rows(target, BT, "target", torch.int64)
    for x, nm in ((student_lse, "student_lse"), (teacher_lse, "teacher_lse"), (sigma, "sigma")):
        _rows(x, BT, nm)
    gce, stride_ce = _upstream(grad_ce, BT, dev, "grad_ce")
    gtvd, stride_tvd = _upstream(grad_tvd, BT, dev, "grad_tvd")
    if stride_ce != stride_tvd:
        gce, gtvd = gce.expand(BT).contiguous(), gtvd.expand(BT).contiguous()
    stride = max(stride_ce, stride_tvd)
    if inplace:
        grad_student = student
    elif grad_student is None:
        grad_student = torch.empty(BT, Vs, device=dev, dtype=student.dtype)
    code_g, ld_g = _logits(grad_student, "grad_student")
    if code_g != code or grad_student.shape != student.shape:
        raise ValueError("grad_student must match the shard's shape and dtype")
    rc = load().fused_ce_tvd_vp_backward(
        _ptr(student), ld_s, _ptr(teacher), ld_t, code, _ptr(target), BT, Vs, int(v_begin), int(V),
        int(ignore_index), _ptr(student_lse), _ptr(teacher_lse), _ptr(sigma), _ptr(gce),
        _ptr(gtvd), stride, _ptr(grad_student), ld_g, _ptr(dev_status), _stream(stream))
    _check(rc, "fused_ce_tvd_vp_backward")
    return grad_student


def _logits_dtype(dtype) -> int:
    if dtype == torch.float32:
        return FCT_F32
    if dtype == torch.bfloat16:
        return FCT_BF16
    raise ValueError("logits_dtype must be torch.float32 or torch.bfloat16")


def fused_linear_ce_tvd_workspace_size(V: int, chunk_rows: int,
                                       logits_dtype=torch.float32) -> int:
    """Bytes of device workspace fused_linear_ce_tvd_forward_backward needs."""
    return int(load().fused_linear_ce_tvd_workspace_size(int(V), int(chunk_rows),
                                                         _logits_dtype(logits_dtype)))


def _mat(x, name):
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or (x.shape[1] > 1 and x.stride(1) != 1):
        raise ValueError(f"{name} must be a 2-D bf16 CUDA tensor with unit stride along columns")
    return max(int(x.stride(0)) if x.shape[0] > 1 else int(x.shape[1]), int(x.shape[1]))


def fused_linear_ce_tvd_forward_backward(h_student, w_student, h_teacher, w_teacher, target,
                                         grad_ce, grad_tvd, ignore_index=IGNORE_INDEX, *,
                                         chunk_rows=2048, logits_dtype=torch.float32,
                                         workspace=None, grad_h=None, grad_w=None,
                                         want_grad_h=True, want_grad_w=True, dev_status=None,
                                         stream=None):
    """Loss from hidden states and lm_head weights, in row blocks (no (BT, V) logits).

    Returns (ce, tvd, student_lse, teacher_lse, sigma, grad_h, grad_w): grad_h
    is d loss / d h_student (bf16), grad_w is d loss / d w_student (fp32,
    accumulated into when passed in; zero-initialised otherwise).
    ``logits_dtype`` (torch.float32 or torch.bfloat16) is the element type of
    the logit blocks the loss kernel reads.  ``chunk_rows`` is the rows per
    block; the results do not depend on it, the workspace grows with it (see
    fused_linear_ce_tvd_workspace_size).  At 8192 rows, hidden 4096 and
    V = 151936 on GB300, 2048 rows took 25.1 ms (bf16 blocks) and 26.4 ms
    (fp32) against 27.2 and 28.1 ms with 1024 rows; 4096 was no faster.
    """
    ld_hs, ld_ws = _mat(h_student, "h_student"), _mat(w_student, "w_student")
    ld_ht, ld_wt = _mat(h_teacher, "h_teacher"), _mat(w_teacher, "w_teacher")
    BT, ds = h_student.shape
    V = w_student.shape[0]
    dt = h_teacher.shape[1]
    if w_student.shape[1] != ds or w_teacher.shape != (V, dt) or h_teacher.shape[0] != BT:
        raise ValueError("inconsistent hidden / weight shapes")
    dev = h_student.device
    _rows(target, BT, "target", torch.int64)
    gce, stride_ce = _upstream(grad_ce, BT, dev, "grad_ce")
    gtvd, stride_tvd = _upstream(grad_tvd, BT, dev, "grad_tvd")
    if stride_ce != stride_tvd:
        gce, gtvd = gce.expand(BT).contiguous(), gtvd.expand(BT).contiguous()
    stride = max(stride_ce, stride_tvd)
    outs = [torch.empty(BT, device=dev, dtype=torch.float32) for _ in range(5)]
    rows = max(1, min(int(chunk_rows), BT))
    code = _logits_dtype(logits_dtype)
    need = fused_linear_ce_tvd_workspace_size(V, rows, logits_dtype)
    if workspace is None:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    if want_grad_h and grad_h is None:
        grad_h = torch.empty_like(h_student)
    if want_grad_w and grad_w is None:
        grad_w = torch.zeros(V, ds, device=dev, dtype=torch.float32)
    ld_gh = _mat(grad_h, "grad_h") if grad_h is not None else ds
    if grad_w is not None and (grad_w.dtype != torch.float32 or grad_w.shape != (V, ds)):
        raise ValueError("grad_w must be (V, d_student) float32")
    ld_gw = int(grad_w.stride(0)) if grad_w is not None else ds
    rc = load().fused_linear_ce_tvd_forward_backward(
        _ptr(h_student), ld_hs, _ptr(w_student), ld_ws, ds, _ptr(h_teacher), ld_ht,
        _ptr(w_teacher), ld_wt, dt, _ptr(target), BT, V, int(ignore_index), _ptr(gce),
        _ptr(gtvd), stride, *map(_ptr, outs), _ptr(grad_h), ld_gh, _ptr(grad_w), ld_gw, code,
        _ptr(workspace), workspace.numel() * workspace.element_size(), rows,
        _ptr(dev_status), _stream(stream))
    _check(rc, "fused_linear_ce_tvd_forward_backward")
    return (*outs, grad_h, grad_w)


GEMM_F32, GEMM_BF16, GEMM_ADD_F32 = 0, 1, 2


def _operand(x: torch.Tensor, name: str):
    """(ld, mn_major) of a 2-D bf16 operand viewed as given: row-major
    (stride (ld, 1)) is K-major, column-major (stride (1, ld)) MN-major."""
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError(f"{name} must be a 2-D bfloat16 CUDA tensor")
    if x.stride(1) == 1:
        return int(x.stride(0)), 0
    if x.stride(0) == 1:
        return int(x.stride(1)), 1
    raise ValueError(f"{name} needs one unit stride")


def fct_gemm_bf16_workspace_size(M: int, N: int) -> int:
    return int(load().fct_gemm_bf16_workspace_size(int(M), int(N)))


def fct_gemm_bf16(a, b, c=None, *, accumulate=False, out_dtype=torch.float32, workspace=None,
                  dev_status=None, stream=None):
    """C = a @ b.T (or C += a @ b.T into an fp32 c) on the library's tcgen05 GEMM.

    a (M, K) and b (N, K) are bf16 CUDA tensors with one unit stride each
    (b.T of a row-major (K, N) tensor is the MN-major case); c is (M, N),
    row-major, fp32 or bf16 (bf16 only without accumulate).  ``workspace``
    (a CUDA tensor, optional) lets a product with few output tiles and a long
    K split K; see fct_gemm_bf16_workspace_size."""
    lda, a_mn = _operand(a, "a")
    ldb, b_mn = _operand(b, "b")
    M, K = a.shape
    N, K2 = b.shape
    if K != K2:
        raise ValueError("a and b differ in K")
    if c is None:
        if accumulate:
            raise ValueError("accumulate needs c")
        c = torch.empty(M, N, device=a.device, dtype=out_dtype)
    if c.dim() != 2 or tuple(c.shape) != (M, N) or (N > 1 and c.stride(1) != 1):
        raise ValueError("c must be a row-major (M, N) tensor")
    if c.dtype == torch.bfloat16 and not accumulate:
        kind = GEMM_BF16
    elif c.dtype == torch.float32:
        kind = GEMM_ADD_F32 if accumulate else GEMM_F32
    else:
        raise ValueError("c must be float32, or bfloat16 without accumulate")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().fct_gemm_bf16(_ptr(a), lda, a_mn, _ptr(b), ldb, b_mn, _ptr(c),
                              int(c.stride(0)) if M > 1 else N, kind, M, N, K,
                              _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(rc, "fct_gemm_bf16")
    return c


def fused_linear_ce_tvd_forward_backward_noalloc(h_student, w_student, h_teacher, w_teacher,
                                                 target, grad_ce, grad_tvd, ce, tvd, student_lse,
                                                 teacher_lse, sigma, grad_h=None, grad_w=None,
                                                 ignore_index=IGNORE_INDEX, *, dev_status=None,
                                                 stream=None):
    """fused_linear_ce_tvd_forward_backward with every buffer supplied by the
    caller, for callers that cannot let a library allocate device memory.

    grad_ce and grad_tvd are fp32 CUDA tensors of BT values or of one value
    (broadcast); ce ... sigma are (BT,) fp32 outputs; grad_h (BT, d_student)
    bf16 and grad_w (V, d_student) fp32 (accumulated into) are optional.
    Nothing is allocated here or in the library call.
    """
    ld_hs, ld_ws = _mat(h_student, "h_student"), _mat(w_student, "w_student")
    ld_ht, ld_wt = _mat(h_teacher, "h_teacher"), _mat(w_teacher, "w_teacher")
    BT, ds = h_student.shape
    V = w_student.shape[0]
    dt = h_teacher.shape[1]
    if w_student.shape[1] != ds or w_teacher.shape != (V, dt) or h_teacher.shape[0] != BT:
        raise ValueError("inconsistent hidden / weight shapes")
    _rows(target, BT, "target", torch.int64)
    strides = []
    for g, name in ((grad_ce, "grad_ce"), (grad_tvd, "grad_tvd")):
        # exactly the tensor handed to the library: a 1-D vector (no reshape,
        # which could silently copy a non-contiguous view)
        if not torch.is_tensor(g) or g.dim() != 1 or g.numel() not in (1, BT):
            raise ValueError(f"{name} must be a 1-D CUDA tensor of {BT} values or of one value")
        strides.append(0 if g.numel() == 1 and BT != 1 else 1)
        _rows(g, g.numel(), name)
    if strides[0] != strides[1]:
        raise ValueError("grad_ce and grad_tvd must both be per-row or both be one value")
    outs = [_rows(x, BT, n) for x, n in ((ce, "ce"), (tvd, "tvd"), (student_lse, "student_lse"),
                                          (teacher_lse, "teacher_lse"), (sigma, "sigma"))]
    ld_gh = _mat(grad_h, "grad_h") if grad_h is not None else ds
    if grad_h is not None and grad_h.shape != (BT, ds):
        raise ValueError("grad_h must be (BT, d_student) bf16")
    if grad_w is not None and (grad_w.dtype != torch.float32 or grad_w.shape != (V, ds)
                               or (ds > 1 and grad_w.stride(1) != 1)):
        raise ValueError("grad_w must be (V, d_student) float32 with unit column stride")
    ld_gw = max(int(grad_w.stride(0)), ds) if grad_w is not None else ds
    rc = load().fused_linear_ce_tvd_forward_backward_noalloc(
        _ptr(h_student), ld_hs, _ptr(w_student), ld_ws, ds, _ptr(h_teacher), ld_ht,
        _ptr(w_teacher), ld_wt, dt, _ptr(target), BT, V, int(ignore_index), _ptr(grad_ce),
        _ptr(grad_tvd), strides[0], *map(_ptr, outs), _ptr(grad_h), ld_gh, _ptr(grad_w), ld_gw,
        _ptr(dev_status), _stream(stream))
    _check(rc, "fused_linear_ce_tvd_forward_backward_noalloc")
    return (*outs, grad_h, grad_w)
