"""torch.autograd wrapper around the fused CE + TVD library calls.

The shape of the PR #1384 analysis's LigerFusedCETVDFunction: the forward
keeps only the O(BT) state (student_lse, teacher_lse, sigma) besides the
inputs, and the backward recomputes p from it.  No (BT, V) intermediate of
the logits' size is saved: the per-row wrapper keeps the sign of p - q as one
bit per element (sign words), so its backward reads the student and those
bits instead of the teacher, with the same gradient bit for bit.
"""
from __future__ import annotations

import torch

from . import binding


class FusedCETVDFunction(torch.autograd.Function):
    """(student, teacher, target) -> per-row (ce, tvd); gradient w.r.t. student only.

    With ``inplace=True`` the backward writes the gradient over the student
    logits' storage (saving a (BT, V) buffer); the student tensor must not be
    used again after the backward.
    """

    @staticmethod
    def forward(ctx, student, teacher, target, ignore_index=binding.IGNORE_INDEX, inplace=False):
        ce, tvd, lse_s, lse_t, sigma, signs = binding.fused_ce_tvd_forward_signs(
            student.detach(), teacher.detach(), target, ignore_index)
        ctx.save_for_backward(student, teacher, target, lse_s, lse_t, sigma, signs)
        ctx.ignore_index = ignore_index
        ctx.inplace = inplace
        return ce, tvd

    @staticmethod
    def backward(ctx, grad_ce, grad_tvd):
        student, teacher, target, lse_s, lse_t, sigma, signs = ctx.saved_tensors
        BT = student.shape[0]
        dev = student.device
        gce = torch.zeros(BT, device=dev) if grad_ce is None else grad_ce.float().contiguous()
        gtvd = torch.zeros(BT, device=dev) if grad_tvd is None else grad_tvd.float().contiguous()
        grad = binding.fused_ce_tvd_backward_signs(
            student.detach(), teacher.detach(), target, lse_s, lse_t, sigma, signs, gce, gtvd,
            ctx.ignore_index, inplace=ctx.inplace)
        return grad, None, None, None, None


def fused_ce_tvd_loss(student, teacher, target, ignore_index=binding.IGNORE_INDEX,
                      inplace=False):
    """Per-row (ce, tvd) with autograd support; reduce them as the caller wishes."""
    return FusedCETVDFunction.apply(student, teacher, target, ignore_index, inplace)


class FusedCETVDMeanLoss(torch.autograd.Function):
    """alpha * mean(ce) + beta * mean(tvd) over the rows not ignored, as a scalar.

    The upstream gradients of a mean are known before the forward (alpha/n and
    beta/n, computed on the device from the targets), so the forward runs the
    single-launch forward + backward and keeps the student gradient; the
    backward only hands it out (scaled by the incoming gradient when that is
    not 1).  With ``inplace=True`` the gradient overwrites the student logits.
    """

    @staticmethod
    def forward(ctx, student, teacher, target, ignore_index=binding.IGNORE_INDEX, alpha=1.0,
                beta=1.0, inplace=False):
        gce, gtvd, _ = binding.fused_ce_tvd_mean_upstream(target, ignore_index, alpha, beta)
        s = student.detach()
        ce, tvd, _, _, _, grad = binding.fused_ce_tvd_forward_backward(
            s, teacher.detach(), target, gce, gtvd, ignore_index, inplace=inplace)
        loss = binding.fused_ce_tvd_mean_loss(ce, tvd, target, ignore_index, alpha, beta)
        ctx.save_for_backward(grad)
        return loss.reshape(())

    @staticmethod
    def backward(ctx, grad_out):
        (grad,) = ctx.saved_tensors
        if not torch.equal(grad_out, torch.ones_like(grad_out)):
            grad = grad * grad_out.to(grad.dtype)
        return grad, None, None, None, None, None, None


def fused_ce_tvd_mean_loss(student, teacher, target, ignore_index=binding.IGNORE_INDEX,
                           alpha=1.0, beta=1.0, inplace=False):
    """Scalar alpha * mean(ce) + beta * mean(tvd) with autograd support."""
    return FusedCETVDMeanLoss.apply(student, teacher, target, ignore_index, alpha, beta, inplace)


class FusedLinearCETVDMeanLoss(torch.autograd.Function):
    """alpha * mean(ce) + beta * mean(tvd) from hidden states and lm_head weights.

    The student's logits are h_student @ w_student.T and the teacher's
    h_teacher @ w_teacher.T, computed in row blocks and never held whole.
    As for FusedCETVDMeanLoss, the upstream gradients of the mean are known
    before the forward, so the forward runs the whole fused-linear forward +
    backward and keeps d loss / d h_student and d loss / d w_student; the
    backward hands them out.  The teacher is frozen.  The weight gradient is
    accumulated in fp32; autograd casts it to the weight's dtype.
    """

    @staticmethod
    def forward(ctx, h_student, w_student, h_teacher, w_teacher, target,
                ignore_index=binding.IGNORE_INDEX, alpha=1.0, beta=1.0, chunk_rows=2048,
                logits_dtype=torch.float32):
        gce, gtvd, _ = binding.fused_ce_tvd_mean_upstream(target, ignore_index, alpha, beta)
        ce, tvd, _, _, _, grad_h, grad_w = binding.fused_linear_ce_tvd_forward_backward(
            h_student.detach(), w_student.detach(), h_teacher.detach(), w_teacher.detach(),
            target, gce, gtvd, ignore_index, chunk_rows=chunk_rows, logits_dtype=logits_dtype,
            want_grad_h=ctx.needs_input_grad[0], want_grad_w=ctx.needs_input_grad[1])
        loss = binding.fused_ce_tvd_mean_loss(ce, tvd, target, ignore_index, alpha, beta)
        ctx.grads = (grad_h, grad_w)
        return loss.reshape(())

    @staticmethod
    def backward(ctx, grad_out):
        grad_h, grad_w = ctx.grads
        if not torch.equal(grad_out, torch.ones_like(grad_out)):
            grad_h = None if grad_h is None else grad_h * grad_out.to(grad_h.dtype)
            grad_w = None if grad_w is None else grad_w * grad_out.to(grad_w.dtype)
        return grad_h, grad_w, None, None, None, None, None, None, None, None


def fused_linear_ce_tvd_mean_loss(h_student, w_student, h_teacher, w_teacher, target,
                                  ignore_index=binding.IGNORE_INDEX, alpha=1.0, beta=1.0,
                                  chunk_rows=2048, logits_dtype=torch.float32):
    """Scalar alpha * mean(ce) + beta * mean(tvd) of the lm_head logits, with
    autograd support for h_student and w_student (2-D bf16 tensors).
    ``logits_dtype`` is the element type of the logit blocks (float32 or
    bfloat16)."""
    return FusedLinearCETVDMeanLoss.apply(h_student, w_student, h_teacher, w_teacher, target,
                                          ignore_index, alpha, beta, chunk_rows, logits_dtype)
