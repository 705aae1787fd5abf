"""torch.autograd wrapper around the fused CE + TVD library calls.

The shape of the PR #1384 analysis's LigerFusedCETVDFunction: the forward
keeps only the O(BT) state (student_lse, teacher_lse, sigma) besides the
inputs, and the backward recomputes p and q from it.  No (BT, V)
intermediate is saved.
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
        ce, tvd, lse_s, lse_t, sigma = binding.fused_ce_tvd_forward(
            student.detach(), teacher.detach(), target, ignore_index)
        ctx.save_for_backward(student, teacher, target, lse_s, lse_t, sigma)
        ctx.ignore_index = ignore_index
        ctx.inplace = inplace
        return ce, tvd

    @staticmethod
    def backward(ctx, grad_ce, grad_tvd):
        student, teacher, target, lse_s, lse_t, sigma = ctx.saved_tensors
        BT = student.shape[0]
        dev = student.device
        gce = torch.zeros(BT, device=dev) if grad_ce is None else grad_ce.float().contiguous()
        gtvd = torch.zeros(BT, device=dev) if grad_tvd is None else grad_tvd.float().contiguous()
        grad = binding.fused_ce_tvd_backward(
            student.detach(), teacher.detach(), target, lse_s, lse_t, sigma, gce, gtvd,
            ctx.ignore_index, inplace=ctx.inplace)
        return grad, None, None, None, None


def fused_ce_tvd_loss(student, teacher, target, ignore_index=binding.IGNORE_INDEX,
                      inplace=False):
    """Per-row (ce, tvd) with autograd support; reduce them as the caller wishes."""
    return FusedCETVDFunction.apply(student, teacher, target, ignore_index, inplace)
