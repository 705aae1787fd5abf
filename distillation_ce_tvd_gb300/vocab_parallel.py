"""Vocabulary-parallel CE + TVD: one step of the loss on a vocabulary shard.

Each device (or, on one device, each shard in turn) holds the columns
[v_begin, v_begin + V_shard) of every row of the student and teacher logits.
A step is three passes of the library over the shard with two exchanges of
per-row partials between them (3 and then 2 floats per row and shard), see
``fused_ce_tvd_vp_*`` in include/fused_ce_tvd.h.  The exchange is the
caller's: an all-gather in shard order across the devices of a vocabulary
group (``gather_across``), or stacking the partials of shards computed on one
device (``forward_backward_local``).  Every device ends with the same per-row
ce, tvd, lse and sigma and the gradient of its own columns.
"""
from __future__ import annotations

import torch

from . import binding


def shard_bounds(V: int, n_shards: int, k: int, elem_bytes: int = 2) -> tuple[int, int]:
    """Columns [begin, end) of shard k of n: contiguous, as equal as possible,
    every start a multiple of the 16-byte vector (8 bf16 or 4 fp32 columns),
    so that a shard of 16-byte-aligned rows keeps the vector path."""
    if not 0 <= k < n_shards:
        raise ValueError("shard index out of range")
    vec = max(1, 16 // elem_bytes)
    per = -(-V // n_shards)          # ceil
    per = -(-per // vec) * vec       # rounded up to whole vectors
    begin = min(V, k * per)
    return begin, min(V, begin + per)


def step(student, teacher, target, v_begin, V, grad_ce, grad_tvd, exchange,
         ignore_index=binding.IGNORE_INDEX, *, ops=binding, dev_status=None, stream=None):
    """One forward + backward step on one shard.

    ``exchange(part)`` returns the partials of every shard stacked in shard
    order, (n_shards, BT, k), with this shard's ``part`` at its own index.
    ``ops`` supplies the shard passes and merges (the library by default).
    Returns (ce, tvd, student_lse, teacher_lse, sigma, grad) with grad the
    gradient of this shard's columns.
    """
    part1 = ops.fused_ce_tvd_vp_lse(student, teacher, target, v_begin, ignore_index, stream=stream)
    ce, lse_s, lse_t = ops.fused_ce_tvd_vp_merge_lse(exchange(part1), target, V, ignore_index,
                                                     dev_status=dev_status, stream=stream)
    part2 = ops.fused_ce_tvd_vp_tvd(student, teacher, target, lse_s, lse_t, ignore_index,
                                    stream=stream)
    tvd, sigma = ops.fused_ce_tvd_vp_merge_tvd(exchange(part2), target, ignore_index,
                                               stream=stream)
    grad = ops.fused_ce_tvd_vp_backward(student, teacher, target, v_begin, V, lse_s, lse_t, sigma,
                                        grad_ce, grad_tvd, ignore_index, dev_status=dev_status,
                                        stream=stream)
    return ce, tvd, lse_s, lse_t, sigma, grad


def gather_across(group=None):
    """An exchange for ``step`` across the ranks of a torch.distributed group:
    the shards are the ranks, in rank order."""
    import torch.distributed as dist

    def exchange(part):
        parts = [torch.empty_like(part) for _ in range(dist.get_world_size(group))]
        dist.all_gather(parts, part.contiguous(), group=group)
        return torch.stack(parts)
    return exchange


def forward_backward_local(student, teacher, target, n_shards, grad_ce, grad_tvd,
                           ignore_index=binding.IGNORE_INDEX, *, dev_status=None, stream=None):
    """The vocabulary-parallel step with all shards on one device, as column
    views of the full (BT, V) logits: pass 1 on every shard, the merge, pass 2
    on every shard, the merge, the backward on every shard.  Returns the
    per-row outputs and the full (BT, V) gradient."""
    BT, V = student.shape
    bounds = [shard_bounds(V, n_shards, k, student.element_size()) for k in range(n_shards)]
    bounds = [(b, e) for b, e in bounds if e > b]
    views = [(student[:, b:e], teacher[:, b:e], b) for b, e in bounds]
    parts1 = torch.stack([binding.fused_ce_tvd_vp_lse(s, t, target, b, ignore_index, stream=stream)
                          for s, t, b in views])
    ce, lse_s, lse_t = binding.fused_ce_tvd_vp_merge_lse(parts1, target, V, ignore_index,
                                                         dev_status=dev_status, stream=stream)
    parts2 = torch.stack([binding.fused_ce_tvd_vp_tvd(s, t, target, lse_s, lse_t, ignore_index,
                                                      stream=stream) for s, t, _ in views])
    tvd, sigma = binding.fused_ce_tvd_vp_merge_tvd(parts2, target, ignore_index, stream=stream)
    grad = torch.empty_like(student)
    for (s, t, b), (_, e) in zip(views, bounds):
        binding.fused_ce_tvd_vp_backward(s, t, target, b, V, lse_s, lse_t, sigma, grad_ce,
                                         grad_tvd, ignore_index, grad_student=grad[:, b:e],
                                         dev_status=dev_status, stream=stream)
    return ce, tvd, lse_s, lse_t, sigma, grad
