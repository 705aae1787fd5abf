"""Model check of the bulk-copy ring's schedule (`forward_tma`, `RingPlan`).

The single-launch kernel's producer lane fills ring slot t % 3 for fill t,
each slot holding a student half and a teacher half; the consumer warps read
a fill after waiting on its `full` barrier and release it on `empty`; the
producer refills a slot only after the release of the slot's previous fill,
and waits on a per-row `carry_bar` before a row's first fill.  Steps carried
from one pass into the next (step 1 -> 2: whole slots, computed first in
step 2; step 2 -> 3: student halves, computed first in step 3, whose other
steps go into the teacher halves) are read from the slots where the earlier
pass left them.

This test restates that schedule on the CPU, independently of the kernel's
code, and checks, for every row length, carry count and pass structure:
each read finds the data it expects in the slot half it reads, that data's
fill was waited on before the read, and no later fill of that half can
start before the read (every such fill is ordered after it by the barriers
above).  A schedule change in the kernel that breaks one of these would be
a race there; the GPU tests check the results.
"""
import itertools

import pytest

KST = 3  # ring slots


def schedule(n, c1_max, c3_max, grad, lse_in, use_bits, rows):
    """Producer fills and consumer events of `rows` rows of n steps."""
    c1 = c1_max if (not lse_in and n >= c1_max + KST) else 0
    c3 = min(c3_max, n - c1) if (grad and use_bits) else 0
    a3 = n - c1 - c3

    def staged3(q):
        return q < a3 or q >= n - c1

    teacher3 = grad and not use_bits
    roles = ([] if lse_in else [0]) + [1] + ([2] if grad else [])
    fills = []  # (slot, {half: (tensor, row, step)}, row)
    for r in range(rows):
        for role in roles:
            for q in range(n):
                if role == 1 and q >= n - c1:
                    continue
                if role == 2 and not staged3(q):
                    continue
                if role == 2 and c3 > 0:
                    content = {"T": ("S", r, q)}  # the student into the teacher half
                else:
                    content = {"S": ("S", r, q)}
                    if role < 2 or teacher3:
                        content["T"] = ("T", r, q)
                fills.append((len(fills) % KST, content, r))
    events = []  # ("wait", f) | ("read", slot, half, want, f) | ("release", f) | ("carry", row)
    nxt = 0
    for r in range(rows):
        for role in roles:
            if role == 0:
                for q in range(n):
                    f, nxt = nxt, nxt + 1
                    events += [("wait", f), ("read", f % KST, "S", ("S", r, q), f),
                               ("read", f % KST, "T", ("T", r, q), f)]
                    if q < n - c1:
                        events.append(("release", f))
            elif role == 1:
                for j in range(c1):  # step 1's last c1 fills, still in their slots
                    f = nxt - c1 + j
                    q = n - c1 + j
                    events += [("read", f % KST, "S", ("S", r, q), f),
                               ("read", f % KST, "T", ("T", r, q), f), ("release", f)]
                for q in range(n - c1):
                    f, nxt = nxt, nxt + 1
                    events += [("wait", f), ("read", f % KST, "S", ("S", r, q), f),
                               ("read", f % KST, "T", ("T", r, q), f), ("release", f)]
            elif c3 > 0:
                for j in range(c3):  # step 2's last c3 fills' student halves
                    f = nxt - c3 + j
                    events.append(("read", f % KST, "S", ("S", r, a3 + j), f))
                events.append(("carry", r))
                for q in range(n):
                    if staged3(q):
                        f, nxt = nxt, nxt + 1
                        events += [("wait", f), ("read", f % KST, "T", ("S", r, q), f),
                                   ("release", f)]
            else:
                for q in range(n):
                    f, nxt = nxt, nxt + 1
                    events += [("wait", f), ("read", f % KST, "S", ("S", r, q), f)]
                    if teacher3:
                        events.append(("read", f % KST, "T", ("T", r, q), f))
                    events.append(("release", f))
    assert nxt == len(fills)
    return fills, events, c3


def check(fills, events, c3, carry_wait=True):
    pos = {}
    for i, e in enumerate(events):
        if e[0] in ("wait", "release", "carry"):
            pos[(e[0], e[1])] = i
    # the consumer event that fill f is ordered after (the producer's waits
    # are in program order, so the gate only grows)
    gate, g, prev_row, row_index = [], -1, None, 0
    for f, (_, _, row) in enumerate(fills):
        if row != prev_row:
            if carry_wait and c3 and row_index > 0:
                g = max(g, pos[("carry", prev_row)])
            prev_row, row_index = row, row_index + 1
        if f >= KST:
            g = max(g, pos[("release", f - KST)])
        gate.append(g)
    for i, e in enumerate(events):
        if e[0] != "read":
            continue
        _, slot, half, want, f0 = e
        assert fills[f0][0] == slot and fills[f0][1].get(half) == want, e
        assert pos[("wait", f0)] < i, ("read before its fill was waited on", e)
        for f in range(f0 + 1, len(fills)):
            if fills[f][0] == slot and half in fills[f][1]:
                assert gate[f] > i, ("overwritten before the read", e, f)


@pytest.mark.parametrize("grad,lse_in", [(False, False), (True, False), (True, True)])
def test_ring_schedule_has_no_race(grad, lse_in):
    for n, c1, c3, use_bits in itertools.product(range(1, 14), range(0, KST), range(0, KST + 1),
                                                 (False, True)):
        check(*schedule(n, c1, c3, grad, lse_in, use_bits, rows=3))


def test_model_catches_a_missing_carry_wait():
    # Without the row-start wait on carry_bar, a short row's next fill can
    # overwrite a carried student half before step 3 reads it.
    fills, events, c3 = schedule(2, 0, 3, True, False, True, rows=3)
    check(fills, events, c3)
    with pytest.raises(AssertionError, match="overwritten"):
        check(fills, events, c3, carry_wait=False)
