"""Seeded synthetic inputs for the fused CE + TVD distillation loss.

This module only draws random numbers and lays them out; it holds none of the
loss arithmetic, so both the CUDA path and the CPU oracle can consume its
output without sharing any of the method's code.  Random draws come from
``torch.Generator`` on the requested device (the CPU and CUDA streams differ,
so a test generates once and hands the same bytes to both sides).

Named workloads (the sizes the loss is tested and measured on):

================================  ======  =======  =====  ==================================
name                              BT      V        dtype  recipe
================================  ======  =======  =====  ==================================
``tiny_bt8_v32_f32``              8       32       f32    s~N(0,2^2); t=s+N(0,1); row 3 t==s;
                                                          row 5 ignored; grads 1
``bt1024_v32000_bf16``            1024    32000    bf16   s~N(0,1.5^2); t=s+N(0,0.5^2); 5%
                                                          ignored; grad_ce=1/BT, grad_tvd=.5/BT
``bt1024_v151936_bf16``           1024    151936   bf16   s,t~N(0,2^2) independent; +6 on t at
                                                          the target in 80% of rows; 5% ignored
``bt8192_v151936_bf16``           8192    151936   bf16   s~N(0,2^2); t=0.7s+N(0,1)+Zipf(1.1)
                                                          bias (max +8) over a vocab permutation;
                                                          targets sampled from softmax(t); 3%
                                                          ignored
``bt4096_v256000_f32``            4096    256000   f32    s,t~N(0,3^2) independent; 10% of rows
                                                          t==s; 5% ignored
================================  ======  =======  =====  ==================================

Teacher rows are derived from the fp32 student and then both are rounded to
bf16 (round to nearest even); "t == s" rows copy the rounded student bytes.
Targets drawn "from the teacher softmax" use the Gumbel-max trick
(argmax of logits plus Gumbel noise), which samples that distribution without
forming it.
"""
from __future__ import annotations

import dataclasses

import torch

IGNORE_INDEX = -100
_CHUNK_ROWS = 512  # rows generated per batch for the large workloads


@dataclasses.dataclass
class Workload:
    name: str
    student: torch.Tensor   # (BT, V) logits, f32 or bf16
    teacher: torch.Tensor   # (BT, V) same dtype
    target: torch.Tensor    # (BT,) int64, IGNORE_INDEX marks ignored rows
    grad_ce: torch.Tensor   # (BT,) f32 upstream gradient of each row's ce
    grad_tvd: torch.Tensor  # (BT,) f32 upstream gradient of each row's tvd
    ignore_index: int = IGNORE_INDEX

    @property
    def BT(self) -> int:
        return self.student.shape[0]

    @property
    def V(self) -> int:
        return self.student.shape[1]


WORKLOADS = {
    "tiny_bt8_v32_f32": dict(BT=8, V=32, dtype=torch.float32, seed=0),
    "bt1024_v32000_bf16": dict(BT=1024, V=32000, dtype=torch.bfloat16, seed=1),
    "bt1024_v151936_bf16": dict(BT=1024, V=151936, dtype=torch.bfloat16, seed=2),
    "bt8192_v151936_bf16": dict(BT=8192, V=151936, dtype=torch.bfloat16, seed=3),
    "bt4096_v256000_f32": dict(BT=4096, V=256000, dtype=torch.float32, seed=4),
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def _rand(shape, g, device):
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32)


def _ignore(target, frac, g, device):
    mask = _rand((target.shape[0],), g, device) < frac
    target[mask] = IGNORE_INDEX
    return target


def _tiny(BT, V, dtype, g, dev):
    s = _randn((BT, V), g, dev) * 2.0
    t = s + _randn((BT, V), g, dev)
    if BT > 3:
        t[3] = s[3]
    target = torch.randint(0, V, (BT,), generator=g, device=dev)
    if BT > 5:
        target[5] = IGNORE_INDEX
    ones = torch.ones(BT, device=dev, dtype=torch.float32)
    return s.to(dtype), t.to(dtype), target, ones, ones.clone()


def _near_teacher(BT, V, dtype, g, dev):
    s = torch.empty((BT, V), device=dev, dtype=dtype)
    t = torch.empty_like(s)
    for r0 in range(0, BT, _CHUNK_ROWS):
        r1 = min(BT, r0 + _CHUNK_ROWS)
        sf = _randn((r1 - r0, V), g, dev) * 1.5
        s[r0:r1] = sf.to(dtype)
        t[r0:r1] = (sf + _randn((r1 - r0, V), g, dev) * 0.5).to(dtype)
    target = _ignore(torch.randint(0, V, (BT,), generator=g, device=dev), 0.05, g, dev)
    gce = torch.full((BT,), 1.0 / BT, device=dev)
    return s, t, target, gce, torch.full((BT,), 0.5 / BT, device=dev)


def _peaked_teacher(BT, V, dtype, g, dev):
    s = torch.empty((BT, V), device=dev, dtype=dtype)
    t = torch.empty_like(s)
    target = torch.randint(0, V, (BT,), generator=g, device=dev)
    peaked = _rand((BT,), g, dev) < 0.8
    for r0 in range(0, BT, _CHUNK_ROWS):
        r1 = min(BT, r0 + _CHUNK_ROWS)
        s[r0:r1] = (_randn((r1 - r0, V), g, dev) * 2.0).to(dtype)
        tf = _randn((r1 - r0, V), g, dev) * 2.0
        rows = torch.arange(r0, r1, device=dev)
        bump = torch.where(peaked[r0:r1], 6.0, 0.0)
        tf[rows - r0, target[r0:r1]] += bump
        t[r0:r1] = tf.to(dtype)
    target = _ignore(target, 0.05, g, dev)
    gce = torch.full((BT,), 1.0 / BT, device=dev)
    return s, t, target, gce, gce.clone()


def _zipf_teacher(BT, V, dtype, g, dev):
    perm = torch.randperm(V, generator=g, device=dev)
    rank = torch.empty(V, device=dev, dtype=torch.float32)
    rank[perm] = torch.arange(1, V + 1, device=dev, dtype=torch.float32)
    bias = 8.0 * rank.pow(-1.1)
    s = torch.empty((BT, V), device=dev, dtype=dtype)
    t = torch.empty_like(s)
    target = torch.empty(BT, device=dev, dtype=torch.int64)
    for r0 in range(0, BT, _CHUNK_ROWS):
        r1 = min(BT, r0 + _CHUNK_ROWS)
        sf = _randn((r1 - r0, V), g, dev) * 2.0
        tq = (0.7 * sf + _randn((r1 - r0, V), g, dev) + bias).to(dtype)
        s[r0:r1] = sf.to(dtype)
        t[r0:r1] = tq
        u = _rand((r1 - r0, V), g, dev).clamp_(min=1e-30, max=1.0 - 1e-7)
        gumbel = -torch.log(-torch.log(u))
        target[r0:r1] = torch.argmax(tq.float() + gumbel, dim=1)
    target = _ignore(target, 0.03, g, dev)
    gce = torch.full((BT,), 1.0 / BT, device=dev)
    return s, t, target, gce, gce.clone()


def _independent_with_ties(BT, V, dtype, g, dev):
    s = torch.empty((BT, V), device=dev, dtype=dtype)
    t = torch.empty_like(s)
    tied = _rand((BT,), g, dev) < 0.10
    for r0 in range(0, BT, _CHUNK_ROWS):
        r1 = min(BT, r0 + _CHUNK_ROWS)
        s[r0:r1] = (_randn((r1 - r0, V), g, dev) * 3.0).to(dtype)
        t[r0:r1] = (_randn((r1 - r0, V), g, dev) * 3.0).to(dtype)
    t[tied] = s[tied]
    target = _ignore(torch.randint(0, V, (BT,), generator=g, device=dev), 0.05, g, dev)
    gce = torch.full((BT,), 1.0 / BT, device=dev)
    return s, t, target, gce, gce.clone()


_RECIPES = {
    "tiny_bt8_v32_f32": _tiny,
    "bt1024_v32000_bf16": _near_teacher,
    "bt1024_v151936_bf16": _peaked_teacher,
    "bt8192_v151936_bf16": _zipf_teacher,
    "bt4096_v256000_f32": _independent_with_ties,
}


def make(name: str, device="cpu", rows: int | None = None, V: int | None = None,
         dtype: torch.dtype | None = None, seed: int | None = None) -> Workload:
    """Generate a named workload on ``device``.

    ``rows``, ``V``, ``dtype`` and ``seed`` override the named sizes while
    keeping the recipe (value distributions, tie/ignore structure), which
    gives smaller cases of the same kind for parity tests and CPU samples.
    """
    cfg = dict(WORKLOADS[name])
    BT = cfg["BT"] if rows is None else int(rows)
    V = cfg["V"] if V is None else int(V)
    dtype = cfg["dtype"] if dtype is None else dtype
    seed = cfg["seed"] if seed is None else int(seed)
    dev = torch.device(device)
    with torch.no_grad():
        s, t, target, gce, gtvd = _RECIPES[name](BT, V, dtype, _gen(dev, seed), dev)
    return Workload(name, s.contiguous(), t.contiguous(), target.contiguous(),
                    gce.float().contiguous(), gtvd.float().contiguous())


LINEAR_WORKLOADS = {
    "linear_bt8192_d4096_v151936_bf16": dict(BT=8192, ds=4096, dt=4096, V=151936, seed=5),
}


@dataclasses.dataclass
class LinearWorkload:
    name: str
    h_student: torch.Tensor  # (BT, ds) bf16
    w_student: torch.Tensor  # (V, ds) bf16
    h_teacher: torch.Tensor  # (BT, dt) bf16
    w_teacher: torch.Tensor  # (V, dt) bf16
    target: torch.Tensor
    grad_ce: torch.Tensor
    grad_tvd: torch.Tensor
    ignore_index: int = IGNORE_INDEX


def make_linear(name: str, device="cpu", rows: int | None = None, V: int | None = None,
                d: int | None = None) -> LinearWorkload:
    """Hidden states ~ N(0, 1) and lm_head weights ~ N(0, (2/sqrt(d))^2), so the
    logits are ~ N(0, 2^2) like the logit workloads; targets uniform with 3%
    ignored; upstream gradients 1/BT.  ``rows``, ``V`` and ``d`` (both hidden
    sizes) override the named sizes, keeping the recipe."""
    cfg = dict(LINEAR_WORKLOADS[name])
    if V is not None:
        cfg["V"] = int(V)
    if d is not None:
        cfg["ds"] = cfg["dt"] = int(d)
    BT = cfg["BT"] if rows is None else int(rows)
    dev = torch.device(device)
    g = _gen(dev, cfg["seed"])
    with torch.no_grad():
        hs = _randn((BT, cfg["ds"]), g, dev).bfloat16()
        ws = (_randn((cfg["V"], cfg["ds"]), g, dev) * (2.0 / cfg["ds"] ** 0.5)).bfloat16()
        ht = _randn((BT, cfg["dt"]), g, dev).bfloat16()
        wt = (_randn((cfg["V"], cfg["dt"]), g, dev) * (2.0 / cfg["dt"] ** 0.5)).bfloat16()
        target = _ignore(torch.randint(0, cfg["V"], (BT,), generator=g, device=dev), 0.03, g, dev)
        gce = torch.full((BT,), 1.0 / BT, device=dev)
    return LinearWorkload(name, hs, ws, ht, wt, target, gce, gce.clone())
