"""The vocabulary-parallel step over gloo ranks on CPU.

Each rank holds one column shard of every row; ``vocab_parallel.step``
exchanges the per-row partials with an all-gather in rank order and merges
them.  The shard passes here are fp64 CPU stand-ins for the library's CUDA
passes (those are checked against the oracle on the GPU): this test checks
the exchange, the shard bounds and the target mapping, by comparing every
rank's per-row outputs and its gradient columns with the oracle on whole
rows."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from distillation_ce_tvd_gb300 import vocab_parallel, workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _lse(x):
    m = x.max()
    return m + np.log(np.exp(x - m).sum()) if np.isfinite(m) else m


class CpuShardOps:
    """fp64 CPU stand-ins with the signatures of the binding's shard calls."""

    @staticmethod
    def fused_ce_tvd_vp_lse(student, teacher, target, v_begin, ignore_index, stream=None):
        s, t, tg = student.double().numpy(), teacher.double().numpy(), target.numpy()
        part = np.zeros((s.shape[0], 3))
        for r in range(s.shape[0]):
            if tg[r] == ignore_index:
                continue
            rel = tg[r] - v_begin
            part[r] = (_lse(s[r]), _lse(t[r]), s[r, rel] if 0 <= rel < s.shape[1] else 0.0)
        return torch.from_numpy(part)

    @staticmethod
    def fused_ce_tvd_vp_merge_lse(parts, target, V, ignore_index, dev_status=None, stream=None):
        p, tg = parts.numpy(), target.numpy()
        BT = p.shape[1]
        ce, ls, lt = np.zeros(BT), np.zeros(BT), np.zeros(BT)
        for r in range(BT):
            if tg[r] == ignore_index:
                continue
            ls[r], lt[r] = _lse(p[:, r, 0]), _lse(p[:, r, 1])
            ce[r] = ls[r] - p[:, r, 2].sum() if 0 <= tg[r] < V else np.nan
        return tuple(torch.from_numpy(x) for x in (ce, ls, lt))

    @staticmethod
    def fused_ce_tvd_vp_tvd(student, teacher, target, lse_s, lse_t, ignore_index, stream=None):
        s, t, tg = student.double().numpy(), teacher.double().numpy(), target.numpy()
        part = np.zeros((s.shape[0], 2))
        for r in range(s.shape[0]):
            if tg[r] == ignore_index:
                continue
            p_, q_ = np.exp(s[r] - lse_s[r].item()), np.exp(t[r] - lse_t[r].item())
            sg = np.sign(p_ - q_)
            part[r] = ((p_ * sg).sum(), (q_ * sg).sum())
        return torch.from_numpy(part)

    @staticmethod
    def fused_ce_tvd_vp_merge_tvd(parts, target, ignore_index, stream=None):
        p, tg = parts.numpy(), target.numpy()
        sig = p[:, :, 0].sum(0)
        tvd = 0.5 * (p[:, :, 0] - p[:, :, 1]).sum(0)
        ign = tg == ignore_index
        sig[ign] = tvd[ign] = 0.0
        return torch.from_numpy(tvd), torch.from_numpy(sig)

    @staticmethod
    def fused_ce_tvd_vp_backward(student, teacher, target, v_begin, V, lse_s, lse_t, sigma,
                                 grad_ce, grad_tvd, ignore_index, dev_status=None, stream=None):
        s, t, tg = student.double().numpy(), teacher.double().numpy(), target.numpy()
        g = np.zeros_like(s)
        for r in range(s.shape[0]):
            if tg[r] == ignore_index:
                continue
            p_ = np.exp(s[r] - lse_s[r].item())
            q_ = np.exp(t[r] - lse_t[r].item())
            gce, gtvd = float(grad_ce[r]), float(grad_tvd[r])
            g[r] = gce * p_ + gtvd * 0.5 * p_ * (np.sign(p_ - q_) - sigma[r].item())
            rel = tg[r] - v_begin
            if 0 <= rel < s.shape[1]:
                g[r, rel] -= gce
        return torch.from_numpy(g)


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = workloads.make("bt1024_v32000_bf16", "cpu", rows=11, V=301, seed=6)
        w.target[3] = 300            # the last column (the last shard)
        w.target[4] = 0              # the first column
        b, e = vocab_parallel.shard_bounds(w.V, world, rank, w.student.element_size())
        out = vocab_parallel.step(w.student[:, b:e], w.teacher[:, b:e], w.target, b, w.V,
                                  w.grad_ce, w.grad_tvd, vocab_parallel.gather_across(),
                                  w.ignore_index, ops=CpuShardOps)
        torch.save({"rows": torch.stack([x.double() for x in out[:5]], 1), "grad": out[5],
                    "bounds": (b, e)}, os.path.join(out_dir, f"r{rank}.pt"))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_hold_vocabulary_shards(tmp_path, world):
    import oracle
    oracle.build()
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [torch.load(os.path.join(tmp_path, f"r{r}.pt")) for r in range(world)]
    w = workloads.make("bt1024_v32000_bf16", "cpu", rows=11, V=301, seed=6)
    w.target[3] = 300
    w.target[4] = 0
    f = oracle.fused_ce_tvd_forward(w.student, w.teacher, w.target, threads=1)
    g, _ = oracle.fused_ce_tvd_backward(w.student, w.teacher, w.target, w.grad_ce, w.grad_tvd,
                                        threads=1)
    ref = np.stack([f[k] for k in ("ce", "tvd", "student_lse", "teacher_lse", "sigma")], 1)
    for r in range(world):  # every rank merged the same per-row values
        assert torch.equal(got[r]["rows"], got[0]["rows"])
    np.testing.assert_allclose(got[0]["rows"].numpy(), ref, rtol=0, atol=1e-12)
    # the shards tile the vocabulary and their gradients tile the oracle's
    assert got[0]["bounds"][0] == 0 and got[-1]["bounds"][1] == w.V
    for a, b in zip(got, got[1:]):
        assert a["bounds"][1] == b["bounds"][0]
    full = np.concatenate([x["grad"].numpy() for x in got], axis=1)
    np.testing.assert_allclose(full, g, rtol=0, atol=1e-12)


def test_shard_bounds_tile_and_align():
    for V in (1, 7, 8, 9, 301, 32000, 151936, 256000):
        for n in (1, 2, 3, 4, 8):
            for e in (2, 4):
                b = [vocab_parallel.shard_bounds(V, n, k, e) for k in range(n)]
                assert b[0][0] == 0 and b[-1][1] == V
                assert all(x[1] == y[0] for x, y in zip(b, b[1:]))
                assert all(lo % (16 // e) == 0 for lo, hi in b if hi > lo)
    with pytest.raises(ValueError):
        vocab_parallel.shard_bounds(10, 2, 2)
