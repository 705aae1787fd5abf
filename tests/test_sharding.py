"""Row sharding over 2 gloo ranks on CPU: the sharded results gathered back
are bitwise the single-process results (rows are independent)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from distillation_ce_tvd_gb300 import sharding, workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = workloads.make("bt1024_v32000_bf16", "cpu", rows=13, V=300, seed=5)
        lo, hi = sharding.row_block(w.BT, rank, world)
        f = oracle.fused_ce_tvd_forward(w.student[lo:hi], w.teacher[lo:hi],
                                        w.target[lo:hi], threads=1)
        g, _ = oracle.fused_ce_tvd_backward(w.student[lo:hi], w.teacher[lo:hi], w.target[lo:hi],
                                            w.grad_ce[lo:hi], w.grad_tvd[lo:hi], threads=1)
        local = torch.from_numpy(np.stack([f[k] for k in ("ce", "tvd", "student_lse",
                                                          "teacher_lse", "sigma")], 1))
        full = sharding.gather_rows(local, w.BT, world)
        grad = sharding.gather_rows(torch.from_numpy(g), w.BT, world)
        mx = sharding.max_over_ranks(float(rank + 1) * 1.5, world)
        if rank == 0:
            torch.save({"rows": full, "grad": grad, "max": mx}, os.path.join(out_dir, "r0.pt"))
    finally:
        dist.destroy_process_group()


def test_row_block_partition():
    for BT in (0, 1, 7, 8192, 8193):
        for world in (1, 2, 3, 8):
            blocks = [sharding.row_block(BT, r, world) for r in range(world)]
            assert blocks[0][0] == 0 and blocks[-1][1] == BT
            assert all(a[1] == b[0] for a, b in zip(blocks, blocks[1:]))
            sizes = [hi - lo for lo, hi in blocks]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        sharding.row_block(4, 2, 2)


def test_two_gloo_ranks_match_single_process(tmp_path):
    import oracle
    oracle.build()
    mp.spawn(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    got = torch.load(os.path.join(tmp_path, "r0.pt"))
    w = workloads.make("bt1024_v32000_bf16", "cpu", rows=13, V=300, seed=5)
    f = oracle.fused_ce_tvd_forward(w.student, w.teacher, w.target, threads=1)
    g, _ = oracle.fused_ce_tvd_backward(w.student, w.teacher, w.target, w.grad_ce, w.grad_tvd,
                                        threads=1)
    ref = np.stack([f[k] for k in ("ce", "tvd", "student_lse", "teacher_lse", "sigma")], 1)
    assert np.array_equal(got["rows"].numpy(), ref)
    assert np.array_equal(got["grad"].numpy(), g)
    assert got["max"] == 3.0
