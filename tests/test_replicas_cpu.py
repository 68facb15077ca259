"""Multi-process (gloo, world size 2, CPU) checks of the replica path.

The MoL path has no exchange step: pairs are independent, so a batch split by
tokens over replicas gives, row for row, the single-replica result, and the
bench combines ranks by the slowest time and the sum of pairs.
"""

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from synth import WORKLOADS, make_layer

        # rank combination used by the bench
        ms, pairs = bench.combine_ranks(1.0 + rank, 100.0 * (rank + 1))
        assert ms == float(world) and pairs == 100.0 * world * (world + 1) / 2

        # a token-sharded layer computed per rank and gathered
        wl = WORKLOADS["tiny"]
        li = make_layer(wl, seed=5)
        st = li.stages[0]
        x, A, B, out0 = st.x.host_all(), st.A.host_all(), st.B.host_all(), st.out0.host_all()
        t0, t1 = bench.shard_tokens(wl.T, world, rank)
        k = wl.topk
        res = oracle.lora_forward_stage(x[t0:t1], st.x_row_div, li.topk_ids[t0:t1], li.lora_ids[t0:t1],
                                        wl.E, wl.L, A, B, st.stage.S, st.stage.r, st.stage.Ns,
                                        wl.scale, None, out0[t0 * k:t1 * k], wl.BM)
        parts = [None] * world
        dist.all_gather_object(parts, res["out"])
        if rank == 0:
            full = oracle.lora_forward_stage(x, st.x_row_div, li.topk_ids, li.lora_ids, wl.E, wl.L,
                                             A, B, st.stage.S, st.stage.r, st.stage.Ns, wl.scale,
                                             None, out0, wl.BM)["out"]
            got = np.concatenate(parts)
            np.save(result_path, np.stack([got, full]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_gloo(tmp_path):
    world = 2
    path = str(tmp_path / "res.npy")
    mp.spawn(_worker, args=(world, _free_port(), path), nprocs=world, join=True)
    got, full = np.load(path)
    import oracle

    g, f = oracle.bf16_to_f64(got), oracle.bf16_to_f64(full)
    assert np.all(np.abs(g - f) <= 1e-2 * (1 + np.abs(f)))
    assert (got == full).mean() > 0.99


def test_shard_tokens_covers_batch():
    import bench

    for T in (0, 1, 5, 23, 4096):
        for world in (1, 2, 3, 8):
            ranges = [bench.shard_tokens(T, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == T
            for (a, b), (c, d) in zip(ranges, ranges[1:]):
                assert b == c and a <= b
            assert max(b - a for a, b in ranges) - min(b - a for a, b in ranges) <= 1
