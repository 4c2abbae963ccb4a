"""Multi-rank paths on CPU ranks (gloo, world_size 2).

1. Head sharding: each rank computes its own (b, h) heads; gathering the
   shards reproduces the whole job with no exchange during the computation.
2. Split keys: each rank attends over its key range only; one all_gather of
   the normalised partials (O_r, LSE_r) and the logsumexp merge reproduce the
   unsplit result.
The arithmetic on every rank is the fp64 oracle; what is under test is the
partitioning and the exchange step.
"""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from exact_attention_20_gb300.shard import heads_for_rank, keys_for_rank, split_range


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    rng = np.random.default_rng(2024)
    q, k, v = (rng.normal(size=(2, 3, 97, 16)) for _ in range(3))
    return q, k, v


def _worker(rank, world, port, out_dir):
    import oracle

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v = _inputs()
        B, H, N, d = q.shape
        # 1. head sharding
        mine = heads_for_rank(B, H, rank, world)
        o_loc = np.stack([oracle.attention(q[b, h], k[b, h], v[b, h], 0.25, True)[0] for b, h in mine])
        gathered = [None] * world
        dist.all_gather_object(gathered, (mine, o_loc))
        # 2. split keys, non-causal, for head (1, 2)
        k0, k1 = keys_for_rank(N, rank, world)
        o_r, l_r = oracle.attention_rows(q[1, 2], k[1, 2, k0:k1], v[1, 2, k0:k1], 0.25, False, np.arange(N))
        t_o = torch.from_numpy(o_r)
        t_l = torch.from_numpy(l_r)
        outs = [torch.empty_like(t_o) for _ in range(world)]
        lses = [torch.empty_like(t_l) for _ in range(world)]
        dist.all_gather(outs, t_o)
        dist.all_gather(lses, t_l)
        o_m, l_m = oracle.merge_partials([x.numpy() for x in outs], [x.numpy() for x in lses])
        if rank == 0:
            full = {}
            for heads, blocks in gathered:
                for (b, h), blk in zip(heads, blocks):
                    full[(b, h)] = blk
            np.savez(os.path.join(out_dir, "result.npz"),
                     heads=np.stack([full[(b, h)] for b in range(B) for h in range(H)]),
                     n_owned=np.array([len(hd) for hd, _ in gathered]),
                     o_merged=o_m, l_merged=l_m)
    finally:
        dist.destroy_process_group()


def test_split_range_partitions_exactly():
    for n in (0, 1, 7, 32, 97):
        for world in (1, 2, 3, 8):
            spans = [split_range(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        split_range(5, 2, 2)


def test_two_gloo_ranks_shard_heads_and_merge_split_keys():
    import oracle

    world = 2
    with tempfile.TemporaryDirectory() as tmp:
        mp.start_processes(_worker, args=(world, _free_port(), tmp), nprocs=world,
                           join=True, start_method="spawn")
        res = np.load(os.path.join(tmp, "result.npz"))
        q, k, v = _inputs()
        B, H, N, d = q.shape
        o_full, _ = oracle.attention(q, k, v, 0.25, True)
        np.testing.assert_array_equal(res["heads"], o_full.reshape(B * H, N, d))
        assert list(res["n_owned"]) == [3, 3]
        o_ref, l_ref = oracle.attention(q[1, 2], k[1, 2], v[1, 2], 0.25, False)
        np.testing.assert_allclose(res["o_merged"], o_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(res["l_merged"], l_ref, rtol=0, atol=1e-12)
