"""kv-head-group sharding of one tree on CPU: two gloo ranks, no GPU.

Each rank takes its kv heads and the q heads that read them, runs the fp64 oracle on its shard
alone (its own tensors, its own head count), and the shards are all-gathered over gloo.  The
concatenation must equal the unsharded oracle for O, LSE, dQ, dK, dV: the tree mask, positions
and loss weights depend on the tree only, and no quantity mixes kv-head groups, so the split
needs no exchange in the data path.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    from workloads import make_tensors, random_tree
    from workloads.trees import Workload
    parent, lens = random_tree(41, 9, max_len=20)
    wl = Workload(name="shard", parent=parent, node_len=lens, Hq=8, Hkv=4, d=16)
    return wl, make_tensors(wl)


def _rank_main(rank, world, port, out_q):
    sys.path.insert(0, ROOT)
    import oracle
    from tree_masked_attention_plan_gb300.shard import kv_head_shard
    torch.distributed.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                                         world_size=world)
    try:
        wl, t = _inputs()
        sh = kv_head_shard(wl.Hq, wl.Hkv, rank, world)
        mine = {"q": t["q"][:, sh.q0:sh.q1], "k": t["k"][:, sh.kv0:sh.kv1], "v": t["v"][:, sh.kv0:sh.kv1],
                "u": t["u"][:, sh.q0:sh.q1]}
        r = oracle.attention_paths(wl.parent, wl.node_len, mine["q"], mine["k"], mine["v"], mine["u"])
        out = {}
        for key in ("o", "dq", "dk", "dv", "lse"):
            x = torch.from_numpy(np.ascontiguousarray(r[key]))
            parts = [torch.empty_like(x) for _ in range(world)]
            torch.distributed.all_gather(parts, x)
            out[key] = torch.cat(parts, dim=0 if key == "lse" else 1).numpy()
        out_q.put((rank, (sh.q0, sh.q1, sh.kv0, sh.kv1), out if rank == 0 else None))
    finally:
        torch.distributed.destroy_process_group()


def test_two_rank_head_shards_reassemble_the_unsharded_oracle():
    sys.path.insert(0, ROOT)
    import oracle
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {rank: (rng, out) for rank, rng, out in (q.get(timeout=300) for _ in range(world))}
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == (0, 4, 0, 2) and res[1][0] == (4, 8, 2, 4)
    wl, t = _inputs()
    full = oracle.attention_paths(wl.parent, wl.node_len, t["q"], t["k"], t["v"], t["u"])
    got = res[0][1]
    for key in ("o", "lse", "dq", "dk", "dv"):
        assert np.abs(got[key] - full[key]).max() < 1e-12, key


def test_shard_ranges_and_rejections():
    sys.path.insert(0, ROOT)
    from tree_masked_attention_plan_gb300.shard import kv_head_shard
    shards = [kv_head_shard(32, 8, r, 4) for r in range(4)]
    assert [(s.q0, s.q1, s.kv0, s.kv1) for s in shards] == [(0, 8, 0, 2), (8, 16, 2, 4), (16, 24, 4, 6),
                                                           (24, 32, 6, 8)]
    # every q head lands on the rank holding its kv head, with the local mapping h // grp
    for s in shards:
        for h in range(s.q0, s.q1):
            assert s.kv0 <= h // 4 < s.kv1 and (h - s.q0) // 4 == h // 4 - s.kv0
    assert kv_head_shard(32, 8, 7, 8).Hq == 4
    with pytest.raises(ValueError):
        kv_head_shard(32, 8, 0, 3)            # 8 kv heads do not split over 3 ranks
    with pytest.raises(ValueError):
        kv_head_shard(30, 8, 0, 2)            # Hq not a multiple of Hkv
    with pytest.raises(ValueError):
        kv_head_shard(32, 8, 2, 2)
