"""The N > 1 host path on CPU: two gloo ranks, each owning a shard of the
heads, compute their part (the float64 oracle stands in for the kernels) with
no data-path collective; gathering the shards reproduces the single-process
result, and the timing reduction returns the maximum over ranks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from attention_kl_divergence_gb300 import dist as kdist
from attention_kl_divergence_gb300 import make_qk


def test_head_range_partitions_exactly():
    for heads in (1, 2, 7, 32, 128):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                a, b = kdist.head_range(heads, r, world)
                seen.extend(range(a, b))
                assert b - a in (heads // world, heads // world + 1)
            assert seen == list(range(heads))
    with pytest.raises(ValueError):
        kdist.head_range(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    try:
        from oracle import oracle
        w, r, _ = kdist.env()
        kdist.init(w, "gloo")
        Q1, K1, Q2, K2 = make_qk(2, 3, 40, 40, 16, 0.5, seed=5)
        mine = [kdist.shard_heads(t, r, w) for t in (Q1, K1, Q2, K2)]
        KL, L1, L2 = oracle.fwd(*mine, causal=True)
        parts = [None] * w
        dist.all_gather_object(parts, (r, KL))
        kdist.barrier(w)
        mx = kdist.max_over_ranks(float(r) + 0.5, w)
        if r == 0:
            full, _, _ = oracle.fwd(Q1, K1, Q2, K2, causal=True)
            got = np.concatenate([p[1].reshape(-1, 40) for p in sorted(parts, key=lambda p: p[0])])
            q.put((np.array_equal(got, full.reshape(-1, 40)), mx))
        dist.destroy_process_group()
    except Exception as e:  # pragma: no cover - reported to the parent
        q.put((repr(e), None))


def test_two_gloo_ranks_shard_heads_without_collectives():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    ok, mx = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
    assert ok is True, ok
    assert mx == 1.5


def test_bench_shards_cover_every_head_of_the_problem_once():
    """bench.py under torchrun splits one problem's heads across the ranks
    (strong scaling): every query and key head is owned by exactly one rank,
    and a shard of the tensors is exactly those heads."""
    import bench
    from attention_kl_divergence_gb300 import WORKLOADS
    for name in ("64k_causal", "64k_causal_gqa", "decode_q1_k512k", "512k_causal"):
        w = WORKLOADS[name]
        hk = w.H_kv or w.H
        group = w.H // hk
        for world in (1, 2, 3, 4, 8):
            keys, queries = [], []
            for r in range(world):
                a, b = bench.rank_heads(w, r, world)
                keys.extend(range(a, b))
                queries.extend(range(a * group, b * group))
            assert keys == list(range(w.B * hk)), (name, world)
            assert queries == list(range(w.B * w.H)), (name, world)
    t = torch.arange(2 * 4 * 3 * 2).reshape(2, 4, 3, 2)
    s = bench.shard(t, 1, 3, group=2)  # key heads 1, 2 -> query heads 2..5 of the flat (b, h) order
    assert s.shape == (1, 4, 3, 2) and s.is_contiguous()
    assert torch.equal(s[0], t.reshape(8, 3, 2)[2:6])
