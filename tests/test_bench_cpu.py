"""Host-side pieces of bench.py (CPU only): the multi-rank timing reduction
under torch.distributed with the gloo backend at world size 2, the reference
arm's rank-0-only rule, the launch count of the attention paths, and the
page-1 explicit mask the bench builds, checked against the oracle's mask."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle as O
from synth import WORKLOADS


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports [1 + r, 10 - r, 3]; the job's times are the per-entry maxima
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.0], world, torch.device("cpu"))
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_size_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 10.0, 3.0]


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks([1.5, 2.5], 1, torch.device("cpu")) == [1.5, 2.5]


def test_reference_arm_runs_on_rank_0_only():
    class A:
        steps, warmup = 1, 0
    assert bench.reference(A(), rank=1, world=2) is None


def test_attention_launch_counts():
    # tensor-core pair path: prep, attention, merge; decode: attention (+ combine with a workspace)
    assert bench.attn_launches(WORKLOADS["long_ctx"], 1) == 3
    assert bench.attn_launches(WORKLOADS["decode"], 1) == 2
    assert bench.attn_launches(WORKLOADS["decode"], 0) == 1


@pytest.mark.parametrize("W", [512, 0])
def test_page1_mask_equals_oracle_mask(W):
    w = WORKLOADS["page1"]
    L, n = int(w.past_lens()[0]), int(w.n_reals()[0])
    m = bench.additive_mask(L, n, w.C, w.P, w.Hq, W)
    assert m.shape == (1, w.Hq, w.C, w.P + w.C) and m.dtype == torch.float32
    ref = O.explicit_mask(L, n, w.C, w.P, W, 1).astype(np.float32)
    for h in range(w.Hq):
        assert np.array_equal(m[0, h].numpy(), ref)
