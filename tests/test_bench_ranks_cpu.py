"""The benchmark's multi-rank host logic on CPU: two gloo ranks, no GPU.

Each rank takes its own block of head-states, the timed region's length is the
maximum over ranks, and the whole-job value counts every rank's head-tokens.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from quantized_linear_attention_gb300 import workload as wlm


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        wl = wlm.WORKLOADS[1]
        s0 = bench.shard_offset(wl, r)
        tk = wlm.tokens(wl, 0, 2, s0, wl.n_states, nthreads=1)
        bench.barrier(w)
        t = bench.max_over_ranks(10.0 + 5.0 * r, w)
        out[r] = (r, w, local, s0, t, float(tk.q.sum()), bench.job_value(wl.n_states, wl.W, 3, w, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_take_the_max():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(out)
    wl = wlm.WORKLOADS[1]
    assert sorted(res) == [0, 1]
    for r in range(world):
        rank, w, local, s0, t, qsum, value = res[r]
        assert (rank, w, local) == (r, world, r)
        assert s0 == r * wl.n_states
        assert t == 15.0  # the slower rank decides
        assert value == pytest.approx(world * wl.n_states * wl.W * 3 / 0.015)
    # the two ranks decoded different head-states
    assert res[0][5] != res[1][5]


def test_shards_are_disjoint_blocks_of_one_stream():
    wl = wlm.WORKLOADS[1]
    both = wlm.tokens(wl, 0, 2, 0, 2 * wl.n_states, nthreads=1)
    r1 = wlm.tokens(wl, 0, 2, bench.shard_offset(wl, 1), wl.n_states, nthreads=1)
    assert np.array_equal(both.q[:, wl.n_states:], r1.q)
    S_both, _ = wlm.initial_state(wlm.WORKLOADS[2], 0, 4, nthreads=1)
    S_r, _ = wlm.initial_state(wlm.WORKLOADS[2], 2, 2, nthreads=1)
    assert np.array_equal(S_both[2:], S_r)


def test_single_rank_is_the_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.shard_offset(wlm.WORKLOADS[4], 0) == 0
    assert bench.job_value(16384, 16, 400, 1, 1000.0) == 16384 * 16 * 400
