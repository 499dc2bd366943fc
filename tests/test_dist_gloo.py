"""World-size-2 gloo tests of the multi-process path (CPU only).

* the benchmark's timing rule: the slowest rank sets the step time and the
  whole-job throughput counts every rank's bytes;
* data-parallel semantics: token shards processed independently, dq and
  dw_o summed across ranks, equal the single-process result (checked with
  the FP64 oracle, which needs no GPU).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from attention_residuals_gb300.dist import (allreduce_param_grads_, max_over_ranks, shard_tokens,
                                            weak_scaling_throughput)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _timing_worker(rank, world, port, out):
    _init(rank, world, port)
    try:
        ms = [1.5 + rank, 0.5 * (rank + 1)]      # per-rank step and kernel times
        mx = max_over_ranks(ms)
        if rank == 0:
            out.put((mx, weak_scaling_throughput(1e9, world, mx[0])))
    finally:
        dist.destroy_process_group()


def _dp_worker(rank, world, port, out):
    _init(rank, world, port)
    try:
        from attention_residuals_gb300.workloads import make_random
        from oracle import attnres_oracle
        wl = make_random(5, 37, 64, 32, key_offset=8, out_norm=True, seed=3)
        a, b = shard_tokens(wl.N, rank, world)
        part = attnres_oracle(wl.values[:, a:b], wl.q, w_o=wl.w_o, dy=wl.dy[a:b], key_offset=8,
                              nthreads=1)
        dq = torch.tensor(part["dq"])
        dw = torch.tensor(part["dw_o"])
        dq16 = dq.to(torch.bfloat16)
        allreduce_param_grads_([dq, dw, dq16, None])
        if rank == 0:
            out.put((dq.numpy(), dw.numpy(), dq16.float().numpy()))
    finally:
        dist.destroy_process_group()


def _run(worker):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = q.get(timeout=120)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return res


def test_shard_tokens_partition():
    for n in (0, 1, 5, 37, 32768):
        for w in (1, 2, 3, 8):
            ranges = [shard_tokens(n, r, w) for r in range(w)]
            assert ranges[0][0] == 0 and ranges[-1][1] == n
            for (a0, b0), (a1, b1) in zip(ranges, ranges[1:]):
                assert b0 == a1
            sizes = [b - a for a, b in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_tokens(4, 2, 2)


def test_max_over_ranks_and_throughput_gloo():
    (mx, gbs) = _run(_timing_worker)
    assert mx == [2.5, 1.0]
    assert gbs == pytest.approx(2 * 1e9 / 2.5e-3 / 1e9)


def test_data_parallel_grads_equal_single_process_gloo():
    dq, dw, dq16 = _run(_dp_worker)
    from attention_residuals_gb300.workloads import make_random
    from oracle import attnres_oracle
    wl = make_random(5, 37, 64, 32, key_offset=8, out_norm=True, seed=3)
    full = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=8, nthreads=1)
    np.testing.assert_allclose(dq, full["dq"], rtol=1e-5, atol=1e-6)   # sum of FP32 partials
    np.testing.assert_allclose(dw, full["dw_o"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(dq16, full["dq"], rtol=1e-2, atol=1e-2)


class _OracleShard:
    """The benchmark's workload interface (fwd, bwd, grads) with the FP64
    oracle standing in for the kernels, on this rank's token shard."""

    def __init__(self, rank, world):
        from attention_residuals_gb300.workloads import make_random
        self.wl = make_random(4, 29, 64, 32, key_offset=16, out_norm=True, seed=9)
        self.a, self.b = shard_tokens(self.wl.N, rank, world)

    def fwd(self, stream):
        return None

    def bwd(self, stream):
        from oracle import attnres_oracle
        wl, a, b = self.wl, self.a, self.b
        r = attnres_oracle(wl.values[:, a:b], wl.q, w_o=wl.w_o, dy=wl.dy[a:b], key_offset=16, nthreads=1)
        return {"dq_f32": torch.tensor(r["dq"], dtype=torch.float32),
                "dw_o_f32": torch.tensor(r["dw_o"], dtype=torch.float32)}

    def grads(self, res):
        return [res["dq_f32"], res["dw_o_f32"]]


def _bench_step_worker(rank, world, port, out):
    _init(rank, world, port)
    try:
        import bench
        work = _OracleShard(rank, world)
        res = bench.run_step(work, None, bench.make_exchange(dist, work))
        if rank == 0:
            out.put((res["dq_f32"].numpy(), res["dw_o_f32"].numpy()))
    finally:
        dist.destroy_process_group()


def test_bench_step_exchange_gloo():
    # The benchmark's data-parallel step (forward, backward, the all-reduce of
    # the FP32 reduced gradients) on two ranks with token shards equals the
    # single-process gradients.
    dq, dw = _run(_bench_step_worker)
    from attention_residuals_gb300.workloads import make_random
    from oracle import attnres_oracle
    wl = make_random(4, 29, 64, 32, key_offset=16, out_norm=True, seed=9)
    full = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=16, nthreads=1)
    np.testing.assert_allclose(dq, full["dq"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(dw, full["dw_o"], rtol=1e-5, atol=1e-6)
