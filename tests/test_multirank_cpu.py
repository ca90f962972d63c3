"""Two-rank (gloo, CPU) checks of the multi-GPU path.

Every chain is independent per row (the Linear chains: GroupNorm and
logsumexp act within a row) or per sample (LayerNorm and the ConvTranspose3d
GroupNorm act within a sample), so N GPUs run replicas with no data
exchange; the only collective is the max of the timings over the ranks.
These tests run two gloo ranks on the CPU: one checks bench.py's reduction
and aggregate, the other that each chain's oracle computed on row / sample
shards by different ranks and gathered equals the oracle on the whole input
(the property that lets the shards run without an exchange).
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


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _timing_worker(rank, world, port, q):
    import bench
    _init(rank, world, port)
    try:
        got = bench.reduce_over_ranks([1.0 + rank, 10.0 - 3 * rank])
        val = bench.job_value(2.0e12, world, got[0], 1e12)
        q.put((rank, got, val))
    finally:
        dist.destroy_process_group()


def test_timing_is_the_max_over_ranks_and_value_counts_all_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    mp.start_processes(_timing_worker, args=(2, port, q), nprocs=2, join=True, start_method="spawn")
    res = sorted(q.get(timeout=60) for _ in range(2))
    for rank, got, val in res:
        assert got == [2.0, 10.0], (rank, got)
        # 2 ranks x 2 TFLOP each in the slowest rank's 2 ms = 2000 units/s
        assert val == pytest.approx(2 * 2.0e12 / 2e-3 / 1e12)


def _shard_worker(rank, world, port, q):
    from conv_activation_normalization_gb300 import synth
    import oracle

    def normal(shape, seed):  # seeded float32 N(0, 1) from the shared input generator
        return synth._normal(synth._rng(seed), shape)

    _init(rank, world, port)
    try:
        out = {}
        # Linear -> Swish -> bias -> GroupNorm: rows
        x, W = normal((6, 16), 1), normal((128, 16), 2) * 0.2
        bl, bias = normal((128,), 3), normal((128,), 4)
        g, b = 1 + 0.1 * normal((128,), 5), 0.1 * normal((128,), 6)
        rows = np.array_split(np.arange(6), world)[rank]
        out["gn"] = oracle.linear_swish_bias_groupnorm(x[rows], W, bl, bias, g, b, 2, 1e-5)
        # Linear -> logsumexp -> LeakyReLU x2 -> GELU x2: rows
        out["lse"] = oracle.linear_lse_act(x[rows], W, bl, 0.01)
        # LayerNorm -> GELU -> Conv1d -> +x: samples
        xs = normal((4, 4, 16), 7)
        cw, cb = normal((4, 4, 3), 8) * 0.3, normal((4,), 9)
        lg, lb = 1 + 0.1 * normal((4, 16), 10), 0.1 * normal((4, 16), 11)
        samp = np.array_split(np.arange(4), world)[rank]
        out["conv"] = oracle.ln_gelu_dconv1d_res(xs[samp], lg, lb, cw, cb, 2, 2, 1e-5)
        # ConvTranspose3d -> Swish -> GroupNorm -> HardSwish: samples
        xt = normal((4, 2, 2, 3, 3), 12)
        wt, bt = normal((2, 16, 3, 3, 3), 13) * 0.2, normal((16,), 14) * 0.1
        gt, btt = 1 + 0.1 * normal((16,), 15), 0.1 * normal((16,), 16)
        out["convt"] = oracle.convt3d_swish_gn_hswish(xt[samp], wt, bt, gt, btt, 2, 1, 4, 1e-5)
        gathered = {}
        for k, v in out.items():
            parts = [None] * world
            dist.all_gather_object(parts, v)
            gathered[k] = np.concatenate(parts, axis=0)
        if rank == 0:
            full = {
                "gn": oracle.linear_swish_bias_groupnorm(x, W, bl, bias, g, b, 2, 1e-5),
                "lse": oracle.linear_lse_act(x, W, bl, 0.01),
                "conv": oracle.ln_gelu_dconv1d_res(xs, lg, lb, cw, cb, 2, 2, 1e-5),
                "convt": oracle.convt3d_swish_gn_hswish(xt, wt, bt, gt, btt, 2, 1, 4, 1e-5),
            }
            # equal up to the fp64 rounding of a BLAS that may block a
            # sub-matrix differently from the whole
            q.put({k: bool(np.allclose(gathered[k], full[k], rtol=1e-12, atol=1e-12)) for k in full})
    finally:
        dist.destroy_process_group()


def test_chains_shard_without_exchange():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    mp.start_processes(_shard_worker, args=(2, port, q), nprocs=2, join=True, start_method="spawn")
    res = q.get(timeout=120)
    assert res == {"gn": True, "lse": True, "conv": True, "convt": True}, res
