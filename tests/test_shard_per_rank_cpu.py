"""The multi-GPU decomposition the single-GPU path stands in for, checked on CPU ranks.

On one GB300 all tp_degree shards run as separate buffers and the pages' All-Reduce is an
on-device sum. Spread over devices, shard i lives on rank i * world // n: X and dZ are
replicated, A_i, a_i, B_i and the saved H_i, Y_i stay local, and exactly one exchange per
direction is needed -- an All-Reduce (SUM) of the row layer's partial output Z (the bias b added
once, after it) and one of the column layer's partial input gradient dX ("Tensor Parallelism:
principle and practice", section 3.1: row-parallel forward summed by All-Reduce, column-parallel
input gradient summed over devices; "PaddlePaddle tensor parallelism: from principle to
industrial deployment": the input gradient of a column-split layer is summed over devices).

Here world_size 2 gloo ranks each hold half of the shards, compute their shards' part with the
oracle's per-shard definitions, and exchange with torch.distributed.all_reduce. Every rank's
Z and dX, and the local weight and bias gradients, must equal the single-process oracle MLP;
sums over ranks change only the fp64 summation order. No GPU is involved.
"""
import os
import socket

import numpy as np
import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


T, H, F, N_SHARDS = 24, 16, 64, 4


def _inputs():
    import workloads as wl

    w = wl.MLP_T4096_H1024_F4096_TP2.with_shape(tokens=T, hidden=H, ffn=F, tp_degree=N_SHARDS)
    return wl.mlp_tensors(w)


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist

    import oracle

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = {k: np.asarray(v, dtype=np.float64) for k, v in _inputs().items()}
    A_s = oracle.split_columns(t["A"], N_SHARDS)
    a_s = oracle.split_vector(t["a"], N_SHARDS)
    B_s = oracle.split_rows(t["B"], N_SHARDS)
    mine = [i for i in range(N_SHARDS) if i * world // N_SHARDS == rank]

    def all_reduce(x):
        v = torch.from_numpy(np.ascontiguousarray(x))
        dist.all_reduce(v, op=dist.ReduceOp.SUM)
        return v.numpy()

    # forward: local column shards, local row partial, one All-Reduce, bias once
    H_, Y_ = oracle.column_parallel_forward(t["X"], [A_s[i] for i in mine],
                                            [a_s[i] for i in mine], "gelu")
    Z = all_reduce(oracle.row_parallel_forward(Y_, [B_s[i] for i in mine], None)) + t["b"]
    # backward: local row-layer gradients, local column-layer gradients, one All-Reduce of dX
    dY, dB, db = oracle.row_parallel_backward(Y_, [B_s[i] for i in mine], t["dZ"])
    dXp, dA, da, _ = oracle.column_parallel_backward(t["X"], [A_s[i] for i in mine], H_, dY,
                                                     "gelu")
    dX = all_reduce(dXp)
    out[rank] = {"mine": mine, "Z": Z, "dX": dX, "dA": dA, "da": da, "dB": dB, "db": db}
    dist.destroy_process_group()


def test_shards_over_two_ranks_compose_to_the_unsharded_mlp():
    mp = pytest.importorskip("torch.multiprocessing")
    import oracle

    ctx = mp.get_context("spawn")
    world, port = 2, _free_port()
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)

    t = {k: np.asarray(v, dtype=np.float64) for k, v in _inputs().items()}
    fwd = oracle.mlp_forward(t["X"], t["A"], t["a"], t["B"], t["b"], N_SHARDS)
    bwd = oracle.mlp_backward(t["X"], t["A"], t["a"], t["B"], t["b"], t["dZ"], N_SHARDS, fwd)
    seen = []
    for r in range(world):
        got = res[r]
        # both ranks hold the whole Z and dX after their All-Reduce
        np.testing.assert_allclose(got["Z"], fwd["Z"], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(got["dX"], bwd["dX"], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(got["db"], bwd["db"], rtol=1e-12, atol=1e-12)
        for j, i in enumerate(got["mine"]):
            np.testing.assert_allclose(got["dA"][j], bwd["dA"][i], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(got["da"][j], bwd["da"][i], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(got["dB"][j], bwd["dB"][i], rtol=1e-12, atol=1e-12)
            seen.append(i)
    assert sorted(seen) == list(range(N_SHARDS))   # every shard lives on exactly one rank


def test_an_unreduced_rank_is_not_the_layer():
    """The exchange is needed: one rank's partial Z (its shards only) is not the layer's Z."""
    import oracle

    t = {k: np.asarray(v, dtype=np.float64) for k, v in _inputs().items()}
    A_s = oracle.split_columns(t["A"], N_SHARDS)
    B_s = oracle.split_rows(t["B"], N_SHARDS)
    _, Y_ = oracle.column_parallel_forward(t["X"], A_s[:2], oracle.split_vector(t["a"], N_SHARDS)[:2],
                                           "gelu")
    partial = oracle.row_parallel_forward(Y_, B_s[:2], t["b"])
    full = oracle.mlp_forward(t["X"], t["A"], t["a"], t["B"], t["b"], N_SHARDS)["Z"]
    assert np.max(np.abs(partial - full)) > 1e-3 * np.max(np.abs(full))
