"""The layer objects over the C ABI: argument checks on the host, and GPU parity against the
oracle on small shapes (including the pages' column-parallel example)."""
import json
import os

import numpy as np
import pytest

import oracle
from harness import TOL_BF16, TOL_F32, np64, rel, rel_shards

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def mods():
    import __graft_entry__

    __graft_entry__.build()
    from tensor_sharded_linear_bias_gb300 import modules

    return modules


def test_shapes_are_checked_by_the_library(mods):
    from tensor_sharded_linear_bias_gb300 import TpError

    with pytest.raises(TpError) as e:
        mods.ColumnParallelLinear(768, 3070, 4, device="cpu")
    assert e.value.name == "TP_ERR_INDIVISIBLE"
    with pytest.raises(TpError):
        mods.RowParallelLinear(770, 768, 4, device="cpu")
    with pytest.raises(TpError):
        mods.TensorParallelMLP(128, 500, 8, device="cpu")


def test_column_weights_are_split_like_the_pages_example(mods):
    import torch

    g = json.load(open(os.path.join(GOLDEN, "csdn_column_example.json")))
    W = torch.randn(g["in_features"], g["out_features"]) * g["weight_init_scale"]
    layer = mods.ColumnParallelLinear(g["in_features"], g["out_features"], g["world_size"],
                                      dtype=torch.float32, device="cpu", weight=W)
    assert [tuple(w.shape) for w in layer.weights] == \
        [(g["in_features"], g["local_out_features"])] * g["world_size"]
    assert torch.equal(torch.cat(layer.weights, 1), W)
    assert all(torch.count_nonzero(b) == 0 for b in layer.biases)


@pytest.mark.gpu
def test_pages_example_through_the_column_layer(mods):
    import torch

    g = json.load(open(os.path.join(GOLDEN, "csdn_column_example.json")))
    gen = torch.Generator().manual_seed(3)
    W = torch.randn(g["in_features"], g["out_features"], generator=gen) * g["weight_init_scale"]
    x = torch.randn(g["batch"], g["in_features"], generator=gen)
    layer = mods.ColumnParallelLinear(g["in_features"], g["out_features"], g["world_size"],
                                      dtype=torch.float32, weight=W)
    y = layer.forward(x.cuda())
    layer.check()
    assert list(y.shape) == g["gathered_output_shape"]
    ref = oracle.concat_columns(oracle.column_parallel_forward(
        x.numpy(), oracle.split_columns(W.numpy(), g["world_size"]), None, "none")[1])
    assert rel(np64(y), ref) <= TOL_F32


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_mlp_and_linears_against_the_oracle(mods, dtype):
    import torch

    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    tol = TOL_BF16 if dtype == "bf16" else TOL_F32
    T, H, F, n = 200, 136, 4 * 88, 4
    gen = torch.Generator().manual_seed(11)
    A = (torch.randn(H, F, generator=gen) * 0.05).to(dt)
    B = (torch.randn(F, H, generator=gen) * 0.05).to(dt)
    a = (torch.randn(F, generator=gen) * 0.1).to(dt)
    b = (torch.randn(H, generator=gen) * 0.1).to(dt)
    x = torch.randn(T, H, generator=gen).to(dt)
    dz = torch.randn(T, H, generator=gen).to(dt)
    f = {k: v.float().numpy() for k, v in dict(A=A, B=B, a=a, b=b, x=x, dz=dz).items()}

    mlp = mods.TensorParallelMLP(H, F, n, dtype=dt, A=A, a=a, B=B, b=b)
    z = mlp.forward(x.cuda())
    dx = mlp.backward(dz.cuda())
    mlp.check()
    rf = oracle.mlp_forward(f["x"], f["A"], f["a"], f["B"], f["b"], n)
    rb = oracle.mlp_backward(f["x"], f["A"], f["a"], f["B"], f["b"], f["dz"], n, rf)
    assert rel(np64(z), rf["Z"]) <= tol
    assert rel(np64(dx), rb["dX"]) <= tol
    assert rel_shards([np64(t) for t in mlp.dA], rb["dA"]) <= tol
    assert rel_shards([np64(t) for t in mlp.dB], rb["dB"]) <= tol
    assert rel_shards([np64(t) for t in mlp.da], rb["da"]) <= tol
    assert rel(np64(mlp.db), rb["db"]) <= tol

    # the same MLP built from the two linears
    col = mods.ColumnParallelLinear(H, F, n, dtype=dt, weight=A, act="gelu", gather=False)
    col.biases = [t.cuda().contiguous() for t in a.split(F // n)]
    row = mods.RowParallelLinear(F, H, n, dtype=dt, weight=B)
    row.bias = b.cuda()
    z2 = row.forward(col.forward(x.cuda()))
    assert rel(np64(z2), rf["Z"]) <= tol
    dys = row.backward(dz.cuda())
    assert rel_shards([np64(t) for t in row.weight_grads], rb["dB"]) <= tol
    dx2 = col.backward([t.to(dt) for t in dys])
    col.check()
    # the row layer hands fp32 dY_i to the column layer, rounded to the input dtype here
    assert rel(np64(dx2), rb["dX"]) <= tol


@pytest.mark.gpu
def test_layernorm_module(mods):
    import torch

    T, H, n = 64, 8 * 128, 8
    gen = torch.Generator().manual_seed(5)
    x = torch.randn(T, H, generator=gen)
    dy = torch.randn(T, H, generator=gen)
    ln = mods.TensorParallelLayerNorm(H, n, dtype=torch.float32)
    ln.gamma = [g + 0.1 * i for i, g in enumerate(ln.gamma)]
    xs = [c.contiguous().cuda() for c in x.split(H // n, 1)]
    ys = ln.forward(xs)
    dxs = ln.backward([c.contiguous().cuda() for c in dy.split(H // n, 1)])
    torch.cuda.synchronize()
    gs = [np64(g) for g in ln.gamma]
    f = oracle.layernorm_forward(oracle.split_hidden(x.numpy(), n), gs, None, 1e-5)
    b = oracle.layernorm_backward(oracle.split_hidden(x.numpy(), n), gs,
                                  oracle.split_hidden(dy.numpy(), n), 1e-5, f)
    assert rel_shards([np64(y) for y in ys], f["Y"]) <= TOL_F32
    assert rel_shards([np64(d) for d in dxs], b["dX"]) <= TOL_F32
    assert rel_shards([np64(g) for g in ln.gamma_grads], b["dgamma"]) <= TOL_F32
    assert rel_shards([np64(g) for g in ln.beta_grads], b["dbeta"]) <= TOL_F32
