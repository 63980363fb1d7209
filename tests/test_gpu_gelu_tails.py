"""GPU parity of the GeLU and GeLU' epilogues over wide pre-activations, element by element.

The random workloads keep pre-activations within a few units of zero (|h| <~ 3), so the far
tails of the activation -- the negative tail where Phi(h) is tiny and GeLU(h) = h Phi(h) with
it, the minimum of GeLU' near h = -0.75, large positive h where GeLU(h) -> h -- are never
exercised by them. Here the pre-activations are placed exactly on a grid over [-12, 12] (and
over the tail alone, [-12, -3], so that the large values of the full range cannot hide a
relative error in the tail behind max|ref|):

  X is a selection matrix (X[t, t] = 1, else 0), so H_i = X A_i + a_i is A_i's row t plus the
  bias, exactly, in every precision. The column GEMM's bias + GeLU epilogue then produces
  Y_i = GeLU(H_i), and with X^T selecting rows again the column weight gradient is the
  activation gradient itself: dA_i[t, :] = dH_i[t, :] = dY_i[t, :] * GeLU'(H_i[t, :]) -- the
  dY GEMM's GeLU' epilogue in the MLP, the stand-alone activation-gradient kernel in the
  column linear's backward. Every output is compared with the fp64 oracle (exact-erf GeLU),
  bf16 at 2e-2 and fp32 at 1e-5 of max|ref| per tensor (per shard for sharded tensors).

"Tensor Parallelism: principle and practice", section 3.1 (the column linear's backward:
weight gradient X^T dL/dY_i); the GeLU of the MLP is the exact erf form.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from harness import TOL_BF16, TOL_F32, compare_full, np64, prepare, rel_shards

pytestmark = pytest.mark.gpu

RANGES = {"wide": (-12.0, 12.0), "tail": (-12.0, -3.0)}


@pytest.fixture(scope="module")
def tp():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import tensor_sharded_linear_bias_gb300 as mod

    return mod


def _bf16_values(x):
    """float32 array -> the nearest bf16 values (as float32), so that sums with them stay
    exact in fp32 and the fp32 path sees the same pre-activations as the bf16 one."""
    return wl.to_bf16(np.ascontiguousarray(x, dtype=np.float32))[1].astype(np.float32)


def _grid_inputs(seed, T, K, N, lo, hi):
    """X: the [T, K] selection matrix (T <= K); W: [K, N], rows < T hold a grid of step 1/16
    over [lo, hi] in a seeded shuffled order, the other rows small random weights; bias: [N],
    multiples of 1/16 in [-0.25, 0.25]. Every pre-activation W[t, j] + bias[j] is then a
    multiple of 1/16 of magnitude <= 12.25: exact in bf16, so the saved bf16 pre-activation
    that the GeLU' epilogue reads is the same number the oracle uses."""
    g = np.random.Generator(np.random.PCG64(seed))
    X = np.zeros((T, K), dtype=np.float32)
    X[np.arange(T), np.arange(T)] = 1.0
    grid = np.round(np.linspace(lo, hi, T * N, dtype=np.float64) * 16.0) / 16.0
    W = (g.standard_normal((K, N)) * 0.02).astype(np.float32)
    W[:T] = g.permutation(grid).reshape(T, N)
    bias = (g.integers(-4, 5, size=N) / 16.0).astype(np.float32)
    return _bf16_values(X), _bf16_values(W), _bf16_values(bias)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("span", ["wide", "tail"])
def test_mlp_gelu_epilogues_on_a_preactivation_grid(tp, dtype, span):
    """The MLP forward + backward: the column GEMM's GeLU epilogue (Y_i) and the dY GEMM's
    GeLU' epilogue (seen exactly through dA_i = X^T dH_i), plus every other output."""
    import torch

    lo, hi = RANGES[span]
    T, H, F, n = 300, 320, 2 * 296, 2
    Fs = F // n
    X, A, a = _grid_inputs(9100, T, H, F, lo, hi)
    g = np.random.Generator(np.random.PCG64(9101))
    raw = {"X": X, "A": A, "a": a,
           "B": (g.standard_normal((F, H)) * 0.05).astype(np.float32),
           "b": (g.standard_normal(H) * 0.01).astype(np.float32),
           "dZ": g.standard_normal((T, H)).astype(np.float32)}
    t, f = prepare(raw, dtype, "cuda")
    bf16 = dtype == "bf16"
    cdt = torch.bfloat16 if bf16 else torch.float32
    As = [t["A"][:, i * Fs:(i + 1) * Fs].contiguous() for i in range(n)]
    as_ = [t["a"][i * Fs:(i + 1) * Fs].contiguous() for i in range(n)]
    Bs = [t["B"][i * Fs:(i + 1) * Fs, :].contiguous() for i in range(n)]
    desc = tp.MlpDesc(tokens=T, hidden=H, ffn=F, tp_degree=n,
                      dtype=tp.TP_BF16 if bf16 else tp.TP_F32, act=tp.TP_ACT_GELU_ERF,
                      reduce=tp.TP_REDUCE_FUSED)
    ws = tp.new_workspace(tp.tp_mlp_workspace_size(desc))
    e = dict(dtype=torch.float32, device="cuda")
    Z = torch.full((T, H), float("nan"), **e)
    Hs = [torch.empty(T, Fs, dtype=cdt, device="cuda") for _ in range(n)]
    Ys = [torch.empty(T, Fs, dtype=cdt, device="cuda") for _ in range(n)]
    dX = torch.full((T, H), float("nan"), **e)
    dA = [torch.full((H, Fs), float("nan"), **e) for _ in range(n)]
    dB = [torch.full((Fs, H), float("nan"), **e) for _ in range(n)]
    da = [torch.full((Fs,), float("nan"), **e) for _ in range(n)]
    db = torch.full((H,), float("nan"), **e)
    tp.tp_mlp_forward(desc, t["X"], As, as_, Bs, t["b"], Z, Hs, Ys, ws)
    tp.tp_mlp_backward(desc, t["X"], As, Bs, Hs, Ys, t["dZ"], dX, dA, da, dB, db, ws)
    tp.tp_check_status(ws)
    torch.cuda.synchronize()

    rf = oracle.mlp_forward(f["X"], f["A"], f["a"], f["B"], f["b"], n)
    rb = oracle.mlp_backward(f["X"], f["A"], f["a"], f["B"], f["b"], f["dZ"], n, rf)
    # the pre-activations really span the range asked for
    h_all = oracle.concat_columns(rf["H"])[:T]
    assert h_all.min() <= lo + 0.3 and h_all.max() >= hi - 0.3
    out = {"Z": np64(Z), "H": [np64(x) for x in Hs], "Y": [np64(x) for x in Ys],
           "dX": np64(dX), "dA": [np64(x) for x in dA], "dB": [np64(x) for x in dB],
           "da": [np64(x) for x in da], "db": np64(db)}
    errs = compare_full(out, rf, rb)
    tol = TOL_BF16 if bf16 else TOL_F32
    assert max(errs.values()) <= tol, errs
    # dA_i's first T rows are dH_i = dY_i * GeLU'(H_i) element by element
    dH_ref = [rb["dA"][i][:T] for i in range(n)]
    assert rel_shards([x[:T] for x in out["dA"]], dH_ref) <= tol


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("span", ["wide", "tail"])
def test_column_linear_gelu_and_activation_gradient_on_a_grid(tp, dtype, span):
    """The column-parallel linear with GeLU: its forward epilogue, and its backward, whose
    activation gradient dH_i = dY_i * GeLU'(H_i) is the stand-alone kernel (seen exactly
    through dW_i = X^T dH_i)."""
    import torch

    lo, hi = RANGES[span]
    T, K, N, n = 200, 264, 4 * 72, 4
    Ns = N // n
    X, W, bias = _grid_inputs(9200, T, K, N, lo, hi)
    g = np.random.Generator(np.random.PCG64(9201))
    raw = {"X": X, "W": W, "bias": bias, "G": g.standard_normal((T, N)).astype(np.float32)}
    t, f = prepare(raw, dtype, "cuda")
    bf16 = dtype == "bf16"
    cdt = torch.bfloat16 if bf16 else torch.float32
    Ws = [t["W"][:, i * Ns:(i + 1) * Ns].contiguous() for i in range(n)]
    bs = [t["bias"][i * Ns:(i + 1) * Ns].contiguous() for i in range(n)]
    desc = tp.LinearDesc(tokens=T, in_features=K, out_features=N, tp_degree=n,
                         dtype=tp.TP_BF16 if bf16 else tp.TP_F32, act=tp.TP_ACT_GELU_ERF,
                         reduce=0, gather=0)
    ws = tp.new_workspace(tp.tp_linear_workspace_size(desc, tp.TP_COLUMN))
    Y = [torch.empty(T, Ns, dtype=cdt, device="cuda") for _ in range(n)]
    Hs = [torch.empty(T, Ns, dtype=cdt, device="cuda") for _ in range(n)]
    tp.tp_linear_column_forward(desc, t["X"], Ws, bs, Y, Hs, ws)
    dY = [t["G"][:, i * Ns:(i + 1) * Ns].contiguous() for i in range(n)]
    dX = torch.full((T, K), float("nan"), dtype=torch.float32, device="cuda")
    dW = [torch.full((K, Ns), float("nan"), dtype=torch.float32, device="cuda") for _ in range(n)]
    db = [torch.full((Ns,), float("nan"), dtype=torch.float32, device="cuda") for _ in range(n)]
    tp.tp_linear_column_backward(desc, t["X"], Ws, Hs, dY, dX, dW, db, ws)
    tp.tp_check_status(ws)
    torch.cuda.synchronize()

    Wr = oracle.split_columns(f["W"], n)
    Hr, Yr = oracle.column_parallel_forward(f["X"], Wr, oracle.split_vector(f["bias"], n),
                                            "gelu")
    dXr, dWr, dbr, dHr = oracle.column_parallel_backward(f["X"], Wr, Hr,
                                                         oracle.split_columns(f["G"], n),
                                                         "gelu")
    tol = TOL_BF16 if bf16 else TOL_F32
    errs = {"Y": rel_shards([np64(y) for y in Y], Yr),
            "H": rel_shards([np64(h) for h in Hs], Hr),
            "dH (dW rows < T)": rel_shards([np64(x)[:T] for x in dW], dHr),
            "dW": rel_shards([np64(x) for x in dW], dWr),
            "db": rel_shards([np64(x) for x in db], dbr)}
    from harness import rel

    errs["dX"] = rel(np64(dX), dXr)
    assert max(errs.values()) <= tol, errs
