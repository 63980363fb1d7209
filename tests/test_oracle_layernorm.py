"""Pins of the LayerNorm oracle (hidden dimension split over the shards) against facts fixed
outside the oracle itself:

* a pure-Python scalar brute force of LayerNorm on tiny shapes;
* invariances of the definition: adding a constant to a row, or (with eps = 0) scaling it,
  leaves the output unchanged; with gamma = 1, beta = 0, eps = 0 every output row has mean 0
  and variance 1;
* the shard count does not change the concatenated result;
* torch fp64 layer_norm and its autograd (a library routine of the same definition);
* central finite differences of L = <dY, Y>;
* planted mistakes (unbiased variance, eps outside the root, per-shard statistics without
  the All-Reduce, a dropped term of the input gradient), each caught by a pin.
"""
import math

import numpy as np
import pytest

from oracle import tp_layernorm as L


def rand(seed, *shape, scale=1.0, shift=0.0):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape) * scale + shift


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / (den if den > 0 else 1.0))


def cat(parts):
    return np.concatenate(parts, axis=-1)


def case(T, H, n, seed, shift=0.0):
    X = rand(seed, T, H, shift=shift)
    g = rand(seed + 1, H, scale=0.5, shift=1.0)
    b = rand(seed + 2, H, scale=0.5)
    dY = rand(seed + 3, T, H)
    return X, g, b, dY, L.split_hidden(X, n), L.split_hidden(g, n), L.split_hidden(b, n), \
        L.split_hidden(dY, n)


# ----------------------------------------------------------------------------- pins
def brute_force(X, g, b, eps):
    """Scalar loops: mean, biased variance, normalise, scale and shift."""
    T, H = len(X), len(X[0])
    out = []
    for t in range(T):
        row = [float(v) for v in X[t]]
        mu = 0.0
        for v in row:
            mu += v
        mu /= H
        var = 0.0
        for v in row:
            var += (v - mu) * (v - mu)
        var /= H
        r = 1.0 / math.sqrt(var + eps)
        out.append([(row[j] - mu) * r * float(g[j]) + float(b[j]) for j in range(H)])
    return np.array(out)


@pytest.mark.parametrize("T,H,n", [(3, 8, 1), (3, 8, 2), (4, 12, 4), (2, 6, 3)])
def test_forward_brute_force(T, H, n):
    X, g, b, _, Xs, gs, bs, _ = case(T, H, n, 10)
    out = L.layernorm_forward(Xs, gs, bs, eps=1e-3)
    assert rel(cat(out["Y"]), brute_force(X, g, b, 1e-3)) < 1e-13


def test_invariances():
    T, H, n = 5, 24, 4
    X, g, b, _, Xs, gs, bs, _ = case(T, H, n, 20)
    y = cat(L.layernorm_forward(Xs, gs, bs, eps=1e-5)["Y"])
    shifted = cat(L.layernorm_forward(L.split_hidden(X + 3.25, n), gs, bs, eps=1e-5)["Y"])
    assert rel(shifted, y) < 1e-12
    y0 = cat(L.layernorm_forward(Xs, None, None, eps=0.0)["Y"])
    scaled = cat(L.layernorm_forward(L.split_hidden(X * 7.5, n), None, None, eps=0.0)["Y"])
    assert rel(scaled, y0) < 1e-12
    assert np.max(np.abs(y0.mean(axis=1))) < 1e-13
    assert np.max(np.abs(y0.var(axis=1) - 1.0)) < 1e-12


def test_shard_count_independence():
    T, H = 6, 24
    ref = None
    for n in (1, 2, 3, 4, 6, 8, 12):
        X, g, b, dY, Xs, gs, bs, dYs = case(T, H, n, 30)
        f = L.layernorm_forward(Xs, gs, bs)
        bw = L.layernorm_backward(Xs, gs, dYs, fwd=f)
        got = np.concatenate([cat(f["Y"]).ravel(), cat(bw["dX"]).ravel(),
                              cat(bw["dgamma"]), cat(bw["dbeta"])])
        if ref is None:
            ref = got
        assert rel(got, ref) < 1e-13


def torch_ref(X, g, b, dY, eps):
    torch = pytest.importorskip("torch")
    Xt = torch.tensor(X, dtype=torch.float64, requires_grad=True)
    gt = torch.tensor(g, dtype=torch.float64, requires_grad=True)
    bt = torch.tensor(b, dtype=torch.float64, requires_grad=True)
    Y = torch.nn.functional.layer_norm(Xt, (X.shape[1],), gt, bt, eps)
    Y.backward(torch.tensor(dY, dtype=torch.float64))
    return Y.detach().numpy(), Xt.grad.numpy(), gt.grad.numpy(), bt.grad.numpy()


def errors_vs_torch(fwd, bwd, T=7, H=24, n=4, seed=40, shift=0.0, eps=1e-5):
    X, g, b, dY, Xs, gs, bs, dYs = case(T, H, n, seed, shift)
    Y, dX, dg, db = torch_ref(X, g, b, dY, eps)
    f = fwd(Xs, gs, bs, eps)
    r = bwd(Xs, gs, dYs, eps, f)
    return {"Y": rel(cat(f["Y"]), Y), "dX": rel(cat(r["dX"]), dX),
            "dgamma": rel(cat(r["dgamma"]), dg), "dbeta": rel(cat(r["dbeta"]), db)}


@pytest.mark.parametrize("shift", [0.0, 40.0])
def test_against_torch_autograd(shift):
    errs = errors_vs_torch(L.layernorm_forward, L.layernorm_backward, shift=shift)
    assert max(errs.values()) < 1e-12, errs


def test_backward_finite_differences():
    T, H, n, eps, h = 3, 8, 2, 1e-3, 1e-6
    X, g, b, dY, Xs, gs, bs, dYs = case(T, H, n, 50)

    def loss(Xv, gv, bv):
        y = cat(L.layernorm_forward(L.split_hidden(Xv, n), L.split_hidden(gv, n),
                                    L.split_hidden(bv, n), eps)["Y"])
        return float(np.sum(y * dY))

    r = L.layernorm_backward(Xs, gs, dYs, eps)
    for name, base, grad in (("X", X, cat(r["dX"])), ("gamma", g, cat(r["dgamma"])),
                             ("beta", b, cat(r["dbeta"]))):
        num = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            up, dn = base.copy(), base.copy()
            up[idx] += h
            dn[idx] -= h
            args = {"X": (X, g, b), "gamma": (X, g, b), "beta": (X, g, b)}[name]
            a_up = [up if k == name else v for k, v in zip(("X", "gamma", "beta"), args)]
            a_dn = [dn if k == name else v for k, v in zip(("X", "gamma", "beta"), args)]
            num[idx] = (loss(*a_up) - loss(*a_dn)) / (2 * h)
        assert rel(grad, num) < 1e-6, name


# ----------------------------------------------------------------------------- mutants
def _fwd_unbiased(Xs, gs, bs, eps):
    X = cat(Xs)
    mean = X.mean(axis=1)
    var = X.var(axis=1, ddof=1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (X - mean[:, None]) * rstd[:, None]
    Y = xhat * cat(gs) + cat(bs)
    return {"Y": L.split_hidden(Y, len(Xs)), "mean": mean, "rstd": rstd, "xhat": xhat}


def _fwd_eps_outside(Xs, gs, bs, eps):
    X = cat(Xs)
    mean = X.mean(axis=1)
    rstd = 1.0 / (np.sqrt(X.var(axis=1)) + eps)
    xhat = (X - mean[:, None]) * rstd[:, None]
    Y = xhat * cat(gs) + cat(bs)
    return {"Y": L.split_hidden(Y, len(Xs)), "mean": mean, "rstd": rstd, "xhat": xhat}


def _fwd_local_stats(Xs, gs, bs, eps):
    """Every shard normalises with its own statistics: the All-Reduce left out."""
    parts, xh = [], []
    for x, g, b in zip(Xs, gs, bs):
        m = x.mean(axis=1)
        r = 1.0 / np.sqrt(x.var(axis=1) + eps)
        h = (x - m[:, None]) * r[:, None]
        xh.append(h)
        parts.append(h * g + b)
    X = cat(Xs)
    return {"Y": parts, "mean": X.mean(axis=1), "rstd": 1.0 / np.sqrt(X.var(axis=1) + eps),
            "xhat": cat(xh)}


def _bwd_no_mean_term(Xs, gs, dYs, eps, fwd):
    xhat, rstd = fwd["xhat"], fwd["rstd"]
    g = cat(dYs) * cat(gs)
    dX = rstd[:, None] * (g - xhat * (g * xhat).mean(axis=1)[:, None])
    r = L.layernorm_backward(Xs, gs, dYs, eps, fwd)
    r["dX"] = L.split_hidden(dX, len(Xs))
    return r


def test_pins_catch_planted_mistakes():
    fwd, bwd = L.layernorm_forward, L.layernorm_backward
    mutants = {
        "unbiased variance": (_fwd_unbiased, bwd),
        "eps outside the root": (_fwd_eps_outside, bwd),
        "per-shard statistics (no All-Reduce)": (_fwd_local_stats, bwd),
        "input gradient without the mean term": (fwd, _bwd_no_mean_term),
    }
    for name, (f, b) in mutants.items():
        errs = errors_vs_torch(f, b, eps=1e-2)
        assert max(errs.values()) > 1e-6, (name, errs)
    assert max(errors_vs_torch(fwd, bwd, eps=1e-2).values()) < 1e-12


def test_divisibility_rule():
    with pytest.raises(ValueError):
        L.split_hidden(np.zeros((2, 10)), 4)


def test_oracle_has_no_cuda_dependency():
    src = open(L.__file__).read()
    assert "tensor_sharded_linear_bias_gb300" not in src
    assert "ctypes" not in src and "cuda" not in src.lower().replace("cuda library", "")
