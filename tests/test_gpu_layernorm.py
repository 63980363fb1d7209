"""GPU parity of the hidden-split LayerNorm (tp_layernorm_forward / tp_layernorm_backward)
against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
from harness import TOL_BF16, TOL_F32, np64, rel, rel_shards

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import tensor_sharded_linear_bias_gb300 as mod

    return mod


def draws(seed, T, H, shift=0.0):
    g = np.random.Generator(np.random.PCG64(seed))
    X = g.standard_normal((T, H)).astype(np.float32) + np.float32(shift)
    gamma = (1.0 + 0.5 * g.standard_normal(H)).astype(np.float32)
    beta = (0.5 * g.standard_normal(H)).astype(np.float32)
    dY = g.standard_normal((T, H)).astype(np.float32)
    return X, gamma, beta, dY


class LnCase:
    def __init__(self, tp, T, H, n, dtype, seed=1, shift=0.0, affine=True, eps=1e-5):
        import torch

        self.tp, self.T, self.H, self.n, self.eps = tp, T, H, n, eps
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        X, g, b, dY = draws(seed, T, H, shift)
        Hs = H // n

        def dev(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to("cuda", tdt)

        def shards(a):
            return [dev(a[..., i * Hs:(i + 1) * Hs]) for i in range(n)]

        self.X, self.dY = shards(X), shards(dY)
        self.g = shards(g) if affine else None
        self.b = shards(b) if affine else None
        # the oracle sees exactly the values handed to the GPU
        host = lambda ts: [np64(t) for t in ts] if ts is not None else None  # noqa: E731
        self.hX, self.hdY, self.hg, self.hb = host(self.X), host(self.dY), host(self.g), host(self.b)
        f32 = dict(dtype=torch.float32, device="cuda")
        self.Y = [torch.full((T, Hs), float("nan"), dtype=tdt, device="cuda") for _ in range(n)]
        self.dX = [torch.full((T, Hs), float("nan"), dtype=tdt, device="cuda") for _ in range(n)]
        self.mean = torch.full((T,), float("nan"), **f32)
        self.rstd = torch.full((T,), float("nan"), **f32)
        self.dg = [torch.full((Hs,), float("nan"), **f32) for _ in range(n)]
        self.db = [torch.full((Hs,), float("nan"), **f32) for _ in range(n)]
        self.desc = tp.LayerNormDesc(tokens=T, hidden=H, tp_degree=n,
                                     dtype=tp.TP_BF16 if dtype == "bf16" else tp.TP_F32, eps=eps)

    def run(self):
        import torch

        tp = self.tp
        tp.tp_layernorm_forward(self.desc, self.X, self.g, self.b, self.Y, self.mean, self.rstd)
        tp.tp_layernorm_backward(self.desc, self.X, self.g, self.mean, self.rstd, self.dY,
                                 self.dX, self.dg, self.db)
        torch.cuda.synchronize()
        return self

    def errors(self):
        f = oracle.layernorm_forward(self.hX, self.hg, self.hb, self.eps)
        b = oracle.layernorm_backward(self.hX, self.hg, self.hdY, self.eps, f)
        return {"Y": rel_shards([np64(y) for y in self.Y], f["Y"]),
                "mean": rel(np64(self.mean), f["mean"]), "rstd": rel(np64(self.rstd), f["rstd"]),
                "dX": rel_shards([np64(x) for x in self.dX], b["dX"]),
                "dgamma": rel_shards([np64(x) for x in self.dg], b["dgamma"]),
                "dbeta": rel_shards([np64(x) for x in self.db], b["dbeta"])}


@pytest.mark.parametrize("dtype,T,H,n", [("bf16", 257, 8 * 72, 8), ("bf16", 96, 4 * 1024, 4),
                                         ("bf16", 33, 16, 1), ("f32", 130, 3 * 77, 3),
                                         ("f32", 64, 8 * 96, 8), ("bf16", 40, 16 * 2048, 16)])
def test_layernorm_matches_oracle(tp, dtype, T, H, n):
    """16-byte accesses for bf16 rows and fp32 rows that allow them (up to 16 shards), and
    the scalar path for fp32 rows that are not 16-byte multiples (77 columns per shard)."""
    errs = LnCase(tp, T, H, n, dtype).run().errors()
    assert max(errs.values()) <= (TOL_BF16 if dtype == "bf16" else TOL_F32), errs


def test_layernorm_shifted_rows_and_no_affine(tp):
    """Rows far from zero mean (the shifted sums keep the statistics accurate) and gamma /
    beta left out (1 and 0)."""
    c = LnCase(tp, 200, 4 * 128, 4, "f32", seed=5, shift=300.0, affine=False).run()
    errs = c.errors()
    errs.pop("dgamma"), errs.pop("dbeta")
    assert max(errs.values()) <= TOL_F32, errs


def test_layernorm_deterministic_and_shard_count(tp):
    import torch

    a = LnCase(tp, 300, 8 * 64, 8, "f32", seed=7).run()
    Y1 = [y.clone() for y in a.Y]
    a.run()
    assert all(torch.equal(p, q) for p, q in zip(Y1, a.Y))
    one = LnCase(tp, 300, 8 * 64, 1, "f32", seed=7).run()
    assert rel(np.concatenate([np64(y) for y in a.Y], 1), np64(one.Y[0])) <= 1e-5
    assert rel(np.concatenate([np64(x) for x in a.dX], 1), np64(one.dX[0])) <= 1e-5


@pytest.mark.parametrize("dtype,T,H,n", [("bf16", 257, 8 * 72, 8), ("bf16", 96, 4 * 1024, 4),
                                         ("bf16", 70, 8 * 1536, 8), ("bf16", 50, 2 * 2048, 2),
                                         ("bf16", 33, 3 * 1000, 3), ("f32", 64, 8 * 96, 8),
                                         ("f32", 40, 8 * 1024, 8)])
def test_layernorm_register_path_matches_two_pass(tp, tune, dtype, T, H, n):
    """Rows whose shards fit in at most 8 16-byte vectors per lane (2, 4, 6 and 8 here, ragged
    last vectors included) run in the register-resident kernels, which do the two-pass
    kernels' arithmetic in the same order: every output bit-identical to knob ln_reg = 0, and
    within tolerance of the oracle."""
    import torch

    cases = {}
    for reg in ("1", "0"):
        tune.set("ln_reg", reg)
        cases[reg] = LnCase(tp, T, H, n, dtype, seed=3).run()
    errs = cases["1"].errors()
    assert max(errs.values()) <= (TOL_BF16 if dtype == "bf16" else TOL_F32), errs
    a, b = cases["1"], cases["0"]
    for name in ("Y", "dX", "dg", "db"):
        assert all(torch.equal(x, y) for x, y in zip(getattr(a, name), getattr(b, name))), name
    assert torch.equal(a.mean, b.mean) and torch.equal(a.rstd, b.rstd)


def test_layernorm_zero_tokens(tp):
    import torch

    c = LnCase(tp, 0, 4 * 64, 4, "bf16")
    c.run()
    assert all(torch.count_nonzero(g) == 0 for g in c.dg)
    assert all(torch.count_nonzero(b) == 0 for b in c.db)


@pytest.mark.slow
def test_layernorm_bench_size(tp):
    """The size bench.py times (T 2048, H 12288, 8 shards, bf16), every output against the
    oracle."""
    errs = LnCase(tp, 2048, 12288, 8, "bf16", seed=11).run().errors()
    assert max(errs.values()) <= TOL_BF16, errs
