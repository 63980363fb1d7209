"""Shared helpers of the GPU parity tests: seeded inputs -> shard buffers on the device ->
calls through the C ABI -> float64 numpy views for comparison with the oracle.

Error metric (per output tensor; per shard for sharded tensors, the worst shard reported):
max |gpu - ref| / max |ref|. Tolerances: bf16 inputs with fp32 accumulation 2e-2, fp32 1e-5,
GPU sharded vs GPU unsharded 1e-3.
"""
from __future__ import annotations

import numpy as np

import workloads as wl

TOL_BF16 = 2e-2
TOL_F32 = 1e-5
TOL_SHARDED_VS_UNSHARDED = 1e-3


def rel(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(x - ref)) / (den if den > 0 else 1.0))


def rel_shards(xs, refs) -> float:
    return max(rel(x, r) for x, r in zip(xs, refs))


def np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def prepare(raw: dict, dtype: str, device):
    """float32 draws -> (device tensors in the compute dtype, float32 host values as given)."""
    import torch

    dev, host = {}, {}
    for k, v in raw.items():
        if dtype == "bf16":
            t, f = wl.to_bf16(v)
        else:
            t, f = torch.from_numpy(np.ascontiguousarray(v)), v
        dev[k] = t.to(device)
        host[k] = f
    return dev, host


class MlpCase:
    """One MLP workload on the device, sharded the way the library expects."""

    def __init__(self, w: wl.MlpWorkload, reduce: int, device="cuda", act=None):
        import torch

        import tensor_sharded_linear_bias_gb300 as tp

        self.tp, self.w, self.device = tp, w, device
        self.bf16 = w.dtype == "bf16"
        self.cdt = torch.bfloat16 if self.bf16 else torch.float32
        raw = wl.mlp_tensors(w)
        self.t, self.f = prepare(raw, w.dtype, device)
        n, T, H, F = w.tp_degree, w.tokens, w.hidden, w.ffn
        self.n, self.T, self.H, self.F, self.Fs = n, T, H, F, F // n
        Fs = self.Fs
        self.A = [self.t["A"][:, i * Fs:(i + 1) * Fs].contiguous() for i in range(n)]
        self.a = [self.t["a"][i * Fs:(i + 1) * Fs].contiguous() for i in range(n)]
        self.B = [self.t["B"][i * Fs:(i + 1) * Fs, :].contiguous() for i in range(n)]
        self.desc = tp.MlpDesc(tokens=T, hidden=H, ffn=F, tp_degree=n,
                               dtype=tp.TP_BF16 if self.bf16 else tp.TP_F32,
                               act=tp.TP_ACT_GELU_ERF if act is None else act, reduce=reduce)
        self.ws = tp.new_workspace(tp.tp_mlp_workspace_size(self.desc), device)
        e = dict(dtype=torch.float32, device=device)
        self.Z = torch.full((T, H), float("nan"), **e)
        self.Hs = [torch.empty(T, Fs, dtype=self.cdt, device=device) for _ in range(n)]
        self.Ys = [torch.empty(T, Fs, dtype=self.cdt, device=device) for _ in range(n)]
        self.dX = torch.full((T, H), float("nan"), **e)
        self.dA = [torch.full((H, Fs), float("nan"), **e) for _ in range(n)]
        self.dB = [torch.full((Fs, H), float("nan"), **e) for _ in range(n)]
        self.da = [torch.full((Fs,), float("nan"), **e) for _ in range(n)]
        self.db = torch.full((H,), float("nan"), **e)

    def forward(self):
        self.tp.tp_mlp_forward(self.desc, self.t["X"], self.A, self.a, self.B, self.t["b"],
                               self.Z, self.Hs, self.Ys, self.ws)

    def backward(self):
        self.tp.tp_mlp_backward(self.desc, self.t["X"], self.A, self.B, self.Hs, self.Ys,
                                self.t["dZ"], self.dX, self.dA, self.da, self.dB, self.db,
                                self.ws)

    def run(self, backward=True):
        import torch

        self.forward()
        if backward:
            self.backward()
        self.tp.tp_check_status(self.ws)
        torch.cuda.synchronize()
        return self

    def outputs(self, backward=True) -> dict:
        out = {"Z": np64(self.Z), "H": [np64(h) for h in self.Hs], "Y": [np64(y) for y in self.Ys]}
        if backward:
            out.update({"dX": np64(self.dX), "dA": [np64(x) for x in self.dA],
                        "dB": [np64(x) for x in self.dB], "da": [np64(x) for x in self.da],
                        "db": np64(self.db)})
        return out


def compare_full(out: dict, ref_f: dict, ref_b=None) -> dict:
    errs = {"Z": rel(out["Z"], ref_f["Z"]), "H": rel_shards(out["H"], ref_f["H"]),
            "Y": rel_shards(out["Y"], ref_f["Y"])}
    if ref_b is not None:
        errs.update({"dX": rel(out["dX"], ref_b["dX"]), "dA": rel_shards(out["dA"], ref_b["dA"]),
                     "dB": rel_shards(out["dB"], ref_b["dB"]),
                     "da": rel_shards(out["da"], ref_b["da"]), "db": rel(out["db"], ref_b["db"])})
    return errs


def sampled_reference(oracle, f: dict, n: int, rows, cols):
    """Oracle values at token rows `rows` (Z, dX, H, Y rows) and ffn columns `cols`
    (dA columns, dB rows, da entries, H / Y columns), plus db."""
    X, A, a, B, b, dZ = f["X"], f["A"], f["a"], f["B"], f["b"], f["dZ"]
    fr = oracle.mlp_forward(X[rows], A, a, B, b, n)
    br = oracle.mlp_backward(X[rows], A, a, B, b, dZ[rows], n, fr)
    cr = oracle.mlp_columns(X, A, a, B, dZ, n, cols)
    return {"Z": fr["Z"], "dX": br["dX"], "Hrows": oracle.concat_columns(fr["H"]),
            "Yrows": oracle.concat_columns(fr["Y"]), "dA": cr["dA"], "dB": cr["dB"],
            "da": cr["da"], "Hcols": cr["H"], "Ycols": cr["Y"], "db": oracle.bias_grad(dZ)}


def sampled_gpu(case: MlpCase, rows, cols) -> dict:
    import torch

    Fs = case.Fs
    ri = torch.as_tensor(rows, device=case.device)
    H = torch.cat(case.Hs, 1)
    Y = torch.cat(case.Ys, 1)
    dA = torch.cat(case.dA, 1)
    dB = torch.cat(case.dB, 0)
    da = torch.cat(case.da, 0)
    ci = torch.as_tensor(cols, device=case.device)
    del Fs
    return {"Z": np64(case.Z[ri]), "dX": np64(case.dX[ri]), "Hrows": np64(H[ri]),
            "Yrows": np64(Y[ri]), "dA": np64(dA[:, ci]), "dB": np64(dB[ci]), "da": np64(da[ci]),
            "Hcols": np64(H[:, ci]), "Ycols": np64(Y[:, ci]), "db": np64(case.db)}


def sample_rows_cols(w: wl.MlpWorkload, nrows=8, ncols=8):
    T, F, Fs = w.tokens, w.ffn, w.ffn // w.tp_degree
    rows = wl.sample_indices(7000 + w.cid, nrows, T, must=[0, T - 1, 127, 128])
    cols = wl.sample_indices(8000 + w.cid, ncols, F, must=[0, F - 1, Fs - 1, Fs, 255, 256])
    return rows, cols
