"""Layer objects over the C ABI: shard buffers, saved activations, gradients and the workspace.

The column-parallel linear plays the part of the custom TensorParallelLinear of "Tensor
parallelism in practice: from theory to complete PyTorch code" (a weight of
[in, out / world_size] per shard, a bias slice per shard, outputs gathered along the last
dimension), except that all tp_degree shards live on the one GPU. The row-parallel linear and
the MLP follow "Tensor Parallelism: principle and practice", section 3.1, the LayerNorm over a
split hidden dimension its section 4.2. Every computation runs in the library's kernels; these
classes only allocate torch tensors and pass pointers.
"""
from __future__ import annotations

from typing import List, Optional

from . import (TP_ACT_GELU_ERF, TP_ACT_NONE, TP_BF16, TP_COLUMN, TP_F32, TP_REDUCE_AUTO, TP_ROW,
               LayerNormDesc, LinearDesc, MlpDesc, new_workspace, tp_check_status,
               tp_layernorm_backward, tp_layernorm_forward, tp_linear_column_backward,
               tp_linear_column_forward, tp_linear_row_backward, tp_linear_row_forward,
               tp_linear_workspace_size, tp_mlp_backward, tp_mlp_forward,
               tp_mlp_workspace_size)

__all__ = ["ColumnParallelLinear", "RowParallelLinear", "TensorParallelMLP",
           "TensorParallelLayerNorm"]


def _dtype_code(dtype) -> int:
    import torch

    if dtype == torch.bfloat16:
        return TP_BF16
    if dtype == torch.float32:
        return TP_F32
    raise ValueError("dtype must be torch.bfloat16 or torch.float32")


def _split_columns(w, n):
    s = w.shape[1] // n
    return [w[:, i * s:(i + 1) * s].contiguous() for i in range(n)]


def _split_rows(w, n):
    s = w.shape[0] // n
    return [w[i * s:(i + 1) * s, :].contiguous() for i in range(n)]


class _Workspaces:
    """One workspace per token count, grown on demand."""

    def __init__(self, device):
        self.device = device
        self.ws = None

    def get(self, nbytes):
        if self.ws is None or self.ws.numel() < nbytes:
            self.ws = new_workspace(nbytes, self.device)
        return self.ws


class ColumnParallelLinear:
    """Y_i = act(X W_i + b_i) for shards i = 0..n-1 of W [in, out] split by columns.

    ``weight``: full [in, out] tensor (split here) or None for ``randn * init_scale``;
    ``gather=True`` returns one [T, out] output (the shards' column blocks), else a list.
    Gradients of the last backward: ``weight_grads`` (list of fp32 [in, out/n]),
    ``bias_grads`` (list of fp32 [out/n])."""

    def __init__(self, in_features: int, out_features: int, tp_degree: int, *,
                 dtype=None, device="cuda", weight=None, bias: bool = True, act: str = "none",
                 gather: bool = True, init_scale: float = 0.01, generator=None):
        import torch

        dtype = torch.bfloat16 if dtype is None else dtype
        self.K, self.N, self.n = in_features, out_features, tp_degree
        self.dtype, self.device, self.gather = dtype, torch.device(device), gather
        self.act = TP_ACT_GELU_ERF if act == "gelu" else TP_ACT_NONE
        self.desc = LinearDesc(tokens=0, in_features=in_features, out_features=out_features,
                               tp_degree=tp_degree, dtype=_dtype_code(dtype), act=self.act,
                               reduce=TP_REDUCE_AUTO if dtype == torch.bfloat16 else 0,
                               gather=int(gather))
        tp_linear_workspace_size(self.desc, TP_COLUMN)  # validates the shape (raises TpError)
        if weight is None:
            weight = torch.randn(in_features, out_features, generator=generator) * init_scale
        self.weights: List = _split_columns(weight.to(self.device, dtype), tp_degree)
        ns = out_features // tp_degree
        self.biases: Optional[List] = (
            [torch.zeros(ns, dtype=dtype, device=self.device) for _ in range(tp_degree)]
            if bias else None)
        self._ws = _Workspaces(self.device)
        self._x = None
        self._h = None

    def _desc(self, T):
        d = LinearDesc.from_buffer_copy(self.desc)
        d.tokens = T
        return d

    def forward(self, x):
        import torch

        T = x.shape[0]
        d = self._desc(T)
        ws = self._ws.get(tp_linear_workspace_size(d, TP_COLUMN))
        ns = self.N // self.n
        y = ([torch.empty(T, self.N, dtype=self.dtype, device=self.device)] if self.gather else
             [torch.empty(T, ns, dtype=self.dtype, device=self.device) for _ in range(self.n)])
        h = ([torch.empty(T, ns, dtype=self.dtype, device=self.device) for _ in range(self.n)]
             if self.act != TP_ACT_NONE else None)
        tp_linear_column_forward(d, x, self.weights, self.biases, y, h, ws)
        self._x, self._h = x, h
        return y[0] if self.gather else y

    def backward(self, dy):
        import torch

        T = self._x.shape[0]
        d = self._desc(T)
        ws = self._ws.get(tp_linear_workspace_size(d, TP_COLUMN))
        ns = self.N // self.n
        f32 = dict(dtype=torch.float32, device=self.device)
        dx = torch.empty(T, self.K, **f32)
        self.weight_grads = [torch.empty(self.K, ns, **f32) for _ in range(self.n)]
        self.bias_grads = ([torch.empty(ns, **f32) for _ in range(self.n)]
                           if self.biases is not None else None)
        dys = [dy] if self.gather else list(dy)
        tp_linear_column_backward(d, self._x, self.weights, self._h, dys, dx, self.weight_grads,
                                  self.bias_grads, ws)
        return dx

    def check(self):
        """Synchronise and raise if a kernel reported a device-side timeout."""
        if self._ws.ws is not None:
            tp_check_status(self._ws.ws)


class RowParallelLinear:
    """Z = sum_i X_i W_i + b for shards of W [in, out] split by rows; X_i are the shard inputs
    (a list of [T, in/n] tensors). ``weight_grads``: fp32 [in/n, out] per shard; ``bias_grad``:
    fp32 [out]."""

    def __init__(self, in_features: int, out_features: int, tp_degree: int, *, dtype=None,
                 device="cuda", weight=None, bias: bool = True, reduce: int = TP_REDUCE_AUTO,
                 init_scale: float = 0.01, generator=None):
        import torch

        dtype = torch.bfloat16 if dtype is None else dtype
        self.K, self.N, self.n = in_features, out_features, tp_degree
        self.dtype, self.device = dtype, torch.device(device)
        if dtype == torch.float32 and reduce == TP_REDUCE_AUTO:
            reduce = 0
        self.desc = LinearDesc(tokens=0, in_features=in_features, out_features=out_features,
                               tp_degree=tp_degree, dtype=_dtype_code(dtype), act=TP_ACT_NONE,
                               reduce=reduce, gather=0)
        tp_linear_workspace_size(self.desc, TP_ROW)
        if weight is None:
            weight = torch.randn(in_features, out_features, generator=generator) * init_scale
        self.weights: List = _split_rows(weight.to(self.device, dtype), tp_degree)
        self.bias = torch.zeros(out_features, dtype=dtype, device=self.device) if bias else None
        self._ws = _Workspaces(self.device)
        self._xs = None

    def _desc(self, T):
        d = LinearDesc.from_buffer_copy(self.desc)
        d.tokens = T
        return d

    def forward(self, xs):
        import torch

        T = xs[0].shape[0]
        d = self._desc(T)
        ws = self._ws.get(tp_linear_workspace_size(d, TP_ROW))
        z = torch.empty(T, self.N, dtype=torch.float32, device=self.device)
        tp_linear_row_forward(d, xs, self.weights, self.bias, z, ws)
        self._xs = list(xs)
        return z

    def backward(self, dz):
        import torch

        T = dz.shape[0]
        d = self._desc(T)
        ws = self._ws.get(tp_linear_workspace_size(d, TP_ROW))
        f32 = dict(dtype=torch.float32, device=self.device)
        ks = self.K // self.n
        dxs = [torch.empty(T, ks, **f32) for _ in range(self.n)]
        self.weight_grads = [torch.empty(ks, self.N, **f32) for _ in range(self.n)]
        self.bias_grad = torch.empty(self.N, **f32) if self.bias is not None else None
        tp_linear_row_backward(d, self._xs, self.weights, dz, dxs, self.weight_grads,
                               self.bias_grad, ws)
        return dxs


class TensorParallelMLP:
    """Column-parallel linear + GeLU -> row-parallel linear (A [H, F] by columns, B [F, H] by
    rows), forward and backward in one library call each. Gradients of the last backward:
    ``dA``, ``da``, ``dB`` (per-shard lists, fp32) and ``db`` (fp32 [H])."""

    def __init__(self, hidden: int, ffn: int, tp_degree: int, *, dtype=None, device="cuda",
                 A=None, a=None, B=None, b=None, reduce: int = TP_REDUCE_AUTO,
                 init_scale: float = 0.02, generator=None):
        import torch

        dtype = torch.bfloat16 if dtype is None else dtype
        self.H, self.F, self.n = hidden, ffn, tp_degree
        self.dtype, self.device = dtype, torch.device(device)
        if dtype == torch.float32 and reduce == TP_REDUCE_AUTO:
            reduce = 0
        self.desc = MlpDesc(tokens=0, hidden=hidden, ffn=ffn, tp_degree=tp_degree,
                            dtype=_dtype_code(dtype), act=TP_ACT_GELU_ERF, reduce=reduce)
        tp_mlp_workspace_size(self.desc)
        A = torch.randn(hidden, ffn, generator=generator) * init_scale if A is None else A
        B = torch.randn(ffn, hidden, generator=generator) * init_scale if B is None else B
        a = torch.zeros(ffn) if a is None else a
        b = torch.zeros(hidden) if b is None else b
        fs = ffn // tp_degree
        self.A = _split_columns(A.to(self.device, dtype), tp_degree)
        self.a = [a.to(self.device, dtype)[i * fs:(i + 1) * fs].contiguous() for i in range(tp_degree)]
        self.B = _split_rows(B.to(self.device, dtype), tp_degree)
        self.b = b.to(self.device, dtype).contiguous()
        self._ws = _Workspaces(self.device)
        self._x = self._h = self._y = None

    def _desc(self, T):
        d = MlpDesc.from_buffer_copy(self.desc)
        d.tokens = T
        return d

    def forward(self, x):
        import torch

        T = x.shape[0]
        d = self._desc(T)
        ws = self._ws.get(tp_mlp_workspace_size(d))
        fs = self.F // self.n
        z = torch.empty(T, self.H, dtype=torch.float32, device=self.device)
        self._h = [torch.empty(T, fs, dtype=self.dtype, device=self.device) for _ in range(self.n)]
        self._y = [torch.empty(T, fs, dtype=self.dtype, device=self.device) for _ in range(self.n)]
        tp_mlp_forward(d, x, self.A, self.a, self.B, self.b, z, self._h, self._y, ws)
        self._x = x
        return z

    def backward(self, dz):
        import torch

        T = self._x.shape[0]
        d = self._desc(T)
        ws = self._ws.get(tp_mlp_workspace_size(d))
        fs = self.F // self.n
        f32 = dict(dtype=torch.float32, device=self.device)
        dx = torch.empty(T, self.H, **f32)
        self.dA = [torch.empty(self.H, fs, **f32) for _ in range(self.n)]
        self.dB = [torch.empty(fs, self.H, **f32) for _ in range(self.n)]
        self.da = [torch.empty(fs, **f32) for _ in range(self.n)]
        self.db = torch.empty(self.H, **f32)
        tp_mlp_backward(d, self._x, self.A, self.B, self._h, self._y, dz, dx, self.dA, self.da,
                        self.dB, self.db, ws)
        return dx

    def check(self):
        """Synchronise and raise if a kernel reported a device-side timeout."""
        if self._ws.ws is not None:
            tp_check_status(self._ws.ws)


class TensorParallelLayerNorm:
    """LayerNorm over a hidden dimension split into tp_degree column shards: inputs and outputs
    are lists of per-shard [T, hidden/n] tensors; gamma / beta are per-shard slices (1 and 0 at
    start). The row statistics cover the whole hidden dimension (combined over the shards on
    the device). Gradients of the last backward: ``gamma_grads``, ``beta_grads`` (fp32 per
    shard)."""

    def __init__(self, hidden: int, tp_degree: int, *, eps: float = 1e-5, dtype=None,
                 device="cuda", affine: bool = True):
        import torch

        dtype = torch.bfloat16 if dtype is None else dtype
        self.H, self.n, self.dtype = hidden, tp_degree, dtype
        self.device = torch.device(device)
        self.desc = LayerNormDesc(tokens=0, hidden=hidden, tp_degree=tp_degree,
                                  dtype=_dtype_code(dtype), eps=eps)
        if hidden % tp_degree != 0:
            raise ValueError(f"hidden {hidden} is not divisible by tp_degree {tp_degree}")
        hs = hidden // tp_degree
        self.gamma = ([torch.ones(hs, dtype=dtype, device=self.device) for _ in range(tp_degree)]
                      if affine else None)
        self.beta = ([torch.zeros(hs, dtype=dtype, device=self.device) for _ in range(tp_degree)]
                     if affine else None)
        self._x = self._mean = self._rstd = None

    def _desc(self, T):
        d = LayerNormDesc.from_buffer_copy(self.desc)
        d.tokens = T
        return d

    def forward(self, xs):
        import torch

        T = xs[0].shape[0]
        f32 = dict(dtype=torch.float32, device=self.device)
        ys = [torch.empty_like(x) for x in xs]
        self._mean, self._rstd = torch.empty(T, **f32), torch.empty(T, **f32)
        tp_layernorm_forward(self._desc(T), xs, self.gamma, self.beta, ys, self._mean, self._rstd)
        self._x = list(xs)
        return ys

    def backward(self, dys):
        import torch

        T = dys[0].shape[0]
        dxs = [torch.empty_like(d) for d in dys]
        hs = self.H // self.n
        f32 = dict(dtype=torch.float32, device=self.device)
        self.gamma_grads = [torch.empty(hs, **f32) for _ in range(self.n)] if self.gamma else None
        self.beta_grads = [torch.empty(hs, **f32) for _ in range(self.n)] if self.beta else None
        tp_layernorm_backward(self._desc(T), self._x, self.gamma, self._mean, self._rstd, dys,
                              dxs, self.gamma_grads, self.beta_grads)
        return dxs
