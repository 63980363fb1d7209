"""Plain fp64 CPU oracle of the tensor-parallel MLP and of its two parallel linears.

TEST INFRASTRUCTURE ONLY. Slow on purpose and written for reading: every step is the plain
definition, in fp64, with the shards cut out explicitly and summed in shard order. It shares
no code with the CUDA library and imports nothing from it.

Pages this follows (cited by title and section):

* [Paddle]  "PaddlePaddle tensor parallelism: from principle to industrial deployment" --
  FFN column split with the outputs gathered; the input gradient of a column-split layer is
  summed over the devices.
* [Lansai]  "What tensor parallelism is: core principles of large-model training" -- section
  "Core working mechanism": X is replicated, A is split by columns, Y_i = X A_i; the next
  linear is split by rows so that Y_i is its shard input.
* [CSDN]    "Tensor parallelism in practice: from theory to complete PyTorch code" -- the
  custom TensorParallelLinear: each shard holds out/world_size columns of the weight and its
  own bias slice, computes X W_i + b_i, and the shard outputs are gathered and concatenated
  along the last dimension; out_features must divide by world_size.
* [Intelli] "Tensor Parallelism: principle and practice" -- section 2.1 (block matrix
  computation and the distributive identity), section 3.1 (Megatron-LM column parallel:
  dL/dW_i = X^T dL/dY_i; row parallel: partial products summed by All-Reduce, input gradient
  (dL/dY) W^T), section 4.2 (QKV projection split by columns / by heads).

Readings taken where the pages are silent, garbled or in conflict:

* R1  The row-parallel bias is added once, after the shard sum (pages silent; the only
      reading under which one shard equals the unsharded layer). Column biases are per
      shard, as in [CSDN].
* R2  In the column layer's gradients dA_i = X^T dY_i and dX = sum_i dY_i A_i^T, "dY_i" is
      the gradient at the column linear's output *before* the activation (dH_i here). The
      pages' layers have no activation, so there the two coincide.
* R3  [Intelli] 3.1 writes the row layer's input gradient as (dL/dY) W^T; read W as the
      shard's own block W_i. The weight gradient of the row layer, dB_i = Y_i^T dZ, is the
      same rule as the column layer's dL/dW_i = X_i^T dL/dY.
* R4  [Lansai] and [Intelli] 2.1 / 4.2 say a column split is combined by a *sum* and write
      XW = X(W1 + ... + Wn); this is garbled. Follow [Paddle] and [CSDN] (column split ->
      concatenate) and [Intelli] 3.1 (row split -> sum): XW = sum_i X_i W_i with X split by
      columns and W by rows.
* R5  The activation is GeLU in its exact erf form (the pages name no activation).
* R6  Shard partials are summed in shard order 0..n-1.
* R8  The fused QKV weight is laid out as [Q | K | V] blocks of H columns each, with heads
      contiguous inside a block; shard s takes the columns of heads s*h/n .. (s+1)*h/n - 1
      from each of the three blocks.
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence

import numpy as np
from scipy.special import erf

__all__ = [
    "gelu", "gelu_grad", "shard_size", "split_columns", "split_rows", "split_vector",
    "concat_columns", "qkv_head_shards", "linear", "bias_grad", "column_parallel_forward",
    "column_parallel_backward", "row_parallel_forward", "row_parallel_backward",
    "mlp_forward", "mlp_backward", "mlp_columns", "attn_forward", "attn_backward",
    "split_tokens", "all_gather_tokens", "mlp_forward_sp", "mlp_backward_sp",
]

_SQRT2 = math.sqrt(2.0)
_INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# ----------------------------------------------------------------------------- activation
def gelu(h):
    """GeLU, exact form: h * Phi(h) with Phi(h) = (1 + erf(h / sqrt 2)) / 2 (reading R5)."""
    h = _f64(h)
    return 0.5 * h * (1.0 + erf(h / _SQRT2))


def gelu_grad(h):
    """d GeLU / dh = Phi(h) + h * phi(h), phi the standard normal density (reading R5)."""
    h = _f64(h)
    return 0.5 * (1.0 + erf(h / _SQRT2)) + h * np.exp(-0.5 * h * h) * _INV_SQRT_2PI


# ----------------------------------------------------------------------------- splitting
def shard_size(total: int, n: int) -> int:
    """Width of one shard; [CSDN] asserts that out_features divides by world_size."""
    if n < 1 or total % n != 0:
        raise ValueError(f"dimension {total} is not divisible by tp_degree {n}")
    return total // n


def split_columns(W, n: int) -> List[np.ndarray]:
    """Column split W = [W_0, ..., W_{n-1}] ([Lansai] core mechanism; [CSDN] weight shard)."""
    w = shard_size(W.shape[1], n)
    return [W[:, i * w:(i + 1) * w] for i in range(n)]


def split_rows(W, n: int) -> List[np.ndarray]:
    """Row split of the next linear's weight ([Intelli] 3.1 row parallel)."""
    w = shard_size(W.shape[0], n)
    return [W[i * w:(i + 1) * w, :] for i in range(n)]


def split_vector(v, n: int) -> List[np.ndarray]:
    """Per-shard slices of a column bias ([CSDN]: a bias of out/world_size per shard)."""
    w = shard_size(v.shape[0], n)
    return [v[i * w:(i + 1) * w] for i in range(n)]


def concat_columns(parts: Sequence[np.ndarray]) -> np.ndarray:
    """The gather + concatenation along the last dimension of [CSDN]'s forward."""
    return np.concatenate([_f64(p) for p in parts], axis=1)


def qkv_head_shards(Wqkv, heads: int, head_dim: int, n: int) -> List[np.ndarray]:
    """Split a fused [Q|K|V] projection by heads ([Paddle]; [Intelli] 4.2; reading R8)."""
    hm = heads * head_dim
    if Wqkv.shape[1] != 3 * hm:
        raise ValueError("fused QKV weight must have 3 * heads * head_dim columns")
    w = shard_size(heads, n) * head_dim
    return [np.concatenate([Wqkv[:, blk * hm + s * w: blk * hm + (s + 1) * w]
                            for blk in range(3)], axis=1) for s in range(n)]


# ----------------------------------------------------------------------------- one linear
def linear(X, W, bias=None) -> np.ndarray:
    """X W (+ bias broadcast over rows), fp64 ([CSDN]: matmul(x, weight) + bias)."""
    out = _f64(X) @ _f64(W)
    if bias is not None:
        out = out + _f64(bias)[None, :]
    return out


def bias_grad(G) -> np.ndarray:
    """Gradient of a bias broadcast over the token rows: the sum over tokens of G."""
    return _f64(G).sum(axis=0)


# ----------------------------------------------------------------------------- column parallel
def column_parallel_forward(X, W_shards, b_shards=None, act: str = "none"):
    """Y_i = act(X W_i + b_i) for every shard i; X is replicated ([Lansai]; [CSDN]).

    Returns (H, Y): the pre-activation outputs H_i and the outputs Y_i, one per shard.
    """
    H, Y = [], []
    for i, Wi in enumerate(W_shards):
        Hi = linear(X, Wi, None if b_shards is None else b_shards[i])
        H.append(Hi)
        Y.append(gelu(Hi) if act == "gelu" else Hi)
    return H, Y


def column_parallel_backward(X, W_shards, H_shards, dY_shards, act: str = "none"):
    """Backward of the column-parallel linear ([Intelli] 3.1; [Paddle]; readings R2, R6).

    ``H_shards`` (the saved pre-activation outputs) is only read when ``act`` is "gelu".
    dH_i = dY_i * act'(H_i); dW_i = X^T dH_i; dbias_i = sum over tokens of dH_i;
    dX = sum_i dH_i W_i^T (the input gradient summed over the shards, in shard order).
    Returns (dX, dW list, dbias list, dH list).
    """
    X = _f64(X)
    dH = []
    for i, dYi in enumerate(dY_shards):
        dH.append(_f64(dYi) * gelu_grad(H_shards[i]) if act == "gelu" else _f64(dYi))
    dW = [X.T @ dHi for dHi in dH]
    dbias = [bias_grad(dHi) for dHi in dH]
    dX = None
    for dHi, Wi in zip(dH, W_shards):
        term = dHi @ _f64(Wi).T
        dX = term if dX is None else dX + term
    return dX, dW, dbias, dH


# ----------------------------------------------------------------------------- row parallel
def row_parallel_forward(X_shards, W_shards, bias=None) -> np.ndarray:
    """Z = sum_i X_i W_i + bias ([Intelli] 3.1 row parallel + All-Reduce SUM; R1, R6)."""
    Z = None
    for Xi, Wi in zip(X_shards, W_shards):
        Pi = linear(Xi, Wi)
        Z = Pi if Z is None else Z + Pi
    if bias is not None:
        Z = Z + _f64(bias)[None, :]
    return Z


def row_parallel_backward(X_shards, W_shards, dZ):
    """Backward of the row-parallel linear ([Intelli] 3.1; reading R3).

    dX_i = dZ W_i^T; dW_i = X_i^T dZ; dbias = sum over tokens of dZ.
    Returns (dX list, dW list, dbias).
    """
    dZ = _f64(dZ)
    dX = [dZ @ _f64(Wi).T for Wi in W_shards]
    dW = [_f64(Xi).T @ dZ for Xi in X_shards]
    return dX, dW, bias_grad(dZ)


# ----------------------------------------------------------------------------- the MLP
def mlp_forward(X, A, a, B, b, n: int):
    """Column-parallel linear + GeLU feeding a row-parallel linear ([Lansai]; [Intelli] 3.1).

    A is split by columns, B by rows; Y_i = GeLU(X A_i + a_i); Z = sum_i Y_i B_i + b.
    Returns a dict with H (list), Y (list) and Z.
    """
    A_s = split_columns(A, n)
    a_s = None if a is None else split_vector(a, n)
    B_s = split_rows(B, n)
    H, Y = column_parallel_forward(X, A_s, a_s, "gelu")
    Z = row_parallel_forward(Y, B_s, b)
    return {"H": H, "Y": Y, "Z": Z}


def mlp_backward(X, A, a, B, b, dZ, n: int, fwd=None):
    """Backward of :func:`mlp_forward` (row layer first, then the column layer).

    Returns a dict with dX, dA (list), da (list), dB (list), db, and dY, dH (lists).
    """
    if fwd is None:
        fwd = mlp_forward(X, A, a, B, b, n)
    A_s = split_columns(A, n)
    B_s = split_rows(B, n)
    dY, dB, db = row_parallel_backward(fwd["Y"], B_s, dZ)
    dX, dA, da, dH = column_parallel_backward(X, A_s, fwd["H"], dY, "gelu")
    return {"dX": dX, "dA": dA, "da": da, "dB": dB, "db": db, "dY": dY, "dH": dH}


def mlp_columns(X, A, a, B, dZ, n: int, cols: Sequence[int]):
    """The MLP's per-ffn-column results for the global ffn columns ``cols`` only.

    Each ffn column j lives in shard j // F_s at local column j % F_s. Its H, Y, dY, dH
    columns, dA column, da entry and dB row depend on no other ffn column, so they are the
    same definitions applied to that one column of the shard. Returns a dict of arrays
    whose last (for dB: first) axis runs over ``cols``: H, Y, dH [T, c], dA [H, c],
    da [c], dB [c, H].
    """
    A_s = split_columns(A, n)
    a_s = None if a is None else split_vector(a, n)
    B_s = split_rows(B, n)
    fs = A_s[0].shape[1]
    T, Hd = X.shape[0], X.shape[1]
    c = len(cols)
    out = {"H": np.zeros((T, c)), "Y": np.zeros((T, c)), "dH": np.zeros((T, c)),
           "dA": np.zeros((Hd, c)), "da": np.zeros(c), "dB": np.zeros((c, B.shape[1]))}
    for pos, j in enumerate(cols):
        i, loc = int(j) // fs, int(j) % fs
        Ai = A_s[i][:, loc:loc + 1]
        ai = None if a_s is None else a_s[i][loc:loc + 1]
        Bi = B_s[i][loc:loc + 1, :]
        (Hi,), (Yi,) = column_parallel_forward(X, [Ai], None if ai is None else [ai], "gelu")
        (dYi,), (dBi,), _ = row_parallel_backward([Yi], [Bi], dZ)
        _, (dAi,), (dai,), (dHi,) = column_parallel_backward(X, [Ai], [Hi], [dYi], "gelu")
        out["H"][:, pos] = Hi[:, 0]
        out["Y"][:, pos] = Yi[:, 0]
        out["dH"][:, pos] = dHi[:, 0]
        out["dA"][:, pos] = dAi[:, 0]
        out["da"][pos] = dai[0]
        out["dB"][pos, :] = dBi[0, :]
    return out


# ----------------------------------------------------------------------------- sequence parallel
def split_tokens(M, n: int) -> List[np.ndarray]:
    """Token (row) split: shard j holds rows j*T/n .. (j+1)*T/n - 1 (sequence parallelism,
    [Lansai] "sequence parallelism", which splits the sequence dimension across devices)."""
    return split_rows(M, n)


def all_gather_tokens(parts: Sequence[np.ndarray]) -> np.ndarray:
    """All-gather of token shards: their rows stacked in shard order."""
    return np.concatenate([_f64(p) for p in parts], axis=0)


def mlp_forward_sp(X_shards, A, a, B, b, n: int):
    """Sequence-parallel MLP forward: the token shards X_j are all-gathered into X, the MLP
    runs as in mlp_forward, and the shard sum Z is reduce-scattered: shard j receives rows
    j*T/n .. (j+1)*T/n - 1 of Z ([Paddle]: ReduceScatter in place of AllReduce).
    Returns a dict with Z (list of token shards), H, Y (lists of shard activations)."""
    X = all_gather_tokens(X_shards)
    out = mlp_forward(X, A, a, B, b, n)
    return {"Z": split_tokens(out["Z"], n), "H": out["H"], "Y": out["Y"]}


def mlp_backward_sp(X_shards, A, a, B, b, dZ_shards, n: int):
    """Backward of mlp_forward_sp: dZ is all-gathered, the weight and bias gradients are those
    of mlp_backward, and dX is reduce-scattered into token shards."""
    X = all_gather_tokens(X_shards)
    dZ = all_gather_tokens(dZ_shards)
    g = mlp_backward(X, A, a, B, b, dZ, n)
    g["dX"] = split_tokens(g["dX"], n)
    return g


# ----------------------------------------------------------------------------- attention projections
def attn_forward(X, Wqkv, C, Wo, heads: int, head_dim: int, n: int):
    """Tensor parallel over heads ([Paddle]; [Intelli] 4.2; [CSDN] "extension" section).

    The fused QKV projection is column parallel (QKV_s = X Wqkv_s, no bias, no activation);
    the output projection is row parallel over the shards' context blocks C_s
    (O = sum_s C_s Wo_s). The attention core between them is not part of this path, so C is
    an input. Returns dict with QKV (list of shard outputs) and O.
    """
    W_s = qkv_head_shards(Wqkv, heads, head_dim, n)
    _, QKV = column_parallel_forward(X, W_s, None, "none")
    O = row_parallel_forward(split_columns(C, n), split_rows(Wo, n), None)
    return {"QKV": QKV, "O": O}


def attn_backward(X, Wqkv, C, Wo, dQKV, dO, heads: int, head_dim: int, n: int):
    """Backward of both projections. dQKV is the upstream gradient in the fused [Q|K|V]
    column layout; shard s sees the same head columns as its weight shard.

    Returns dX (sum over shards), dWqkv (list), dC (list of shard blocks), dWo (list).
    """
    W_s = qkv_head_shards(Wqkv, heads, head_dim, n)
    dQKV_s = qkv_head_shards(dQKV, heads, head_dim, n)
    dX, dWqkv, _, _ = column_parallel_backward(X, W_s, None, dQKV_s, "none")
    dC, dWo, _ = row_parallel_backward(split_columns(C, n), split_rows(Wo, n), dO)
    return {"dX": dX, "dWqkv": dWqkv, "dC": dC, "dWo": dWo}
