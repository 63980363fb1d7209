"""Seeded synthetic inputs for the tensor-parallel MLP and attention-projection workloads.

This module draws random numbers and nothing else: it holds no step of the method (no
split, no product, no activation, no sum). Both the CPU oracle (``oracle/``) and the CUDA
path are fed from it, so that they see the same values.

Recipe (one rule for every workload): tensor ``k`` of workload ``c`` is drawn from
``numpy.random.Generator(PCG64(1000 * c + k))`` as a standard normal in float32, multiplied
by the workload's standard deviation for that tensor (a standard deviation of 0 gives
zeros), and, for bf16 workloads, rounded to bf16 (round to nearest even) by
:func:`to_bf16`. Tensor order ``k``: for the MLP workloads X=0, A=1, a=2, B=3, b=4, dZ=5;
for the attention-projection workload X=0, W_qkv=1, C=2, W_o=3, dQKV=4, dO=5.

The shapes and distributions are the synthetic stand-ins for the pages' workloads: the
column-parallel example of "Tensor parallelism in practice: from theory to PyTorch code"
(a 768 -> 3072 linear, batch 32, weights drawn as ``randn * 0.01``, zero bias, 4 shards),
and GPT-3-175B-, attention- and sweep-shaped slices. No dataset and no trained weight is
involved.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

# Tensor order inside a workload's seed space.
MLP_TENSORS = ("X", "A", "a", "B", "b", "dZ")
ATTN_TENSORS = ("X", "Wqkv", "C", "Wo", "dQKV", "dO")


@dataclasses.dataclass(frozen=True)
class MlpWorkload:
    """One MLP workload: shapes, shard count, dtype and the standard deviation per tensor."""

    cid: int            # workload number (seed space 1000 * cid + k)
    name: str
    tokens: int         # T
    hidden: int         # H
    ffn: int            # F
    tp_degree: int      # n
    dtype: str          # "f32" or "bf16"
    sigma: Dict[str, float]
    backward: bool = True

    def with_shape(self, tokens=None, hidden=None, ffn=None, tp_degree=None):
        return dataclasses.replace(
            self,
            tokens=self.tokens if tokens is None else tokens,
            hidden=self.hidden if hidden is None else hidden,
            ffn=self.ffn if ffn is None else ffn,
            tp_degree=self.tp_degree if tp_degree is None else tp_degree,
        )

    @property
    def flops_fwd(self) -> int:
        """Algorithmic forward flops: two GEMMs of 2*T*H*F."""
        return 4 * self.tokens * self.hidden * self.ffn

    @property
    def flops_fwd_bwd(self) -> int:
        """Algorithmic forward + backward flops: six GEMMs of 2*T*H*F."""
        return 12 * self.tokens * self.hidden * self.ffn


@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    """Attention projections split over heads: fused QKV (column) and output (row)."""

    cid: int
    name: str
    tokens: int
    hidden: int
    heads: int
    head_dim: int
    tp_degree: int
    dtype: str
    sigma: Dict[str, float]

    def with_shape(self, tokens=None, heads=None, head_dim=None, tp_degree=None):
        heads = self.heads if heads is None else heads
        head_dim = self.head_dim if head_dim is None else head_dim
        return dataclasses.replace(
            self,
            tokens=self.tokens if tokens is None else tokens,
            heads=heads,
            head_dim=head_dim,
            hidden=heads * head_dim,
            tp_degree=self.tp_degree if tp_degree is None else tp_degree,
        )

    @property
    def flops_fwd_bwd(self) -> int:
        """QKV projection (H -> 3H) and output projection (H -> H), forward + backward."""
        T, H = self.tokens, self.hidden
        return 6 * T * H * (3 * H) + 6 * T * H * H


# Workload 1: the pages' column-parallel example (768 -> 3072, batch 32, 4 shards) closed by
# a row-parallel 3072 -> 768 layer, fp32, forward only.
P3_FP32_FWD = MlpWorkload(
    cid=1, name="p3_mlp_fp32_fwd_T32_H768_F3072_tp4", tokens=32, hidden=768, ffn=3072,
    tp_degree=4, dtype="f32",
    sigma={"X": 1.0, "A": 0.01, "a": 0.0, "B": 0.01, "b": 0.0, "dZ": 1.0}, backward=False)

# Workload 2: a mid-sized MLP, two shards.
MLP_T4096_H1024_F4096_TP2 = MlpWorkload(
    cid=2, name="mlp_bf16_T4096_H1024_F4096_tp2", tokens=4096, hidden=1024, ffn=4096,
    tp_degree=2, dtype="bf16",
    sigma={"X": 1.0, "A": 0.02, "a": 0.01, "B": 0.02, "b": 0.01, "dZ": 1.0})

# Workload 3: a GPT-3-175B-shaped MLP slice: one sequence of 2048 tokens, hidden 12288,
# ffn 4 * 12288, eight shards.
GPT3_MLP_T2048_TP8 = MlpWorkload(
    cid=3, name="gpt3_175b_mlp_bf16_T2048_H12288_F49152_tp8", tokens=2048, hidden=12288,
    ffn=49152, tp_degree=8, dtype="bf16",
    sigma={"X": 1.0, "A": 0.006, "a": 0.0, "B": 0.006, "b": 0.0, "dZ": 1.0})

# Workload 4: attention projections over 40 heads of 128, eight shards of 5 heads.
ATTN_T4096_H5120_TP8 = AttnWorkload(
    cid=4, name="attn_proj_bf16_T4096_H5120_40x128_tp8", tokens=4096, hidden=5120,
    heads=40, head_dim=128, tp_degree=8, dtype="bf16",
    sigma={"X": 1.0, "Wqkv": 0.02, "C": 1.0, "Wo": 0.02, "dQKV": 1.0, "dO": 1.0})

# Workload 5: the sharding sweep (hidden 8192, ffn 28672); the shard count and the token
# count are the sweep's two axes.
SWEEP_H8192_F28672 = MlpWorkload(
    cid=5, name="sweep_bf16_H8192_F28672", tokens=2048, hidden=8192, ffn=28672,
    tp_degree=8, dtype="bf16",
    sigma={"X": 1.0, "A": 0.01, "a": 0.0, "B": 0.01, "b": 0.0, "dZ": 1.0})
SWEEP_TP = (1, 2, 4, 8)
SWEEP_TOKENS = (512, 2048, 8192, 16384)

WORKLOADS = {w.cid: w for w in (P3_FP32_FWD, MLP_T4096_H1024_F4096_TP2, GPT3_MLP_T2048_TP8,
                                 ATTN_T4096_H5120_TP8, SWEEP_H8192_F28672)}


def normal(seed: int, shape, sigma: float) -> np.ndarray:
    """float32 draw of N(0, sigma^2) from PCG64(seed); sigma == 0 gives zeros."""
    if sigma == 0.0:
        return np.zeros(shape, dtype=np.float32)
    rng = np.random.Generator(np.random.PCG64(seed))
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        out *= np.float32(sigma)
    return out


def to_bf16(x: np.ndarray):
    """Round float32 values to bf16 (nearest even). Returns (torch bf16 tensor, float32 copy).

    The float32 copy holds exactly the bf16 values, so the oracle and the GPU see the same
    numbers.
    """
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)
    return t, t.to(torch.float32).numpy()


def mlp_tensors(w: MlpWorkload, which=MLP_TENSORS) -> Dict[str, np.ndarray]:
    """float32 draws for an MLP workload (not yet rounded to bf16)."""
    T, H, F = w.tokens, w.hidden, w.ffn
    shapes = {"X": (T, H), "A": (H, F), "a": (F,), "B": (F, H), "b": (H,), "dZ": (T, H)}
    out = {}
    for k, name in enumerate(MLP_TENSORS):
        if name in which:
            out[name] = normal(1000 * w.cid + k, shapes[name], w.sigma[name])
    return out


def attn_tensors(w: AttnWorkload, which=ATTN_TENSORS) -> Dict[str, np.ndarray]:
    """float32 draws for the attention-projection workload.

    C is the attention core's output (the input of the output projection); the core itself
    is not part of this path, so C is drawn directly, like the upstream gradients dQKV and dO.
    """
    T, H = w.tokens, w.hidden
    shapes = {"X": (T, H), "Wqkv": (H, 3 * H), "C": (T, H), "Wo": (H, H),
              "dQKV": (T, 3 * H), "dO": (T, H)}
    out = {}
    for k, name in enumerate(ATTN_TENSORS):
        if name in which:
            out[name] = normal(1000 * w.cid + k, shapes[name], w.sigma[name])
    return out


def sample_indices(seed: int, count: int, upto: int, must: Optional[list] = None) -> np.ndarray:
    """Sorted distinct indices in [0, upto) for sampled checks; ``must`` entries are kept."""
    rng = np.random.Generator(np.random.PCG64(seed))
    k = min(count, upto)
    idx = set(int(i) for i in rng.choice(upto, size=k, replace=False))
    for m in must or []:
        if 0 <= m < upto:
            idx.add(int(m))
    return np.array(sorted(idx), dtype=np.int64)
