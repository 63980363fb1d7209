"""The row-parallel forward for callers that cannot allocate device memory.

tp_linear_row_forward_noalloc keeps its scratch (status word and per-shard partials) in a
static device array inside the library instead of a caller-allocated workspace. It is meant
for callers with no device allocator of their own, such as a plug-in inside an application
that owns all device memory. This test calls it through the C ABI (ctypes, no workspace
argument) and checks its output against tp_linear_row_forward, the workspace-based entry
point, on two calls in a row with different inputs, so that contents left in the shared
static array by the first call cannot leak into the second.

The file name puts it last in collection order.
"""
import ctypes

import numpy as np
import pytest

import workloads as wl
from harness import np64, prepare, rel

pytestmark = pytest.mark.gpu

TOL_GPU_VS_GPU = 1e-5   # two GPU paths over the same bf16 / fp32 inputs (fp32 outputs)


def _inputs(seed, T, K, N, dtype):
    raw = {"X": wl.normal(seed, (T, K), 1.0), "W": wl.normal(seed + 1, (K, N), 0.05),
           "bias": wl.normal(seed + 2, (N,), 0.1)}
    return prepare(raw, dtype, "cuda")[0]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_row_forward_without_allocation_matches_workspace_path(dtype):
    import torch

    import tensor_sharded_linear_bias_gb300 as tp

    fn = tp.lib.tp_linear_row_forward_noalloc
    T, K, N, n = 200, 4 * 88, 264, 4
    Ks = K // n
    desc = tp.LinearDesc(tokens=T, in_features=K, out_features=N, tp_degree=n,
                         dtype=tp.TP_BF16 if dtype == "bf16" else tp.TP_F32, act=0,
                         reduce=tp.TP_REDUCE_PARTIALS, gather=0)
    ws = tp.new_workspace(tp.tp_linear_workspace_size(desc, tp.TP_ROW))
    stream = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((501, 611)):
        t = _inputs(seed, T, K, N, dtype)
        X = [t["X"][:, i * Ks:(i + 1) * Ks].contiguous() for i in range(n)]
        W = [t["W"][i * Ks:(i + 1) * Ks, :].contiguous() for i in range(n)]
        Z_ref = torch.empty(T, N, dtype=torch.float32, device="cuda")
        tp.tp_linear_row_forward(desc, X, W, t["bias"], Z_ref, ws)
        Z = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
        st = fn(ctypes.byref(desc), tp._arr(X), tp._arr(W), t["bias"].data_ptr(), Z.data_ptr(),
                stream)
        assert st == 0, tp.tp_last_error()
        torch.cuda.synchronize()
        got, ref = np64(Z), np64(Z_ref)
        assert np.isfinite(got).all(), f"call {call}: unwritten outputs"
        assert rel(got, ref) <= TOL_GPU_VS_GPU, f"call {call}"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_row_forward_without_allocation_allocates_nothing(dtype):
    """The entry point's contract: after a first call (which looks up the static array's
    address and loads the kernels), further calls leave the device's free memory and torch's
    allocator untouched -- everything is allocated before the measured call."""
    import torch

    import tensor_sharded_linear_bias_gb300 as tp

    fn = tp.lib.tp_linear_row_forward_noalloc
    T, K, N, n = 300, 4 * 64, 512, 4
    Ks = K // n
    desc = tp.LinearDesc(tokens=T, in_features=K, out_features=N, tp_degree=n,
                         dtype=tp.TP_BF16 if dtype == "bf16" else tp.TP_F32, act=0,
                         reduce=tp.TP_REDUCE_PARTIALS, gather=0)
    t = _inputs(733, T, K, N, dtype)
    X = [t["X"][:, i * Ks:(i + 1) * Ks].contiguous() for i in range(n)]
    W = [t["W"][i * Ks:(i + 1) * Ks, :].contiguous() for i in range(n)]
    Zs = [torch.empty(T, N, dtype=torch.float32, device="cuda") for _ in range(2)]
    stream = torch.cuda.current_stream().cuda_stream
    xs, ws, b = tp._arr(X), tp._arr(W), t["bias"].data_ptr()
    assert fn(ctypes.byref(desc), xs, ws, b, Zs[0].data_ptr(), stream) == 0, tp.tp_last_error()
    torch.cuda.synchronize()
    free0, allocated0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    reserved0 = torch.cuda.memory_reserved()
    assert fn(ctypes.byref(desc), xs, ws, b, Zs[1].data_ptr(), stream) == 0, tp.tp_last_error()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == allocated0
    assert torch.cuda.memory_reserved() == reserved0
    assert torch.equal(Zs[0], Zs[1])


def test_row_forward_without_allocation_rejects_oversize():
    import tensor_sharded_linear_bias_gb300 as tp

    # 4 shards x 4096 tokens x 1024 outputs x 4 bytes = 64 MiB of partials > 32 MiB
    desc = tp.LinearDesc(tokens=4096, in_features=4 * 64, out_features=1024, tp_degree=4,
                         dtype=tp.TP_BF16, act=0, reduce=0, gather=0)
    fake = [0x7F0000000000] * 4
    st = tp.lib.tp_linear_row_forward_noalloc(ctypes.byref(desc), tp._arr(fake), tp._arr(fake),
                                              None, 0x7F0000000000, 0)
    assert tp.STATUS_NAMES[st] == "TP_ERR_WORKSPACE"
    assert "32" in tp.tp_last_error() or "scratch" in tp.tp_last_error()
