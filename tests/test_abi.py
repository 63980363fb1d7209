"""Host-side checks of the C ABI: the library builds and loads, exports every symbol the header
declares, and rejects bad arguments with the documented status before touching the GPU.

No test here launches a kernel or dereferences a pointer: every call either fails validation
(which runs before any CUDA call) or, on a machine without a CUDA device, stops at the
device check.
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tp_mlp.h")
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))


@pytest.fixture(scope="module")
def tp():
    import __graft_entry__

    __graft_entry__.build()
    import tensor_sharded_linear_bias_gb300 as mod

    return mod


def header_functions():
    """Every function declared by a header under include/."""
    names = set()
    for h in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(tp_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_what_the_binding_exports(tp):
    assert header_functions() == sorted(tp.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(tp):
    out = subprocess.run(["nm", "-D", "--defined-only", tp.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(tp_\w+)", out))
    for name in header_functions():
        assert name in exported, name
        assert hasattr(tp.lib, name)


def test_version_and_error_string(tp):
    assert tp.tp_version() == 100
    assert isinstance(tp.tp_last_error(), str)


def mlp(tp, **kw):
    d = dict(tokens=64, hidden=128, ffn=512, tp_degree=4, dtype=tp.TP_BF16,
             act=tp.TP_ACT_GELU_ERF, reduce=tp.TP_REDUCE_FUSED)
    d.update(kw)
    return tp.MlpDesc(**d)


def status_of(fn):
    from tensor_sharded_linear_bias_gb300 import TpError

    try:
        fn()
    except TpError as e:
        return e.name
    return "TP_OK"


def test_workspace_sizes(tp):
    T, H, F, n = 64, 128, 512, 4
    tail = tp.TP_BF16_TAIL_SCRATCH_BYTES   # bf16: split tail tiles after the status block
    assert tail == 80 * 256 * 256 * 4 + 4096
    assert tp.tp_mlp_workspace_size(mlp(tp)) == 256 + tail + T * F * 2
    assert tp.tp_mlp_workspace_size(mlp(tp, dtype=tp.TP_F32)) == 256 + T * F * 4
    part = n * T * H * 4
    assert tp.tp_mlp_workspace_size(mlp(tp, reduce=tp.TP_REDUCE_PARTIALS)) == 256 + tail + T * F * 2 + part
    assert tp.tp_mlp_workspace_size(mlp(tp, reduce=tp.TP_REDUCE_AUTO)) == 256 + tail + T * F * 2 + part
    assert tp.tp_mlp_workspace_size(mlp(tp, reduce=tp.TP_REDUCE_PARTIALS_BF16)) == \
        256 + tail + T * F * 2 + part // 2
    counters = 256   # (64 / 32) x (128 / 256 -> 1) ints, rounded up to 256 bytes
    assert tp.tp_mlp_workspace_size(mlp(tp, reduce=tp.TP_REDUCE_OVERLAP)) == \
        256 + tail + T * F * 2 + part + counters
    col = tp.LinearDesc(tokens=32, in_features=768, out_features=3072, tp_degree=4,
                        dtype=tp.TP_F32, act=0, reduce=0, gather=1)
    assert tp.tp_linear_workspace_size(col, tp.TP_COLUMN) == 256
    row = tp.LinearDesc(tokens=32, in_features=3072, out_features=768, tp_degree=4,
                        dtype=tp.TP_F32, act=0, reduce=tp.TP_REDUCE_PARTIALS, gather=0)
    assert tp.tp_linear_workspace_size(row, tp.TP_ROW) == 256 + 4 * 32 * 768 * 4


@pytest.mark.parametrize("kw,expected", [
    (dict(tp_degree=0), "TP_ERR_SHAPE"),
    (dict(tp_degree=65), "TP_ERR_SHAPE"),
    (dict(ffn=510), "TP_ERR_INDIVISIBLE"),
    (dict(hidden=0), "TP_ERR_SHAPE"),
    (dict(tokens=-1), "TP_ERR_SHAPE"),
    (dict(hidden=130), "TP_ERR_ALIGN"),          # bf16 widths must be multiples of 8
    (dict(ffn=4 * 130), "TP_ERR_ALIGN"),         # ... including the shard width
    (dict(dtype=7), "TP_ERR_DTYPE"),
    (dict(act=3), "TP_ERR_DTYPE"),
    (dict(reduce=5), "TP_ERR_DTYPE"),
    (dict(reduce=4, dtype=0), "TP_ERR_DTYPE"),     # the overlapped sum needs bf16 inputs
    (dict(reduce=3, dtype=0), "TP_ERR_DTYPE"),     # bf16 partials need bf16 inputs
])
def test_mlp_desc_validation(tp, kw, expected):
    assert status_of(lambda: tp.tp_mlp_workspace_size(mlp(tp, **kw))) == expected


def test_sequence_parallel_workspace(tp):
    d = mlp(tp)   # T=64, H=128, F=512, n=4, bf16
    base = tp.tp_mlp_workspace_size(d)
    base += (-base) % 256
    assert tp.tp_mlp_sp_workspace_size(d) == base + 2 * (64 * 128 * 2) + 2 * (64 * 128 * 4)
    assert status_of(lambda: tp.tp_mlp_sp_workspace_size(mlp(tp, tokens=66))) == "TP_ERR_INDIVISIBLE"


def test_fp32_has_no_width_rule(tp):
    assert tp.tp_mlp_workspace_size(mlp(tp, hidden=130, ffn=4 * 131, dtype=tp.TP_F32)) > 0


def test_linear_desc_validation(tp):
    base = dict(tokens=8, in_features=64, out_features=96, tp_degree=4, dtype=tp.TP_BF16,
                act=0, reduce=0, gather=0)
    ok = tp.LinearDesc(**base)
    assert tp.tp_linear_workspace_size(ok, tp.TP_COLUMN) == 256 + tp.TP_BF16_TAIL_SCRATCH_BYTES
    assert status_of(lambda: tp.tp_linear_workspace_size(
        tp.LinearDesc(**{**base, "out_features": 98}), tp.TP_COLUMN)) == "TP_ERR_INDIVISIBLE"
    assert status_of(lambda: tp.tp_linear_workspace_size(
        tp.LinearDesc(**{**base, "in_features": 66}), tp.TP_ROW)) == "TP_ERR_INDIVISIBLE"
    assert status_of(lambda: tp.tp_linear_workspace_size(
        tp.LinearDesc(**{**base, "act": 1}), tp.TP_ROW)) == "TP_ERR_DTYPE"
    assert status_of(lambda: tp.tp_linear_workspace_size(
        tp.LinearDesc(**{**base, "gather": 1}), tp.TP_ROW)) == "TP_ERR_DTYPE"
    assert status_of(lambda: tp.tp_linear_workspace_size(ok, 5)) == "TP_ERR_DTYPE"


# Fake device addresses: validation rejects the call before anything could use them.
ALIGNED = 0x7F0000000000
WS = 0x7F0000100000


def forward_args(tp, desc, **over):
    n = desc.tp_degree
    args = dict(X=ALIGNED, A=[ALIGNED] * n, a=None, B=[ALIGNED] * n, b=None, Z=ALIGNED,
                Hsave=[ALIGNED] * n, Ysave=[ALIGNED] * n, ws=None)
    args.update(over)
    return args


def call_forward(tp, desc, ws_bytes, **over):
    a = forward_args(tp, desc, **over)
    p = tp._arr
    st = tp.lib.tp_mlp_forward(ctypes.byref(desc), a["X"], p(a["A"]), p(a["a"]), p(a["B"]),
                               a["b"], a["Z"], p(a["Hsave"]), p(a["Ysave"]),
                               a.get("wsp", WS), ws_bytes, 0)
    return tp.STATUS_NAMES[st]


def test_forward_argument_checks(tp):
    d = mlp(tp)
    need = tp.tp_mlp_workspace_size(d)
    assert call_forward(tp, d, need, X=None) == "TP_ERR_NULL"
    assert call_forward(tp, d, need, A=None) == "TP_ERR_NULL"
    assert call_forward(tp, d, need, A=[ALIGNED, ALIGNED, None, ALIGNED]) == "TP_ERR_NULL"
    assert call_forward(tp, d, need, Ysave=None) == "TP_ERR_NULL"
    assert call_forward(tp, d, need, Hsave=None) == "TP_ERR_NULL"   # GeLU needs H saved
    assert call_forward(tp, d, need, X=ALIGNED + 8) == "TP_ERR_ALIGN"
    assert call_forward(tp, d, need, B=[ALIGNED] * 3 + [ALIGNED + 2]) == "TP_ERR_ALIGN"
    assert call_forward(tp, d, need - 1) == "TP_ERR_WORKSPACE"
    assert call_forward(tp, d, need, wsp=None) == "TP_ERR_WORKSPACE"
    assert call_forward(tp, d, need, wsp=WS + 16) == "TP_ERR_ALIGN"
    assert "workspace" in tp.tp_last_error()


def test_valid_call_without_a_device_is_refused(tp):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present: fake pointers must not reach it")
    d = mlp(tp)
    assert call_forward(tp, d, tp.tp_mlp_workspace_size(d)) == "TP_ERR_ARCH"


def test_selftest_argument_checks(tp):
    assert tp.STATUS_NAMES[tp.lib.tp_selftest_wait_timeout(WS, 256, 0, 0)] == "TP_ERR_SHAPE"
    assert tp.STATUS_NAMES[tp.lib.tp_selftest_wait_timeout(None, 256, 10, 0)] == "TP_ERR_WORKSPACE"
    assert tp.STATUS_NAMES[tp.lib.tp_check_status(WS, 16, 0)] == "TP_ERR_WORKSPACE"


def test_product_path_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "tensor_sharded_linear_bias_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.replace("oracle-free", ""), f


def test_header_tail_scratch_matches_binding(tp):
    import re

    text = open(os.path.join(ROOT, "include", "tp_mlp.h")).read()
    m = re.search(r"#define TP_BF16_TAIL_SCRATCH_BYTES \(\(size_t\)([0-9 *+]+)\)", text)
    assert m is not None
    assert eval(m.group(1)) == tp.TP_BF16_TAIL_SCRATCH_BYTES
    kinds = dict((int(v), k) for k, v in re.findall(r"(TP_K_\w+) = (\d+)", text))
    assert {k: v.lower()[5:] for k, v in kinds.items()} == {
        k: v for k, v in tp.KERNEL_NAMES.items()}


def test_layernorm_desc_validation(tp):
    ok = dict(tokens=0, hidden=64, tp_degree=4, dtype=tp.TP_BF16, eps=1e-5)

    def fwd(**kw):
        return status_of(lambda: tp.tp_layernorm_forward(tp.LayerNormDesc(**{**ok, **kw}), None,
                                                         None, None, None, None, None, 0))
    assert fwd(hidden=66) == "TP_ERR_INDIVISIBLE"
    assert fwd(hidden=4 * 12) == "TP_ERR_ALIGN"       # bf16 shard width must be a multiple of 8
    assert fwd(eps=0.0) == "TP_ERR_SHAPE"
    assert fwd(tp_degree=65) == "TP_ERR_SHAPE"
    assert fwd(dtype=9) == "TP_ERR_DTYPE"
    assert fwd(tokens=8) == "TP_ERR_NULL"              # X is required when there are tokens
    assert fwd(dtype=tp.TP_F32, hidden=4 * 12) in ("TP_OK", "TP_ERR_ARCH")  # fp32: any width


def test_binding_refuses_strided_views():
    """Every buffer is read as dense row-major: a column slice or a transpose is refused by the
    binding (ValueError) before any call; raw int addresses and None pass through."""
    import torch

    import tensor_sharded_linear_bias_gb300 as tpm

    base = torch.zeros(4, 6)
    for view in (base[:, :3], base.t(), base[:, ::2]):
        with pytest.raises(ValueError, match="not contiguous"):
            tpm._ptr(view)
    # a row range is still dense: only the device check (no GPU here) refuses it
    with pytest.raises(ValueError, match="device memory"):
        tpm._ptr(base[1:3])
    assert tpm._ptr(None) is None and tpm._ptr(1234) == 1234


def test_binding_checks_device_and_dtype():
    """A host tensor is refused (the kernels read device memory only), and so is a tensor whose
    dtype is not the one its role has for the call's dtype (bf16 inputs with an fp32
    descriptor would be read past their end): ValueError before anything reaches the library."""
    import torch

    import tensor_sharded_linear_bias_gb300 as tpm

    with pytest.raises(ValueError, match="device memory"):
        tpm._ptr(torch.zeros(4, 4))
    tpm._need(torch.bfloat16, "X", None, 7, [None, torch.zeros(2, dtype=torch.bfloat16)])
    with pytest.raises(ValueError, match="X must be torch.bfloat16"):
        tpm._need(torch.bfloat16, "X", [torch.zeros(2, dtype=torch.bfloat16), torch.zeros(2)])
    d = tpm.MlpDesc(tokens=8, hidden=64, ffn=128, tp_degree=2, dtype=tpm.TP_F32, act=1, reduce=0)
    bf = torch.zeros(8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="must be torch.float32"):
        tpm.tp_mlp_forward(d, bf, [bf], [bf], [bf], None, bf, [bf], [bf], None)


def test_tuning_hook_without_environment(tp):
    """Kernel-variant overrides go through the tuning entry points only: setting and reading a
    knob needs no GPU, unknown knobs and values are refused, and no environment variable
    changes what the library picks."""
    src = "".join(open(os.path.join(ROOT, "tensor_sharded_linear_bias_gb300", "csrc", f)).read()
                  for f in os.listdir(os.path.join(ROOT, "tensor_sharded_linear_bias_gb300", "csrc"))
                  if f.endswith((".cu", ".cuh", ".h")))
    assert "getenv" not in src
    for name in tp.TUNE_KNOBS:
        assert tp.tp_tuning_get(name) == tp.TP_TUNE_AUTO
    with tp.tuning(raster=1, tail_waves=3):
        assert tp.tp_tuning_get("raster") == 1 and tp.tp_tuning_get("tail_waves") == 3
    assert tp.tp_tuning_get("raster") == tp.TP_TUNE_AUTO
    assert tp.lib.tp_tuning_set(len(tp.TUNE_KNOBS), 0) == 5       # TP_ERR_DTYPE
    assert tp.lib.tp_tuning_set(-1, 0) == 5
    assert tp.lib.tp_tuning_set(0, -2) == 2                        # TP_ERR_SHAPE
    assert tp.lib.tp_tuning_get(99) == tp.TP_TUNE_AUTO - 1
    assert tp.tp_tuning_get("gemm_pair") == tp.TP_TUNE_AUTO
