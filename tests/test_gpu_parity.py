"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle, element by element.

Small and ragged shapes are compared in full (several 128 x 256 output tiles, partial tiles in
M, N and K); the full-size workloads are compared on sampled token rows and ffn columns that
the oracle computes one by one; plus the invariants (sharded vs unsharded, fused vs partials,
run-to-run determinism, every output element written, zero tokens).
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from harness import (TOL_BF16, TOL_F32, TOL_SHARDED_VS_UNSHARDED, MlpCase, compare_full, np64,
                     prepare, rel, rel_shards, sample_rows_cols, sampled_gpu, sampled_reference)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import tensor_sharded_linear_bias_gb300 as mod

    return mod


SMALL = wl.MLP_T4096_H1024_F4096_TP2


def full_reference(case):
    f = case.f
    rf = oracle.mlp_forward(f["X"], f["A"], f["a"], f["B"], f["b"], case.n)
    rb = oracle.mlp_backward(f["X"], f["A"], f["a"], f["B"], f["b"], f["dZ"], case.n, rf)
    return rf, rb


# ----------------------------------------------------------------------------- device status
def test_wait_timeout_is_reported(tp):
    import torch

    ws = tp.new_workspace(256)
    tp.tp_check_status(ws)
    tp.tp_selftest_wait_timeout(ws, 2000)
    with pytest.raises(tp.TpError) as e:
        tp.tp_check_status(ws)
    assert e.value.name == "TP_ERR_DEVICE_TIMEOUT"
    tp.tp_workspace_init(ws)
    tp.tp_check_status(ws)
    # the context is still usable
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0


# ----------------------------------------------------------------------------- small MLPs
@pytest.mark.parametrize("T,H,F,n", [
    (128, 64, 512, 2),        # one tile in M, exact K block
    (300, 136, 2 * 296, 2),   # ragged M (300), ragged N (296 of 256), ragged K (136 of 64)
    (513, 264, 4 * 136, 4),   # 4 shards, ragged everywhere
    (64, 512, 520, 1),        # one shard: the unsharded layer
    (1, 8, 16, 2),            # a single token, widths at the minimum
    (130, 72, 8 * 40, 8),     # 8 shards of 40 columns
])
@pytest.mark.parametrize("reduce", [0, 1, 2, 3, 4])
def test_mlp_bf16_small(tp, T, H, F, n, reduce):
    w = SMALL.with_shape(tokens=T, hidden=H, ffn=F, tp_degree=n)
    case = MlpCase(w, reduce).run()
    errs = compare_full(case.outputs(), *full_reference(case))
    assert max(errs.values()) <= TOL_BF16, errs


@pytest.mark.parametrize("reduce", [2, 4])
@pytest.mark.parametrize("split", ["1", "2", "4", "8"])
def test_shard_sum_in_groups(tp, tune, split, reduce):
    """The shard sum split into `split` partial outputs (groups of 8 / split shards each),
    reduced after the GEMM (AUTO) or inside it (OVERLAP); twice in a row, so the second launch
    starts from counters the first one reset."""
    tune.set("shard_split", split)
    w = SMALL.with_shape(tokens=300, hidden=136, ffn=8 * 136, tp_degree=8)
    case = MlpCase(w, reduce).run()
    first = case.outputs()
    errs = compare_full(first, *full_reference(case))
    assert max(errs.values()) <= TOL_BF16, errs
    second = case.run().outputs()
    assert np.array_equal(first["Z"], second["Z"]) and np.array_equal(first["dX"], second["dX"])


@pytest.mark.parametrize("tma3d", ["0", "1"])
@pytest.mark.parametrize("raster", ["0", "1"])
@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("T,H,F,n", [(96, 72, 2 * 136, 2), (300, 136, 2 * 296, 2),
                                     (640, 264, 4 * 392, 4), (392, 192, 2 * 320, 2),
                                     (520, 320, 4 * 448, 4)])
def test_gemm_kernel_variants(tp, tune, pair, raster, tma3d, T, H, F, n):
    """Both tensor-core kernels on every GEMM of the MLP: one SM per 128 x 256 tile, and SM
    pairs (tcgen05 cta_group::2) per 256 x 256 tile, including pairs whose second half of
    the rows lies beyond M; in both tile orders (m fastest, n fastest)."""
    tune.set("gemm_pair", pair)
    tune.set("raster", raster)
    # MN-major operands whose MN size is a multiple of 64 (H = 192, 320; F/n = 320, 448) are
    # loaded as one 3-D TMA box per tile, or as 64-wide 2-D boxes
    tune.set("tma_3d", tma3d)
    for reduce in (0, 2):
        case = MlpCase(SMALL.with_shape(tokens=T, hidden=H, ffn=F, tp_degree=n), reduce).run()
        errs = compare_full(case.outputs(), *full_reference(case))
        assert max(errs.values()) <= TOL_BF16, (reduce, errs)


def test_mlp_fp32_small(tp):
    w = wl.P3_FP32_FWD.with_shape(tokens=70, hidden=100, ffn=4 * 33, tp_degree=4)
    w = wl.dataclasses.replace(w, sigma={**w.sigma, "a": 0.05, "b": 0.05})
    for reduce in (0, 1):
        case = MlpCase(w, reduce).run()
        errs = compare_full(case.outputs(), *full_reference(case))
        assert max(errs.values()) <= TOL_F32, errs


def test_p3_shapes_fp32_forward(tp):
    """The pages' example shapes (768 -> 3072, batch 32, 4 shards) closed by the row layer."""
    w = wl.P3_FP32_FWD
    for reduce in (0, 1):
        case = MlpCase(w, reduce).run(backward=False)
        f = case.f
        rf = oracle.mlp_forward(f["X"], f["A"], f["a"], f["B"], f["b"], w.tp_degree)
        errs = compare_full(case.outputs(backward=False), rf)
        assert max(errs.values()) <= TOL_F32, errs


def test_fp32_split_k(tp, tune):
    """Few tokens: the FFMA GEMMs whose tiles cannot fill the GPU cut their K range over the
    CTAs of a cluster (column forward, row forward with the shard sum, the dY GEMM with the
    GeLU' epilogue, the input gradient) and add the partial tiles in CTA order through
    distributed shared memory. Ragged K per slice and ragged tiles match the oracle to fp32
    accuracy; repeated runs are bit-identical; the unsplit kernel (knob simt_split = 0) agrees
    to fp32 rounding but not bit for bit (the split path did run)."""
    import torch

    w = wl.P3_FP32_FWD.with_shape(tokens=9, hidden=1000, ffn=4 * 300, tp_degree=4)
    w = wl.dataclasses.replace(w, sigma={**w.sigma, "a": 0.05, "b": 0.05})
    case = MlpCase(w, 0).run()
    errs = compare_full(case.outputs(), *full_reference(case))
    assert max(errs.values()) <= TOL_F32, errs
    Z1, dX1, Y1 = case.Z.clone(), case.dX.clone(), [y.clone() for y in case.Ys]
    case.run()
    assert torch.equal(Z1, case.Z) and torch.equal(dX1, case.dX)
    tune.set("simt_split", 0)
    case.run()
    assert rel(np64(case.Z), np64(Z1)) <= TOL_F32 and rel(np64(case.dX), np64(dX1)) <= TOL_F32
    assert not (torch.equal(Z1, case.Z) and torch.equal(dX1, case.dX)
                and all(torch.equal(a, b) for a, b in zip(Y1, case.Ys)))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bias_grads_many_tokens(tp, dtype):
    """Column sums over many tokens and few columns: each 256-column strip is summed by a
    cluster of blocks (ragged row ranges per block, a ragged last strip), then the blocks'
    sums are added in block order; matches the oracle's bias gradients."""
    base = wl.P3_FP32_FWD if dtype == "f32" else SMALL
    w = base.with_shape(tokens=3000, hidden=264, ffn=4 * 72, tp_degree=4)
    case = MlpCase(w, 0).run()
    f = case.f
    fr = oracle.mlp_forward(f["X"], f["A"], f["a"], f["B"], f["b"], case.n)
    br = oracle.mlp_backward(f["X"], f["A"], f["a"], f["B"], f["b"], f["dZ"], case.n, fr)
    tol = TOL_BF16 if dtype == "bf16" else TOL_F32
    errs = {"db": rel(np64(case.db), br["db"]), "da": rel_shards([np64(x) for x in case.da], br["da"])}
    assert max(errs.values()) <= tol, errs


@pytest.mark.parametrize("epi_warps", ["4", "8", "12"])
@pytest.mark.parametrize("T,H,F,n", [(300, 264, 2 * 392, 2), (520, 136, 4 * 136, 4)])
def test_epilogue_warps(tp, tune, epi_warps, T, H, F, n):
    """The SM-pair kernel with 4 epilogue warps (each on all 256 columns of its 32 rows), 8
    (two per TMEM lane quadrant, 128 columns each) or 12 (three per quadrant: 96, 96 and 64
    columns, a ring of 5 K blocks), every epilogue and reduce mode, ragged tiles: matches the
    oracle."""
    tune.set("epi_warps", epi_warps)
    tune.set("gemm_pair", 1)
    for reduce in (0, 2, 4):
        case = MlpCase(SMALL.with_shape(tokens=T, hidden=H, ffn=F, tp_degree=n), reduce).run()
        errs = compare_full(case.outputs(), *full_reference(case))
        assert max(errs.values()) <= TOL_BF16, (reduce, errs)


def test_epilogue_warps_bit_identical(tp, tune):
    """4, 8 and 12 epilogue warps split the same accumulators differently among warps; the
    arithmetic is the same, so every output is bit-identical (GeLU and GeLU' epilogues, fused
    and overlapped shard sums, a ragged last tile)."""
    tune.set("gemm_pair", 1)
    w = SMALL.with_shape(tokens=600, hidden=392, ffn=2 * 264, tp_degree=2)
    for reduce in (0, 4):
        outs = {}
        for e in (4, 8, 12):
            with tp.tuning(epi_warps=e):
                outs[e] = MlpCase(w, reduce).run().outputs()
        for e in (8, 12):
            for k, v in outs[4].items():
                pairs = zip(v, outs[e][k]) if isinstance(v, list) else [(v, outs[e][k])]
                assert all(np.array_equal(a, b) for a, b in pairs), (reduce, e, k)


_ISSUE_VARIANTS = [{"split_loads": 1}, {"split_loads": 0},
                   {"mma_probe": 0, "load_probe": 0},
                   {"mma_probe": 1, "load_probe": 1},
                   {"pdl": 1}, {"pdl": 0}, {"stage_blocks": 1}, {"stage_blocks": 2}]


@pytest.mark.parametrize("epi_warps", ["4", "8", "12"])
def test_issue_loop_variants(tp, tune, epi_warps):
    """The SM-pair kernel's issue loops in every variant: A and B loads from one producer thread
    or two (warp 0 and the last warp), with and without the early looks at the next block's
    barriers (MMA issuer and producers), launched with and without programmatic stream
    serialisation (set-up overlapping the previous kernel), with one or two 64-deep K blocks
    per operand-ring stage (odd K-block counts end on a half stage), for all three operand layouts
    (forward, input-gradient and
    weight-gradient GEMMs), ragged tiles, fused and overlapped shard sums.
    The default matches the oracle; every variant is bit-identical to it (they change which
    thread issues what and when, not the arithmetic)."""
    tune.set("epi_warps", epi_warps)
    tune.set("gemm_pair", 1)
    w = SMALL.with_shape(tokens=600, hidden=392, ffn=2 * 264, tp_degree=2)
    for reduce in (0, 4):
        case = MlpCase(w, reduce).run()
        base = case.outputs()
        errs = compare_full(base, *full_reference(case))
        assert max(errs.values()) <= TOL_BF16, (reduce, errs)
        for env in _ISSUE_VARIANTS:
            with tp.tuning(**env):
                out = MlpCase(w, reduce).run().outputs()
            for k, v in base.items():
                pairs = zip(v, out[k]) if isinstance(v, list) else [(v, out[k])]
                assert all(np.array_equal(a, b) for a, b in pairs), (reduce, env, k)


@pytest.mark.parametrize("T,H,F,n", [
    (300, 136, 2 * 296, 2),    # ragged M, N and K in all four GEMMs
    (600, 392, 2 * 264, 2),
    (520, 264, 4 * 136, 4),
    (257, 200, 16 * 136, 16),  # 16 shards: the most one shared launch takes
    (2048, 512, 2 * 1024, 2),  # more units than pairs: some pairs take two
])
def test_two_gemm_launches(tp, tune, T, H, F, n):
    """The backward's independent GEMMs in one SM-pair launch (dB_i with dY_i, dA_i with dX and
    its shard sum), with the GeLU' epilogue and without an activation: matches the oracle, and
    is bit-identical to separate launches (every tile runs the same K loop and epilogue; the
    split tail, which adds K pieces in another order, is off in both); three steps in a row
    give the same outputs."""
    tune.set("tail_split", 0)
    w = SMALL.with_shape(tokens=T, hidden=H, ffn=F, tp_degree=n)
    for act in (None, tp.TP_ACT_NONE):
        outs = {}
        for dual in (0, 1):
            with tp.tuning(dual=dual):
                case = MlpCase(w, 0, act=act)
                tp.tp_trace_start(64)
                case.run()
                tags = [r["tag"] for r in tp.tp_trace_stop(64)]
                first = case.outputs()
                for _ in range(2):
                    case.run()
                    again = case.outputs()
                    for k, v in first.items():
                        pairs = zip(v, again[k]) if isinstance(v, list) else [(v, again[k])]
                        assert all(np.array_equal(a, b) for a, b in pairs), (dual, act, k)
            shared = {"row_grads", "column_grads"}
            assert shared & set(tags) == (shared if dual else set()), (dual, tags)
            outs[dual] = first
            if act is None and dual:
                errs = compare_full(outs[dual], *full_reference(case))
                assert max(errs.values()) <= TOL_BF16, errs
        for k, v in outs[0].items():
            pairs = zip(v, outs[1][k]) if isinstance(v, list) else [(v, outs[1][k])]
            assert all(np.array_equal(a, b) for a, b in pairs), (act, k)


@pytest.mark.parametrize("dtype,T,H,F,n", [("bf16", 600, 392, 2 * 264, 2),     # shared backward launches
                                           ("bf16", 2048, 512, 8 * 512, 8),    # split tail tiles
                                           ("f32", 32, 768, 4 * 768, 4)])      # few-row fp32 kernel
def test_step_captures_into_a_cuda_graph(tp, dtype, T, H, F, n):
    """A whole step (forward and, for bf16, backward) can be captured into a CUDA graph: the
    library makes no host synchronisation, allocation or device query on the launch path once
    a first call has run, and a replay gives the eager step's outputs bit for bit."""
    import torch

    base = wl.P3_FP32_FWD if dtype == "f32" else SMALL
    w = base.with_shape(tokens=T, hidden=H, ffn=F, tp_degree=n)
    case = MlpCase(w, 2)
    backward = dtype == "bf16"
    case.run(backward=backward)
    eager = case.outputs(backward=backward)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        case.forward()
        if backward:
            case.backward()
    torch.cuda.synchronize()
    for t in [case.Z, case.dX] + case.dA + case.dB + case.da + [case.db]:
        t.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    tp.tp_check_status(case.ws)
    replayed = case.outputs(backward=backward)
    for k, v in eager.items():
        pairs = zip(v, replayed[k]) if isinstance(v, list) else [(v, replayed[k])]
        assert all(np.array_equal(a, b) for a, b in pairs), k


_TAIL_REF = {}


@pytest.mark.parametrize("stage_blocks", [1, 2])
@pytest.mark.parametrize("reduce", [0, 2, 4])
def test_tail_split(tp, tune, reduce, stage_blocks):
    """Tiles of a GEMM's partial last wave of SM pairs run as K pieces on the idle pairs and are
    added in piece order before the epilogue. Ragged tiles in M and N, ragged K per piece, and
    every epilogue (bias + GeLU, fused or grouped shard sum, overlapped sum, GeLU', plain fp32):
    matches the oracle, matches the unsplit kernel (knob tail_split = 0) to fp32 rounding, and
    repeats bit for bit."""
    import torch

    # 81-90 tiles of 256 x 256 per GEMM, K of 33-34 blocks: the tiles beyond the first wave of
    # pairs are split in two on a 76-pair GB300
    w = SMALL.with_shape(tokens=2080, hidden=2056, ffn=2 * 1040, tp_degree=2)
    tune.set("stage_blocks", stage_blocks)   # pieces of odd K-block counts end on a half stage
    outs = {}
    for split in ("1", "0"):
        tune.set("tail_split", split)
        case = MlpCase(w, reduce).run()
        outs[split] = case.outputs()
        if split == "1":
            if "ref" not in _TAIL_REF:
                _TAIL_REF["ref"] = full_reference(case)
            errs = compare_full(outs[split], *_TAIL_REF["ref"])
            assert max(errs.values()) <= TOL_BF16, errs
            Z1, dA1 = case.Z.clone(), [x.clone() for x in case.dA]
            case.run()
            assert torch.equal(Z1, case.Z) and all(torch.equal(a, b) for a, b in zip(dA1, case.dA))
    a, b = outs["1"], outs["0"]
    for k in ("Z", "dX", "db"):
        assert rel(a[k], b[k]) <= TOL_SHARDED_VS_UNSHARDED, k
    for k in ("dA", "dB", "da"):
        assert rel_shards(a[k], b[k]) <= TOL_SHARDED_VS_UNSHARDED, k
    for k in ("H", "Y"):
        assert rel_shards(a[k], b[k]) <= 1e-2, k


# ----------------------------------------------------------------------------- invariants
def test_sharded_matches_unsharded(tp):
    T, H, F = 384, 256, 1024
    outs = {}
    for n in (1, 2, 4, 8):
        w = SMALL.with_shape(tokens=T, hidden=H, ffn=F, tp_degree=n)
        c = MlpCase(w, 0).run()
        o = c.outputs()
        outs[n] = {"Z": o["Z"], "dX": o["dX"], "dA": np.concatenate(o["dA"], 1),
                   "dB": np.concatenate(o["dB"], 0), "da": np.concatenate(o["da"]),
                   "db": o["db"], "H": np.concatenate(o["H"], 1), "Y": np.concatenate(o["Y"], 1)}
    for n in (2, 4, 8):
        for k in outs[1]:
            e = rel(outs[n][k], outs[1][k])
            assert e <= TOL_SHARDED_VS_UNSHARDED, (n, k, e)
        # the column layer's K order does not depend on n: saved activations are identical
        assert np.array_equal(outs[n]["H"], outs[1]["H"])
        assert np.array_equal(outs[n]["Y"], outs[1]["Y"])


def test_fused_matches_partials(tp):
    w = SMALL.with_shape(tokens=320, hidden=200, ffn=4 * 264, tp_degree=4)
    a = MlpCase(w, 0).run().outputs()
    b = MlpCase(w, 1).run().outputs()
    for k in ("Z", "dX"):
        assert rel(a[k], b[k]) <= 1e-5, k
    for k in ("dA", "dB", "da", "H", "Y"):
        assert all(np.array_equal(x, y) for x, y in zip(a[k], b[k])), k


def test_bf16_partials_error_vs_bytes(tp):
    """bf16 shard partials halve the partial bytes; their rounding error stays far inside the
    bf16 tolerance (it is recorded against the fp32-partials error of the same inputs)."""
    w = SMALL.with_shape(tokens=512, hidden=256, ffn=8 * 256, tp_degree=8)
    ref_f, ref_b = None, None
    errs = {}
    for reduce in (1, 3):
        case = MlpCase(w, reduce).run()
        if ref_f is None:
            ref_f, ref_b = full_reference(case)
        o = case.outputs()
        errs[reduce] = (rel(o["Z"], ref_f["Z"]), rel(o["dX"], ref_b["dX"]))
    assert max(errs[3]) <= TOL_BF16, errs
    # the bf16 partials add at most a few bf16 ulps (2^-8 relative) to the fp32-partials error
    assert errs[3][0] <= errs[1][0] + 8 * 2.0 ** -8, errs


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T,H,F,n", [(300, 136, 4 * 88, 4), (4096, 1024, 4096, 2)])
def test_sequence_parallel_mlp(tp, dtype, T, H, F, n):
    """Token-sharded X and dZ in, token-sharded Z and dX out (all-gather before the column
    GEMM, reduce-scatter after the row GEMM), against the oracle's sequence-parallel MLP."""
    import torch

    base = wl.P3_FP32_FWD if dtype == "f32" else SMALL
    w = base.with_shape(tokens=T, hidden=H, ffn=F, tp_degree=n)
    w = wl.dataclasses.replace(w, sigma={**w.sigma, "A": 0.02, "B": 0.02, "a": 0.01, "b": 0.01})
    t, f = prepare(wl.mlp_tensors(w), w.dtype, "cuda")
    cdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    code = tp.TP_BF16 if dtype == "bf16" else tp.TP_F32
    Fs, Ts = F // n, T // n
    A = [t["A"][:, i * Fs:(i + 1) * Fs].contiguous() for i in range(n)]
    a = [t["a"][i * Fs:(i + 1) * Fs].contiguous() for i in range(n)]
    B = [t["B"][i * Fs:(i + 1) * Fs, :].contiguous() for i in range(n)]
    Xs = [t["X"][j * Ts:(j + 1) * Ts].contiguous() for j in range(n)]
    dZs = [t["dZ"][j * Ts:(j + 1) * Ts].contiguous() for j in range(n)]
    desc = tp.MlpDesc(tokens=T, hidden=H, ffn=F, tp_degree=n, dtype=code,
                      act=tp.TP_ACT_GELU_ERF, reduce=tp.TP_REDUCE_AUTO)
    ws = tp.new_workspace(tp.tp_mlp_sp_workspace_size(desc))
    f32 = dict(dtype=torch.float32, device="cuda")
    Zs = [torch.full((Ts, H), float("nan"), **f32) for _ in range(n)]
    Hs = [torch.empty(T, Fs, dtype=cdt, device="cuda") for _ in range(n)]
    Ys = [torch.empty(T, Fs, dtype=cdt, device="cuda") for _ in range(n)]
    tp.tp_mlp_forward_sp(desc, Xs, A, a, B, t["b"], Zs, Hs, Ys, ws)
    dXs = [torch.full((Ts, H), float("nan"), **f32) for _ in range(n)]
    dA = [torch.empty(H, Fs, **f32) for _ in range(n)]
    dB = [torch.empty(Fs, H, **f32) for _ in range(n)]
    da = [torch.empty(Fs, **f32) for _ in range(n)]
    db = torch.empty(H, **f32)
    tp.tp_mlp_backward_sp(desc, Xs, A, B, Hs, Ys, dZs, dXs, dA, da, dB, db, ws)
    tp.tp_check_status(ws)
    torch.cuda.synchronize()
    xs = [f["X"][j * Ts:(j + 1) * Ts] for j in range(n)]
    dzs = [f["dZ"][j * Ts:(j + 1) * Ts] for j in range(n)]
    rf = oracle.mlp_forward_sp(xs, f["A"], f["a"], f["B"], f["b"], n)
    rb = oracle.mlp_backward_sp(xs, f["A"], f["a"], f["B"], f["b"], dzs, n)
    tol = TOL_BF16 if dtype == "bf16" else TOL_F32
    errs = {"Z": rel_shards([np64(z) for z in Zs], rf["Z"]),
            "dX": rel_shards([np64(x) for x in dXs], rb["dX"]),
            "dA": rel_shards([np64(x) for x in dA], rb["dA"]),
            "dB": rel_shards([np64(x) for x in dB], rb["dB"]),
            "da": rel_shards([np64(x) for x in da], rb["da"]), "db": rel(np64(db), rb["db"])}
    assert max(errs.values()) <= tol, errs


def test_deterministic(tp):
    w = SMALL.with_shape(tokens=257, hidden=128, ffn=2 * 384, tp_degree=2)
    for reduce in (0, 1):
        c = MlpCase(w, reduce)
        c.run()
        first = c.outputs()
        c.run()
        second = c.outputs()
        for k, v in first.items():
            if isinstance(v, list):
                assert all(np.array_equal(x, y) for x, y in zip(v, second[k])), k
            else:
                assert np.array_equal(v, second[k]), k


def test_every_output_written(tp):
    w = SMALL.with_shape(tokens=200, hidden=136, ffn=2 * 264, tp_degree=2)
    for reduce in (0, 1):
        o = MlpCase(w, reduce).run().outputs()   # outputs start as NaN
        for k, v in o.items():
            vs = v if isinstance(v, list) else [v]
            assert all(np.isfinite(x).all() for x in vs), k


def test_zero_tokens(tp):
    import torch

    w = SMALL.with_shape(tokens=0, hidden=64, ffn=2 * 64, tp_degree=2)
    c = MlpCase(w, 0).run()
    assert torch.all(torch.cat([x.flatten() for x in c.dA + c.dB + c.da]) == 0)
    assert torch.all(c.db == 0)


# ----------------------------------------------------------------------------- parallel linears
def _lin_inputs(seed, T, K, N, dtype, device):
    raw = {"X": wl.normal(seed, (T, K), 1.0), "W": wl.normal(seed + 1, (K, N), 0.05),
           "bias": wl.normal(seed + 2, (N,), 0.1), "G": wl.normal(seed + 3, (T, N), 1.0)}
    return prepare(raw, dtype, device)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("gather", [0, 1])
@pytest.mark.parametrize("act", [0, 1])
def test_column_linear(tp, dtype, gather, act):
    import torch

    T, K, N, n = 200, 136, 4 * 72, 4
    t, f = _lin_inputs(31, T, K, N, dtype, "cuda")
    Ns = N // n
    cdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    W = [t["W"][:, i * Ns:(i + 1) * Ns].contiguous() for i in range(n)]
    bias = [t["bias"][i * Ns:(i + 1) * Ns].contiguous() for i in range(n)]
    desc = tp.LinearDesc(tokens=T, in_features=K, out_features=N, tp_degree=n,
                         dtype=tp.TP_BF16 if dtype == "bf16" else tp.TP_F32, act=act,
                         reduce=0, gather=gather)
    ws = tp.new_workspace(tp.tp_linear_workspace_size(desc, tp.TP_COLUMN))
    Y = [torch.empty(T, N, dtype=cdt, device="cuda")] if gather else \
        [torch.empty(T, Ns, dtype=cdt, device="cuda") for _ in range(n)]
    Hs = [torch.empty(T, Ns, dtype=cdt, device="cuda") for _ in range(n)] if act else None
    tp.tp_linear_column_forward(desc, t["X"], W, bias, Y, Hs, ws)
    G = t["G"]
    dY = [G] if gather else [G[:, i * Ns:(i + 1) * Ns].contiguous() for i in range(n)]
    dX = torch.empty(T, K, dtype=torch.float32, device="cuda")
    dW = [torch.empty(K, Ns, dtype=torch.float32, device="cuda") for _ in range(n)]
    db = [torch.empty(Ns, dtype=torch.float32, device="cuda") for _ in range(n)]
    tp.tp_linear_column_backward(desc, t["X"], W, Hs, dY, dX, dW, db, ws)
    tp.tp_check_status(ws)
    torch.cuda.synchronize()

    a = "gelu" if act else "none"
    Wr = oracle.split_columns(f["W"], n)
    Hr, Yr = oracle.column_parallel_forward(f["X"], Wr, oracle.split_vector(f["bias"], n), a)
    dXr, dWr, dbr, _ = oracle.column_parallel_backward(f["X"], Wr, Hr,
                                                       oracle.split_columns(f["G"], n), a)
    tol = TOL_BF16 if dtype == "bf16" else TOL_F32
    ygpu = [np64(Y[0])[:, i * Ns:(i + 1) * Ns] for i in range(n)] if gather else \
        [np64(y) for y in Y]
    assert rel_shards(ygpu, Yr) <= tol
    if act:
        assert rel_shards([np64(h) for h in Hs], Hr) <= tol
    assert rel(np64(dX), dXr) <= tol
    assert rel_shards([np64(x) for x in dW], dWr) <= tol
    assert rel_shards([np64(x) for x in db], dbr) <= tol


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("reduce", [0, 1, 2, 3, 4])
def test_row_linear(tp, dtype, reduce):
    if reduce in (3, 4) and dtype == "f32":
        pytest.skip("this reduce mode needs bf16 inputs")
    import torch

    T, K, N, n = 190, 4 * 88, 264, 4
    t, f = _lin_inputs(41, T, K, N, dtype, "cuda")
    Ks = K // n
    X = [t["X"][:, i * Ks:(i + 1) * Ks].contiguous() for i in range(n)]
    W = [t["W"][i * Ks:(i + 1) * Ks, :].contiguous() for i in range(n)]
    desc = tp.LinearDesc(tokens=T, in_features=K, out_features=N, tp_degree=n,
                         dtype=tp.TP_BF16 if dtype == "bf16" else tp.TP_F32, act=0,
                         reduce=reduce, gather=0)
    ws = tp.new_workspace(tp.tp_linear_workspace_size(desc, tp.TP_ROW))
    Z = torch.empty(T, N, dtype=torch.float32, device="cuda")
    tp.tp_linear_row_forward(desc, X, W, t["bias"], Z, ws)
    dX = [torch.empty(T, Ks, dtype=torch.float32, device="cuda") for _ in range(n)]
    dW = [torch.empty(Ks, N, dtype=torch.float32, device="cuda") for _ in range(n)]
    db = torch.empty(N, dtype=torch.float32, device="cuda")
    tp.tp_linear_row_backward(desc, X, W, t["G"], dX, dW, db, ws)
    tp.tp_check_status(ws)
    torch.cuda.synchronize()

    Xr, Wr = oracle.split_columns(f["X"], n), oracle.split_rows(f["W"], n)
    Zr = oracle.row_parallel_forward(Xr, Wr, f["bias"])
    dXr, dWr, dbr = oracle.row_parallel_backward(Xr, Wr, f["G"])
    tol = TOL_BF16 if dtype == "bf16" else TOL_F32
    assert rel(np64(Z), Zr) <= tol
    assert rel_shards([np64(x) for x in dX], dXr) <= tol
    assert rel_shards([np64(x) for x in dW], dWr) <= tol
    assert rel(np64(db), dbr) <= tol


@pytest.mark.parametrize("kind,gather,act", [("column", 0, 0), ("column", 1, 1), ("column", 0, 1),
                                             ("row", 0, 0)])
def test_linear_backward_shared_launches(tp, tune, kind, gather, act):
    """The linear layers' backward with its weight-gradient and input-gradient GEMMs in one
    SM-pair launch (column: dW_i with dX and its shard sum; row: dW_i with dX_i), gathered or
    per-shard dY, with and without the activation: bit-identical to separate launches, and the
    oracle's values."""
    import torch

    tune.set("tail_split", 0)
    n = 4
    if kind == "column":
        T, K, N = 520, 264, 4 * 200
    else:
        T, K, N = 300, 4 * 136, 264
    t, f = _lin_inputs(53, T, K, N, "bf16", "cuda")
    desc = tp.LinearDesc(tokens=T, in_features=K, out_features=N, tp_degree=n, dtype=tp.TP_BF16,
                         act=act, reduce=0, gather=gather)
    ws = tp.new_workspace(tp.tp_linear_workspace_size(desc, tp.TP_COLUMN if kind == "column" else tp.TP_ROW))
    f32 = dict(dtype=torch.float32, device="cuda")
    outs = {}
    for dual in (0, 1):
        with tp.tuning(dual=dual):
            tp.tp_trace_start(16)
            if kind == "column":
                Ns = N // n
                W = [t["W"][:, i * Ns:(i + 1) * Ns].contiguous() for i in range(n)]
                bias = [t["bias"][i * Ns:(i + 1) * Ns].contiguous() for i in range(n)]
                Y = [torch.empty(T, N, dtype=torch.bfloat16, device="cuda")] if gather else \
                    [torch.empty(T, Ns, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
                Hs = [torch.empty(T, Ns, dtype=torch.bfloat16, device="cuda") for _ in range(n)] if act else None
                tp.tp_linear_column_forward(desc, t["X"], W, bias, Y, Hs, ws)
                G = t["G"]
                dY = [G] if gather else [G[:, i * Ns:(i + 1) * Ns].contiguous() for i in range(n)]
                dX = torch.full((T, K), float("nan"), **f32)
                dW = [torch.full((K, Ns), float("nan"), **f32) for _ in range(n)]
                db = [torch.full((Ns,), float("nan"), **f32) for _ in range(n)]
                tp.tp_linear_column_backward(desc, t["X"], W, Hs, dY, dX, dW, db, ws)
                got = [dX] + dW + db
            else:
                Ks = K // n
                X = [t["X"][:, i * Ks:(i + 1) * Ks].contiguous() for i in range(n)]
                W = [t["W"][i * Ks:(i + 1) * Ks, :].contiguous() for i in range(n)]
                dX = [torch.full((T, Ks), float("nan"), **f32) for _ in range(n)]
                dW = [torch.full((Ks, N), float("nan"), **f32) for _ in range(n)]
                db = torch.full((N,), float("nan"), **f32)
                tp.tp_linear_row_backward(desc, X, W, t["G"], dX, dW, db, ws)
                got = dX + dW + [db]
            tags = [r["tag"] for r in tp.tp_trace_stop(16)]
        tp.tp_check_status(ws)
        torch.cuda.synchronize()
        want = "column_grads" if kind == "column" else "row_grads"
        assert (want in tags) == bool(dual), (dual, tags)
        outs[dual] = [np64(x) for x in got]
    assert all(np.array_equal(a, b) for a, b in zip(outs[0], outs[1]))
    a = "gelu" if act else "none"
    if kind == "column":
        Wr = oracle.split_columns(f["W"], n)
        Hr, _ = oracle.column_parallel_forward(f["X"], Wr, oracle.split_vector(f["bias"], n), a)
        dXr, dWr, dbr, _ = oracle.column_parallel_backward(f["X"], Wr, Hr,
                                                           oracle.split_columns(f["G"], n), a)
        assert rel(outs[1][0], dXr) <= TOL_BF16
        assert rel_shards(outs[1][1:1 + n], dWr) <= TOL_BF16
        assert rel_shards(outs[1][1 + n:], dbr) <= TOL_BF16
    else:
        Xr, Wr = oracle.split_columns(f["X"], n), oracle.split_rows(f["W"], n)
        dXr, dWr, dbr = oracle.row_parallel_backward(Xr, Wr, f["G"])
        assert rel_shards(outs[1][:n], dXr) <= TOL_BF16
        assert rel_shards(outs[1][n:2 * n], dWr) <= TOL_BF16
        assert rel(outs[1][-1], dbr) <= TOL_BF16


def test_many_shards(tp):
    w = SMALL.with_shape(tokens=96, hidden=64, ffn=64 * 8, tp_degree=64)
    case = MlpCase(w, 0).run()
    errs = compare_full(case.outputs(), *full_reference(case))
    assert max(errs.values()) <= TOL_BF16, errs


# ----------------------------------------------------------------------------- full-size workloads
@pytest.mark.slow
def test_workload_mlp_4096_1024_4096_tp2_full(tp):
    w = wl.MLP_T4096_H1024_F4096_TP2
    case = MlpCase(w, 0).run()
    errs = compare_full(case.outputs(), *full_reference(case))
    assert max(errs.values()) <= TOL_BF16, errs


@pytest.mark.slow
@pytest.mark.parametrize("reduce", [0, 1, 2, 3, 4])
def test_workload_gpt3_mlp_slice_sampled(tp, reduce):
    """The bench's workload and launch configuration (reduce=2 is the AUTO mode it times)."""
    w = wl.GPT3_MLP_T2048_TP8
    case = MlpCase(w, reduce).run()
    rows, cols = sample_rows_cols(w)
    ref = sampled_reference(oracle, case.f, w.tp_degree, rows, cols)
    got = sampled_gpu(case, rows, cols)
    errs = {k: rel(got[k], ref[k]) for k in ref}
    assert max(errs.values()) <= TOL_BF16, errs


@pytest.mark.slow
@pytest.mark.parametrize("n,T", [(1, 512), (8, 16384), (2, 2048), (4, 8192)])
def test_workload_sweep_sampled(tp, n, T):
    w = wl.SWEEP_H8192_F28672.with_shape(tokens=T, tp_degree=n)
    case = MlpCase(w, 2).run()
    rows, cols = sample_rows_cols(w, nrows=4, ncols=4)
    ref = sampled_reference(oracle, case.f, n, rows, cols)
    got = sampled_gpu(case, rows, cols)
    errs = {k: rel(got[k], ref[k]) for k in ref}
    assert max(errs.values()) <= TOL_BF16, errs


@pytest.mark.slow
@pytest.mark.parametrize("reduce", [0, 1, 2, 4])
def test_workload_attention_projections(tp, reduce):
    """Fused QKV (column parallel over heads) and output projection (row parallel), with the
    shard sums fused, as fp32 partials, as AUTO picks them, and overlapped with the GEMM."""
    import torch

    w = wl.ATTN_T4096_H5120_TP8
    n, T, Hm, hd, heads = w.tp_degree, w.tokens, w.hidden, w.head_dim, w.heads
    raw = wl.attn_tensors(w)
    t, f = prepare(raw, "bf16", "cuda")
    # shard buffers (head-split of the fused [Q|K|V] weight), made on the device by slicing
    hw = heads // n * hd
    Wq = [torch.cat([t["Wqkv"][:, blk * Hm + s * hw: blk * Hm + (s + 1) * hw] for blk in range(3)],
                    1).contiguous() for s in range(n)]
    dQ = [torch.cat([t["dQKV"][:, blk * Hm + s * hw: blk * Hm + (s + 1) * hw] for blk in range(3)],
                    1).contiguous() for s in range(n)]
    Cs = [t["C"][:, s * hw:(s + 1) * hw].contiguous() for s in range(n)]
    Wo = [t["Wo"][s * hw:(s + 1) * hw, :].contiguous() for s in range(n)]
    f32 = dict(dtype=torch.float32, device="cuda")
    col = tp.LinearDesc(tokens=T, in_features=Hm, out_features=3 * Hm, tp_degree=n,
                        dtype=tp.TP_BF16, act=0, reduce=reduce, gather=0)
    row = tp.LinearDesc(tokens=T, in_features=Hm, out_features=Hm, tp_degree=n,
                        dtype=tp.TP_BF16, act=0, reduce=reduce, gather=0)
    ws = tp.new_workspace(max(tp.tp_linear_workspace_size(col, tp.TP_COLUMN),
                              tp.tp_linear_workspace_size(row, tp.TP_ROW)))
    QKV = [torch.empty(T, 3 * hw, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    tp.tp_linear_column_forward(col, t["X"], Wq, None, QKV, None, ws)
    O = torch.empty(T, Hm, **f32)
    tp.tp_linear_row_forward(row, Cs, Wo, None, O, ws)
    dX = torch.empty(T, Hm, **f32)
    dWq = [torch.empty(Hm, 3 * hw, **f32) for _ in range(n)]
    tp.tp_linear_column_backward(col, t["X"], Wq, None, dQ, dX, dWq, None, ws)
    dC = [torch.empty(T, hw, **f32) for _ in range(n)]
    dWo = [torch.empty(hw, Hm, **f32) for _ in range(n)]
    tp.tp_linear_row_backward(row, Cs, Wo, t["dO"], dC, dWo, None, ws)
    tp.tp_check_status(ws)
    torch.cuda.synchronize()

    rows = wl.sample_indices(9004, 8, T, must=[0, T - 1])
    fr = oracle.attn_forward(f["X"][rows], f["Wqkv"], f["C"][rows], f["Wo"], heads, hd, n)
    br = oracle.attn_backward(f["X"][rows], f["Wqkv"], f["C"][rows], f["Wo"], f["dQKV"][rows],
                              f["dO"][rows], heads, hd, n)
    errs = {"QKV": rel_shards([np64(q)[rows] for q in QKV], fr["QKV"]),
            "O": rel(np64(O)[rows], fr["O"]),
            "dX": rel(np64(dX)[rows], br["dX"]),
            "dC": rel_shards([np64(c)[rows] for c in dC], br["dC"])}
    # weight gradients: full oracle over all tokens for a few columns of each shard
    Wsh = oracle.qkv_head_shards(f["Wqkv"], heads, hd, n)
    dQsh = oracle.qkv_head_shards(f["dQKV"], heads, hd, n)
    qcols = [0, 1, hw, 2 * hw, 3 * hw - 1]   # first / last column of Q, K and V blocks
    ocols = [0, 1, hw - 1]
    for s in (0, n - 1):
        _, (dw,), _, _ = oracle.column_parallel_backward(f["X"], [Wsh[s][:, qcols]], None,
                                                         [dQsh[s][:, qcols]], "none")
        errs[f"dWqkv{s}"] = rel(np64(dWq[s])[:, qcols], dw)
        Csh = oracle.split_columns(f["C"], n)[s]
        Wosh = oracle.split_rows(f["Wo"], n)[s]
        _, (dwo,), _ = oracle.row_parallel_backward([Csh[:, ocols]], [Wosh[ocols, :]], f["dO"])
        errs[f"dWo{s}"] = rel(np64(dWo[s])[ocols], dwo)
    assert max(errs.values()) <= TOL_BF16, errs


def test_trace_records_every_launch(tp):
    T, H, F, n = 256, 128, 2 * 256, 2
    c = MlpCase(SMALL.with_shape(tokens=T, hidden=H, ffn=F, tp_degree=n), 0)
    with tp.tuning(dual=0):
        tp.tp_trace_start(64)
        c.run()
        recs = tp.tp_trace_stop(64)
    assert [r["tag"] for r in recs] == ["column_fwd", "row_fwd", "row_dgrad", "row_wgrad",
                                        "column_wgrad", "column_dgrad", "bias_grad"]
    assert sum(r["flops"] for r in recs if r["kernel"] == "gemm_tc") == 12 * T * H * F
    assert all(r["ms"] > 0 for r in recs)
    # the backward's independent GEMMs in shared launches: dB_i with dY_i, dA_i with dX
    H = 256
    c = MlpCase(SMALL.with_shape(tokens=T, hidden=H, ffn=F, tp_degree=n), 0)
    with tp.tuning(dual=1):
        tp.tp_trace_start(64)
        c.run()
        recs = tp.tp_trace_stop(64)
    assert [r["tag"] for r in recs] == ["column_fwd", "row_fwd", "row_grads", "column_grads",
                                        "bias_grad"]
    assert sum(r["flops"] for r in recs if r["kernel"] == "gemm_tc") == 12 * T * H * F


# ----------------------------------------------------------------------------- few-token fp32
@pytest.mark.parametrize("few_rows", [None, 0], ids=["auto", "general"])
@pytest.mark.parametrize("T,K,N,n", [
    (32, 768, 4 * 768, 4),     # the pages' example shapes (column: 4 x [768, 768])
    (1, 136, 4 * 72, 4),       # one token, ragged widths (K % 64 != 0: general kernel)
    (7, 3000, 2 * 1030, 2),    # long K split over a cluster, ragged N
    (32, 64, 8 * 40, 8),       # K too short to split
    (19, 1024, 1 * 520, 1),    # one shard
    (17, 640, 2 * 264, 2),     # ragged column tiles (264 = 4 x 64 + 8)
    (32, 4096, 4 * 256, 4),    # 8 K chunks per slice: the whole operand ring
    (8, 8192, 64, 1),          # 16 K chunks per slice: the operand ring wraps twice
    (1, 64, 64, 1),            # one chunk, one tile, one token
])
def test_few_token_fp32_linears(tp, tune, T, K, N, n, few_rows):
    """fp32 linears over at most 32 tokens (the bulk-copy few-row kernel where the shapes fit it,
    else the FFMA GEMM's K split over a cluster; `general` forces the latter): the column
    linear with bias + GeLU (per-shard outputs, and gathered into one buffer), the row linear
    with the shard sum and its bias, against the oracle at the fp32 tolerance; repeated calls
    bit-identical."""
    import torch

    if few_rows is not None:
        tune.set("few_rows", few_rows)

    t, f = _lin_inputs(57, T, K, N, "f32", "cuda")
    Ns, Ks = N // n, K // n if K % n == 0 else None
    desc = tp.LinearDesc(tokens=T, in_features=K, out_features=N, tp_degree=n, dtype=tp.TP_F32,
                         act=tp.TP_ACT_GELU_ERF, reduce=0, gather=0)
    ws = tp.new_workspace(tp.tp_linear_workspace_size(desc, tp.TP_COLUMN))
    W = [t["W"][:, i * Ns:(i + 1) * Ns].contiguous() for i in range(n)]
    bias = [t["bias"][i * Ns:(i + 1) * Ns].contiguous() for i in range(n)]
    Y = [torch.full((T, Ns), float("nan"), device="cuda") for _ in range(n)]
    Hs = [torch.full((T, Ns), float("nan"), device="cuda") for _ in range(n)]
    tp.tp_linear_column_forward(desc, t["X"], W, bias, Y, Hs, ws)
    gdesc = tp.LinearDesc(tokens=T, in_features=K, out_features=N, tp_degree=n, dtype=tp.TP_F32,
                          act=tp.TP_ACT_GELU_ERF, reduce=0, gather=1)
    Yg = torch.full((T, N), float("nan"), device="cuda")
    Hg = [torch.empty(T, Ns, device="cuda") for _ in range(n)]
    tp.tp_linear_column_forward(gdesc, t["X"], W, bias, [Yg], Hg, ws)
    Wc = oracle.split_columns(f["W"], n)
    Hr, Yr = oracle.column_parallel_forward(f["X"], Wc, oracle.split_vector(f["bias"], n), "gelu")
    if Ks is not None:
        rdesc = tp.LinearDesc(tokens=T, in_features=K, out_features=N, tp_degree=n,
                              dtype=tp.TP_F32, act=0, reduce=0, gather=0)
        Xs = [t["X"][:, i * Ks:(i + 1) * Ks].contiguous() for i in range(n)]
        Wr = [t["W"][i * Ks:(i + 1) * Ks, :].contiguous() for i in range(n)]
        Z = torch.full((T, N), float("nan"), device="cuda")
        tp.tp_linear_row_forward(rdesc, Xs, Wr, t["bias"], Z, ws)
        Z2 = torch.empty_like(Z)
        tp.tp_linear_row_forward(rdesc, Xs, Wr, t["bias"], Z2, ws)
    tp.tp_check_status(ws)
    torch.cuda.synchronize()
    assert rel_shards([np64(y) for y in Y], Yr) <= TOL_F32
    assert rel_shards([np64(h) for h in Hs], Hr) <= TOL_F32
    assert rel(np64(Yg), oracle.concat_columns(Yr)) <= TOL_F32
    if Ks is not None:
        assert torch.equal(Z, Z2)
        Zr = oracle.row_parallel_forward(oracle.split_columns(f["X"], n), oracle.split_rows(f["W"], n),
                                         f["bias"])
        assert rel(np64(Z), Zr) <= TOL_F32


@pytest.mark.parametrize("T,K,N,n", [(32, 768, 4 * 768, 4), (5, 1024, 2 * 264, 2)])
def test_few_token_fp32_no_bias_no_act(tp, tune, T, K, N, n):
    """The few-row fp32 kernel's other epilogues: the column linear without bias or
    activation, the row linear without bias (shard sum and per-shard partials), against the
    oracle at the fp32 tolerance, and bit-identical to themselves on a second call."""
    import torch

    t, f = _lin_inputs(91, T, K, N, "f32", "cuda")
    Ns, Ks = N // n, K // n
    desc = tp.LinearDesc(tokens=T, in_features=K, out_features=N, tp_degree=n, dtype=tp.TP_F32,
                         act=0, reduce=0, gather=0)
    ws = tp.new_workspace(max(tp.tp_linear_workspace_size(desc, tp.TP_COLUMN),
                              tp.tp_linear_workspace_size(
                                  tp.LinearDesc(tokens=T, in_features=K, out_features=N,
                                                tp_degree=n, dtype=tp.TP_F32, act=0, reduce=1,
                                                gather=0), tp.TP_ROW)))
    W = [t["W"][:, i * Ns:(i + 1) * Ns].contiguous() for i in range(n)]
    Y = [torch.full((T, Ns), float("nan"), device="cuda") for _ in range(n)]
    tp.tp_linear_column_forward(desc, t["X"], W, None, Y, None, ws)
    Wc = oracle.split_columns(f["W"], n)
    _, Yr = oracle.column_parallel_forward(f["X"], Wc, None, "none")
    Xs = [t["X"][:, i * Ks:(i + 1) * Ks].contiguous() for i in range(n)]
    Wr = [t["W"][i * Ks:(i + 1) * Ks, :].contiguous() for i in range(n)]
    Zr = oracle.row_parallel_forward(oracle.split_columns(f["X"], n), oracle.split_rows(f["W"], n),
                                     None)
    for reduce in (0, 1):
        rdesc = tp.LinearDesc(tokens=T, in_features=K, out_features=N, tp_degree=n,
                              dtype=tp.TP_F32, act=0, reduce=reduce, gather=0)
        Z = torch.full((T, N), float("nan"), device="cuda")
        tp.tp_linear_row_forward(rdesc, Xs, Wr, None, Z, ws)
        Z2 = torch.empty_like(Z)
        tp.tp_linear_row_forward(rdesc, Xs, Wr, None, Z2, ws)
        tp.tp_check_status(ws)
        torch.cuda.synchronize()
        assert torch.equal(Z, Z2), reduce
        assert rel(np64(Z), Zr) <= TOL_F32, reduce
    assert rel_shards([np64(y) for y in Y], Yr) <= TOL_F32
