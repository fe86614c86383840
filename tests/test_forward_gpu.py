"""Fused router_forward / router_forward_ex against the oracle.

Expert ids must equal the oracle's except on rows whose oracle key gap is
below 1e-5 (counted); weights within 2e-5 absolute. The fused selection is
also checked bit-exactly against the oracle run on the kernel's own FP32
logits (the telemetry tap), and the fused M=2 table bit-exactly against the
oracle table of the kernel's ids."""
import numpy as np
import pytest

import oracle
from moe_expert_router_02_gb300 import router as R
from moe_expert_router_02_gb300 import synth
from tests.helpers import W_TOL, check_routes, dev, empty_outputs

pytestmark = pytest.mark.gpu


def upload(case):
    t = dict(x=dev(case["x"]), W=dev(case["W"]))
    t["bias"] = None if case["bias"] is None else dev(case["bias"])
    t["scales"] = None if case["scales"] is None else dev(case["scales"])
    return t


def run_case(case, flags=0, table=False, tap=False, t=None):
    import torch
    M, H, E, k = case["M"], case["H"], case["E"], case["k"]
    t = t or upload(case)
    idx, w = empty_outputs(M, k)
    tbl = None
    if table:
        n = 2 * k
        tbl = (torch.full((M // 2, n), -9, dtype=torch.int32, device="cuda"),
               torch.full((M // 2, n), 0xEE, dtype=torch.uint8, device="cuda"),
               torch.full((M // 2, 2, k), 0xEE, dtype=torch.uint8, device="cuda"),
               torch.full((M // 2,), -9, dtype=torch.int32, device="cuda"))
    logits = torch.full((M, E), float("nan"), device="cuda") if tap else None
    opts = R.make_opts(x_dtype=case["x_dtype"], w_dtype=case["w_dtype"], w_scales=t["scales"],
                       w_global_scale=case["g"], table=tbl, out_logits=logits, flags=flags)
    R.router_forward_ex(t["x"], t["W"], t["bias"], M, H, E, k, case["act"], idx, w, opts)
    torch.cuda.synchronize()
    out = dict(idx=idx.cpu().numpy(), w=w.cpu().numpy())
    if table:
        out["table"] = [x.cpu().numpy() for x in tbl]
    if tap:
        out["logits"] = logits.cpu().numpy()
    return out


def run_select_on(lg, k, act, bias):
    import torch
    M, E = lg.shape
    idx, w = empty_outputs(M, k)
    R.router_select(dev(np.ascontiguousarray(lg, dtype=np.float32)),
                    None if bias is None else dev(bias), M, E, k, act, idx, w)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


def check_case(case, flags=0, table=False, expect_regime=None):
    if expect_regime is not None:
        o = R.make_opts(x_dtype=case["x_dtype"], w_dtype=case["w_dtype"],
                        w_scales=1 if case["scales"] is not None else None, flags=flags)
        want = expect_regime if isinstance(expect_regime, tuple) else (expect_regime,)
        assert R.router_regime(case["M"], case["H"], case["E"], case["k"], o) in want
    got = run_case(case, flags=flags, table=table, tap=True)
    ref = oracle.router(case)
    k = case["k"]
    differ = check_routes(got["idx"], got["w"], ref, case)
    # selection stage on the kernel's own logits: bit-exact ids
    lg = got["logits"]
    assert np.all(np.isfinite(lg))
    np.testing.assert_allclose(lg, ref["logits"], rtol=0, atol=1e-4)
    oi, ow, _ = oracle.select(lg.astype(np.float64), k, case["act"], bias=case["bias"])
    assert np.array_equal(got["idx"], oi)
    assert np.max(np.abs(got["w"] - ow)) <= W_TOL
    # qwisp #145 G-A: the fused kernel and the unfused selection stage give
    # bit-identical ids and weights on the same FP32 logits
    si, sw = run_select_on(lg, k, case["act"], case["bias"])
    assert np.array_equal(got["idx"], si)
    assert np.array_equal(got["w"].view(np.uint32), sw.view(np.uint32))
    if table:
        tref = oracle.route_table(got["idx"].reshape(-1, 2, k))
        for name, g, r in zip(("unique", "mask", "map", "count"), got["table"], tref):
            assert np.array_equal(g, r), name
    return differ


C = synth.CONFIGS
SMALL = (R.GBR_REGIME_GEMV, R.GBR_REGIME_GEMV1C)


def test_tiny_fp32_case():
    check_case(synth.make_case(C["C0"], seed=0), expect_regime=R.GBR_REGIME_GENERIC)


@pytest.mark.parametrize("M", [1, 2, 8])
@pytest.mark.parametrize("dup", [0.0, 0.1])
def test_decode_softmax(M, dup):
    case = synth.make_case(C["C1"], M=M, seed=M, dup_frac=dup)
    check_case(case, expect_regime=R.GBR_REGIME_GEMV1C)
    check_case(case, flags=R.GBR_FLAG_NO_SINGLE_CLUSTER, expect_regime=R.GBR_REGIME_GEMV)
    check_case(case, flags=R.GBR_FLAG_FORCE_GENERIC)


@pytest.mark.parametrize("M", [1, 16, 64])
def test_sqrt_softplus_bias(M):
    case = synth.make_case(C["C2"], M=M, seed=10 + M, dup_frac=0.1)
    # one cluster per 4 (M <= 16), 8 (M <= 32) or 16 rows
    check_case(case, expect_regime=R.GBR_REGIME_GEMV1C)
    check_case(case, flags=R.GBR_FLAG_NO_SINGLE_CLUSTER, expect_regime=R.GBR_REGIME_GEMV)


@pytest.mark.parametrize("M", [3, 5, 7, 9, 13, 16, 17, 25, 31, 33, 37, 63])
def test_ragged_M(M):
    check_case(synth.make_case(C["C2"], M=M, seed=M))
    check_case(synth.make_case(C["C1"], M=M, seed=M), flags=R.GBR_FLAG_NO_SINGLE_CLUSTER)


def test_m2_route_table_fused():
    cfg = C["C4"]
    for seed in range(6):
        case = synth.make_case(cfg, M=2, seed=seed)
        if seed % 2 == 0:
            x = case["x"].copy()
            x[1] = x[0]  # identical rows: identical expert sets
            case["x"] = x
        check_case(case, table=True, expect_regime=R.GBR_REGIME_GEMV1C)
        check_case(case, table=True, flags=R.GBR_FLAG_NO_SINGLE_CLUSTER)
        check_case(case, table=True, flags=R.GBR_FLAG_FORCE_GENERIC)
    for M in (4, 6, 8, 10, 16, 18, 26, 64):  # row pairs across 4-, 8- and 16-row groups
        check_case(synth.make_case(cfg, M=M, seed=M), table=True)
        check_case(synth.make_case(cfg, M=M, seed=M), table=True,
                   flags=R.GBR_FLAG_NO_SINGLE_CLUSTER)


def test_exact_tie_from_duplicated_weights_goes_to_lower_index():
    cfg = dict(C["C1"])
    case = synth.make_case(cfg, M=4, seed=3)
    W = synth.bf16_bits_to_f32(case["W"]).copy()
    W[200] = W[37]  # experts 37 and 200 now have identical logits
    x = np.tile(W[37] / np.sqrt(np.mean(W[37] ** 2)), (4, 1)).astype(np.float32)
    case["W"] = synth.f32_to_bf16_bits(W)
    case["x"] = synth.f32_to_bf16_bits(x)
    for k in (1, 2, 8):
        case["k"] = k
        got = run_case(case)
        assert np.all(got["idx"][:, 0] == 37)
        if k >= 2:
            assert np.all(got["idx"][:, 1] == 200)
            np.testing.assert_allclose(got["w"][:, 0], got["w"][:, 1], rtol=0, atol=0)


def test_unfused_pair_matches_fused_bitwise():
    # the unfused pair runs the split-cluster logits kernel, then router_select
    case = synth.make_case(C["C1"], M=8, seed=5)
    a = run_case(case, flags=R.GBR_FLAG_NO_SINGLE_CLUSTER)
    b = run_case(case, flags=R.GBR_FLAG_UNFUSED)
    assert np.array_equal(a["idx"], b["idx"])
    assert np.array_equal(a["w"], b["w"])


@pytest.mark.parametrize("H", [64, 96, 160, 100, 2056])
def test_odd_hidden_sizes(H):
    cfg = dict(C["C1"], H=H)
    check_case(synth.make_case(cfg, M=8, seed=H))


@pytest.mark.parametrize("E,k", [(16, 2), (64, 16), (128, 4), (512, 8), (48, 3), (256, 1)])
def test_expert_counts(E, k):
    cfg = dict(C["C2"], E=E, k=k, H=512)
    check_case(synth.make_case(cfg, M=8, seed=E))
    check_case(synth.make_case(cfg, M=12, seed=E + 2), flags=R.GBR_FLAG_NO_SINGLE_CLUSTER)
    check_case(synth.make_case(cfg, M=33, seed=E + 1))


@pytest.mark.parametrize("H", [32, 6144, 7168])
def test_single_cluster_hidden_limits(H):
    cfg = dict(C["C1"], H=H)
    check_case(synth.make_case(cfg, M=4, seed=H))


@pytest.mark.parametrize("M", [1, 2, 5, 8, 16, 20])
def test_nvfp4_weights_small_M(M):
    case = synth.make_case(C["C2"], M=M, seed=4 + M, w_dtype=synth.NVFP4)
    check_case(case, expect_regime=R.GBR_REGIME_GEMV1C)
    case = synth.make_case(C["C2"], M=M, seed=4, w_dtype=synth.NVFP4, nvfp4_global=0.5)
    check_case(case, table=(M % 2 == 0))
    softmax = dict(C["C1"], H=2048)
    check_case(synth.make_case(softmax, M=M, seed=M, w_dtype=synth.NVFP4))


def test_nvfp4_small_M_other_paths():
    # 32 < M <= 64: a cluster per 16 rows (the last one ragged); H not a
    # multiple of 256 takes the generic kernel
    check_case(synth.make_case(C["C2"], M=33, seed=1, w_dtype=synth.NVFP4),
               expect_regime=R.GBR_REGIME_GEMV1C)
    check_case(synth.make_case(C["C2"], M=64, seed=7, w_dtype=synth.NVFP4), table=True,
               expect_regime=R.GBR_REGIME_GEMV1C)
    check_case(synth.make_case(dict(C["C2"], H=1056), M=4, seed=2, w_dtype=synth.NVFP4),
               expect_regime=R.GBR_REGIME_GENERIC)


def test_repeated_calls_reuse_workspace_and_ticket():
    import torch
    case = synth.make_case(C["C1"], M=8, seed=1)
    t = upload(case)
    first = run_case(case, t=t)
    for _ in range(20):
        again = run_case(case, t=t)
        assert np.array_equal(first["idx"], again["idx"])
        assert np.array_equal(first["w"], again["w"])
    # explicit caller workspace, zero-filled once
    need = R.router_workspace_size(8, case["H"], case["E"], case["k"])
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    idx, w = empty_outputs(8, case["k"])
    for _ in range(3):
        R.router_forward_ex(t["x"], t["W"], None, 8, case["H"], case["E"], case["k"], case["act"],
                            idx, w, R.make_opts(workspace=ws, workspace_bytes=need))
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), first["idx"])


def test_graph_replay_with_changing_inputs():
    import torch
    cfg = C["C4"]
    M, H, E, k = 2, cfg["H"], cfg["E"], cfg["k"]
    base = synth.make_case(cfg, M=M, seed=0)
    # same W and bias in every replay; only the token rows change
    cases = [dict(base, x=synth.make_case(cfg, M=M, seed=s)["x"]) for s in range(8)]
    t = upload(cases[0])
    idx, w = empty_outputs(M, k)
    tbl = (torch.zeros((1, 2 * k), dtype=torch.int32, device="cuda"),
           torch.zeros((1, 2 * k), dtype=torch.uint8, device="cuda"),
           torch.zeros((1, 2, k), dtype=torch.uint8, device="cuda"),
           torch.zeros((1,), dtype=torch.int32, device="cuda"))
    opts = R.make_opts(table=tbl)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        R.router_forward_ex(t["x"], t["W"], t["bias"], M, H, E, k, cfg["act"], idx, w, opts,
                            stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):  # three back-to-back calls inside one graph
            R.router_forward_ex(t["x"], t["W"], t["bias"], M, H, E, k, cfg["act"], idx, w, opts,
                                stream=s)
    for case in cases[1:]:
        t["x"].copy_(dev(case["x"]))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.router(case)
        check_routes(idx.cpu().numpy(), w.cpu().numpy(), ref, case)
        tref = oracle.route_table(idx.cpu().numpy().reshape(1, 2, k))
        for got, r in zip(tbl, tref):
            assert np.array_equal(got.cpu().numpy(), r)
