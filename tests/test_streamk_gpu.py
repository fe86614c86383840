"""Stream-K form of the tcgen05 prefill router. With fewer 256-row tiles
than CTA pairs the device can hold, the tiles x k-steps units are split
evenly over up to one CTA pair per two SMs (as many as keep each tile
within four groups): a group finishes at most one tile, adding the partial
accumulators other groups published in the workspace.
Every case here is checked against the oracle as in the other prefill tests
(ids, weights, logits, the selection on the kernel's own logits bit-exact,
the unfused selection bit-identical)."""
import os

import numpy as np
import pytest

import oracle
from moe_expert_router_02_gb300 import router as R
from moe_expert_router_02_gb300 import synth
from tests.helpers import check_routes, dev, empty_outputs
from tests.test_forward_gpu import check_case, upload
from tests.test_prefill_gpu import small_prefill

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def groups(case, flags=0):
    o = R.make_opts(x_dtype=case["x_dtype"], w_dtype=case["w_dtype"],
                    w_scales=1 if case["scales"] is not None else None, flags=flags)
    return R.router_tc_groups(case["M"], case["H"], case["E"], case["k"], o)


def test_engaged_on_the_prefill_workload():
    # 64 tiles of 256 rows x 112 k-steps over the device's CTA pairs
    g = R.router_tc_groups(16384, 7168, 256, 8)
    assert 64 < g <= 80
    assert R.router_tc_groups(8192, 7168, 256, 8) == g
    # fewer tiles: fewer groups, so that no tile is split more than four ways
    g16 = R.router_tc_groups(4096, 7168, 256, 8)
    assert 16 < g16 <= 64 and g16 < g
    g2 = R.router_tc_groups(300, 7168, 256, 8)
    assert 2 < g2 <= 8
    # below 256 rows: a pair per tile
    assert R.router_tc_groups(200, 7168, 256, 8) == 0
    # not the prefill kernel
    assert R.router_tc_groups(8, 2048, 256, 8) == 0
    assert R.router_tc_groups(1, 64, 16, 17) == -1


@pytest.mark.parametrize("M,H,E,k,act,bias", [
    (8192 + 77, 1024, 256, 8, synth.SQRT_SOFTPLUS, True),   # ragged last tile
    (8192, 512, 256, 8, synth.SOFTMAX, False),
    (7000, 1024, 128, 6, synth.SIGMOID, True),
    (9000, 768, 64, 4, synth.SQRT_SOFTPLUS, False),
    (6000, 2048, 256, 16, synth.SQRT_SOFTPLUS, True),       # KC = 18 list
    (12000, 512, 256, 2, synth.SOFTMAX, False),
    (300, 2048, 256, 8, synth.SQRT_SOFTPLUS, True),          # two tiles, few groups
    (2000, 7168, 256, 8, synth.SOFTMAX, False),             # eight tiles, long K
])
def test_parity(M, H, E, k, act, bias):
    case = small_prefill(M, H=H, E=E, k=k, act=act, bias=bias, seed=M + H + E + k)
    assert groups(case) > 0
    check_case(case, expect_regime=R.GBR_REGIME_TC)


@pytest.mark.parametrize("glob", [None, 0.25])
def test_nvfp4(glob):
    case = small_prefill(8192 + 130, H=1024, seed=31, w_dtype=synth.NVFP4, glob=glob)
    assert groups(case) > 0
    check_case(case, expect_regime=R.GBR_REGIME_TC)


def test_table_and_tap():
    case = small_prefill(8192, H=1024, k=6, seed=33)
    assert groups(case) > 0
    check_case(case, table=True)


def test_exact_ties_across_partials():
    # duplicated expert rows: equal keys must still go to the lower index
    # when the two logits are summed from different groups' partials
    cfg = dict(synth.CONFIGS["C3"], H=1024)
    case = synth.make_case(cfg, M=8192, seed=5, dup_frac=0.2)
    assert groups(case) > 0
    check_case(case)


def test_epochs_across_launches_and_regimes():
    """Back-to-back launches on one caller workspace: stream-K shapes of
    different sizes (different groups finish different tiles), the M <= 64
    kernels (which use the front of the same workspace), NVFP4 decoding and
    a pair-per-tile launch in between. A partial or a flag left from an
    earlier launch would show up as a wrong route."""
    import torch
    cases = [small_prefill(8192, H=1024, seed=40),
             synth.make_case(synth.CONFIGS["C1"], M=8, seed=41),
             small_prefill(9000, H=768, E=256, seed=42),
             small_prefill(8192 + 130, H=1024, seed=43, w_dtype=synth.NVFP4),
             small_prefill(1000, H=1024, seed=44),
             small_prefill(8192, H=1024, seed=45),
             small_prefill(8192, H=1024, seed=45)]
    probes = [R.make_opts(x_dtype=c["x_dtype"], w_dtype=c["w_dtype"],
                          w_scales=1 if c["scales"] is not None else None) for c in cases]
    need = max(R.router_workspace_size(c["M"], c["H"], c["E"], c["k"], o)
               for c, o in zip(cases, probes))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for c in cases:
        t = upload(c)
        idx, w = empty_outputs(c["M"], c["k"])
        opts = R.make_opts(x_dtype=c["x_dtype"], w_dtype=c["w_dtype"], w_scales=t["scales"],
                           w_global_scale=c["g"], workspace=ws, workspace_bytes=need)
        R.router_forward_ex(t["x"], t["W"], t["bias"], c["M"], c["H"], c["E"], c["k"],
                            c["act"], idx, w, opts)
        torch.cuda.synchronize()
        ref = oracle.router(c)
        check_routes(idx.cpu().numpy(), w.cpu().numpy(), ref, c)
    assert R.router_device_status(clear=True) == R.GBR_OK


def test_graph_replay():
    """Captured launches replayed with new inputs: each launch runs a new
    epoch, so no finisher may take a partial from the launch before."""
    import torch
    c = small_prefill(8192, H=1024, seed=50)
    M, H, E, k = c["M"], c["H"], c["E"], c["k"]
    t = upload(c)
    idx, w = empty_outputs(M, k)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        R.router_forward(t["x"], t["W"], t["bias"], M, H, E, k, c["act"], idx, w, s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(2):  # back to back: the second waits on the first (PDL)
                R.router_forward(t["x"], t["W"], t["bias"], M, H, E, k, c["act"], idx, w, s)
    for seed in (51, 52, 53):
        c2 = small_prefill(8192, H=1024, seed=seed)
        t["x"].copy_(dev(c2["x"]))
        g.replay()
        torch.cuda.synchronize()
        c3 = dict(c, x=c2["x"])
        check_routes(idx.cpu().numpy(), w.cpu().numpy(), oracle.router(c3), c3)
    assert R.router_device_status(clear=True) == R.GBR_OK


def test_single_cta_groups():
    """GBR_FLAG_TC_SINGLE_CTA: one CTA per SM is a group (M = 128 MMAs)."""
    f = R.GBR_FLAG_TC_SINGLE_CTA
    c = small_prefill(8192 + 77, H=1024, seed=60)
    g = groups(c, flags=f)
    assert g > 80, g
    check_case(c, flags=f)
    c = small_prefill(7000, H=1024, E=48, k=3, seed=61)
    assert groups(c, flags=f) > 0
    check_case(c, flags=f)


def test_disabled_by_flag():
    c = small_prefill(8192, H=1024, seed=62)
    assert groups(c, flags=R.GBR_FLAG_TC_NO_STREAMK) == 0
    check_case(c, flags=R.GBR_FLAG_TC_NO_STREAMK)


def test_bitwise_repeatable():
    """Partials reach the finishing pair by two routes (prefetched during the
    main loop, or bulk-copied after it), depending on timing; the additions
    and their order are the same either way, so repeated launches on the
    same inputs give bit-identical logits, ids and weights."""
    import torch
    c = small_prefill(8192 + 77, H=2048, seed=70)
    assert groups(c) > 0
    t = upload(c)
    M, H, E, k = c["M"], c["H"], c["E"], c["k"]
    outs = []
    for _ in range(4):
        idx, w = empty_outputs(M, k)
        lg = torch.full((M, E), float("nan"), device="cuda")
        opts = R.make_opts(out_logits=lg)
        R.router_forward_ex(t["x"], t["W"], t["bias"], M, H, E, k, c["act"], idx, w, opts)
        torch.cuda.synchronize()
        outs.append((lg.cpu().numpy().view(np.uint32), idx.cpu().numpy(),
                     w.cpu().numpy().view(np.uint32)))
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert np.array_equal(a, b)
