"""The sigmoid score with a selection bias (a = 1 / (1 + exp(-z)), key =
a + bias, weights the unbiased a renormalised): the selection stage on
identical FP32 logits bit-exact against the oracle (constructed exact and
one-ulp ties at the k / k+1 boundary, random rows), and the fused kernels
of every regime against the oracle end to end."""
import numpy as np
import pytest

import oracle
from moe_expert_router_02_gb300 import router as R
from moe_expert_router_02_gb300 import synth
from tests.test_forward_gpu import check_case
from tests.test_select_gpu import assert_exact

pytestmark = pytest.mark.gpu

C = synth.CONFIGS
SIG = synth.SIGMOID


def test_select_boundary_ties():
    rows, bias, kinds = synth.tie_rows_sqrt_softplus(60, 256, 6, seed=13, std=0.5)
    for r in range(len(rows)):  # the bias differs per row: one call per row
        assert_exact(rows[r:r + 1], 6, SIG, bias[r])


def test_select_random_rows_and_shapes():
    gen = synth.rng(29)
    rows = synth.normal(gen, (2000, 256), 1.3)
    assert_exact(rows, 6, SIG, synth.make_bias(256, 5))
    assert_exact(rows, 8, SIG, None)
    for E, k in ((16, 16), (40, 3), (512, 9), (1, 1)):
        rows = gen.integers(-3, 4, size=(37, E)).astype(np.float32)  # many ties
        assert_exact(rows, k, SIG, synth.make_bias(E, 2))


def sig_case(cfg_name, M, seed, **kw):
    cfg = dict(C[cfg_name], act=SIG, bias=True, **kw)
    return synth.make_case(cfg, M=M, seed=seed)


@pytest.mark.parametrize("M", [1, 8, 16])
def test_decode_single_cluster(M):
    check_case(sig_case("C2", M, seed=M), expect_regime=(R.GBR_REGIME_GEMV1C, R.GBR_REGIME_GEMV))


def test_decode_split_clusters_and_table():
    check_case(sig_case("C2", 40, seed=3), expect_regime=R.GBR_REGIME_GEMV1C)
    check_case(sig_case("C2", 40, seed=3), flags=R.GBR_FLAG_NO_SINGLE_CLUSTER,
               expect_regime=R.GBR_REGIME_GEMV)
    check_case(sig_case("C4", 2, seed=4), table=True)


@pytest.mark.parametrize("M", [130, 300])
def test_prefill(M):
    check_case(sig_case("C3", M, seed=M, H=512), expect_regime=R.GBR_REGIME_TC)


def test_prefill_nvfp4_and_generic():
    cfg = dict(C["C3"], act=SIG, bias=True, H=1024)
    check_case(synth.make_case(cfg, M=200, seed=5, w_dtype=synth.NVFP4),
               expect_regime=R.GBR_REGIME_TC)
    check_case(sig_case("C2", 4, seed=6), flags=R.GBR_FLAG_FORCE_GENERIC,
               expect_regime=R.GBR_REGIME_GENERIC)


def test_no_timeout_recorded():
    assert R.router_device_status(clear=True) == R.GBR_OK
