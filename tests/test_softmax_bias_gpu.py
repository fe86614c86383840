"""Softmax with a selection bias (key = the full-E softmax probability +
bias, weights the unbiased probabilities renormalised; the bias variant of
the softmax route in qwisp issue #145, "Gates", G-C): the selection stage
on identical FP32 logits bit-exact against the oracle, with constructed
exact and one-ulp ties at the k / k+1 boundary for M in {1, 2, 8} (G-A),
and the fused kernels of every small-M regime, the unfused pair and the
generic kernel end to end."""
import numpy as np
import pytest

from moe_expert_router_02_gb300 import router as R
from moe_expert_router_02_gb300 import synth
from tests.test_forward_gpu import check_case
from tests.test_select_gpu import assert_exact

pytestmark = pytest.mark.gpu

C = synth.CONFIGS
SM = synth.SOFTMAX


def test_select_boundary_ties_one_row_per_call():
    rows, bias, kinds = synth.tie_rows_softmax_bias(60, 256, 8, seed=3)
    for r in range(len(rows)):  # the bias differs per row: one call per row
        assert_exact(rows[r:r + 1], 8, SM, bias[r])


@pytest.mark.parametrize("M", [1, 2, 8])
def test_select_boundary_ties_batched(M):
    for seed in range(6):  # every bias kind twice
        rows, bias, kinds = synth.tie_rows_softmax_bias_shared(24, 256, 8, seed=10 * M + seed)
        for s in range(0, len(rows), M):
            assert_exact(rows[s:s + M], 8, SM, bias)


def test_select_random_rows_and_shapes():
    gen = synth.rng(31)
    rows = synth.normal(gen, (3000, 256), 1.0)
    assert_exact(rows, 8, SM, synth.make_bias(256, 6))
    assert_exact(rows, 6, SM, synth.make_bias(256, 7) * 10)  # the bias dominates
    for E, k in ((16, 16), (40, 3), (100, 7), (512, 9), (33, 1), (1, 1)):
        rows = gen.integers(-3, 4, size=(37, E)).astype(np.float32)  # many ties
        assert_exact(rows, k, SM, synth.make_bias(E, 2))
        assert_exact(rows, k, SM, np.zeros(E, dtype=np.float32))


def test_select_special_values():
    E = 64
    rows = np.zeros((6, E), dtype=np.float32)
    rows[0] = 0.5                                          # all equal
    rows[1, ::2] = -0.0                                    # signed zeros
    rows[2] = np.where(np.arange(E) % 3 == 0, 80.0, -80.0)  # probabilities underflow in FP32
    rows[3] = np.where(np.arange(E) % 5 == 0, 1e4, -1e4)
    rows[4] = -np.arange(E, dtype=np.float32) - 1.0
    rows[5] = np.arange(E, dtype=np.float32)
    for k in (1, 4, 8):
        assert_exact(rows, k, SM, np.zeros(E, dtype=np.float32))
        assert_exact(rows, k, SM, synth.make_bias(E, 9))


def sm_case(cfg_name, M, seed, **kw):
    cfg = dict(C[cfg_name], act=SM, bias=True, **kw)
    return synth.make_case(cfg, M=M, seed=seed, dup_frac=0.1)


@pytest.mark.parametrize("M", [1, 2, 8])
def test_decode_every_small_M_kernel(M):
    case = sm_case("C1", M, seed=M)
    check_case(case, expect_regime=R.GBR_REGIME_GEMV1C)
    check_case(case, flags=R.GBR_FLAG_NO_SINGLE_CLUSTER, expect_regime=R.GBR_REGIME_GEMV)
    check_case(case, flags=R.GBR_FLAG_FORCE_GENERIC)
    check_case(case, flags=R.GBR_FLAG_UNFUSED)


def test_split_clusters_table_and_nvfp4():
    check_case(sm_case("C2", 40, seed=4), expect_regime=R.GBR_REGIME_GEMV1C)
    check_case(sm_case("C2", 40, seed=4), flags=R.GBR_FLAG_NO_SINGLE_CLUSTER,
               expect_regime=R.GBR_REGIME_GEMV)
    check_case(sm_case("C4", 2, seed=5), table=True)
    cfg = dict(C["C2"], act=SM, bias=True)
    check_case(synth.make_case(cfg, M=8, seed=6, w_dtype=synth.NVFP4),
               expect_regime=R.GBR_REGIME_GEMV1C)


def test_large_M_falls_back_to_the_generic_kernel():
    # the prefill kernel's epilogue does not take the probability key: the
    # call runs the generic kernel, exactly
    check_case(sm_case("C3", 130, seed=7, H=512))
