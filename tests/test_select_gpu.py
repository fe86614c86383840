"""router_select (the selection stage alone) against the oracle on identical
FP32 logits: expert ids bit-exact, weights within 2e-5. Adversarial exact
and one-ulp ties at the k / k+1 boundary for M in {1, 2, 8} follow qwisp
issue #145, "Gates" (G-A)."""
import numpy as np
import pytest

import oracle
from moe_expert_router_02_gb300 import router as R
from moe_expert_router_02_gb300 import synth
from tests.helpers import W_TOL, dev, empty_outputs
from tests.test_oracle import _read_golden_ties

pytestmark = pytest.mark.gpu


def run_select(lg32, k, act, bias=None):
    import torch
    M, E = lg32.shape
    idx, w = empty_outputs(M, k)
    R.router_select(dev(lg32), None if bias is None else dev(bias), M, E, k, act, idx, w)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


def assert_exact(lg32, k, act, bias=None):
    gi, gw = run_select(lg32, k, act, bias)
    oi, ow, _ = oracle.select(lg32.astype(np.float64), k, act, bias=bias)
    bad = np.nonzero(np.any(gi != oi, axis=1))[0]
    assert len(bad) == 0, f"rows {bad[:8]}: gpu {gi[bad[:2]]} oracle {oi[bad[:2]]}"
    assert np.max(np.abs(gw - ow)) <= W_TOL


def test_golden_hand_built_rows():
    rows, expect = _read_golden_ties()
    gi, _ = run_select(rows, 2, synth.SOFTMAX)
    assert np.array_equal(gi, expect)


def test_tiny_case_64_tie_rows():
    rows, _ = synth.tie_rows_softmax(64, 16, 2, seed=0)
    assert_exact(rows, 2, synth.SOFTMAX)


@pytest.mark.parametrize("M", [1, 2, 8])
def test_decode_tie_rows_softmax(M):
    gen = synth.rng(M)
    rows = synth.normal(gen, (max(M, 10) * 10, 256), 0.9)
    rows = synth.inject_tie_rows(rows, 0.1, 8, seed=M)
    for s in range(0, len(rows), M):
        assert_exact(rows[s:s + M], 8, synth.SOFTMAX)


@pytest.mark.parametrize("M", [1, 2, 8])
def test_all_boundary_tie_kinds_softmax(M):
    rows, kinds = synth.tie_rows_softmax(40, 256, 8, seed=100 + M)
    for s in range(0, len(rows), M):
        assert_exact(rows[s:s + M], 8, synth.SOFTMAX)


@pytest.mark.parametrize("spacing", [1, 3, 255, 256, 257, 4096])
@pytest.mark.parametrize("E,k", [(256, 8), (128, 6), (64, 4)])
def test_softmax_keys_close_in_their_top_bits(spacing, E, k):
    """The softmax selection ranks 32-bit words holding a key's top 24 bits
    and falls back to (key, index) rounds when two of its picks, or its
    last pick and the best word left, share those bits. Rows whose 2k
    largest logits sit a multiple of `spacing` ulps apart (some equal,
    spread over lanes and slots) take the fallback (spacing < 256), the
    32-bit rounds alone (spacing >= 256, multiples that cross the
    truncation step) or both; the ids equal the oracle's either way."""
    gen = synth.rng(spacing * 7 + E + k)
    M = 96
    rows = gen.normal(0.0, 1.0, size=(M, E)).astype(np.float32)
    n = 2 * k
    for r in range(M):
        cols = gen.choice(E, n, replace=False)
        steps = np.cumsum(gen.integers(0, 3, size=n))  # some equal neighbours
        base = np.array([4.0 + 0.5 * (r % 5)], dtype=np.float32).view(np.int32)[0]
        rows[r, cols] = (base + steps * spacing).astype(np.int32).view(np.float32)
    assert_exact(rows, k, synth.SOFTMAX)


def test_sqrt_softplus_bias_boundary_ties():
    rows, bias, kinds = synth.tie_rows_sqrt_softplus(60, 256, 6, seed=3)
    for r in range(len(rows)):  # the bias differs per row: one call per row
        assert_exact(rows[r:r + 1], 6, synth.SQRT_SOFTPLUS, bias[r])


def test_sqrt_softplus_bias_random_rows():
    gen = synth.rng(17)
    rows = synth.normal(gen, (2000, 256), 1.3)
    assert_exact(rows, 6, synth.SQRT_SOFTPLUS, synth.make_bias(256, 5))
    assert_exact(rows, 8, synth.SQRT_SOFTPLUS, None)


@pytest.mark.parametrize("E,k", [(16, 16), (8, 8), (40, 3), (100, 7), (300, 16), (512, 9),
                                 (33, 1), (1, 1)])
def test_shapes_and_k_edges(E, k):
    gen = synth.rng(E * 31 + k)
    rows = gen.integers(-3, 4, size=(37, E)).astype(np.float32)  # many ties
    assert_exact(rows, k, synth.SOFTMAX)
    assert_exact(rows, k, synth.SQRT_SOFTPLUS, synth.make_bias(E, 2))
    rows = synth.normal(gen, (37, E), 1.0)
    assert_exact(rows, k, synth.SOFTMAX)


def test_special_values():
    E = 64
    rows = np.zeros((8, E), dtype=np.float32)
    rows[0] = 0.5                                 # all equal
    rows[1, ::2] = -0.0                           # signed zeros
    rows[2] = np.where(np.arange(E) % 3 == 0, 80.0, -80.0)
    rows[3] = np.where(np.arange(E) % 5 == 0, 1e4, -1e4)
    rows[4] = np.float32(1e-45) * (np.arange(E) % 4)  # subnormals
    rows[5] = -np.arange(E, dtype=np.float32) - 1.0  # negative only, decreasing
    rows[6] = np.arange(E, dtype=np.float32)         # increasing ramp
    rows[7] = -1e4                                    # sqrt-softplus scores underflow to 0
    for k in (1, 4, 8):
        assert_exact(rows, k, synth.SOFTMAX)
        assert_exact(rows, k, synth.SQRT_SOFTPLUS)


def test_large_batch_ragged():
    gen = synth.rng(99)
    rows = synth.normal(gen, (4099, 256), 1.0)
    assert_exact(rows, 8, synth.SOFTMAX)
