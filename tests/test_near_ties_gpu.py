"""Near ties between experts with different logits and different biases.

The sqrt-softplus + bias ranking re-keys experts inside the FP32 error band
of the k-th key with double-float keys and sends pairs still too close to
call to FP64 (router_near_tie_keys exposes the double-float key). Here:
the key's error against the oracle's FP64 sqrt(softplus), and boundary
pairs whose FP64 keys differ by 1e-7 down to ~1e-13 (below the
double-float distinctness bound, so the FP64 fallback decides), through
router_select, the small-M fused kernels and the tcgen05 prefill kernel.
The fused kernels see the constructed logits exactly: x and W_gate encode
each logit as three BF16 pieces (W_gate[e, 3e + t] = 2^-8t), and the
logits tap confirms it."""
import functools

import numpy as np
import pytest

import oracle
from moe_expert_router_02_gb300 import router as R
from moe_expert_router_02_gb300 import synth
from tests.helpers import W_TOL, dev, empty_outputs

pytestmark = pytest.mark.gpu

E, K = 256, 6
I_EXP, J_EXP = 10, 200          # the boundary pair; ties go to I_EXP
B_I, B_J = np.float32(0.0125), np.float32(-0.0375)
GAPS = (1e-7, -1e-7, 1e-9, -1e-9, 3e-11, -3e-11, 1e-12, -1e-12, 2e-13, -2e-13)


def near_keys(z, b, act=synth.SQRT_SOFTPLUS):
    import torch
    n = len(z)
    hi = torch.empty(n, dtype=torch.float32, device="cuda")
    lo = torch.empty(n, dtype=torch.float32, device="cuda")
    R.router_near_tie_keys(dev(z), None if b is None else dev(b), n, hi, lo, act=act)
    torch.cuda.synchronize()
    return hi.cpu().numpy(), lo.cpu().numpy()


@pytest.mark.parametrize("act", [synth.SQRT_SOFTPLUS, synth.SIGMOID])
def test_near_tie_key_error_against_fp64(act):
    gen = synth.rng(5)
    z = np.concatenate([gen.uniform(-30, 30, 6000), synth.normal(gen, 6000, 2.0),
                        np.array([0.0, -0.0, 1e-30, -1e-30, 1e-8, -1e-8, 30.0, -30.0,
                                  30.5, -30.5, 45.0, -45.0, 80.0, -80.0])]).astype(np.float32)
    b = np.where(np.arange(len(z)) % 3 == 0, 0.0, gen.uniform(-0.05, 0.05, len(z)))
    b = b.astype(np.float32)
    hi, lo = near_keys(z, b, act)
    f = oracle.sigmoid if act == synth.SIGMOID else oracle.sqrt_softplus
    s = np.array([f(float(v)) for v in z])
    ref = s + b.astype(np.float64)
    got = hi.astype(np.float64) + lo.astype(np.float64)
    err = np.abs(got - ref) / (s + np.abs(ref))
    assert np.max(err) <= 2.0 ** -40, (np.max(err), z[np.argmax(err)])
    # normalised pairs: |lo| <= ulp(hi) / 2
    assert np.all(np.abs(lo) <= np.spacing(np.abs(hi)) / 2)


def test_near_tie_keys_without_bias_and_empty():
    z = np.linspace(-5, 5, 101).astype(np.float32)
    hi, lo = near_keys(z, None)
    s = np.array([oracle.sqrt_softplus(float(v)) for v in z])
    assert np.max(np.abs(hi.astype(np.float64) + lo - s) / s) <= 2.0 ** -40
    R.router_near_tie_keys(None, None, 0, None, None)  # n == 0: no launch, ok


def _s64(z):
    z = np.asarray(z, dtype=np.float64)
    return np.sqrt(np.maximum(z, 0.0) + np.log1p(np.exp(-np.abs(z))))


def boundary_rows(gaps, seed):
    rows, bias, got = _boundary_rows(tuple(gaps), seed)
    return rows.copy(), bias.copy(), got.copy()


@functools.lru_cache(maxsize=None)
def _boundary_rows(gaps, seed):
    """One row per requested key gap g = key_J - key_I (FP64, as the oracle
    computes it): five experts far above, the pair (I_EXP, J_EXP) at ranks
    6/7 with biases B_I, B_J, the rest far below. The pair is found by
    scanning z_I over many floats and solving for z_J."""
    gen = synth.rng(seed)
    rows = np.clip(synth.normal(gen, (len(gaps), E), 0.5), -1.5, 1.5).astype(np.float32)
    got_gaps = []
    zi_all = (np.float32(2.5) + np.arange(2000000, dtype=np.float32) *
              np.float32(2.0 ** -21)).astype(np.float32)
    si = _s64(zi_all)
    # z_J from key_J = key_I + g by Newton on s, then the float neighbours
    for r, g in enumerate(gaps):
        target = si + float(B_I) - float(B_J) + g
        zj = zi_all.astype(np.float64) + (float(B_I) - float(B_J))
        for _ in range(6):
            sp = _s64(zj)
            d = (1.0 / (1.0 + np.exp(-zj))) / (2.0 * sp)
            zj = zj - (sp - target) / d
        best = None
        for step in (-1, 0, 1):
            zj32 = np.nextafter(zj.astype(np.float32), np.float32(np.inf * step)) if step else \
                zj.astype(np.float32)
            res = (_s64(zj32) + float(B_J)) - (si + float(B_I))
            ok = (np.sign(res) == np.sign(g)) & (np.abs(res) <= 2 * abs(g)) & \
                 (np.abs(res) >= abs(g) / 2)
            if np.any(ok):
                c = np.nonzero(ok)[0][0]
                best = (zi_all[c], zj32[c])
                break
        assert best is not None, f"no pair found for gap {g}"
        zi, zj = best
        # the oracle's own FP64 key gap
        gap = (oracle.sqrt_softplus(float(zj)) + float(B_J)) - \
              (oracle.sqrt_softplus(float(zi)) + float(B_I))
        assert np.sign(gap) == np.sign(g) and abs(gap) <= 4 * abs(g), (g, gap)
        got_gaps.append(gap)
        top = gen.choice([e for e in range(E) if e not in (I_EXP, J_EXP)], K - 1, replace=False)
        rows[r, top] = np.float32(6.0) + gen.uniform(0, 2, K - 1).astype(np.float32)
        rows[r, I_EXP], rows[r, J_EXP] = zi, zj
    bias = synth.make_bias(E, seed + 1)
    bias[I_EXP], bias[J_EXP] = B_I, B_J
    return rows, bias, np.array(got_gaps)


def assert_select_exact(rows, bias):
    import torch
    M = rows.shape[0]
    idx, w = empty_outputs(M, K)
    R.router_select(dev(rows), dev(bias), M, E, K, synth.SQRT_SOFTPLUS, idx, w)
    torch.cuda.synchronize()
    oi, ow, _ = oracle.select(rows.astype(np.float64), K, synth.SQRT_SOFTPLUS, bias=bias)
    gi = idx.cpu().numpy()
    assert np.array_equal(gi, oi), (gi, oi)
    assert np.max(np.abs(w.cpu().numpy() - ow)) <= W_TOL
    return oi


def test_select_cross_input_near_ties():
    rows, bias, gaps = boundary_rows(GAPS, seed=11)
    oi = assert_select_exact(rows, bias)
    # the pair really sits at the boundary: rank 6 is J when key_J > key_I
    for r, g in enumerate(gaps):
        assert oi[r, K - 1] == (J_EXP if g > 0 else I_EXP)


def encode_exact(Z):
    """x [M, 3E] and W_gate [E, 3E] BF16 bit patterns with x . W_gate^T = Z
    exactly: Z = p0 + p1 + p2, each piece a BF16 value, x[m, 3e+t] = p_t
    2^8t, W_gate[e, 3e+t] = 2^-8t."""
    M = Z.shape[0]
    H = 3 * E
    x = np.zeros((M, H), dtype=np.float32)
    rest = Z.astype(np.float32)
    for t in range(3):
        piece = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(rest))
        x[:, t::3] = piece * np.float32(2.0 ** (8 * t))
        rest = (rest - piece).astype(np.float32)
    assert np.all(rest == 0)
    W = np.zeros((E, H), dtype=np.float32)
    for t in range(3):
        W[np.arange(E), 3 * np.arange(E) + t] = np.float32(2.0 ** (-8 * t))
    return synth.f32_to_bf16_bits(x), synth.f32_to_bf16_bits(W)


@pytest.mark.parametrize("M,flags,regimes", [
    (8, 0, (R.GBR_REGIME_GEMV1C, R.GBR_REGIME_GEMV)),
    (40, 0, (R.GBR_REGIME_GEMV1C,)),
    (40, R.GBR_FLAG_NO_SINGLE_CLUSTER, (R.GBR_REGIME_GEMV,)),
    (130, 0, (R.GBR_REGIME_TC,)),
])
def test_fused_cross_input_near_ties(M, flags, regimes):
    import torch
    base, bias, _ = boundary_rows(GAPS, seed=23)
    reps = -(-M // len(GAPS))
    Z = np.tile(base, (reps, 1))[:M]
    xb, wb = encode_exact(Z)
    H = xb.shape[1]
    o = R.make_opts(flags=flags)
    assert R.router_regime(M, H, E, K, o) in regimes
    idx, w = empty_outputs(M, K)
    lg = torch.full((M, E), float("nan"), device="cuda")
    opts = R.make_opts(out_logits=lg, flags=flags)
    R.router_forward_ex(dev(xb), dev(wb), dev(bias), M, H, E, K, synth.SQRT_SOFTPLUS, idx, w, opts)
    torch.cuda.synchronize()
    assert np.array_equal(lg.cpu().numpy(), Z), "logits not exact"
    oi, ow, _ = oracle.select(Z.astype(np.float64), K, synth.SQRT_SOFTPLUS, bias=bias)
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert np.max(np.abs(w.cpu().numpy() - ow)) <= W_TOL
    assert R.router_device_status(clear=True) == R.GBR_OK


@pytest.mark.parametrize("act,with_bias", [(synth.SQRT_SOFTPLUS, True), (synth.SQRT_SOFTPLUS, False),
                                           (synth.SOFTMAX, False), (synth.SIGMOID, True)])
def test_prefill_extreme_logits(act, with_bias):
    """Logits far outside the usual range reach the prefill kernel exactly:
    its candidate threshold must hold where expm1f(y^2) overflows (large
    keys), and ties among equal large logits keep the lower index."""
    import torch
    M = 130
    gen = synth.rng(41)
    Z = synth.normal(gen, (M, E), 1.0).astype(np.float32)
    big = np.array([1e4, -1e4, 100.0, -100.0, 88.5, -88.5, 80.0, 30.5, -30.5, 9.5], np.float32)
    for r in range(M):
        kind = r % 5
        cols = gen.choice(E, 12, replace=False)
        if kind == 0:
            Z[r, cols] = gen.choice(big, 12)
        elif kind == 1:
            Z[r] = np.float32(-1e4)
            Z[r, cols] = np.float32(100.0)          # twelve-way tie at the top
        elif kind == 2:
            Z[r] = np.float32(95.0) + gen.uniform(0, 1, E).astype(np.float32)
        elif kind == 3:
            Z[r] = -np.float32(200.0) - gen.uniform(0, 1, E).astype(np.float32)
    bias = synth.make_bias(E, 43) if with_bias else None
    xb, wb = encode_exact(Z)
    H = xb.shape[1]
    assert R.router_regime(M, H, E, K, R.make_opts()) == R.GBR_REGIME_TC
    idx, w = empty_outputs(M, K)
    lg = torch.full((M, E), float("nan"), device="cuda")
    R.router_forward_ex(dev(xb), dev(wb), None if bias is None else dev(bias), M, H, E, K, act,
                        idx, w, R.make_opts(out_logits=lg))
    torch.cuda.synchronize()
    assert np.array_equal(lg.cpu().numpy(), Z), "logits not exact"
    oi, ow, _ = oracle.select(Z.astype(np.float64), K, act, bias=bias)
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert np.max(np.abs(w.cpu().numpy() - ow)) <= W_TOL
    assert R.router_device_status(clear=True) == R.GBR_OK


@pytest.mark.parametrize("act", [synth.SQRT_SOFTPLUS, synth.SIGMOID])
@pytest.mark.parametrize("lo,hi", [(-201.0, -200.0), (-110.0, -95.0)])
def test_select_underflowing_activations(lo, hi, act):
    """Rows whose chosen sqrt-softplus activations are all below FP32's
    range: the weights are ratios of exp(z/2) and come from the log domain
    (to 2e-5 of the oracle's FP64 weights)."""
    import torch
    gen = synth.rng(int(-lo))
    M = 16
    Z = gen.uniform(lo, hi, (M, E)).astype(np.float32)
    for bias in (None, synth.make_bias(E, 3)):
        idx, w = empty_outputs(M, K)
        R.router_select(dev(Z), None if bias is None else dev(bias), M, E, K, act, idx, w)
        torch.cuda.synchronize()
        oi, ow, _ = oracle.select(Z.astype(np.float64), K, act, bias=bias)
        assert np.array_equal(idx.cpu().numpy(), oi)
        assert np.max(np.abs(w.cpu().numpy() - ow)) <= W_TOL
