"""Pins for the FP64 CPU oracle, against things other than the oracle itself:
brute force, closed forms, high-precision decimal evaluation, independent
library routines (numpy argmax/matmul, torch's FP8 decoder), invariants and
the hand-built tie rows in ``tests/golden``. CPU only."""
import decimal
import itertools
import math
import os

import numpy as np
import pytest

import oracle
from moe_expert_router_02_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers
def _dec_sqrt_softplus(z: float) -> decimal.Decimal:
    """sqrt(ln(1 + e^z)) evaluated directly (not the stable form) in decimal
    arithmetic with enough digits that 1 + e^z keeps e^z to 60 digits."""
    with decimal.localcontext() as c:
        c.prec = 60 + int(abs(z) / 2.3)
        zd = decimal.Decimal(z)
        return (decimal.Decimal(1) + zd.exp()).ln().sqrt()


def _brute_topk(keys, k):
    """The ordered k-tuple of distinct experts that is lexicographically
    best under (key desc, index asc), found by enumerating all of them."""
    E = len(keys)
    best = None
    for tup in itertools.permutations(range(E), k):
        score = tuple((-keys[e], e) for e in tup)
        if best is None or score < best[0]:
            best = (score, tup)
    return list(best[1])


def _read_golden_ties():
    rows, expect = [], []
    with open(os.path.join(GOLDEN, "tie_rows_e8_k2.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            lhs, rhs = line.split("|")
            rows.append([float.fromhex(t) if "0x" in t else float(t) for t in lhs.split()])
            expect.append([int(t) for t in rhs.split()])
    return np.array(rows, dtype=np.float32), np.array(expect, dtype=np.int32)


# ---------------------------------------------------------------- number formats
def test_e2m1_all_codes_match_bitfield_definition():
    # E2M1: sign bit 3, exponent bits 2:1 with bias 1, mantissa bit 0;
    # exponent 0 is subnormal (m * 0.5).
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        v = (m * 0.5) if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        assert oracle.e2m1(code) == (-v if s else v)


def test_e4m3_all_codes_match_torch_fp8():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3(c)
        if np.isnan(ref[c]):
            assert np.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])


def test_nvfp4_decoded_products_are_bf16_exact():
    # e2m1 x e4m3 has at most 5 significant bits and stays inside BF16's
    # exponent range, so a BF16 tile holds the product exactly.
    for q in range(16):
        for s in range(256):
            v = oracle.e2m1(q) * oracle.e4m3(s)
            if np.isnan(v):
                continue
            f = np.float32(v)
            assert float(f) == v
            assert synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.array([f])))[0] == f


# ---------------------------------------------------------------- activation
@pytest.mark.parametrize("z", [0.0, 1e-8, -1e-8, 0.5, -0.5, 1.0, -1.0, 2.5, -3.0, 10.0,
                               -10.0, 30.0, -30.0, 80.0, -80.0, 300.0, -300.0])
def test_sqrt_softplus_matches_60_digit_decimal(z):
    ref = float(_dec_sqrt_softplus(z))
    assert oracle.sqrt_softplus(z) == pytest.approx(ref, rel=4e-16, abs=0)


def test_sqrt_softplus_closed_forms():
    assert oracle.sqrt_softplus(0.0) == pytest.approx(math.sqrt(math.log(2.0)), rel=1e-16)
    assert abs(oracle.sqrt_softplus(0.0) - 0.8325546111576977) < 2e-16
    # softplus(z) -> z for large z; -> exp(z) for very negative z
    assert oracle.sqrt_softplus(50.0) == pytest.approx(math.sqrt(50.0), rel=1e-16)
    assert oracle.sqrt_softplus(-60.0) == pytest.approx(math.exp(-30.0), rel=1e-15)


def test_sqrt_softplus_strictly_increasing():
    zs = np.linspace(-40, 40, 20001)
    a = np.array([oracle.sqrt_softplus(z) for z in zs])
    assert np.all(np.diff(a) > 0)


def _dec_sigmoid(z):
    """sigmoid(z) = 1 / (1 + e^-z) in 60-digit decimal."""
    with decimal.localcontext() as c:
        c.prec = 60 + int(abs(z) / 2.3)
        return 1 / (1 + (-decimal.Decimal(float(z))).exp())


@pytest.mark.parametrize("z", [0.0, 1e-8, -1e-8, 0.5, -0.5, 1.0, -1.0, 2.5, -3.0, 10.0,
                               -10.0, 30.0, -30.0, 80.0, -80.0, 300.0, -300.0])
def test_sigmoid_matches_60_digit_decimal(z):
    ref = float(_dec_sigmoid(z))
    assert oracle.sigmoid(z) == pytest.approx(ref, rel=4e-16, abs=0)


def test_sigmoid_closed_forms_and_symmetry():
    assert oracle.sigmoid(0.0) == 0.5
    assert oracle.sigmoid(800.0) == 1.0 and oracle.sigmoid(-800.0) == 0.0
    assert oracle.sigmoid(-60.0) == pytest.approx(math.exp(-60.0), rel=1e-15)
    for z in np.linspace(-20, 20, 401):
        assert oracle.sigmoid(z) + oracle.sigmoid(-z) == pytest.approx(1.0, abs=5e-16)
    zs = np.linspace(-30, 30, 20001)
    a = np.array([oracle.sigmoid(z) for z in zs])
    assert np.all(np.diff(a) > 0)


def test_constructed_sigmoid_bias_rows_against_decimal_brute_force():
    E, k = 12, 3
    rows, bias, kinds = synth.tie_rows_sqrt_softplus(30, E, k, seed=7, std=0.4)
    idx, w, _ = oracle.select(rows.astype(np.float64), k, synth.SIGMOID, bias=bias)
    for r in range(len(rows)):
        a = [_dec_sigmoid(float(z)) for z in rows[r]]
        keys = [a[e] + decimal.Decimal(float(bias[r, e])) for e in range(E)]
        assert list(idx[r]) == _brute_topk(keys, k), kinds[r]
        tot = sum(a[e] for e in idx[r])
        for j, e in enumerate(idx[r]):
            assert w[r, j] == pytest.approx(float(a[e] / tot), rel=1e-14)


# ---------------------------------------------------------------- selection
@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (6, 3), (7, 2), (7, 3)])
def test_topk_matches_brute_force_with_ties(E, k):
    gen = synth.rng(E * 10 + k)
    lg = gen.integers(-2, 3, size=(200, E)).astype(np.float64)  # ties are common
    idx, w, _ = oracle.select(lg, k, synth.SOFTMAX)
    for r in range(len(lg)):
        assert list(idx[r]) == _brute_topk(list(lg[r]), k)


def test_k1_is_first_argmax():
    gen = synth.rng(7)
    lg = gen.integers(-3, 4, size=(500, 16)).astype(np.float64)
    idx, w, _ = oracle.select(lg, 1, synth.SOFTMAX)
    assert np.array_equal(idx[:, 0], np.argmax(lg, axis=1))  # numpy: first max wins
    assert np.all(w == 1.0)


def test_k_equals_E_gives_full_softmax_in_comparator_order():
    scipy_special = pytest.importorskip("scipy.special")
    gen = synth.rng(3)
    lg = gen.normal(size=(50, 12))
    lg[:, 5] = lg[:, 2]  # a tie inside the full order
    idx, w, _ = oracle.select(lg, 12, synth.SOFTMAX)
    p = scipy_special.softmax(lg, axis=1)
    for r in range(len(lg)):
        order = np.lexsort((np.arange(12), -lg[r]))
        assert np.array_equal(idx[r], order)
        np.testing.assert_allclose(w[r], p[r][order], rtol=1e-13)


def test_all_equal_row():
    for act in (synth.SOFTMAX, synth.SQRT_SOFTPLUS):
        lg = np.full((3, 10), 0.25)
        idx, w, _ = oracle.select(lg, 4, act)
        assert np.array_equal(idx, np.tile(np.arange(4), (3, 1)))
        np.testing.assert_allclose(w, 0.25, rtol=1e-15)


def test_golden_hand_built_tie_rows():
    rows, expect = _read_golden_ties()
    idx, w, _ = oracle.select(rows.astype(np.float64), 2, synth.SOFTMAX)
    assert np.array_equal(idx, expect)


@pytest.mark.parametrize("E,k", [(16, 2), (10, 3)])
def test_constructed_softmax_tie_rows_brute_force(E, k):
    rows, kinds = synth.tie_rows_softmax(40, E, k, seed=11)
    idx, w, _ = oracle.select(rows.astype(np.float64), k, synth.SOFTMAX)
    for r in range(len(rows)):
        assert list(idx[r]) == _brute_topk([float(v) for v in rows[r]], k), kinds[r]


def test_constructed_sqrt_softplus_bias_rows_against_decimal_brute_force():
    E, k = 12, 3
    rows, bias, kinds = synth.tie_rows_sqrt_softplus(30, E, k, seed=5)
    idx, w, _ = oracle.select(rows.astype(np.float64), k, synth.SQRT_SOFTPLUS, bias=bias)
    for r in range(len(rows)):
        a = [_dec_sqrt_softplus(float(z)) for z in rows[r]]
        keys = [a[e] + decimal.Decimal(float(bias[r, e])) for e in range(E)]
        assert list(idx[r]) == _brute_topk(keys, k), kinds[r]
        tot = sum(a[e] for e in idx[r])
        for j, e in enumerate(idx[r]):
            assert w[r, j] == pytest.approx(float(a[e] / tot), rel=1e-14)


def _dec_softmax(row):
    """Full-E softmax of one row in 60-digit decimal."""
    with decimal.localcontext() as c:
        c.prec = 60
        ex = [decimal.Decimal(float(z)).exp() for z in row]
        tot = sum(ex)
        return [v / tot for v in ex]


@pytest.mark.parametrize("E,k", [(12, 3), (9, 1), (16, 8)])
def test_constructed_softmax_bias_rows_against_decimal_brute_force(E, k):
    # key = the softmax probability + the bias, found by enumerating every
    # ordered k-tuple in 60-digit decimal; weights the unbiased probabilities
    # renormalised over the chosen k
    rows, bias, kinds = synth.tie_rows_softmax_bias(25, E, k, seed=E + k)
    idx, w, _ = oracle.select(rows.astype(np.float64), k, synth.SOFTMAX, bias=bias)
    for r in range(len(rows)):
        p = _dec_softmax(rows[r])
        keys = [p[e] + decimal.Decimal(float(bias[r, e])) for e in range(E)]
        if k <= 3:
            assert list(idx[r]) == _brute_topk(keys, k), kinds[r]
        else:  # the same order by sorting (key desc, index asc) in decimal
            assert list(idx[r]) == sorted(range(E), key=lambda e: (-keys[e], e))[:k], kinds[r]
        tot = sum(p[e] for e in idx[r])
        for j, e in enumerate(idx[r]):
            assert w[r, j] == pytest.approx(float(p[e] / tot), rel=1e-14)


def test_softmax_bias_random_rows_against_decimal():
    gen = synth.rng(17)
    E, k = 10, 3
    lg = gen.normal(size=(40, E)) * 1.5
    bias = gen.uniform(-0.05, 0.05, size=(40, E)).astype(np.float32)
    idx, w, keys = oracle.select(lg, k, synth.SOFTMAX, bias=bias)
    kfull, score = oracle.keys(lg, synth.SOFTMAX, bias=bias)
    for r in range(len(lg)):
        p = _dec_softmax(lg[r])
        dk = [p[e] + decimal.Decimal(float(bias[r, e])) for e in range(E)]
        assert list(idx[r]) == _brute_topk(dk, k)
        for e in range(E):  # every expert's key and score
            assert kfull[r, e] == pytest.approx(float(dk[e]), rel=0, abs=5e-16)
            assert score[r, e] == pytest.approx(float(p[e]), rel=1e-14)
        np.testing.assert_array_equal(keys[r], kfull[r][np.concatenate([idx[r], [
            sorted(range(E), key=lambda e: (-dk[e], e))[k]]])])


def test_softmax_bias_flips_the_order_but_not_the_weights():
    # expert 1 has the larger probability; expert 0 wins through its bias
    lg = np.array([[1.0, 1.2, -5.0, -5.0]])
    bias = np.array([0.1, 0.0, 0.0, 0.0], dtype=np.float32)
    idx, w, _ = oracle.select(lg, 2, synth.SOFTMAX, bias=bias)
    assert list(idx[0]) == [0, 1]
    np.testing.assert_allclose(w[0], [math.exp(1.0) / (math.exp(1.0) + math.exp(1.2)),
                                      math.exp(1.2) / (math.exp(1.0) + math.exp(1.2))],
                               rtol=1e-14)
    # a zero bias ranks by probability, the order of the logits
    gen = synth.rng(23)
    lg = gen.normal(size=(200, 32))
    a, _, _ = oracle.select(lg, 4, synth.SOFTMAX)
    b, _, _ = oracle.select(lg, 4, synth.SOFTMAX, bias=np.zeros(32, dtype=np.float32))
    assert np.array_equal(a, b)


def test_keys_agree_with_select_for_every_activation():
    gen = synth.rng(29)
    lg = gen.normal(size=(50, 64))
    for act, bias in ((synth.SOFTMAX, None), (synth.SOFTMAX, synth.make_bias(64, 3)),
                      (synth.SQRT_SOFTPLUS, synth.make_bias(64, 4)),
                      (synth.SIGMOID, None)):
        idx, w, skeys = oracle.select(lg, 6, act, bias=bias)
        key, score = oracle.keys(lg, act, bias=bias)
        # the sorted keys are the keys of the chosen experts, then the next
        np.testing.assert_array_equal(np.take_along_axis(key, idx.astype(np.int64), 1),
                                      skeys[:, :6])
        sc = np.take_along_axis(score, idx.astype(np.int64), 1)
        np.testing.assert_allclose(w, sc / sc.sum(axis=1, keepdims=True), rtol=1e-14)


def test_bias_selects_but_does_not_weight():
    # Expert 1 has the larger activation but expert 0 wins through its bias;
    # the weights are the unbiased activations renormalised.
    lg = np.array([[1.0, 1.2, -5.0, -5.0]])
    bias = np.array([0.3, 0.0, 0.0, 0.0], dtype=np.float32)
    idx, w, _ = oracle.select(lg, 2, synth.SQRT_SOFTPLUS, bias=bias)
    assert list(idx[0]) == [0, 1]
    a0, a1 = float(_dec_sqrt_softplus(1.0)), float(_dec_sqrt_softplus(1.2))
    np.testing.assert_allclose(w[0], [a0 / (a0 + a1), a1 / (a0 + a1)], rtol=1e-14)


def test_renormalisation_invariants():
    gen = synth.rng(9)
    lg = gen.normal(size=(300, 256)) * 0.9
    for act, bias in ((synth.SOFTMAX, None),
                      (synth.SOFTMAX, synth.make_bias(256, 3)),
                      (synth.SQRT_SOFTPLUS, synth.make_bias(256, 1)),
                      (synth.SIGMOID, synth.make_bias(256, 2))):
        idx, w, keys = oracle.select(lg, 8, act, bias=bias)
        np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-12)
        assert all(len(set(r)) == 8 for r in idx)
        assert idx.min() >= 0 and idx.max() < 256
        assert np.all(np.diff(keys, axis=1) <= 0)
        if act == synth.SOFTMAX and bias is None:
            assert np.all(np.diff(w, axis=1) <= 0)


def test_softmax_key_is_the_logit_not_the_probability():
    # Far below the maximum, FP64 probabilities underflow to 0 and would
    # tie; the logits still order the experts.
    lg = np.array([[0.0, -800.0, -760.0, -900.0]])
    by_logit, _, _ = oracle.select(lg, 2, synth.SOFTMAX)
    by_prob = oracle.select_by_prob(lg, 2)
    assert list(by_logit[0]) == [0, 2]
    assert list(by_prob[0]) == [0, 1]  # the collapsed tie falls to index order


def test_zero_scores_renormalise_to_uniform():
    lg = np.array([[-1e4, -1e4, -2e4]])
    idx, w, _ = oracle.select(lg, 2, synth.SQRT_SOFTPLUS)
    assert list(idx[0]) == [0, 1]
    np.testing.assert_array_equal(w[0], [0.5, 0.5])


# ---------------------------------------------------------------- gate projection
def test_logits_integer_inputs_exact_against_numpy_int_matmul():
    gen = synth.rng(21)
    M, H, E = 5, 96, 24
    xi = gen.integers(-8, 9, size=(M, H))
    wi = gen.integers(-8, 9, size=(E, H))
    ref = (xi @ wi.T).astype(np.float64)
    for xd, wd in ((synth.F32, synth.F32), (synth.BF16, synth.BF16), (synth.F32, synth.BF16)):
        x = xi.astype(np.float32) if xd == synth.F32 else synth.f32_to_bf16_bits(xi.astype(np.float32))
        w = wi.astype(np.float32) if wd == synth.F32 else synth.f32_to_bf16_bits(wi.astype(np.float32))
        got = oracle.logits(x, xd, w, wd, M, H, E)
        assert np.array_equal(got, ref)


def test_logits_identity_and_single_hot():
    gen = synth.rng(4)
    H = E = 32
    x = gen.normal(size=(3, H)).astype(np.float32)
    got = oracle.logits(x, synth.F32, np.eye(E, dtype=np.float32), synth.F32, 3, H, E)
    assert np.array_equal(got, x.astype(np.float64))
    W = gen.normal(size=(E, H)).astype(np.float32)
    hot = np.zeros((1, H), dtype=np.float32)
    hot[0, 7] = 1.0
    got = oracle.logits(hot, synth.F32, W, synth.F32, 1, H, E)
    assert np.array_equal(got[0], W[:, 7].astype(np.float64))


def test_nvfp4_logits_against_torch_decoded_weights():
    torch = pytest.importorskip("torch")
    gen = synth.rng(8)
    M, H, E = 3, 64, 8
    q = gen.integers(0, 256, size=(E, H // 2)).astype(np.uint8)
    s = gen.integers(0, 0x7F, size=(E, H // 16)).astype(np.uint8)  # no NaN code
    g = 0.75
    xi = gen.integers(-4, 5, size=(M, H)).astype(np.float32)
    e2m1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])
    codes = np.empty((E, H), dtype=np.int64)
    codes[:, 0::2] = q & 15
    codes[:, 1::2] = q >> 4
    sv = torch.from_numpy(s).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    wdec = e2m1[codes] * np.repeat(sv, 16, axis=1)
    ref = g * (xi.astype(np.float64) @ wdec.T)
    got = oracle.logits(xi, synth.F32, q, synth.NVFP4, M, H, E, scales=s, g=g)
    np.testing.assert_allclose(got, ref, rtol=1e-15, atol=0)


def test_nvfp4_rejects_nan_scale():
    q = np.zeros((1, 8), dtype=np.uint8)
    s = np.array([[0x7F]], dtype=np.uint8)
    with pytest.raises(ValueError):
        oracle.logits(np.zeros((1, 16), np.float32), synth.F32, q, synth.NVFP4, 1, 16, 1,
                      scales=s)


# ---------------------------------------------------------------- route table
def _check_table(idx, unique, mask, mp, count):
    G, T, k = idx.shape
    for g in range(G):
        rows = idx[g]
        seen = []
        for t in range(T):
            for s in range(k):
                if rows[t, s] not in seen:
                    seen.append(int(rows[t, s]))
        U = len(seen)
        assert count[g] == U
        assert list(unique[g, :U]) == seen  # encounter order
        assert np.all(unique[g, U:] == -1) and np.all(mask[g, U:] == 0)
        for u, e in enumerate(seen):
            bits = sum(1 << t for t in range(T) if e in rows[t])
            assert mask[g, u] == bits
        for t in range(T):
            for s in range(k):
                u = mp[g, t, s]
                assert unique[g, u] == rows[t, s]  # round trip
                assert (mask[g, u] >> t) & 1


@pytest.mark.parametrize("k", [1, 2, 3])
def test_route_table_exhaustive_pairs_E6(k):
    perms = list(itertools.permutations(range(6), k))
    idx = np.array([[a, b] for a in perms for b in perms], dtype=np.int32)
    unique, mask, mp, count = oracle.route_table(idx)
    assert len(idx) == len(perms) ** 2
    for g in range(len(idx)):
        r0, r1 = set(idx[g, 0]), set(idx[g, 1])
        assert count[g] == len(r0 | r1)
        assert sum(bin(int(m)).count("1") for m in mask[g]) == 2 * k
        assert int(np.sum(mask[g] == 3)) == len(r0 & r1)
    sample = np.random.default_rng(0).choice(len(idx), size=min(len(idx), 1500), replace=False)
    _check_table(idx[sample], unique[sample], mask[sample], mp[sample], count[sample])


def test_route_table_duplicates_and_wider_groups():
    gen = synth.rng(13)
    for T, k in ((2, 6), (1, 4), (4, 3), (8, 16), (3, 5)):
        idx = gen.integers(0, 5, size=(200, T, k)).astype(np.int32)  # heavy duplication
        _check_table(idx, *oracle.route_table(idx))
    dup = np.array([[[3, 3, 3], [3, 3, 3]]], dtype=np.int32)
    unique, mask, mp, count = oracle.route_table(dup)
    assert count[0] == 1 and unique[0, 0] == 3 and mask[0, 0] == 3
    assert np.all(mp == 0)


def test_route_table_generator_categories():
    idx = synth.table_pairs(400, 6, 256, seed=1)
    unique, mask, mp, count = oracle.route_table(idx)
    cat = np.arange(400) % 4
    assert np.all(count[cat == 0] == 6)
    assert np.all(count[cat == 1] == 12)
    assert np.all((count[cat == 2] > 6) & (count[cat == 2] < 12))
    _check_table(idx[:80], unique[:80], mask[:80], mp[:80], count[:80])


# ---------------------------------------------------------------- whole router
def test_router_tiny_case_consistency():
    case = synth.make_case(synth.CONFIGS["C0"], seed=0)
    out = oracle.router(case)
    x = case["x"].astype(np.float64)
    W = case["W"].astype(np.float64)
    np.testing.assert_allclose(out["logits"], x @ W.T, rtol=1e-12, atol=1e-12)
    for r in range(case["M"]):
        assert list(out["idx"][r]) == _brute_topk(list(out["logits"][r]), case["k"])


# ---------------------------------------------------------------- table consumer
def _bits(v):
    return synth.f32_to_bf16_bits(np.asarray(v, dtype=np.float32))


def _val(b):
    return synth.bf16_bits_to_f32(np.asarray(b, dtype=np.uint16))


def test_gather_add_exact_integer_case_through_the_table():
    """Integer expert outputs, weights 1 or 2 and integer shared outputs keep
    every step exact, so the result must be the integer sum over the routes
    read through idx directly; a wrong map (token and slot swapped, the wrong
    unique row) changes it."""
    G, k, D, E = 60, 6, 32, 256
    gen = synth.rng(3)
    idx = synth.table_pairs(G, k, E, seed=4)
    unique, mask, mp, count = oracle.route_table(idx)
    Y = gen.integers(-8, 9, size=(G, E, 2, D)).astype(np.float32)  # every expert's output
    y = np.full((G, 2 * k, 2, D), np.nan, dtype=np.float32)          # unused rows: NaN
    for g in range(G):
        for u in range(count[g]):
            for t in range(2):
                if mask[g, u] >> t & 1:
                    y[g, u, t] = Y[g, unique[g, u], t]
    w = gen.choice([1.0, 2.0], size=(G, 2, k)).astype(np.float32)
    sh = gen.integers(-8, 9, size=(G, 2, D)).astype(np.float32)
    out = _val(oracle.gather_add(_bits(y), mp, w, _bits(sh)))
    want = np.zeros((G, 2, D))
    for g in range(G):
        for t in range(2):
            for s in range(k):
                want[g, t] += w[g, t, s] * Y[g, idx[g, t, s], t]
    np.testing.assert_array_equal(out, want + sh)


def test_gather_add_rounding_chain_and_fma():
    """Hand-worked values. Routed sum 1 + 2^-8 is a BF16 halfway case and
    rounds to 1.0 (even) before the shared 2^-9 is added, so the chain gives
    1.0 where one rounding of the whole sum would give 1 + 2^-7. Slots
    -(1 + 2^-23) and (1 + 2^-23) times 1 + 2^-7 leave 2^-30 with FMA
    accumulation (a separate multiply would round it away to 0)."""
    y = np.zeros((1, 4, 2, 2), dtype=np.float32)
    y[0, 0, 0, 0] = 1.0
    y[0, 1, 0, 0] = 1.0
    y[0, 0, 0, 1] = 1.0 + 2.0 ** -7
    y[0, 1, 0, 1] = 1.0 + 2.0 ** -7
    mp = np.array([[[0, 1], [2, 3]]], dtype=np.uint8)
    w = np.zeros((1, 2, 2), dtype=np.float32)
    sh = np.zeros((1, 2, 2), dtype=np.float32)
    # column 0: weights 1 and 2^-8, shared 2^-9
    # column 1 uses the same weights, so give column 1 its own case via token 1 below
    w[0, 0] = [1.0, 2.0 ** -8]
    sh[0, 0, 0] = 2.0 ** -9
    out = _val(oracle.gather_add(_bits(y), mp, w, _bits(sh)))
    assert out[0, 0, 0] == 1.0
    # token 1: rows 2 and 3 hold 1 + 2^-7; weights -(1 + 2^-23), 1 + 2^-23
    y[0, 2, 1, 0] = 1.0 + 2.0 ** -7
    y[0, 3, 1, 0] = 1.0 + 2.0 ** -7
    w[0, 1] = [-(1.0 + 2.0 ** -23), 1.0 + 2.0 ** -23]
    out = _val(oracle.gather_add(_bits(y), mp, w, _bits(sh)))
    assert out[0, 1, 0] == 2.0 ** -30


def test_gather_add_within_rounding_of_exact_and_row_permutation():
    G, k, D = 40, 6, 64
    y, w, sh = synth.gather_inputs(G, k, D, seed=8)
    idx = synth.table_pairs(G, k, 256, seed=9)
    unique, mask, mp, count = oracle.route_table(idx)
    out = _val(oracle.gather_add(y, mp, w, sh)).astype(np.float64)
    yv = _val(y).astype(np.float64)
    exact = np.zeros((G, 2, D))
    mag = np.zeros((G, 2, D))
    for g in range(G):
        for t in range(2):
            for s in range(k):
                r = yv[g, mp[g, t, s], t]
                exact[g, t] += w[g, t, s] * r
                mag[g, t] += abs(w[g, t, s] * r)
    exact += _val(sh)
    # BF16 rounding twice (2^-9 relative each) plus FP32 accumulation error
    bound = 2.0 ** -8 * (np.abs(exact) + mag) + 2.0 ** -20 * mag + 1e-30
    assert np.all(np.abs(out - exact) <= bound)
    # relabelling the unique rows consistently leaves the result unchanged
    perm = synth.rng(10).permutation(2 * k)
    inv = np.argsort(perm)
    y2 = y[:, perm]
    mp2 = inv[mp].astype(np.uint8)
    np.testing.assert_array_equal(oracle.gather_add(y2, mp2, w, sh), oracle.gather_add(y, mp, w, sh))
