"""Seeded synthetic inputs for the fused MoE router.

This module builds inputs only. It holds none of the router's arithmetic
(no gate projection, no activation, no selection, no renormalisation, no
route table), so the oracle and the CUDA path can both take their inputs
from here without sharing any of the method.

Everything is numpy on the host and deterministic for a given seed.
Distributions follow the workloads of the router pages:

* x rows are post-RMSNorm hidden states (qwisp issue #145, "Observation":
  the gate matvec reads ``postNorm[H]``), drawn N(0,1) and divided by their
  root-mean-square, then rounded to BF16 with round-to-nearest-even.
* W_gate is expert-major ``[E, H]`` with N(0, sigma) entries; sigma is the
  standard deviation.
* The selection bias is U(-0.05, 0.05) in FP32 (dense_router_decode commit
  page, "DenseRouterDecodeKernel ... sqrt(softplus) + bias + top-k").
* NVFP4 weights: E2M1 codes, one E4M3 scale per 16-element block along H and
  an FP32 global scale (dense_router_decode commit page, "NVFP4 blockscaled
  GEMM"). Packing: element 2j in the low nibble of byte j, 2j+1 in the high
  nibble; scales are ``[E, H/16]`` row-major.
* Adversarial selection rows place exact ties and one-ulp near ties at the
  k / k+1 boundary by construction (qwisp issue #145, "Gates", G-A).
* M=2 route-table inputs mix identical, disjoint, partly overlapping and
  random expert sets (b70 lab note, "Unique-route router screen").
"""
from __future__ import annotations

import numpy as np

F32, BF16, NVFP4 = 0, 1, 2
SOFTMAX, SQRT_SOFTPLUS, SIGMOID = 0, 1, 2


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------- number formats
def f32_to_bf16_bits(a) -> np.ndarray:
    """Round FP32 values to BF16 (round-to-nearest-even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    """Exact widening of BF16 bit patterns to FP32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _e4m3_positive_values() -> np.ndarray:
    """All finite positive E4M3 magnitudes indexed by their 7-bit code (OCP FP8)."""
    codes = np.arange(127)  # 0x7F is NaN
    e = codes >> 3
    m = codes & 7
    return np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))


def f64_to_e4m3_code(v) -> np.ndarray:
    """Encode non-negative values to E4M3 codes, nearest with ties to even code,
    saturating at 448. Input preparation for NVFP4 scales."""
    tab = _e4m3_positive_values()
    v = np.minimum(np.asarray(v, dtype=np.float64), tab[-1])
    hi = np.clip(np.searchsorted(tab, v, side="left"), 0, len(tab) - 1)
    lo = np.clip(hi - 1, 0, len(tab) - 1)
    dlo = np.abs(v - tab[lo])
    dhi = np.abs(tab[hi] - v)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    return np.where(pick_hi, hi, lo).astype(np.uint8)


_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def f64_to_e2m1_code(v) -> np.ndarray:
    """Encode values to E2M1 4-bit codes, nearest with ties to even code,
    saturating at 6."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), 6.0)
    hi = np.clip(np.searchsorted(_E2M1_MAG, a, side="left"), 0, 7)
    lo = np.clip(hi - 1, 0, 7)
    dlo = np.abs(a - _E2M1_MAG[lo])
    dhi = np.abs(_E2M1_MAG[hi] - a)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    return (code | np.where((v < 0) & (code != 0), 8, 0)).astype(np.uint8)


def quantize_nvfp4(w: np.ndarray, global_scale: float | None = None):
    """Quantise an FP32 ``[E, H]`` matrix to NVFP4.

    Returns ``(q, s, g)``: packed E2M1 bytes ``[E, H/2]``, E4M3 block-scale
    codes ``[E, H/16]`` and the FP32 global scale ``g``. When ``global_scale``
    is None, ``g = amax / (448 * 6)`` so the block scales use the normal E4M3
    range; ``s = E4M3(amax_block / (6 g))`` and ``q = E2M1(w / (s g))``.
    """
    E, H = w.shape
    assert H % 16 == 0
    w64 = w.astype(np.float64)
    g = float(np.float32(global_scale if global_scale is not None
                         else max(np.abs(w64).max(), 1e-30) / (448.0 * 6.0)))
    blocks = w64.reshape(E, H // 16, 16)
    amax = np.abs(blocks).max(axis=2)
    s_code = f64_to_e4m3_code(amax / (6.0 * g))
    s_val = np.concatenate([_e4m3_positive_values(), [np.nan]])[s_code]
    denom = (s_val * g)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = np.where(denom > 0, blocks / denom, 0.0)
    codes = f64_to_e2m1_code(scaled).reshape(E, H)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return np.ascontiguousarray(packed), np.ascontiguousarray(s_code), g


# ---------------------------------------------------------------- tensors
def normal(gen: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return (gen.standard_normal(shape) * std).astype(np.float32)


def rms_rows(x: np.ndarray) -> np.ndarray:
    """Divide each row by its root-mean-square (input recipe for post-norm x)."""
    x64 = x.astype(np.float64)
    r = np.sqrt(np.mean(x64 * x64, axis=1, keepdims=True))
    return (x64 / np.maximum(r, 1e-30)).astype(np.float32)


def make_x(M: int, H: int, seed: int, dtype: int = BF16, rms: bool = True):
    """Token activations ``[M, H]``: FP32 array, or BF16 bits (uint16)."""
    x = normal(rng(seed), (M, H), 1.0)
    if rms:
        x = rms_rows(x)
    return x if dtype == F32 else f32_to_bf16_bits(x)


def make_w(E: int, H: int, seed: int, std: float, dtype: int = BF16):
    """Gate weights ``[E, H]`` expert-major: FP32 array or BF16 bits."""
    w = normal(rng(seed), (E, H), std)
    return w if dtype == F32 else f32_to_bf16_bits(w)


def make_bias(E: int, seed: int, lo: float = -0.05, hi: float = 0.05) -> np.ndarray:
    return rng(seed).uniform(lo, hi, size=E).astype(np.float32)


def duplicate_experts(w: np.ndarray, frac: float, seed: int):
    """Copy row e onto row e' for a fraction of experts so their logits tie
    exactly. Returns the new matrix and the list of (source, copy) pairs."""
    E = w.shape[0]
    gen = rng(seed)
    n = max(1, int(round(frac * E)))
    perm = gen.permutation(E)
    pairs = [(int(perm[2 * i]), int(perm[2 * i + 1])) for i in range(min(n, E // 2))]
    w = w.copy()
    for a, b in pairs:
        w[b] = w[a]
    return w, pairs


# ---------------------------------------------------------------- adversarial rows
TIE_KINDS = ("exact", "near_up", "near_down", "exact_lowfirst", "three_way")


def tie_rows_softmax(n: int, E: int, k: int, seed: int, std: float = 1.0):
    """FP32 logit rows with a constructed tie or one-ulp near tie between the
    k-th and (k+1)-th largest logits. Returns (rows [n, E] float32, kinds).

    Construction (no sorting): the bulk is N(0, std) clipped to
    [-4 std, 4 std]; the two boundary experts get v = 4 std + 1; k-1 "top"
    experts get distinct values above v + 1. Exact ties use the same float;
    near ties move one of the pair by one ulp with nextafter.
    """
    gen = rng(seed)
    rows = np.clip(normal(gen, (n, E), std), -4 * std, 4 * std).astype(np.float32)
    kinds = []
    for r in range(n):
        kind = TIE_KINDS[r % len(TIE_KINDS)]
        kinds.append(kind)
        need = k + 1 + (1 if kind == "three_way" else 0)
        if need > E:
            continue
        perm = gen.permutation(E)
        top, (i, j) = perm[: k - 1], perm[k - 1: k + 1]
        v = np.float32(4 * std + 1.0)
        for t, e in enumerate(top):
            rows[r, e] = np.float32(v + 1.0 + 0.25 * t + gen.uniform(0, 0.1))
        rows[r, i] = v
        if kind in ("exact", "exact_lowfirst"):
            rows[r, j] = v
        elif kind == "near_up":
            rows[r, j] = np.nextafter(v, np.float32(np.inf))
        elif kind == "near_down":
            rows[r, j] = np.nextafter(v, np.float32(-np.inf))
        elif kind == "three_way":
            rows[r, j] = v
            rows[r, perm[k + 1]] = v
    return rows, kinds


def tie_rows_sqrt_softplus(n: int, E: int, k: int, seed: int, std: float = 1.0):
    """Logit rows plus a per-row bias for the sqrt(softplus)+bias key, with
    constructed exact and near ties at the k / k+1 boundary.

    Returns (rows [n, E] float32, bias [n, E] float32, kinds). Boundary pair
    (i, j): equal logit and equal bias (exact key tie); logit one ulp apart
    with equal bias; or equal logit with bias one ulp apart. The bias of
    every other expert is U(-0.05, 0.05).
    """
    gen = rng(seed)
    rows = np.clip(normal(gen, (n, E), std), -4 * std, 4 * std).astype(np.float32)
    bias = gen.uniform(-0.05, 0.05, size=(n, E)).astype(np.float32)
    kinds_all = ("exact", "near_logit_up", "near_logit_down", "near_bias_up", "near_bias_down")
    kinds = []
    for r in range(n):
        kind = kinds_all[r % len(kinds_all)]
        kinds.append(kind)
        if k + 1 > E:
            continue
        perm = gen.permutation(E)
        top, (i, j) = perm[: k - 1], perm[k - 1: k + 1]
        v = np.float32(4 * std + 1.0)
        for t, e in enumerate(top):
            rows[r, e] = np.float32(v + 2.0 + 1.0 * t + gen.uniform(0, 0.1))
        rows[r, i] = v
        rows[r, j] = v
        bias[r, j] = bias[r, i]
        if kind == "near_logit_up":
            rows[r, j] = np.nextafter(v, np.float32(np.inf))
        elif kind == "near_logit_down":
            rows[r, j] = np.nextafter(v, np.float32(-np.inf))
        elif kind == "near_bias_up":
            bias[r, j] = np.nextafter(bias[r, i], np.float32(np.inf))
        elif kind == "near_bias_down":
            bias[r, j] = np.nextafter(bias[r, i], np.float32(-np.inf))
    return rows, bias, kinds


def tie_rows_softmax_bias(n: int, E: int, k: int, seed: int, std: float = 1.0):
    """Logit rows plus a per-row bias for the softmax-probability + bias key,
    with constructed exact and near ties at the k / k+1 boundary.

    Returns (rows [n, E] float32, bias [n, E] float32, kinds). Placement (no
    arithmetic of the key): the bulk is N(0, std) clipped to [-4 std, 4 std]
    with bias U(-0.05, -0.02); the boundary pair (i, j) sits at logit
    v = 4 std + 1 with a common bias b0 ~ U(0.005, 0.015); k-1 top experts
    sit at logits v + 3 + t with bias U(0.04, 0.05). Every top expert's
    probability is then at least e^3 times the pair's and every bulk
    expert's at most 1/e of it, so the pair holds ranks k and k+1 whatever
    the row's denominator. Kinds: equal logit and bias (exact key tie),
    logit one ulp apart, bias one ulp apart.
    """
    gen = rng(seed)
    rows = np.clip(normal(gen, (n, E), std), -4 * std, 4 * std).astype(np.float32)
    bias = gen.uniform(-0.05, -0.02, size=(n, E)).astype(np.float32)
    kinds_all = ("exact", "near_logit_up", "near_logit_down", "near_bias_up", "near_bias_down")
    kinds = []
    for r in range(n):
        kind = kinds_all[r % len(kinds_all)]
        kinds.append(kind)
        if k + 1 > E:
            continue
        perm = gen.permutation(E)
        top, (i, j) = perm[: k - 1], perm[k - 1: k + 1]
        v = np.float32(4 * std + 1.0)
        for t, e in enumerate(top):
            rows[r, e] = np.float32(v + 3.0 + 1.0 * t + gen.uniform(0, 0.1))
            bias[r, e] = np.float32(gen.uniform(0.04, 0.05))
        b0 = np.float32(gen.uniform(0.005, 0.015))
        rows[r, i] = rows[r, j] = v
        bias[r, i] = bias[r, j] = b0
        if kind == "near_logit_up":
            rows[r, j] = np.nextafter(v, np.float32(np.inf))
        elif kind == "near_logit_down":
            rows[r, j] = np.nextafter(v, np.float32(-np.inf))
        elif kind == "near_bias_up":
            bias[r, j] = np.nextafter(b0, np.float32(np.inf))
        elif kind == "near_bias_down":
            bias[r, j] = np.nextafter(b0, np.float32(-np.inf))
    return rows, bias, kinds


def tie_rows_softmax_bias_shared(n: int, E: int, k: int, seed: int, std: float = 1.0):
    """As ``tie_rows_softmax_bias`` with one bias vector for all n rows (a
    batch shares its bias). The boundary pair and the top experts are the
    same in every row; the pair's bias is equal, or one ulp apart up or
    down (by seed); each row's pair logits are equal, or one ulp apart up
    or down (by row). Returns (rows [n, E] float32, bias [E] float32,
    kinds)."""
    gen = rng(seed)
    rows = np.clip(normal(gen, (n, E), std), -4 * std, 4 * std).astype(np.float32)
    bias = gen.uniform(-0.05, -0.02, size=E).astype(np.float32)
    perm = gen.permutation(E)
    top, (i, j) = perm[: k - 1], perm[k - 1: k + 1]
    bias[top] = gen.uniform(0.04, 0.05, size=k - 1).astype(np.float32)
    b0 = np.float32(gen.uniform(0.005, 0.015))
    bias[i] = b0
    bias_kind = ("bias_equal", "bias_up", "bias_down")[seed % 3]
    bias[j] = {"bias_equal": b0, "bias_up": np.nextafter(b0, np.float32(np.inf)),
               "bias_down": np.nextafter(b0, np.float32(-np.inf))}[bias_kind]
    v = np.float32(4 * std + 1.0)
    kinds = []
    for r in range(n):
        logit_kind = ("logit_equal", "logit_up", "logit_down")[r % 3]
        kinds.append(bias_kind + "/" + logit_kind)
        for t, e in enumerate(top):
            rows[r, e] = np.float32(v + 3.0 + 1.0 * t + gen.uniform(0, 0.1))
        rows[r, i] = v
        rows[r, j] = {"logit_equal": v, "logit_up": np.nextafter(v, np.float32(np.inf)),
                      "logit_down": np.nextafter(v, np.float32(-np.inf))}[logit_kind]
    return rows, bias, kinds


def inject_tie_rows(rows: np.ndarray, frac: float, k: int, seed: int) -> np.ndarray:
    """Replace a fraction of logit rows with constructed boundary-tie rows
    (same E, same scale)."""
    n, E = rows.shape
    n_tie = int(round(frac * n))
    if n_tie == 0:
        return rows
    std = float(np.std(rows)) or 1.0
    t, _ = tie_rows_softmax(n_tie, E, k, seed, std)
    out = rows.copy()
    pick = rng(seed + 1).choice(n, size=n_tie, replace=False)
    out[pick] = t
    return out


# ---------------------------------------------------------------- route-table input
def table_pairs(G: int, k: int, E: int, seed: int) -> np.ndarray:
    """``[G, 2, k]`` int32 expert ids (distinct within a row), G groups in
    four equal categories: identical sets (row 1 is a permutation of row 0),
    disjoint sets, sets overlapping in u ~ U{1..k-1} experts, and independent
    random sets."""
    gen = rng(seed)
    out = np.empty((G, 2, k), dtype=np.int32)
    for g in range(G):
        cat = g % 4
        perm = gen.permutation(E)
        r0 = perm[:k]
        if cat == 0:
            r1 = gen.permutation(r0)
        elif cat == 1:
            r1 = perm[k: 2 * k]
        elif cat == 2:
            u = int(gen.integers(1, k)) if k > 1 else 1
            shared = gen.choice(r0, size=u, replace=False)
            r1 = gen.permutation(np.concatenate([shared, perm[k: 2 * k - u]]))
        else:
            r1 = gen.permutation(E)[:k]
        out[g, 0] = r0
        out[g, 1] = r1
    return out


# ---------------------------------------------------------------- workloads
def gather_inputs(G: int, k: int, D: int, seed: int, T: int = 2):
    """Inputs of the table's consumer for G groups of T tokens: expert output
    rows y BF16 bits [G, T*k, T, D] ~ N(0, 1), router weights w FP32
    [G, T, k] (positive, each token's summing to 1), shared expert output
    BF16 bits [G, T, D] ~ N(0, 1)."""
    gen = rng(seed)
    y = f32_to_bf16_bits(normal(gen, (G, T * k, T, D), 1.0))
    w = gen.uniform(0.05, 1.0, size=(G, T, k))
    w = (w / w.sum(axis=2, keepdims=True)).astype(np.float32)
    shared = f32_to_bf16_bits(normal(gen, (G, T, D), 1.0))
    return y, w, shared


CONFIGS = {
    # tiny correctness case: FP32 x and W, softmax, top-2
    "C0": dict(M=4, H=256, E=16, k=2, act=SOFTMAX, x_dtype=F32, w_dtype=F32,
               x_std=1.0, w_std=0.05, rms=False, bias=False),
    # decode / verify widths, softmax, top-8
    "C1": dict(M=8, Ms=(1, 2, 8), H=2048, E=256, k=8, act=SOFTMAX, x_dtype=BF16,
               w_dtype=BF16, x_std=1.0, w_std=0.02, rms=True, bias=False),
    # sqrt(softplus) with selection bias, top-6
    "C2": dict(M=64, Ms=(1, 16, 64), H=4096, E=256, k=6, act=SQRT_SOFTPLUS,
               x_dtype=BF16, w_dtype=BF16, x_std=1.0, w_std=0.02, rms=True, bias=True),
    # prefill on tensor cores (BF16 or NVFP4 W)
    "C3": dict(M=16384, H=7168, E=256, k=8, act=SQRT_SOFTPLUS, x_dtype=BF16,
               w_dtype=BF16, x_std=1.0, w_std=0.02, rms=False, bias=True),
    # M=2 router with the unique-route table
    "C4": dict(M=2, H=4096, E=256, k=6, act=SQRT_SOFTPLUS, x_dtype=BF16,
               w_dtype=BF16, x_std=1.0, w_std=0.02, rms=True, bias=True, table=True,
               table_groups=100000),
}


def make_case(cfg: dict, M: int | None = None, seed: int = 0, w_dtype: int | None = None,
              dup_frac: float = 0.0, nvfp4_global: float | None = None):
    """Inputs for one router call: dict with x, W (and q/s/g for NVFP4),
    bias (or None) and the shape/act fields."""
    M = cfg["M"] if M is None else M
    H, E = cfg["H"], cfg["E"]
    w_dtype = cfg["w_dtype"] if w_dtype is None else w_dtype
    x = make_x(M, H, seed, cfg["x_dtype"], rms=cfg["rms"])
    w32 = normal(rng(seed + 1000), (E, H), cfg["w_std"])
    if dup_frac > 0:
        w32, _ = duplicate_experts(w32, dup_frac, seed + 2000)
    case = dict(M=M, H=H, E=E, k=cfg["k"], act=cfg["act"], x_dtype=cfg["x_dtype"],
                w_dtype=w_dtype, x=x, scales=None, g=1.0)
    if w_dtype == F32:
        case["W"] = w32
    elif w_dtype == BF16:
        case["W"] = f32_to_bf16_bits(w32)
    else:
        q, s, g = quantize_nvfp4(w32, nvfp4_global)
        case.update(W=q, scales=s, g=g)
    case["bias"] = make_bias(E, seed + 3000) if cfg.get("bias") else None
    return case
