"""Python access to the FP64 CPU oracle of the fused MoE router.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package smoke check
and by the benchmark's CPU-baseline leg. The product path never imports it.

The oracle itself is plain C++ in ``oracle.cpp`` (compiled here with g++,
``-O2 -ffp-contract=off`` so that x86_64 and aarch64 hosts give the same
FP64 results). This module only marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, NVFP4 = 0, 1, 2
SOFTMAX, SQRT_SOFTPLUS, SIGMOID = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` if it is missing or older than its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC",
                               "-shared", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            L.orc_e2m1.argtypes, L.orc_e2m1.restype = [I], D
            L.orc_e4m3.argtypes, L.orc_e4m3.restype = [I], D
            L.orc_sqrt_softplus.argtypes, L.orc_sqrt_softplus.restype = [D], D
            L.orc_sigmoid.argtypes, L.orc_sigmoid.restype = [D], D
            L.orc_logits.argtypes = [P, I, P, I, P, D, I, I, I, P]
            L.orc_select.argtypes = [P, P, I, I, I, I, I, P, P, P]
            L.orc_keys.argtypes = [P, P, I, I, I, I, P, P]
            L.orc_select_by_prob.argtypes = [P, I, I, I, P]
            L.orc_route_table.argtypes = [P, I, I, I, P, P, P, P]
            L.orc_gather_add.argtypes = [P, P, P, P, I, I, I, I, P]
            for f in (L.orc_logits, L.orc_select, L.orc_keys, L.orc_select_by_prob,
                      L.orc_route_table, L.orc_gather_add):
                f.restype = I
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def e2m1(code: int) -> float:
    return lib().orc_e2m1(int(code))


def e4m3(code: int) -> float:
    return lib().orc_e4m3(int(code))


def sqrt_softplus(z: float) -> float:
    return lib().orc_sqrt_softplus(float(z))


def sigmoid(z: float) -> float:
    return lib().orc_sigmoid(float(z))


def logits(x, x_dtype, W, w_dtype, M, H, E, scales=None, g=1.0) -> np.ndarray:
    """FP64 gate logits ``[M, E]``."""
    x = np.ascontiguousarray(x)
    W = np.ascontiguousarray(W)
    scales = None if scales is None else np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.empty((M, E), dtype=np.float64)
    rc = lib().orc_logits(_p(x), x_dtype, _p(W), w_dtype, _p(scales), float(g), M, H, E, _p(out))
    if rc != 0:
        raise ValueError("oracle: bad logits arguments")
    return out


def select(lg, k, act, bias=None):
    """Top-k + renormalise on logits ``[M, E]`` (widened exactly to FP64).

    ``bias`` is None, ``[E]`` or ``[M, E]`` FP32. Returns
    ``(idx int32 [M,k], w float64 [M,k], keys float64 [M, min(k+1,E)])``.
    """
    lg = np.ascontiguousarray(lg, dtype=np.float64)
    M, E = lg.shape
    per_row = 0
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
        per_row = 1 if bias.ndim == 2 else 0
    kk = min(k + 1, E)
    idx = np.empty((M, k), dtype=np.int32)
    w = np.empty((M, k), dtype=np.float64)
    keys = np.empty((M, kk), dtype=np.float64)
    rc = lib().orc_select(_p(lg), _p(bias), per_row, M, E, k, act, _p(idx), _p(w), _p(keys))
    if rc != 0:
        raise ValueError("oracle: bad select arguments")
    return idx, w, keys


def keys(lg, act, bias=None):
    """Every expert's selection key and weight score, ``(key [M, E], score
    [M, E])`` float64, as :func:`select` ranks and weights them."""
    lg = np.ascontiguousarray(lg, dtype=np.float64)
    M, E = lg.shape
    per_row = 0
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
        per_row = 1 if bias.ndim == 2 else 0
    key = np.empty((M, E), dtype=np.float64)
    score = np.empty((M, E), dtype=np.float64)
    if lib().orc_keys(_p(lg), _p(bias), per_row, M, E, act, _p(key), _p(score)) != 0:
        raise ValueError("oracle: bad keys arguments")
    return key, score


def select_by_prob(lg, k):
    lg = np.ascontiguousarray(lg, dtype=np.float64)
    M, E = lg.shape
    idx = np.empty((M, k), dtype=np.int32)
    if lib().orc_select_by_prob(_p(lg), M, E, k, _p(idx)) != 0:
        raise ValueError("oracle: bad select_by_prob arguments")
    return idx


def route_table(idx):
    """Serial unique-route table for ``idx [G, T, k]`` int32.

    Returns ``(unique [G,T*k] int32, mask [G,T*k] uint8, map [G,T,k] uint8,
    count [G] int32)``.
    """
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    G, T, k = idx.shape
    n = T * k
    unique = np.empty((G, n), dtype=np.int32)
    mask = np.empty((G, n), dtype=np.uint8)
    mp = np.empty((G, T, k), dtype=np.uint8)
    count = np.empty((G,), dtype=np.int32)
    if lib().orc_route_table(_p(idx), G, T, k, _p(unique), _p(mask), _p(mp), _p(count)) != 0:
        raise ValueError("oracle: bad route_table arguments")
    return unique, mask, mp, count


def gather_add(y, mp, w, shared):
    """The table's consumer: ``y`` BF16 bits ``[G, T*k, T, D]`` (row (u, t) =
    unique expert u's output for token t), ``mp`` uint8 ``[G, T, k]``, ``w``
    FP32 ``[G, T, k]``, ``shared`` BF16 bits ``[G, T, D]``. Returns the BF16
    bits ``[G, T, D]`` of bf16(bf16(FP32 fma sum in slot order) + shared)."""
    y = np.ascontiguousarray(y, dtype=np.uint16)
    mp = np.ascontiguousarray(mp, dtype=np.uint8)
    w = np.ascontiguousarray(w, dtype=np.float32)
    shared = np.ascontiguousarray(shared, dtype=np.uint16)
    G, T, k = mp.shape
    D = shared.shape[-1]
    assert y.shape == (G, T * k, T, D) and w.shape == (G, T, k) and shared.shape == (G, T, D)
    out = np.empty((G, T, D), dtype=np.uint16)
    if lib().orc_gather_add(_p(y), _p(mp), _p(w), _p(shared), G, T, k, D, _p(out)) != 0:
        raise ValueError("oracle: bad gather_add arguments")
    return out


def router(case: dict):
    """Whole router on one synthetic case from ``synth.make_case``.

    Returns dict with logits (FP64), idx, w, keys (first k+1 sorted keys)
    and, when the case asks for it, the M=2 route table. ``keys(...)`` of the
    returned logits gives every expert's key and score.
    """
    lg = logits(case["x"], case["x_dtype"], case["W"], case["w_dtype"], case["M"], case["H"],
                case["E"], scales=case.get("scales"), g=case.get("g", 1.0))
    idx, w, skeys = select(lg, case["k"], case["act"], case.get("bias"))
    out = dict(logits=lg, idx=idx, w=w, keys=skeys)
    if case.get("table"):
        M, k = case["M"], case["k"]
        out["table"] = route_table(idx.reshape(M // 2, 2, k))
    return out
