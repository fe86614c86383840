"""Python binding of the ``gbrouter`` C ABI (``include/gbrouter.h``).

Argument marshalling only: every step of the router runs in the CUDA
library. The functions carry the C names and take torch CUDA tensors (or
``None`` for nullable pointers) and an optional ``torch.cuda.Stream``. A
non-zero status raises :class:`RouterError`. There is no fallback: if the
library is missing and cannot be built, loading raises.
"""
from __future__ import annotations

import ctypes
import threading

from . import build as _build

GBR_OK, GBR_EINVAL, GBR_EUNSUPPORTED, GBR_ECUDA, GBR_EWORKSPACE, GBR_ETIMEOUT = range(6)
GBR_ACT_SOFTMAX, GBR_ACT_SQRT_SOFTPLUS, GBR_ACT_SIGMOID = 0, 1, 2
GBR_F32, GBR_BF16, GBR_NVFP4 = 0, 1, 2
GBR_FLAG_NO_PDL, GBR_FLAG_FORCE_GENERIC, GBR_FLAG_FORCE_GEMV, GBR_FLAG_FORCE_TC, \
    GBR_FLAG_UNFUSED, GBR_FLAG_NO_SINGLE_CLUSTER, GBR_FLAG_TC_NO_STREAMK, \
    GBR_FLAG_TC_SINGLE_CTA = 1, 2, 4, 8, 16, 32, 64, 128
GBR_REGIME_GENERIC, GBR_REGIME_GEMV, GBR_REGIME_TC, GBR_REGIME_UNFUSED, GBR_REGIME_GEMV1C = \
    0, 1, 2, 3, 4

EXPORTS = ("router_forward", "router_forward_ex", "router_workspace_size", "router_regime",
           "router_tc_groups", "router_select", "route_table", "router_strerror", "router_device_status",
           "router_forward_noalloc", "router_near_tie_keys", "route_gather_add", "gbr_diag_chain",
           "gbr_diag_act_sweep", "gbr_diag_act_coef", "gbr_diag_near_key_cycles")


class RouterError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {router_strerror(status)} (status {status})")


class GbrOpts(ctypes.Structure):
    _fields_ = [("x_dtype", ctypes.c_int), ("w_dtype", ctypes.c_int),
                ("w_scales", ctypes.c_void_p), ("w_global_scale", ctypes.c_float),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("tbl_unique", ctypes.c_void_p), ("tbl_mask", ctypes.c_void_p),
                ("tbl_map", ctypes.c_void_p), ("tbl_count", ctypes.c_void_p),
                ("out_logits", ctypes.c_void_p), ("flags", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


_variant = None


def use_variant(variant) -> None:
    """Load the named build variant (``"stamps"``: the measurement build with
    per-phase timestamps) instead of the library; call before the first
    router call of the process."""
    global _variant
    with _lock:
        if _lib is not None:
            raise RuntimeError("the router library is already loaded")
        _variant = variant


def lib() -> ctypes.CDLL:
    """Load (building first if stale) the in-tree ``libgbrouter.so``."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build(variant=_variant)
            L = ctypes.CDLL(path)
            P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            L.router_forward.argtypes = [P, P, P, I, I, I, I, I, P, P, P]
            L.router_forward_ex.argtypes = [P, P, P, I, I, I, I, I, P, P,
                                            ctypes.POINTER(GbrOpts), P]
            L.router_workspace_size.argtypes = [I, I, I, I, ctypes.POINTER(GbrOpts)]
            L.router_workspace_size.restype = S
            L.router_regime.argtypes = [I, I, I, I, ctypes.POINTER(GbrOpts)]
            L.router_tc_groups.argtypes = [I, I, I, I, ctypes.POINTER(GbrOpts)]
            L.router_select.argtypes = [P, P, I, I, I, I, P, P, P]
            L.route_table.argtypes = [P, I, I, I, P, P, P, P, P]
            L.router_forward_noalloc.argtypes = [P, P, P, I, I, I, I, I, P, P, P]
            L.router_near_tie_keys.argtypes = [P, P, I, I, P, P, P]
            L.route_gather_add.argtypes = [P, P, P, P, I, I, I, I, P, P]
            L.router_strerror.argtypes = [I]
            L.router_strerror.restype = ctypes.c_char_p
            L.router_device_status.argtypes = [I]
            L.gbr_diag_chain.argtypes = [I, I, P, S, P, P]
            L.gbr_diag_chain.restype = I
            L.gbr_diag_act_sweep.argtypes = [I, ctypes.c_ulonglong, ctypes.c_ulonglong, P, P]
            L.gbr_diag_act_sweep.restype = I
            L.gbr_diag_act_coef.argtypes = [I]
            L.gbr_diag_act_coef.restype = ctypes.c_float
            L.gbr_diag_near_key_cycles.argtypes = [I, I, P, P]
            L.gbr_diag_near_key_cycles.restype = I
            if _variant == "stamps":
                L.router_phase_stamps.argtypes = [P, P, P, P]
                L.router_phase_stamps.restype = I
                L.router_tc_phase_stamps.argtypes = [P, P, P]
                L.router_tc_phase_stamps.restype = I
                L.router_split_phase_stamps.argtypes = [P, P, P, P]
                L.router_split_phase_stamps.restype = I
            for f in (L.router_forward, L.router_forward_ex, L.router_regime, L.router_tc_groups,
                      L.router_select,
                      L.route_table, L.router_device_status, L.router_forward_noalloc,
                      L.router_near_tie_keys, L.route_gather_add):
                f.restype = I
            _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(rc: int, where: str):
    if rc != GBR_OK:
        raise RouterError(rc, where)


def make_opts(x_dtype=GBR_BF16, w_dtype=GBR_BF16, w_scales=None, w_global_scale=1.0,
              workspace=None, workspace_bytes=0, table=None, out_logits=None, flags=0) -> GbrOpts:
    """``table`` is None or a tuple (unique, mask, map, count) of tensors."""
    o = GbrOpts()
    o.x_dtype, o.w_dtype = x_dtype, w_dtype
    o.w_scales = _ptr(w_scales)
    o.w_global_scale = float(w_global_scale)
    o.workspace = _ptr(workspace)
    o.workspace_bytes = int(workspace_bytes)
    if table is not None:
        o.tbl_unique, o.tbl_mask, o.tbl_map, o.tbl_count = (_ptr(t) for t in table)
    o.out_logits = _ptr(out_logits)
    o.flags = int(flags)
    return o


def router_strerror(status: int) -> str:
    return lib().router_strerror(int(status)).decode()


def router_forward(x, W_gate, bias, M, H, E, k, act, out_idx, out_w, stream=None):
    _check(lib().router_forward(_ptr(x), _ptr(W_gate), _ptr(bias), M, H, E, k, act,
                                _ptr(out_idx), _ptr(out_w), _stream(stream)), "router_forward")


def router_forward_ex(x, W_gate, bias, M, H, E, k, act, out_idx, out_w, opts=None, stream=None):
    _check(lib().router_forward_ex(_ptr(x), _ptr(W_gate), _ptr(bias), M, H, E, k, act,
                                   _ptr(out_idx), _ptr(out_w),
                                   ctypes.byref(opts) if opts is not None else None,
                                   _stream(stream)), "router_forward_ex")


def router_forward_noalloc(x, W_gate, bias, M, H, E, k, act, out_idx, out_w, stream=None):
    """router_forward without any device allocation: the library's static
    scratch array serves as the workspace (M <= 64, E <= 512)."""
    _check(lib().router_forward_noalloc(_ptr(x), _ptr(W_gate), _ptr(bias), M, H, E, k, act,
                                        _ptr(out_idx), _ptr(out_w), _stream(stream)),
           "router_forward_noalloc")


def router_workspace_size(M, H, E, k, opts=None) -> int:
    return lib().router_workspace_size(M, H, E, k, ctypes.byref(opts) if opts is not None else None)


def router_regime(M, H, E, k, opts=None) -> int:
    return lib().router_regime(M, H, E, k, ctypes.byref(opts) if opts is not None else None)


def router_tc_groups(M, H, E, k, opts=None) -> int:
    """Stream-K work groups of the prefill kernel for this shape (0: none)."""
    return lib().router_tc_groups(M, H, E, k, ctypes.byref(opts) if opts is not None else None)


def router_select(logits, bias, M, E, k, act, out_idx, out_w, stream=None):
    _check(lib().router_select(_ptr(logits), _ptr(bias), M, E, k, act, _ptr(out_idx),
                               _ptr(out_w), _stream(stream)), "router_select")


def router_near_tie_keys(z, bias, n, key_hi, key_lo, act=GBR_ACT_SQRT_SOFTPLUS, stream=None):
    _check(lib().router_near_tie_keys(_ptr(z), _ptr(bias), n, act, _ptr(key_hi), _ptr(key_lo),
                                      _stream(stream)), "router_near_tie_keys")


def route_table(idx, groups, tokens_per_group, k, out_unique, out_mask, out_map, out_count,
                stream=None):
    _check(lib().route_table(_ptr(idx), groups, tokens_per_group, k, _ptr(out_unique),
                             _ptr(out_mask), _ptr(out_map), _ptr(out_count), _stream(stream)),
           "route_table")


def route_gather_add(y, mp, w, shared, groups, tokens_per_group, k, D, out, stream=None):
    _check(lib().route_gather_add(_ptr(y), _ptr(mp), _ptr(w), _ptr(shared), groups,
                                  tokens_per_group, k, D, _ptr(out), _stream(stream)),
           "route_gather_add")


def router_device_status(clear: bool = False) -> int:
    return lib().router_device_status(1 if clear else 0)


def diag_chain(kind, n, x, sink, stream=None):
    """Launch-chain floor (``include/gbrouter_diag.h``): n PDL launches of the
    single-cluster router's shape; kind 0 waits only, kind 1 also reads x."""
    xb = 0 if x is None else x.numel() * x.element_size()
    rc = lib().gbr_diag_chain(int(kind), int(n), _ptr(x), xb, _ptr(sink), _stream(stream))
    if rc != 0:
        raise RuntimeError(f"gbr_diag_chain failed ({rc})")


def diag_act_sweep(act, first, count, out, stream=None):
    """Error sweep of the FP32 score ``act`` over the FP32 bit patterns
    [first, first + count) (``include/gbrouter_diag.h``); out: device float32
    tensor of 2, written asynchronously."""
    rc = lib().gbr_diag_act_sweep(int(act), int(first), int(count), _ptr(out), _stream(stream))
    if rc != 0:
        raise RuntimeError(f"gbr_diag_act_sweep failed ({rc})")


def diag_near_key_cycles(act, reps=64):
    """SM cycles per near-tie key evaluation (one warp, dependent chain)."""
    import torch
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    rc = lib().gbr_diag_near_key_cycles(int(act), int(reps), _ptr(out), _stream(None))
    if rc != 0:
        raise RuntimeError(f"gbr_diag_near_key_cycles failed ({rc})")
    torch.cuda.synchronize()
    return int(out[0])


def diag_act_coef(act):
    """The coefficient c of the kernels' FP32 score bound c 2^-23 a + 2^-60."""
    return float(lib().gbr_diag_act_coef(int(act)))


def phase_stamps(with_refines=False):
    """Measurement build only: the single-cluster kernel's phase stamps as a
    numpy array [calls, ctas, phases] of %globaltimer ns (0 = not stamped),
    and the last selection's sub-phase stamps per CTA rank [16, 5]; with
    with_refines, also the counts of warp selections (small-M kernels) that
    re-ranked near ties, that went on to FP64, and whose 32-bit rounds ran
    again on (key, index) pairs since the previous read."""
    import numpy as np
    L = lib()
    c, t, p = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    L.router_phase_stamps(None, ctypes.byref(c), ctypes.byref(t), ctypes.byref(p))
    n = c.value * t.value * p.value
    buf = np.zeros(n + 16 * 5 + 3, dtype=np.uint64)
    if L.router_phase_stamps(buf.ctypes.data_as(ctypes.c_void_p), ctypes.byref(c), ctypes.byref(t),
                             ctypes.byref(p)) != 0:
        raise RuntimeError("router_phase_stamps failed")
    st, sel = buf[:n].reshape(c.value, t.value, p.value), buf[n:n + 80].reshape(16, 5)
    if with_refines:
        return st, sel, (int(buf[n + 80]), int(buf[n + 81]), int(buf[n + 82]))
    return st, sel


def tc_phase_stamps():
    """Measurement build only: the phase stamps of the prefill launches since
    the previous read as a numpy array [ctas, phases] (%globaltimer ns, 0 =
    not stamped; see the prefill kernel); reading clears them."""
    import numpy as np
    L = lib()
    c, p = ctypes.c_int(), ctypes.c_int()
    L.router_tc_phase_stamps(None, ctypes.byref(c), ctypes.byref(p))
    out = np.zeros((c.value, p.value), dtype=np.uint64)
    if L.router_tc_phase_stamps(out.ctypes.data_as(ctypes.c_void_p), ctypes.byref(c),
                                ctypes.byref(p)) != 0:
        raise RuntimeError("router_tc_phase_stamps failed")
    return out


def split_phase_stamps():
    """Measurement build only: the split-cluster kernel's phase stamps as a
    numpy array [calls, ctas, phases] (%globaltimer ns, 0 = not stamped)."""
    import numpy as np
    L = lib()
    c, t, p = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    L.router_split_phase_stamps(None, ctypes.byref(c), ctypes.byref(t), ctypes.byref(p))
    out = np.zeros((c.value, t.value, p.value), dtype=np.uint64)
    if L.router_split_phase_stamps(out.ctypes.data_as(ctypes.c_void_p), ctypes.byref(c),
                                   ctypes.byref(t), ctypes.byref(p)) != 0:
        raise RuntimeError("router_split_phase_stamps failed")
    return out
