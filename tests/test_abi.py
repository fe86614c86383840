"""The C-ABI library builds, loads and exports every declared entry point;
host-side argument checks reject bad calls without touching the GPU."""
import ctypes
import os
import re

import pytest

from moe_expert_router_02_gb300 import router as R

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADERS = [os.path.join(INCLUDE, h) for h in ("gbrouter.h", "gbrouter_diag.h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\**\s+\**([a-z_0-9]+)\s*\(", text,
                                flags=re.M))
    return sorted(names)


def test_header_declares_the_binding_names():
    assert sorted(declared_functions()) == sorted(R.EXPORTS)


def test_library_exports_every_declared_symbol():
    L = R.lib()
    for name in declared_functions():
        assert hasattr(L, name), name


def test_strerror():
    assert R.router_strerror(R.GBR_OK) == "ok"
    assert "invalid" in R.router_strerror(R.GBR_EINVAL)
    assert R.router_strerror(99) == "unknown status"


def test_empty_calls_return_ok_without_launch():
    L = R.lib()
    assert L.router_forward(None, None, None, 0, 64, 16, 2, 0, None, None, None) == R.GBR_OK
    assert L.router_select(None, None, 0, 16, 2, 0, None, None, None) == R.GBR_OK
    assert L.route_table(None, 0, 2, 6, None, None, None, None, None) == R.GBR_OK


@pytest.mark.parametrize("args,expect", [
    ((1, 64, 16, 0, 0), R.GBR_EINVAL),      # k < 1
    ((1, 64, 16, 17, 0), R.GBR_EINVAL),     # k > E
    ((1, 64, 16, 2, 3), R.GBR_EINVAL),      # bad act
    ((-1, 64, 16, 2, 0), R.GBR_EINVAL),     # M < 0
    ((1, 0, 16, 2, 0), R.GBR_EINVAL),       # H < 1
    ((1, 64, 1024, 2, 0), R.GBR_EUNSUPPORTED),  # E > 512
    ((1, 64, 64, 17, 0), R.GBR_EUNSUPPORTED),   # k > 16
    ((1, 64, 16, 2, 0), R.GBR_EINVAL),      # null pointers
])
def test_router_forward_argument_errors(args, expect):
    M, H, E, k, act = args
    assert R.lib().router_forward(None, None, None, M, H, E, k, act, None, None, None) == expect


def test_bias_with_softmax_accepted_by_the_argument_checks():
    # softmax with a bias is a valid call (key = probability + bias); these
    # calls return before any CUDA call: M == 0 launches nothing, and the
    # shape errors are still reported
    L = R.lib()
    fake = ctypes.c_void_p(16)  # never dereferenced: the checks come first
    assert L.router_forward(fake, fake, fake, 0, 64, 16, 2, R.GBR_ACT_SOFTMAX, fake, fake,
                            None) == R.GBR_OK
    assert L.router_forward(fake, fake, fake, 1, 64, 16, 17, R.GBR_ACT_SOFTMAX, fake, fake,
                            None) == R.GBR_EINVAL
    assert L.router_select(fake, fake, 0, 16, 2, R.GBR_ACT_SOFTMAX, fake, fake,
                           None) == R.GBR_OK
    assert L.router_select(fake, fake, 1, 1024, 2, R.GBR_ACT_SOFTMAX, fake, fake,
                           None) == R.GBR_EUNSUPPORTED
    assert L.router_forward_noalloc(fake, fake, fake, 65, 64, 16, 2, R.GBR_ACT_SOFTMAX, fake,
                                    fake, None) == R.GBR_EWORKSPACE


def test_partial_table_and_odd_M_rejected():
    L = R.lib()
    fake = ctypes.c_void_p(256)
    o = R.make_opts()
    o.tbl_unique = 256
    assert L.router_forward_ex(fake, fake, None, 2, 64, 16, 2, 0, fake, fake, ctypes.byref(o),
                               None) == R.GBR_EINVAL
    o = R.make_opts(table=(256, 256, 256, 256))
    assert L.router_forward_ex(fake, fake, None, 3, 64, 16, 2, 0, fake, fake, ctypes.byref(o),
                               None) == R.GBR_EINVAL


def test_nvfp4_needs_scales_and_h16():
    L = R.lib()
    fake = ctypes.c_void_p(256)
    o = R.make_opts(w_dtype=R.GBR_NVFP4)
    assert L.router_forward_ex(fake, fake, None, 2, 64, 16, 2, 0, fake, fake, ctypes.byref(o),
                               None) == R.GBR_EINVAL
    o = R.make_opts(w_dtype=R.GBR_NVFP4, w_scales=256)
    assert L.router_forward_ex(fake, fake, None, 2, 72, 16, 2, 0, fake, fake, ctypes.byref(o),
                               None) == R.GBR_EINVAL


def test_workspace_too_small_rejected():
    L = R.lib()
    fake = ctypes.c_void_p(256)
    need = R.router_workspace_size(8, 2048, 256, 8)
    assert need > 0
    o = R.make_opts(workspace=256, workspace_bytes=need - 1)
    assert L.router_forward_ex(fake, fake, None, 8, 2048, 256, 8, 0, fake, fake, ctypes.byref(o),
                               None) == R.GBR_EWORKSPACE


def test_route_table_argument_errors():
    L = R.lib()
    fake = ctypes.c_void_p(256)
    assert L.route_table(fake, 4, 0, 6, fake, fake, fake, fake, None) == R.GBR_EINVAL
    assert L.route_table(fake, 4, 9, 6, fake, fake, fake, fake, None) == R.GBR_EINVAL
    assert L.route_table(fake, 4, 2, 17, fake, fake, fake, fake, None) == R.GBR_EINVAL
    assert L.route_table(fake, -1, 2, 6, fake, fake, fake, fake, None) == R.GBR_EINVAL
    assert L.route_table(None, 4, 2, 6, fake, fake, fake, fake, None) == R.GBR_EINVAL


def test_regime_choice():
    # the single-cluster kernel is chosen only where a device can schedule it
    assert R.router_regime(8, 2048, 256, 8) in (R.GBR_REGIME_GEMV, R.GBR_REGIME_GEMV1C)
    # a cluster per row group where the device can hold one, else split clusters
    assert R.router_regime(64, 4096, 256, 6) in (R.GBR_REGIME_GEMV, R.GBR_REGIME_GEMV1C)
    f32 = R.make_opts(x_dtype=R.GBR_F32, w_dtype=R.GBR_F32)
    assert R.router_regime(4, 256, 16, 2, f32) == R.GBR_REGIME_GENERIC
    assert R.router_regime(8, 100, 256, 8) == R.GBR_REGIME_GENERIC  # H % 32 != 0
    assert R.router_regime(16384, 7168, 256, 8) in (R.GBR_REGIME_TC, R.GBR_REGIME_GENERIC)
    assert R.router_regime(8, 2048, 256, 8, R.make_opts(flags=R.GBR_FLAG_FORCE_GENERIC)) == \
        R.GBR_REGIME_GENERIC
    assert R.router_regime(1, 64, 16, 17) == -1


def test_prefill_workspace_layout():
    # the prefill kernel's part of a workspace starts past the M <= 64
    # kernels' ticket and logits (256 + 64 * 512 * 4 bytes); from 256 rows
    # it holds 160 stream-K partial accumulators of E x 128 FP32
    small = 256 + 64 * 512 * 4
    assert R.router_workspace_size(200, 7168, 256, 8) == 0
    assert R.router_workspace_size(256, 7168, 256, 8) >= small + 160 * 256 * 128 * 4
    big = R.router_workspace_size(16384, 7168, 256, 8)
    assert big >= small + 160 * 256 * 128 * 4
    assert big < small + 160 * 256 * 128 * 4 + 4096
    fp4 = R.make_opts(w_dtype=R.GBR_NVFP4, w_scales=1)
    assert R.router_workspace_size(1000, 7168, 256, 8, fp4) >= small + 256 * 7168 * 2
    assert R.router_workspace_size(16384, 7168, 256, 8, fp4) >= big + 256 * 7168 * 2
    # stream-K groups: none outside the prefill kernel, -1 for rejected shapes
    assert R.router_tc_groups(8, 2048, 256, 8) == 0
    assert R.router_tc_groups(1, 64, 16, 17) == -1


def test_act_sweep_argument_errors_and_coefficients():
    """The score sweep rejects bad calls before any CUDA call; the kernels'
    score-bound coefficients leave room above the reference compositions'
    own bounds (2.25 and 3)."""
    L = R.lib()
    fake = ctypes.c_void_p(16)
    assert L.gbr_diag_act_sweep(R.GBR_ACT_SOFTMAX, 0, 16, fake, None) == 1
    assert L.gbr_diag_act_sweep(R.GBR_ACT_SIGMOID, 0, 16, None, None) == 1
    assert L.gbr_diag_act_sweep(R.GBR_ACT_SIGMOID, 1 << 32, 1, fake, None) == 1
    assert L.gbr_diag_act_sweep(R.GBR_ACT_SIGMOID, 5, (1 << 32) - 4, fake, None) == 1
    assert R.diag_act_coef(R.GBR_ACT_SQRT_SOFTPLUS) > 2.25
    assert R.diag_act_coef(R.GBR_ACT_SIGMOID) > 3.0
