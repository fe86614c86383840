"""A bounded device-side wait that runs out, on purpose and without any
fault: the NVFP4 prefill kernel decodes W once per launch, its CTAs
claiming column blocks from a counter in the caller's workspace, and its
producers wait (bounded, about a second) for each block's flag. Here the
host sets that counter past every block before the call, so no CTA decodes
anything: every producer's flag wait, the MMA warp's wait for the first
tile and the epilogue's wait for the accumulator give up, the kernel
records GBR_ETIMEOUT in the device status word, frees its tensor memory and
returns. The status is read through router_device_status, and the context
stays usable (the same call on a fresh workspace then matches the oracle)."""
import numpy as np
import pytest

from moe_expert_router_02_gb300 import router as R
from moe_expert_router_02_gb300 import synth
from tests.test_forward_gpu import check_case, upload
from tests.test_prefill_gpu import small_prefill

pytestmark = pytest.mark.gpu

# The prefill kernel's part of a workspace starts past the small-M kernels'
# ticket and logits (256 + 64 * 512 * 4 bytes); its first word is the NVFP4
# column-block claim counter.
PREFILL_PART_OFFSET = 256 + 64 * 512 * 4


def test_bounded_wait_expires_and_reports_timeout():
    import torch
    assert R.router_device_status(clear=True) == R.GBR_OK
    M, H = 200, 1024  # one CTA pair, one tile, 16 column blocks; no stream-K (M < 256)
    case = small_prefill(M, H=H, seed=3, w_dtype=synth.NVFP4)
    E, k = case["E"], case["k"]
    t = upload(case)
    probe = R.make_opts(w_dtype=synth.NVFP4, w_scales=1)
    need = R.router_workspace_size(M, H, E, k, probe)
    assert need > PREFILL_PART_OFFSET
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ws.view(torch.int32)[PREFILL_PART_OFFSET // 4] = 0x40000000  # every claim fails
    idx = torch.zeros((M, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((M, k), dtype=torch.float32, device="cuda")
    opts = R.make_opts(x_dtype=case["x_dtype"], w_dtype=case["w_dtype"], w_scales=t["scales"],
                       w_global_scale=case["g"], workspace=ws, workspace_bytes=need)
    assert R.router_regime(M, H, E, k, opts) == R.GBR_REGIME_TC
    R.router_forward_ex(t["x"], t["W"], t["bias"], M, H, E, k, case["act"], idx, w, opts)
    torch.cuda.synchronize()  # returns after the waits gave up (a few seconds)
    assert R.router_device_status(clear=True) == R.GBR_ETIMEOUT
    assert R.router_device_status() == R.GBR_OK
    # the context is intact: the same call with the library's own workspace
    check_case(case, expect_regime=R.GBR_REGIME_TC)
    assert R.router_device_status(clear=True) == R.GBR_OK
