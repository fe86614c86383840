"""router_forward_noalloc, the entry point for callers that cannot allocate
device memory, gives the same routes as router_forward.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test. It passes both alone in a
fresh process and after the rest of the suite."""
import ctypes

import numpy as np
import pytest

from moe_expert_router_02_gb300 import router as R
from moe_expert_router_02_gb300 import synth
import oracle
from tests.helpers import GAP_TOL, W_TOL, check_routes, dev, empty_outputs

pytestmark = pytest.mark.gpu


C = synth.CONFIGS
CASES = {
    "C1_M8": (C["C1"], 8),
    "C2_M64": (C["C2"], 64),
    "C4_M2": (C["C4"], 2),
    # E = 512 at M = 64 fills the whole array (16 logits per lane in selection)
    "E512_M64": (dict(C["C2"], E=512, k=8, H=2048), 64),
    "sigmoid_bias_M16": (dict(C["C2"], act=synth.SIGMOID), 16),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_matches_router_forward_on_two_calls(name):
    import torch
    cfg, M = CASES[name]
    H, E, k, act = cfg["H"], cfg["E"], cfg["k"], cfg["act"]
    case = synth.make_case(cfg, M=M, seed=21)
    x, W = dev(case["x"]), dev(case["W"])
    bias = None if case["bias"] is None else dev(case["bias"])
    ref_idx, ref_w = empty_outputs(M, k)
    R.router_forward(x, W, bias, M, H, E, k, act, ref_idx, ref_w)
    torch.cuda.synchronize()
    ri, rw = ref_idx.cpu().numpy(), ref_w.cpu().numpy()
    orc = oracle.router(case)
    for _ in range(2):  # the second call reuses the array the first one left behind
        idx, w = empty_outputs(M, k)
        rc = R.lib().router_forward_noalloc(x.data_ptr(), W.data_ptr(),
                                            None if bias is None else bias.data_ptr(),
                                            M, H, E, k, act, idx.data_ptr(), w.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)
        assert rc == R.GBR_OK, R.router_strerror(rc)
        torch.cuda.synchronize()
        gi, gw = idx.cpu().numpy(), w.cpu().numpy()
        # the two entry points may run different kernels (different FP32
        # summation order): ids must agree except on rows whose oracle key gap
        # at the k / k+1 boundary is below the tests' gap tolerance
        same = np.all(gi == ri, axis=1)
        if not np.all(same):
            gap = orc["keys"][:, k - 1] - orc["keys"][:, k]
            assert np.all(gap[~same] < GAP_TOL)
        assert np.max(np.abs(gw[same] - rw[same])) <= W_TOL
        # and every row against the oracle, differing rows included
        check_routes(gi, gw, orc, case)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fake = ctypes.c_void_p(256)
    L = R.lib()
    assert L.router_forward_noalloc(fake, fake, None, 65, 2048, 256, 8, 0, fake, fake,
                                    None) == R.GBR_EWORKSPACE
    assert L.router_forward_noalloc(fake, fake, None, 8, 2048, 1024, 8, 0, fake, fake,
                                    None) == R.GBR_EUNSUPPORTED
