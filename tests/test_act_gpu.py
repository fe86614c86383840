"""The FP32 scores the kernels compute (branch-free sqrt(softplus) and
sigmoid built on the PTX ex2/rcp/rsqrt approximations) against the same
scores composed of CUDA's expf, log1pf, sqrtf and division, at EVERY finite
FP32 input. The near-tie guard band rests on the bound
|a32 - a| <= c 2^-23 a + 2^-60 (c from gbr_diag_act_coef): with the sweep's
largest relative distance m to the composition, and the composition's own
documented bound r (2.25 for sqrt-softplus: expf 2 ulp, log1pf 1 ulp, a
correctly rounded add and square root; 3 for the sigmoid), the bound holds
when m (1 + 2^-20) + r <= c. Inputs whose reference is below 2^-62 are held
to an absolute 2^-61 instead."""
import json

import pytest

from moe_expert_router_02_gb300 import router as R

pytestmark = pytest.mark.gpu

REF_BOUND = {R.GBR_ACT_SQRT_SOFTPLUS: 2.25, R.GBR_ACT_SIGMOID: 3.0}


@pytest.mark.parametrize("act", [R.GBR_ACT_SQRT_SOFTPLUS, R.GBR_ACT_SIGMOID],
                         ids=["sqrt_softplus", "sigmoid"])
def test_every_fp32_input_within_the_bound(act):
    import torch
    out = torch.zeros(2, dtype=torch.float32, device="cuda")
    R.diag_act_sweep(act, 0, 1 << 32, out)
    torch.cuda.synchronize()
    m, absmax = (float(v) for v in out.cpu())
    c = R.diag_act_coef(act)
    print("ACT_SWEEP " + json.dumps({"act": act, "max_rel_2^-23": m, "max_abs_tiny": absmax,
                                     "coef": c}))
    assert m * (1.0 + 2.0 ** -20) + REF_BOUND[act] <= c
    assert absmax <= 2.0 ** -61


def test_sweep_sees_a_planted_difference():
    """The sweep covers the inputs it is given: over [1.0, 2.0) alone the
    sqrt-softplus distance is nonzero (the two forms round differently
    somewhere in that binade), and an empty range gives zero."""
    import torch
    out = torch.zeros(2, dtype=torch.float32, device="cuda")
    R.diag_act_sweep(R.GBR_ACT_SQRT_SOFTPLUS, 0x3F800000, 1 << 23, out)
    torch.cuda.synchronize()
    assert float(out[0]) > 0.0
    R.diag_act_sweep(R.GBR_ACT_SQRT_SOFTPLUS, 0x3F800000, 0, out)
    torch.cuda.synchronize()
    assert float(out[0]) == 0.0 and float(out[1]) == 0.0
