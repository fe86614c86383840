"""route_gather_add (the unique-route table's consumer) against the oracle,
bit for bit: random expert outputs routed through tables of the four pair
categories, duplicate slots, groups of up to 8 tokens, D with a ragged
tail and the element-wise path (D % 8 != 0, unaligned rows)."""
import numpy as np
import pytest

import oracle
from moe_expert_router_02_gb300 import router as R
from moe_expert_router_02_gb300 import synth
from tests.helpers import dev

pytestmark = pytest.mark.gpu


def run_gather(y, mp, w, sh, offset=0):
    import torch
    G, T, k = mp.shape
    D = sh.shape[-1]
    out = torch.full((G * T * D + offset,), 0x7fc0, dtype=torch.int16, device="cuda")
    if offset:  # shift every buffer by `offset` elements (2-byte aligned only)
        ybuf = torch.zeros(y.size + offset, dtype=torch.int16, device="cuda")
        ybuf[offset:] = dev(y.view(np.int16).reshape(-1))
        sbuf = torch.zeros(sh.size + offset, dtype=torch.int16, device="cuda")
        sbuf[offset:] = dev(sh.view(np.int16).reshape(-1))
        yp, sp, op = ybuf[offset:], sbuf[offset:], out[offset:]
    else:
        yp, sp, op = dev(y.view(np.int16)), dev(sh.view(np.int16)), out
    R.route_gather_add(yp, dev(mp), dev(w), sp, G, T, k, D, op)
    torch.cuda.synchronize()
    return op.cpu().numpy().view(np.uint16).reshape(G, T, D)


def table_for(G, k, seed, T=2):
    if T == 2:
        idx = synth.table_pairs(G, k, 256, seed)
    else:
        gen = synth.rng(seed)
        idx = np.stack([np.stack([gen.choice(24, k, replace=False) for _ in range(T)])
                        for _ in range(G)]).astype(np.int32)
    return oracle.route_table(idx)


@pytest.mark.parametrize("D", [4096, 7168, 264])
def test_pairs_bit_exact(D):
    G, k = 64, 6
    y, w, sh = synth.gather_inputs(G, k, D, seed=D)
    _, _, mp, _ = table_for(G, k, seed=D + 1)
    assert np.array_equal(run_gather(y, mp, w, sh), oracle.gather_add(y, mp, w, sh))


def test_duplicate_slots_and_wide_groups():
    G, k, D = 24, 4, 256
    for T in (1, 3, 8):
        y, w, sh = synth.gather_inputs(G, k, D, seed=T, T=T)
        _, _, mp, _ = table_for(G, k, seed=T + 10, T=T)
        mp = mp.copy()
        mp[:, 0, 1] = mp[:, 0, 0]  # a slot reusing its neighbour's row
        assert np.array_equal(run_gather(y, mp, w, sh), oracle.gather_add(y, mp, w, sh))


@pytest.mark.parametrize("D,offset", [(250, 0), (256, 1), (7, 3)])
def test_element_path(D, offset):
    G, k = 16, 6
    y, w, sh = synth.gather_inputs(G, k, D, seed=D + offset)
    _, _, mp, _ = table_for(G, k, seed=D)
    assert np.array_equal(run_gather(y, mp, w, sh, offset), oracle.gather_add(y, mp, w, sh))


def test_many_groups_grid_stride():
    G, k, D = 70000, 2, 8
    y, w, sh = synth.gather_inputs(G, k, D, seed=5)
    _, _, mp, _ = table_for(G, k, seed=6)
    assert np.array_equal(run_gather(y, mp, w, sh), oracle.gather_add(y, mp, w, sh))


def test_argument_errors_and_empty():
    L = R.lib()
    assert L.route_gather_add(None, None, None, None, 0, 2, 6, 64, None, None) == R.GBR_OK
    assert L.route_gather_add(None, None, None, None, -1, 2, 6, 64, None, None) == R.GBR_EINVAL
    assert L.route_gather_add(None, None, None, None, 1, 9, 6, 64, None, None) == R.GBR_EINVAL
    assert L.route_gather_add(None, None, None, None, 1, 2, 17, 64, None, None) == R.GBR_EINVAL
    assert L.route_gather_add(None, None, None, None, 1, 2, 6, 64, None, None) == R.GBR_EINVAL
