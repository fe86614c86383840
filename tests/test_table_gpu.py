"""route_table against the oracle's serial table builder, bit-exact; and
under CUDA-graph replay with changing inputs (b70 lab note, "Unique-route
router screen": eager and graph replays exact for every emitted field)."""
import itertools

import numpy as np
import pytest

import oracle
from moe_expert_router_02_gb300 import router as R
from moe_expert_router_02_gb300 import synth
from tests.helpers import dev

pytestmark = pytest.mark.gpu


def alloc(G, T, k):
    import torch
    n = T * k
    return (torch.full((G, n), -9, dtype=torch.int32, device="cuda"),
            torch.full((G, n), 0xEE, dtype=torch.uint8, device="cuda"),
            torch.full((G, T, k), 0xEE, dtype=torch.uint8, device="cuda"),
            torch.full((G,), -9, dtype=torch.int32, device="cuda"))


def run_table(idx):
    import torch
    G, T, k = idx.shape
    out = alloc(G, T, k)
    R.route_table(dev(idx), G, T, k, *out)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in out]


def assert_table_equal(idx):
    got = run_table(idx)
    ref = oracle.route_table(idx)
    for name, g, r in zip(("unique", "mask", "map", "count"), got, ref):
        assert np.array_equal(g, r), name


@pytest.mark.parametrize("k", [1, 2, 3])
def test_exhaustive_pairs_E6(k):
    perms = list(itertools.permutations(range(6), k))
    idx = np.array([[a, b] for a in perms for b in perms], dtype=np.int32)
    assert_table_equal(idx)


def test_1e5_seeded_pairs():
    assert_table_equal(synth.table_pairs(100000, 6, 256, seed=0))


@pytest.mark.parametrize("T,k", [(2, 6), (1, 1), (1, 16), (4, 3), (8, 16), (3, 5), (2, 16),
                                 (2, 2), (2, 4), (4, 2), (8, 2), (1, 4), (4, 4), (8, 1), (1, 12)])
def test_duplicates_and_group_sizes(T, k):
    gen = synth.rng(T * 100 + k)
    assert_table_equal(gen.integers(0, 5, size=(333, T, k)).astype(np.int32))
    assert_table_equal(gen.integers(0, 1000, size=(333, T, k)).astype(np.int32))


@pytest.mark.parametrize("T,k", [(2, 6), (1, 7), (4, 8), (2, 16), (8, 16)])
@pytest.mark.parametrize("G", [1, 2, 3, 17, 31, 1000])
def test_ragged_group_counts(T, k, G):
    # counts that leave the last warp's groups partly empty
    gen = synth.rng(G * 7 + T + k)
    assert_table_equal(gen.integers(0, 9, size=(G, T, k)).astype(np.int32))


@pytest.mark.parametrize("T,k", [(2, 6), (2, 8), (4, 1)])
def test_unaligned_buffers(T, k):
    """Group sizes that take 16-byte loads and stores (T*k a multiple of 4)
    on buffers offset by one element: the same table through the general
    kernel."""
    import torch
    G = 77
    n = T * k
    host = synth.rng(T + 10 * k).integers(0, 7, size=(G, T, k)).astype(np.int32)
    src = torch.zeros(G * n + 1, dtype=torch.int32, device="cuda")
    src[1:] = dev(host.reshape(-1))
    un = torch.full((G * n + 1,), -9, dtype=torch.int32, device="cuda")
    mk = torch.full((G * n + 1,), 0xEE, dtype=torch.uint8, device="cuda")
    mp = torch.full((G * n + 1,), 0xEE, dtype=torch.uint8, device="cuda")
    cnt = torch.full((G,), -9, dtype=torch.int32, device="cuda")
    R.route_table(src[1:], G, T, k, un[1:], mk[1:], mp[1:], cnt)
    torch.cuda.synchronize()
    ref = oracle.route_table(host)
    got = (un[1:].cpu().numpy().reshape(G, n), mk[1:].cpu().numpy().reshape(G, n),
           mp[1:].cpu().numpy().reshape(G, T, k), cnt.cpu().numpy())
    for name, g, r in zip(("unique", "mask", "map", "count"), got, ref):
        assert np.array_equal(g, r), name
    assert int(un[0]) == -9 and int(mk[0]) == 0xEE and int(mp[0]) == 0xEE


def test_graph_replay_with_changing_inputs():
    import torch
    G, T, k = 4096, 2, 6
    src = dev(synth.table_pairs(G, k, 256, seed=1))
    out = alloc(G, T, k)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        R.route_table(src, G, T, k, *out, stream=s)  # warm up outside capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        R.route_table(src, G, T, k, *out, stream=s)
    for seed in range(2, 12):
        host = synth.table_pairs(G, k, 256, seed=seed)
        src.copy_(dev(host))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.route_table(host)
        for got, r in zip(out, ref):
            assert np.array_equal(got.cpu().numpy(), r)
