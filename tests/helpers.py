"""Shared test helpers: device upload and the route comparison rule."""
import numpy as np

GAP_TOL = 1e-5  # oracle key gap below which a row's experts may legitimately differ
W_TOL = 2e-5    # absolute tolerance on renormalised weights


def dev(a):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def empty_outputs(M, k):
    import torch
    idx = torch.full((M, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((M, k), float("nan"), dtype=torch.float32, device="cuda")
    return idx, w


def check_routes(gi, gw, oi, ow, okeys, k, gap_tol=GAP_TOL, w_tol=W_TOL):
    """Compare GPU routes with the oracle's.

    Rows with identical experts must have weights within ``w_tol``. A row
    may differ only where the oracle's keys are within ``gap_tol``: at the
    k / k+1 boundary (counted, not compared further), or inside the top k
    (same set; every slot's oracle key within ``gap_tol`` of the oracle's
    key at that slot; weights compared per expert). Returns the number of
    rows that differed.
    """
    gi, gw, oi, ow, okeys = map(np.asarray, (gi, gw, oi, ow, okeys))
    differ = 0
    for r in range(len(gi)):
        assert len(set(gi[r].tolist())) == k, f"row {r}: repeated experts {gi[r]}"
        if np.array_equal(gi[r], oi[r]):
            err = np.max(np.abs(gw[r] - ow[r]))
            assert err <= w_tol, f"row {r}: weight error {err}"
            continue
        differ += 1
        boundary_gap = okeys[r, k - 1] - okeys[r, k] if okeys.shape[1] > k else np.inf
        if boundary_gap < gap_tol:
            continue
        assert set(gi[r].tolist()) == set(oi[r].tolist()), \
            f"row {r}: experts {gi[r]} vs oracle {oi[r]} with boundary gap {boundary_gap}"
        key_of = dict(zip(oi[r].tolist(), okeys[r, :k].tolist()))
        w_of = dict(zip(oi[r].tolist(), ow[r].tolist()))
        for j in range(k):
            e = int(gi[r, j])
            assert abs(key_of[e] - okeys[r, j]) < gap_tol, f"row {r}: slot {j} misordered"
            assert abs(gw[r, j] - w_of[e]) <= w_tol, f"row {r}: weight of expert {e}"
    return differ
