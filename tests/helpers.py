"""Shared test helpers: device upload, the route comparison rule, and the
record of rows whose experts differ from the oracle's."""
import os

import numpy as np

GAP_TOL = 1e-5  # oracle key gap below which a row's experts may legitimately differ
W_TOL = 2e-5    # absolute tolerance on renormalised weights

# (test id, rows checked, rows with an oracle gap below GAP_TOL at the k / k+1
# boundary, rows whose ids differed); printed by conftest at the end of a run
PARITY_LOG = []


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


def _test_id():
    t = os.environ.get("PYTEST_CURRENT_TEST", "")
    return t.rsplit(" ", 1)[0] if t else "?"


def check_routes(gi, gw, ref, case, label=None, gap_tol=GAP_TOL, w_tol=W_TOL):
    """Compare GPU routes (ids ``gi``, weights ``gw``) with the oracle's.

    ``ref`` is ``oracle.router(case)`` (or any dict with the oracle's
    ``idx``, ``w``, sorted ``keys`` and FP64 ``logits``). Every row must hold
    k distinct experts in [0, E). A row with the oracle's ids must have
    weights within ``w_tol``. A row whose ids differ is still checked in
    full against the oracle's key and score of every expert:

    * experts in one set but not the other have oracle keys within
      ``gap_tol`` of the oracle's k-th key (only a near tie at the k / k+1
      boundary may change the set);
    * consecutive slots are ordered by the oracle's keys within ``gap_tol``;
    * each weight is within ``w_tol`` of the oracle's FP64 score of that
      expert renormalised over the GPU's chosen set.

    Counts go to ``PARITY_LOG`` under ``label`` (default: the test id).
    Returns the number of rows whose ids differed.
    """
    import oracle
    k = case["k"]
    gi, gw = np.asarray(gi), np.asarray(gw)
    oi, ow, okeys = (np.asarray(ref[n]) for n in ("idx", "w", "keys"))
    E = np.asarray(ref["logits"]).shape[1]
    kfull, score = oracle.keys(ref["logits"], case["act"], case.get("bias"))
    gap = okeys[:, k - 1] - okeys[:, k] if okeys.shape[1] > k else np.full(len(gi), np.inf)
    differ = 0
    for r in range(len(gi)):
        row = gi[r].tolist()
        assert len(set(row)) == k, f"row {r}: repeated experts {row}"
        assert min(row) >= 0 and max(row) < E, f"row {r}: expert out of range {row}"
        if np.array_equal(gi[r], oi[r]):
            err = np.max(np.abs(gw[r] - ow[r]))
            assert err <= w_tol, f"row {r}: weight error {err}"
            continue
        differ += 1
        kth = okeys[r, k - 1]
        swapped = set(row) ^ set(oi[r].tolist())
        for e in swapped:
            assert abs(kfull[r, e] - kth) < gap_tol, \
                f"row {r}: expert {e} (key {kfull[r, e]!r}) vs oracle k-th key {kth!r}; " \
                f"ids {row} vs oracle {oi[r].tolist()}"
        for j in range(k - 1):
            a, b = kfull[r, row[j]], kfull[r, row[j + 1]]
            assert a >= b - gap_tol, f"row {r}: slots {j}, {j + 1} misordered ({a!r} < {b!r})"
        s = score[r, gi[r]]
        tot = s.sum()
        expect = s / tot if tot > 0 else np.full(k, 1.0 / k)
        err = np.max(np.abs(gw[r] - expect))
        assert err <= w_tol, f"row {r}: weight error {err} against the oracle's scores"
    PARITY_LOG.append((label or _test_id(), int(len(gi)), int(np.sum(gap < gap_tol)), differ))
    return differ
