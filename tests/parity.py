"""Shared helpers of the GPU parity tests: tolerances and the routing rule.

Tolerances follow the layer's accuracy contract: max |err| <= 2e-3 * max |ref|
on the fp32-accumulate GEMV path, <= 1e-2 * max |ref| on the bf16 tensor-core
path. Expert ids must equal the oracle's exactly, as a set, on every row whose
oracle gap between the k-th and (k+1)-th logit is at least 1e-5; the slot
order must match too where every adjacent gap among the top k+1 is at least
1e-5. Rows under the gap are excused from the id and value comparison (at most one
in a hundred of the checked rows, or one), and their GPU ids must still be a
valid top-k of the oracle's logits to within 1e-5.
"""

import numpy as np

TOL_GEMV = 2e-3
TOL_TC = 1e-2
GAP = 1e-5


def check_routes(ids_gpu: np.ndarray, ids_ref: np.ndarray, gap: np.ndarray,
                 logits: np.ndarray) -> np.ndarray:
    """Asserts the routing rule; returns the boolean mask of rows that count."""
    T, k = ids_ref.shape
    ok = gap >= GAP
    for t in range(T):
        if ok[t]:
            assert sorted(ids_gpu[t]) == sorted(ids_ref[t]), (t, ids_gpu[t], ids_ref[t])
            srt = -np.sort(-logits[t])[: k + 1]
            if np.all(-np.diff(srt) >= GAP):
                assert list(ids_gpu[t]) == list(ids_ref[t]), (t, ids_gpu[t], ids_ref[t])
        else:
            # a valid top-k: every chosen logit within GAP of the k-th largest or above
            kth = -np.sort(-logits[t])[k - 1]
            assert len(set(ids_gpu[t].tolist())) == k
            assert np.all(logits[t, ids_gpu[t]] >= kth - GAP)
    # the excuse is for rare accidental near-ties, not a loophole: at most one
    # row in a hundred (or one row) may take it
    assert int((~ok).sum()) <= max(1, T // 100), f"{int((~ok).sum())} of {T} rows excused"
    return ok


def assert_close(got: np.ndarray, ref: np.ndarray, tol: float, rows=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if rows is not None:
        got, ref = got[rows], ref[rows]
    if ref.size == 0:
        return
    scale = np.max(np.abs(ref))
    err = np.max(np.abs(got - ref))
    assert np.all(np.isfinite(got)), "non-finite output"
    assert err <= tol * scale, f"max|err| {err:.3e} > {tol:g} * max|ref| {scale:.3e} (ratio {err / scale:.2e})"
