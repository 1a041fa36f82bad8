"""Shared helpers of the parity tests: tolerance checks and oracle runs.

Inputs come from synthetic_inputs; the oracle side runs oracle/ on CPU copies
of exactly those inputs. Nothing here feeds a GPU result into the oracle.
"""
import numpy as np
import torch

import oracle as O
import synthetic_inputs as SI

# bf16 logits and fused rows: |gpu - oracle| <= ATOL + RTOL * |oracle|
ATOL = 2e-2
RTOL = 1e-2


def tol_report(gpu, ref, atol=ATOL, rtol=RTOL):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    err = np.abs(g - r)
    bound = atol + rtol * np.abs(r)
    bad = err > bound
    return {
        "mean_abs": float(err.mean()) if err.size else 0.0,
        "p999_ratio": float(np.quantile(err / bound, 0.999)) if err.size else 0.0,
        "max_abs": float(err.max()) if err.size else 0.0,
        "n_bad": int(bad.sum()),
        "n": int(err.size),
        "worst": float((err / bound).max()) if err.size and np.all(bound > 0) else (0.0 if not err.any() else float("inf")),
    }


def assert_close(gpu, ref, what, atol=ATOL, rtol=RTOL):
    rep = tol_report(gpu, ref, atol, rtol)
    assert rep["n_bad"] == 0, f"{what}: {rep}"
    return rep


def f64(t):
    return O.to_f64(t)


def gpu_weights(model, seed, device="cuda"):
    return SI.make_weights(model, seed, device=device)


def topk_ids_match(gpu_ids, ref_logits, k, margin):
    """Compare GPU top-k ids with the oracle's ranking where it is clear.

    A rank j is checked when the oracle's values at ranks j-1, j, j+1 are
    more than `margin` apart from its own; otherwise it is a near-tie and is
    only counted. Returns (checked, near_ties, mismatches)."""
    checked = near = bad = 0
    for r in range(ref_logits.shape[0]):
        row = ref_logits[r]
        order = np.lexsort((np.arange(row.shape[0]), -row))[: k + 1]
        vals = row[order]
        for j in range(k):
            gap_prev = vals[j - 1] - vals[j] if j > 0 else np.inf
            gap_next = vals[j] - vals[j + 1]
            if min(gap_prev, gap_next) <= margin:
                near += 1
                continue
            checked += 1
            bad += int(gpu_ids[r, j] != order[j])
    return checked, near, bad


def check_topk_consistent(logits, ids, vals):
    """GPU top-k against its own GPU logits: values equal the logits at the
    ids, descending, ties in ascending id, and nothing outside is larger
    than the k-th value (or equal with a lower id)."""
    lg = logits.float()
    k = ids.shape[1]
    got = torch.gather(lg, 1, ids.long())
    assert torch.equal(got, vals), "top-k values differ from the logits at the ids"
    assert torch.all(vals[:, :-1] >= vals[:, 1:])
    eq = vals[:, :-1] == vals[:, 1:]
    assert torch.all(~eq | (ids[:, :-1] < ids[:, 1:]))
    kth = vals[:, -1:]
    mask = torch.ones_like(lg, dtype=torch.bool)
    mask.scatter_(1, ids.long(), False)
    above = (lg > kth) & mask
    assert not above.any(), "a logit outside the top-k is larger than the k-th"
    tie = (lg == kth) & mask
    if tie.any():
        r, c = torch.nonzero(tie, as_tuple=True)
        assert torch.all(c > ids[r, -1]), "a tie with a lower id was left out"
