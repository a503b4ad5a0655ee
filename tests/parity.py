"""Parity checks shared by the CPU pin tests and the GPU tests.

Acceptance (the layer's stated tolerances):
  * forced routing: ids bit-exact;
  * free routing: ids bit-exact except at near-ties, i.e. where the reference probabilities
    of the two candidates differ by at most 1e-4 (exact ties must go to the lowest index);
  * outputs: max|err| <= 2e-2 * max|y_ref| and relative L2 error <= 5e-3.
"""
from __future__ import annotations

import numpy as np

TIE_TOL = 1e-4
MAX_ERR_FRAC = 2e-2
REL_L2 = 5e-3


def rel_l2(a: np.ndarray, ref: np.ndarray) -> float:
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref.ravel())
    return float(np.linalg.norm((a - ref).ravel()) / (den if den > 0 else 1.0))


def output_errors(y: np.ndarray, y_ref: np.ndarray):
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    maxabs = float(np.max(np.abs(y - y_ref))) if y.size else 0.0
    scale = float(np.max(np.abs(y_ref))) if y.size else 0.0
    return maxabs, scale, rel_l2(y, y_ref)


def outputs_ok(y, y_ref, max_frac=MAX_ERR_FRAC, rl2=REL_L2):
    if np.asarray(y).size == 0:
        return True, "empty"
    if not np.all(np.isfinite(y)):
        return False, "non-finite output"
    maxabs, scale, r = output_errors(y, y_ref)
    ok = maxabs <= max_frac * scale and r <= rl2
    return ok, f"max|err|={maxabs:.3e} (limit {max_frac * scale:.3e}), relL2={r:.3e} (limit {rl2:.1e})"


def ids_ok(ids: np.ndarray, ids_ref: np.ndarray, p_ref: np.ndarray, E: int, tol: float = TIE_TOL):
    """Free-routing id check.  For every token: the ids are distinct and in range; where a
    slot differs from the reference, both candidates' reference probabilities are within
    `tol` of each other and not exactly equal (an exact tie must pick the lower index, as the
    reference does), and the set stays a valid top-k: every chosen id's probability is at
    least the reference's k-th largest minus `tol`."""
    ids = np.asarray(ids)
    ids_ref = np.asarray(ids_ref)
    T, k = ids_ref.shape
    bad = []
    for t in range(T):
        row = ids[t]
        if len(set(row.tolist())) != k or row.min() < 0 or row.max() >= E:
            bad.append((t, "invalid ids"))
            continue
        if np.array_equal(row, ids_ref[t]):
            continue
        p = p_ref[t]
        kth = p[ids_ref[t]].min()
        for i in range(k):
            a, b = int(row[i]), int(ids_ref[t, i])
            if a == b:
                continue
            if abs(float(p[a]) - float(p[b])) > tol or p[a] == p[b]:
                bad.append((t, f"slot {i}: id {a} (p={p[a]:.6g}) vs ref {b} (p={p[b]:.6g})"))
                break
        else:
            if p[row].min() < kth - tol:
                bad.append((t, "not a top-k set"))
    return len(bad) == 0, bad[:5], T - sum(np.array_equal(ids[t], ids_ref[t]) for t in range(T))


def weights_ok(w, w_ref, tol=1e-5):
    w = np.asarray(w, np.float64)
    w_ref = np.asarray(w_ref, np.float64)
    if w.size == 0:
        return True, "empty"
    err = float(np.max(np.abs(w - w_ref)))
    return err <= tol, f"max|w err|={err:.3e}"


def routing_diagnostics(logits, ids, logits_ref, ids_ref) -> dict:
    """The router comparison the pages report ("We Ported Aleph Alpha's Kolibri to a MacBook.
    Our Own Gate Said No.", section "Taking it apart"): the router-logit error normalised by the
    spread of each reference row (max |dlogit| / std of the reference logits), and how often the
    selected experts disagree: as sets per token, and slot by slot."""
    lg = np.asarray(logits, np.float64)
    lr = np.asarray(logits_ref, np.float64)
    sigma = lr.std(axis=1)
    sig_err = np.max(np.abs(lg - lr), axis=1) / np.where(sigma > 0, sigma, 1.0)
    ids = np.asarray(ids)
    ids_ref = np.asarray(ids_ref)
    set_diff = np.array([set(a) != set(b) for a, b in zip(ids.tolist(), ids_ref.tolist())])
    return {"sigma_err_max": float(sig_err.max()), "sigma_err_mean": float(sig_err.mean()),
            "token_set_disagreement": float(set_diff.mean()),
            "slot_disagreement": float(np.mean(ids != ids_ref))}
