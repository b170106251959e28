"""Comparison helpers for the GPU-vs-oracle parity tests.

Error measure (per output row i of each head):

    err_i = ||y_i - yref_i||_inf / ||yref_i||_inf

must satisfy err_i <= tol * max(1, kappa_i), where

    kappa_i = sum_j M_ij (|phi(q_i)| . |phi(k_j)|) / |sum_j M_ij s_ij|

is the componentwise condition number of the row sum under relative
perturbations of the features: a tensor-core path rounds phi(q) and phi(k)
to 16-bit operands, and the error of each score s_ij is bounded by that
rounding times |phi(q_i)| . |phi(k_j)| (the standard dot-product bound), not
by |s_ij|.  kappa_i = 1 whenever the features are non-negative (elu+1); with
SiLU features scores and row sums can cancel and the bound widens
accordingly.  kappa is only computed (by the oracle, O(L d) per row) for rows
that miss the plain bound, which keeps full-size checks fast.

Tolerances: 2e-3 for bfloat16 inputs with float32 accumulation, 1e-5 for
float32 inputs.
"""
import numpy as np

TOL_BF16 = 2e-3
TOL_FP32 = 1e-5

# One line per labelled check, printed at the end of the pytest run (see
# conftest.pytest_terminal_summary): how much of the per-row bound each case
# used and how many rows needed the conditioning factor.
STATS = []


def row_errors(y, ref):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.max(np.abs(y - ref), axis=-1)
    den = np.max(np.abs(ref), axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        e = num / den
    e[~np.isfinite(y).all(axis=-1)] = np.inf
    e[(den == 0) & (num == 0)] = 0.0
    return e


def check_rows(oracle, y, ref, tol, q64, k64, ll64, mask_kind, phi_kind=0, max_kappa_rows=4096,
               label=None):
    """Assert the per-row bound over y, ref of shape [B, H, L, d].  Returns a
    summary dict: rows, the worst plain error, the rows that needed kappa
    (plain error above tol), the largest kappa among them, and the worst
    error as a fraction of its row's bound.  With a label the summary is
    also recorded in STATS."""
    e = row_errors(y, ref)
    bad = np.argwhere(e > tol)
    worst_scaled = float(np.max(np.minimum(e, 1e300))) / tol if e.size else 0.0
    if len(bad) > max_kappa_rows:
        raise AssertionError(f"{len(bad)} rows exceed tol {tol} before conditioning "
                             f"(worst {float(np.max(e)):.3e})")
    scaled = []
    max_kappa = 0.0
    for b, h, i in bad:
        kap = oracle.row_kappa(q64, k64, ll64, mask_kind, int(b), int(h), int(i), int(i) + 1,
                               phi_kind)[0]
        max_kappa = max(max_kappa, float(kap))
        s = e[b, h, i] / (tol * max(1.0, kap))
        scaled.append(s)
        assert s <= 1.0, (f"row (b={b}, h={h}, i={i}): err {e[b, h, i]:.3e} > "
                          f"{tol:.1e} * max(1, kappa={kap:.3e})")
    if scaled:
        worst_scaled = max(float(np.max(np.where(e <= tol, e, 0))) / tol, max(scaled))
    summary = {"rows": int(e.size), "max_err": float(np.max(e)), "kappa_rows": len(bad),
               "max_kappa": max_kappa, "worst_scaled": worst_scaled}
    if label is not None:
        STATS.append((label, summary))
    return summary


def format_stats(label, st):
    if "worst_scaled" not in st:
        return f"{label}: " + ", ".join(f"{k} {v:.3g}" if isinstance(v, float) else f"{k} {v}"
                                        for k, v in st.items())
    return (f"{label}: rows {st['rows']}, max plain err {st['max_err']:.2e}, "
            f"rows needing kappa {st['kappa_rows']} (largest kappa {st['max_kappa']:.1f}), "
            f"worst err / bound {st['worst_scaled']:.3f}")
