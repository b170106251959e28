"""Pins for the float64 oracle: each checks it against something other than
itself -- a closed form, an invariant, a special case that reduces to a
textbook formula, exact rational arithmetic on tiny inputs, or another form
of the same operator -- so that a dropped term, a wrong sign or index, or a
transposed operand fails at least one of them.

Page passages (LION rebuttal page on paperhub.cn, "LION: A bidirectional
framework that trains like a Transformer and infers like an RNN"):
  * Theorem 3.3: full form Y = SCALE(QK^T (.) M) V (Eq 25) equals the
    bidirectional RNN (Eq 20-24) -- reply "Concern 1".
  * Causal Linear-Transformer recurrence and its two-direction extension that
    removes the diagonal once -- reply "1: Recurrence Form ...".
  * All-ones mask when lambda_i = 1; scaling does not change the result --
    reply "5) Mask M for Linear Transformer".
  * Feature maps elu+1 (LIT) and normalised SiLU (LION-S) -- reply "4)".
  * Mask built from a cumulative sum -- reply "P3: LION-S uses cumsum".
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

MASKS = (0, 1, 2)


def _inputs(rng, B, H, L, d, mask_kind, lam_lo=0.3, lam_hi=0.99):
    q = rng.standard_normal((B, H, L, d))
    k = rng.standard_normal((B, H, L, d))
    v = rng.standard_normal((B, H, L, d))
    if mask_kind == 0:
        ll = None
    elif mask_kind == 1:
        ll = np.log(rng.uniform(lam_lo, lam_hi, size=H))
    else:
        ll = np.log(rng.uniform(lam_lo, lam_hi, size=(B, H, L)))
    return q, k, v, ll


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def _rel_rows_kappa(o, y, ref, q, k, ll, mask_kind, phi_kind):
    """max over rows of ||y_i - ref_i||_inf / (||ref_i||_inf * max(1, kappa_i)):
    features that can be negative (SiLU) may make a row sum cancel."""
    B, H, L, _ = q.shape
    worst = 0.0
    for b in range(B):
        for h in range(H):
            kap = o.row_kappa(q, k, ll, mask_kind, b, h, 0, L, phi_kind)
            err = np.max(np.abs(y[b, h] - ref[b, h]), axis=-1)
            nrm = np.max(np.abs(ref[b, h]), axis=-1)
            worst = max(worst, float(np.max(err / (nrm * np.maximum(1.0, kap)))))
    return worst


# ---------------------------------------------------------------- P1 -----
@pytest.mark.parametrize("mask_kind", MASKS)
@pytest.mark.parametrize("phi_kind", (0, 1, 2, 3))
def test_three_forms_agree_small(oracle_mod, mask_kind, phi_kind):
    """Theorem 3.3: full == bidirectional RNN == chunkwise for L <= 16, every
    chunk length (including 1, non-divisors and C >= L)."""
    o = oracle_mod
    rng = np.random.default_rng(100 + mask_kind * 10 + phi_kind)
    for L in (1, 2, 3, 5, 8, 13, 16):
        for d in (1, 3, 4):
            q, k, v, ll = _inputs(rng, 2, 2, L, d, mask_kind)
            if phi_kind == 3:           # identity features: keep row sums away from 0
                q, k = np.abs(q) + 0.1, np.abs(k) + 0.1
            silu = phi_kind == 2 or (phi_kind == 0 and mask_kind == 2)
            if silu and d == 1:
                continue                # phi = sign(x): row sums are exactly 0 or +-L
            yf = o.full(q, k, v, ll, mask_kind, phi_kind)
            yr = o.rnn(q, k, v, ll, mask_kind, phi_kind)
            err = (lambda y: _rel_rows_kappa(o, y, yf, q, k, ll, mask_kind, phi_kind)) if silu \
                else (lambda y: _rel(y, yf))
            assert err(yr) < 1e-11, (L, d)
            for C in sorted({1, 2, 3, 4, 5, L, L + 3}):
                yc = o.chunk(q, k, v, ll, mask_kind, C, phi_kind)
                assert err(yc) < 1e-11, (L, d, C)


# ---------------------------------------------------------------- P2 -----
@pytest.mark.parametrize("phi_kind", (1, 2))
def test_lit_closed_form(oracle_mod, phi_kind):
    """All-ones mask: y_i = phi(q_i)^T (sum_j phi(k_j) v_j^T) / phi(q_i)^T sum_j phi(k_j)
    (linear attention by associativity; no L x L matrix)."""
    o = oracle_mod
    rng = np.random.default_rng(7)
    q, k, v, _ = _inputs(rng, 2, 3, 37, 8, 0)
    fq = torch.nn.functional.elu(torch.from_numpy(q)) + 1.0 if phi_kind == 1 else None
    if phi_kind == 1:
        fk = torch.nn.functional.elu(torch.from_numpy(k)) + 1.0
    else:
        fq = torch.nn.functional.normalize(torch.nn.functional.silu(torch.from_numpy(q)), dim=-1, eps=1e-12)
        fk = torch.nn.functional.normalize(torch.nn.functional.silu(torch.from_numpy(k)), dim=-1, eps=1e-12)
    kv = torch.einsum("bhjm,bhjn->bhmn", fk, torch.from_numpy(v))
    ksum = fk.sum(dim=2)
    num = torch.einsum("bhim,bhmn->bhin", fq, kv)
    den = torch.einsum("bhim,bhm->bhi", fq, ksum)
    ref = (num / den[..., None]).numpy()
    for y in (o.full(q, k, v, None, 0, phi_kind), o.rnn(q, k, v, None, 0, phi_kind),
              o.chunk(q, k, v, None, 0, 5, phi_kind)):
        assert _rel(y, ref) < 1e-11


# ---------------------------------------------------------------- P3 -----
def test_d_mask_is_symmetric_toeplitz(oracle_mod):
    """LION-D: M_ij = lambda^|i-j| for a fixed per-head lambda."""
    o = oracle_mod
    L = 23
    for lam in (0.5, 0.9, 0.999):
        ll = np.array([0.0, np.log(lam)])
        M = o.mask(1, ll, L, b=0, h=1, H=2)
        i = np.arange(L)
        ref = lam ** np.abs(i[:, None] - i[None, :]).astype(np.float64)
        assert np.allclose(M, ref, rtol=1e-13, atol=0)
        assert np.array_equal(M, M.T)
        for off in range(-L + 1, L):   # Toeplitz: constant along each diagonal
            dg = np.diagonal(M, off)
            assert np.allclose(dg, dg[0], rtol=1e-13, atol=0)


def test_s_mask_index_convention(oracle_mod):
    """LION-S reading: M_ij = prod_{k=min(i,j)+1}^{max(i,j)} lambda_k, M_ii = 1,
    symmetric, lambda_0 unused, and equal to exp of cumsum differences."""
    o = oracle_mod
    lam = np.array([0.11, 0.5, 0.25, 0.8, 0.9])
    ll = np.log(lam)[None, None, :]
    M = o.mask(2, ll, 5, b=0, h=0, H=1)
    assert np.allclose(np.diag(M), 1.0)
    assert np.isclose(M[0, 1], 0.5) and np.isclose(M[1, 0], 0.5)
    assert np.isclose(M[0, 2], 0.5 * 0.25) and np.isclose(M[2, 0], 0.5 * 0.25)
    assert np.isclose(M[1, 4], 0.25 * 0.8 * 0.9)
    assert np.isclose(M[4, 1], 0.25 * 0.8 * 0.9)
    assert np.allclose(M, M.T, rtol=1e-14)
    P = np.cumsum(np.log(lam))
    i = np.arange(5)
    ref = np.exp(-np.abs(P[:, None] - P[None, :]))
    assert np.allclose(M, ref, rtol=1e-13)
    ll2 = ll.copy()
    ll2[0, 0, 0] = np.log(0.999)     # lambda_0 never enters the mask
    assert np.array_equal(o.mask(2, ll2, 5, H=1), M)
    del i


# ---------------------------------------------------------------- P4 -----
@pytest.mark.parametrize("mask_kind", MASKS)
def test_convex_hull_positive_features(oracle_mod, mask_kind):
    """elu+1 features give s_ij > 0 and M_ij > 0, so y_i is a convex
    combination of the v_j: each coordinate lies in [min_j v_jn, max_j v_jn]."""
    o = oracle_mod
    rng = np.random.default_rng(11 + mask_kind)
    q, k, v, ll = _inputs(rng, 2, 2, 40, 6, mask_kind)
    y = o.chunk(q, k, v, ll, mask_kind, 7, 1)
    lo = v.min(axis=2, keepdims=True)
    hi = v.max(axis=2, keepdims=True)
    assert np.all(y >= lo - 1e-12) and np.all(y <= hi + 1e-12)


# ---------------------------------------------------------------- P5 -----
def test_unit_decay_reduces_to_lit(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(21)
    q, k, v, _ = _inputs(rng, 2, 2, 19, 5, 0)
    ref = o.full(q, k, v, None, 0, 1)
    yd = o.rnn(q, k, v, np.zeros(2), 1, 1)
    ys = o.chunk(q, k, v, np.zeros((2, 2, 19)), 2, 4, 1)
    assert _rel(yd, ref) < 1e-12 and _rel(ys, ref) < 1e-12


@pytest.mark.parametrize("mask_kind", (1, 2))
def test_vanishing_decay_gives_identity(oracle_mod, mask_kind):
    """lambda -> 0 (log lambda = -1e4): M = I, so y_i = s_ii v_i / s_ii = v_i."""
    o = oracle_mod
    rng = np.random.default_rng(31)
    q, k, v, _ = _inputs(rng, 1, 2, 12, 4, 0)
    ll = np.full(2, -1e4) if mask_kind == 1 else np.full((1, 2, 12), -1e4)
    for y in (o.full(q, k, v, ll, mask_kind, 1), o.rnn(q, k, v, ll, mask_kind, 1),
              o.chunk(q, k, v, ll, mask_kind, 5, 1)):
        assert _rel(y, v) < 1e-12


def test_forward_half_is_causal_linear_transformer(oracle_mod):
    """With lambda = 1 the forward recurrence is the causal Linear Transformer:
    S_i = S_{i-1} + k_i v_i^T, z_i = z_{i-1} + k_i, y_i = q_i^T S_i / q_i^T z_i
    (rebuttal page, reply "1: Recurrence Form"), here unrolled with cumsum."""
    o = oracle_mod
    rng = np.random.default_rng(41)
    q, k, v, _ = _inputs(rng, 1, 2, 30, 6, 0)
    yF, cF = o.rnn_forward_half(q, k, v, None, 0, 1)
    fq = np.where(q > 0, q + 1, np.exp(q))
    fk = np.where(k > 0, k + 1, np.exp(k))
    S = np.cumsum(fk[..., :, None] * v[..., None, :], axis=2)   # [B,H,L,d,d]
    z = np.cumsum(fk, axis=2)
    num = np.einsum("bhim,bhimn->bhin", fq, S)
    den = np.einsum("bhim,bhim->bhi", fq, z)
    assert _rel(yF, num) < 1e-12 and _rel(cF, den) < 1e-12


# ---------------------------------------------------------------- P6 -----
@pytest.mark.parametrize("mask_kind", MASKS)
def test_sequence_reversal(oracle_mod, mask_kind):
    """Reversing the tokens and using l'_k = l_{L-k} (k >= 1) reverses the output."""
    o = oracle_mod
    rng = np.random.default_rng(51 + mask_kind)
    L = 17
    q, k, v, ll = _inputs(rng, 1, 2, L, 4, mask_kind)
    y = o.full(q, k, v, ll, mask_kind)
    rq, rk, rv = q[:, :, ::-1], k[:, :, ::-1], v[:, :, ::-1]
    if mask_kind == 2:
        rll = np.empty_like(ll)
        rll[..., 0] = -0.3                     # unused
        rll[..., 1:] = ll[..., :0:-1]          # l'_k = l_{L-k}
    else:
        rll = ll
    yr = o.rnn(rq, rk, rv, rll, mask_kind)
    assert _rel(yr[:, :, ::-1], y) < 1e-12


# ---------------------------------------------------------------- P7 -----
@pytest.mark.parametrize("mask_kind", MASKS)
def test_query_scale_invariance(oracle_mod, mask_kind):
    """Row-sum normalisation: scaling q_i by c_i > 0 (identity features) leaves
    y unchanged -- no temperature, no epsilon in the denominator."""
    o = oracle_mod
    rng = np.random.default_rng(61 + mask_kind)
    q, k, v, ll = _inputs(rng, 1, 2, 14, 3, mask_kind)
    q, k = np.abs(q) + 0.1, np.abs(k) + 0.1
    c = rng.uniform(0.01, 100.0, size=(1, 2, 14, 1))
    y1 = o.chunk(q, k, v, ll, mask_kind, 4, 3)
    y2 = o.chunk(q * c, k, v, ll, mask_kind, 4, 3)
    assert _rel(y2, y1) < 1e-12


# ------------------------------------------------- exact tiny cases -----
def _exact_bruteforce(q, k, v, lam):
    """Exact rational y for one head with identity features."""
    L, d = len(q), len(q[0])
    y = []
    for i in range(L):
        num = [Fraction(0)] * d
        den = Fraction(0)
        for j in range(L):
            m = Fraction(1)
            for t in range(min(i, j) + 1, max(i, j) + 1):
                m *= lam[t]
            s = sum(q[i][a] * k[j][a] for a in range(d))
            den += m * s
            for n in range(d):
                num[n] += m * s * v[j][n]
        y.append([float(x / den) for x in num])
    return np.array(y)


def test_exact_rational_tiny(oracle_mod):
    o = oracle_mod
    q = [[Fraction(1), Fraction(2)], [Fraction(3), Fraction(1)], [Fraction(1, 2), Fraction(5)]]
    k = [[Fraction(2), Fraction(1)], [Fraction(1), Fraction(1)], [Fraction(4), Fraction(1, 3)]]
    v = [[Fraction(1), Fraction(-2)], [Fraction(-3), Fraction(1)], [Fraction(2), Fraction(7)]]
    lam = [Fraction(1, 3), Fraction(1, 2), Fraction(1, 4)]
    ref = _exact_bruteforce(q, k, v, lam)
    arr = lambda m: np.array([[float(x) for x in r] for r in m])[None, None]  # noqa: E731
    ll = np.log(np.array([float(x) for x in lam]))[None, None]
    for y in (o.full(arr(q), arr(k), arr(v), ll, 2, 3), o.rnn(arr(q), arr(k), arr(v), ll, 2, 3),
              o.chunk(arr(q), arr(k), arr(v), ll, 2, 2, 3)):
        assert _rel(y[0, 0], ref) < 1e-14
    # L = 2, d = 1 by hand: y_0 = (s00 v0 + lam1 s01 v1) / (s00 + lam1 s01)
    q2, k2, v2 = np.array([[[[2.0], [1.0]]]]), np.array([[[[3.0], [5.0]]]]), np.array([[[[1.0], [4.0]]]])
    ll2 = np.log(np.array([[[0.7, 0.25]]]))
    y = o.full(q2, k2, v2, ll2, 2, 3)
    y0 = (6 * 1 + 0.25 * 10 * 4) / (6 + 0.25 * 10)
    y1 = (0.25 * 3 * 1 + 5 * 4) / (0.25 * 3 + 5)
    assert np.allclose(y[0, 0, :, 0], [y0, y1], rtol=1e-14)


# ---------------------------------------------------------------- phi ----
def test_feature_maps(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(71)
    x = rng.standard_normal((9, 16)) * 3
    t = torch.from_numpy(x)
    assert np.allclose(o.phi(1, x), (torch.nn.functional.elu(t) + 1).numpy(), rtol=1e-14, atol=1e-15)
    ref = torch.nn.functional.normalize(torch.nn.functional.silu(t), dim=-1, eps=1e-12).numpy()
    assert np.allclose(o.phi(2, x), ref, rtol=1e-13, atol=1e-16)
    assert np.array_equal(o.phi(3, x), x)
    z = np.zeros((2, 8))
    assert np.array_equal(o.phi(2, z), z)       # ||u|| clamped at 1e-12, no NaN


# ------------------------------------------------------ sampled rows -----
@pytest.mark.parametrize("mask_kind", MASKS)
def test_sampled_rows_match_full(oracle_mod, mask_kind):
    o = oracle_mod
    rng = np.random.default_rng(81 + mask_kind)
    q, k, v, ll = _inputs(rng, 2, 3, 29, 5, mask_kind)
    y = o.full(q, k, v, ll, mask_kind)
    idx = [0, 7, 28, 13]
    yr = o.rows(q, k, v, ll, mask_kind, 1, 2, idx)
    assert _rel(yr, y[1, 2, idx]) < 1e-13


def test_kappa_is_one_for_positive_features(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(91)
    q, k, v, ll = _inputs(rng, 1, 1, 20, 4, 2)
    kap = o.row_kappa(q, k, ll, 2, 0, 0, 0, 20, phi_kind=1)
    assert np.allclose(kap, 1.0, rtol=1e-12)
    kap2 = o.row_kappa(q, k, ll, 2, 0, 0, 0, 20)    # SiLU features may cancel
    assert np.all(kap2 >= 1.0 - 1e-12)


def test_kappa_hand_cases(oracle_mod):
    """Identity features, LIT mask (M = 1), values worked by hand.
    One token, q = (2, -1), k = (1, 1): s = 1, |q|.|k| = 3, kappa = 3.
    Two tokens, q_0 = (1, 1), k_0 = (1, 1), k_1 = (-0.5, 3): s_00 = 2,
    s_01 = 2.5, |q_0|.|k_1| = 3.5, kappa_0 = (2 + 3.5) / (2 + 2.5) = 11/9."""
    o = oracle_mod
    q = np.array([2.0, -1.0]).reshape(1, 1, 1, 2)
    k = np.array([1.0, 1.0]).reshape(1, 1, 1, 2)
    assert o.row_kappa(q, k, None, 0, 0, 0, 0, 1, phi_kind=3)[0] == pytest.approx(3.0, rel=1e-15)
    q = np.array([[1.0, 1.0], [0.3, 0.7]]).reshape(1, 1, 2, 2)
    k = np.array([[1.0, 1.0], [-0.5, 3.0]]).reshape(1, 1, 2, 2)
    assert o.row_kappa(q, k, None, 0, 0, 0, 0, 1, phi_kind=3)[0] == pytest.approx(11.0 / 9.0, rel=1e-15)


def test_invalid_arguments(oracle_mod):
    o = oracle_mod
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(ValueError):
        o.full(q, q, q, None, 1)                      # LION-D without decays
    with pytest.raises(ValueError):
        o.chunk(q, q, q, None, 0, 0)                  # chunk < 1


# ------------------------------------------------------ backward (full form) --
# The gradients of sum(dy * y) with respect to q, k, v and log lambda: the
# operator is the pages' training path (the full form trains like a
# Transformer, rebuttal page reply "Concern 1", Theorem 3.3 Eq 25).

def _fd_loss(oracle_mod, q, k, v, ll, dy, mask_kind, phi_kind):
    return float((oracle_mod.full(q, k, v, ll, mask_kind, phi_kind) * dy).sum())


@pytest.mark.parametrize("mask_kind", MASKS)
@pytest.mark.parametrize("phi_kind", (1, 2, 3))
def test_full_bwd_matches_finite_differences(oracle_mod, mask_kind, phi_kind):
    """Every element of dq, dk, dv (and dlog_lambda) against central
    differences of the forward oracle (step 1e-6, float64)."""
    rng = np.random.default_rng(40 + 3 * mask_kind + phi_kind)
    q, k, v, ll = _inputs(rng, 1, 2, 6, 4, mask_kind, lam_lo=0.5)
    if phi_kind == 3:   # identity features: keep the row sums away from zero
        q, k = np.abs(q) + 0.3, np.abs(k) + 0.3
    dy = rng.standard_normal(q.shape)
    dq, dk, dv, dll = oracle_mod.full_bwd(q, k, v, ll, dy, mask_kind, phi_kind)
    eps = 1e-6
    named = {"q": (q, dq), "k": (k, dk), "v": (v, dv)}
    if ll is not None:
        named["ll"] = (ll, dll)
    for name, (arr, grad) in named.items():
        for idx in np.ndindex(arr.shape):
            args = {"q": q, "k": k, "v": v, "ll": ll}
            a = arr.copy()
            a[idx] += eps
            args[name] = a
            fp = _fd_loss(oracle_mod, args["q"], args["k"], args["v"], args["ll"], dy, mask_kind, phi_kind)
            a[idx] -= 2 * eps
            fm = _fd_loss(oracle_mod, args["q"], args["k"], args["v"], args["ll"], dy, mask_kind, phi_kind)
            fd = (fp - fm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 2e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])
    if mask_kind == 2:
        assert np.all(dll[..., 0] == 0.0)   # l_0 never enters the mask


@pytest.mark.parametrize("mask_kind", MASKS)
def test_full_bwd_euler_identity_in_v(oracle_mod, mask_kind):
    """y is homogeneous of degree 1 in v, so <dy, y> = <dv, v>."""
    rng = np.random.default_rng(50 + mask_kind)
    q, k, v, ll = _inputs(rng, 2, 2, 13, 5, mask_kind)
    dy = rng.standard_normal(q.shape)
    _, _, dv, _ = oracle_mod.full_bwd(q, k, v, ll, dy, mask_kind)
    y = oracle_mod.full(q, k, v, ll, mask_kind)
    assert abs((dy * y).sum() - (dv * v).sum()) <= 1e-10 * max(1.0, abs((dy * y).sum()))


@pytest.mark.parametrize("mask_kind", MASKS)
def test_full_bwd_query_scale_invariance(oracle_mod, mask_kind):
    """With identity features y_i does not change when q_i is scaled, so the
    gradient with respect to q_i is orthogonal to q_i."""
    rng = np.random.default_rng(60 + mask_kind)
    q, k, v, ll = _inputs(rng, 1, 3, 11, 6, mask_kind)
    q, k = np.abs(q) + 0.2, np.abs(k) + 0.2
    dy = rng.standard_normal(q.shape)
    dq, _, _, _ = oracle_mod.full_bwd(q, k, v, ll, dy, mask_kind, 3)
    dots = (dq * q).sum(-1)
    assert np.abs(dots).max() <= 1e-10 * max(1.0, np.abs(dq).max() * np.abs(q).max())


def test_full_bwd_d_is_the_sum_of_s(oracle_mod):
    """LION-D is LION-S with every position carrying log lambda_h: its
    gradient is the sum over batch and positions of the per-token ones, and
    the other gradients coincide."""
    rng = np.random.default_rng(70)
    q, k, v, ll_d = _inputs(rng, 2, 3, 9, 4, 1)
    ll_s = np.broadcast_to(ll_d[None, :, None], (2, 3, 9)).copy()
    dy = rng.standard_normal(q.shape)
    gd = oracle_mod.full_bwd(q, k, v, ll_d, dy, 1, 1)
    gs = oracle_mod.full_bwd(q, k, v, ll_s, dy, 2, 1)
    for a, b in zip(gd[:3], gs[:3]):
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(a).max())
    assert np.abs(gd[3] - gs[3].sum(axis=(0, 2))).max() <= 1e-10 * max(1.0, np.abs(gd[3]).max())


# ------------------------------------------------- reordered full form ----
# The mask averaged over two traversal orders of the tokens (rebuttal page,
# reply "P2: Comparison against vision SSMs", item 1: the two masks of its
# Figure 7 b and c are averaged; results page "LION Part IV - Results",
# "Model Comparisons", the reordered-patch models).  Along an order the mask
# is LION's mask of the reordered sequence.

def _non_involution(rng, L):
    while True:
        p = rng.permutation(L)
        if np.any(p[p] != np.arange(L)):
            return p


@pytest.mark.parametrize("mask_kind", MASKS)
def test_reordered_one_order_twice_is_lion_on_the_reordered_sequence(oracle_mod, mask_kind):
    """Both orders equal to pi: the plain operator run on the tokens (with
    their decays) taken in the order pi, its output put back in place."""
    rng = np.random.default_rng(900 + mask_kind)
    B, H, L, d = 2, 2, 11, 5
    q, k, v, ll = _inputs(rng, B, H, L, d, mask_kind)
    pi = _non_involution(rng, L)
    got = oracle_mod.full_reordered(q, k, v, ll, np.stack([pi, pi]), mask_kind)
    llp = ll[..., pi] if mask_kind == 2 else ll
    yp = oracle_mod.full(q[:, :, pi], k[:, :, pi], v[:, :, pi], llp, mask_kind)
    want = np.empty_like(yp)
    want[:, :, pi] = yp
    assert _rel(got, want) < 1e-12


def test_reordered_order_swap_and_lit(oracle_mod):
    rng = np.random.default_rng(910)
    L = 13
    o1, o2 = rng.permutation(L), rng.permutation(L)
    q, k, v, ll = _inputs(rng, 1, 2, L, 4, 2)
    a = oracle_mod.full_reordered(q, k, v, ll, np.stack([o1, o2]), 2)
    b = oracle_mod.full_reordered(q, k, v, ll, np.stack([o2, o1]), 2)
    assert _rel(a, b) < 1e-14
    # LIT: every order gives the all-ones mask
    got = oracle_mod.full_reordered(q, k, v, None, np.stack([o1, o2]), 0)
    assert _rel(got, oracle_mod.full(q, k, v, None, 0)) < 1e-13


def test_reordered_d_with_reversal_is_plain_d(oracle_mod):
    """LION-D along the reversed order keeps every distance |i - j|."""
    rng = np.random.default_rng(920)
    L = 12
    q, k, v, ll = _inputs(rng, 2, 3, L, 4, 1)
    orders = np.stack([np.arange(L), np.arange(L)[::-1]])
    got = oracle_mod.full_reordered(q, k, v, ll, orders, 1)
    assert _rel(got, oracle_mod.full(q, k, v, ll, 1)) < 1e-13


def test_reordered_s_with_reversal_closed_form(oracle_mod):
    """LION-S, orders (identity, reversal): for i < j the reversed traversal
    multiplies lambda_i .. lambda_{j-1} instead of lambda_{i+1} .. lambda_j,
    so M_ij = (prod_{i<t<=j} lambda_t + prod_{i<=t<j} lambda_t) / 2 (and
    symmetric).  Identity features, written out with explicit products."""
    rng = np.random.default_rng(930)
    B, H, L, d = 1, 2, 10, 3
    q, k, v, ll = _inputs(rng, B, H, L, d, 2)
    q, k = np.abs(q) + 0.25, np.abs(k) + 0.25
    orders = np.stack([np.arange(L), np.arange(L)[::-1]])
    got = oracle_mod.full_reordered(q, k, v, ll, orders, 2, phi_kind=3)
    lam = np.exp(ll)
    for b in range(B):
        for h in range(H):
            M = np.ones((L, L))
            for i in range(L):
                for j in range(i + 1, L):
                    fwd = np.prod(lam[b, h, i + 1:j + 1])
                    rev = np.prod(lam[b, h, i:j])
                    M[i, j] = M[j, i] = 0.5 * (fwd + rev)
            A = (q[b, h] @ k[b, h].T) * M
            want = (A @ v[b, h]) / A.sum(axis=1, keepdims=True)
            assert _rel(got[b, h], want) < 1e-12


def test_reordered_s_matches_cumsum_route(oracle_mod):
    """General orders, LION-S: the mask along an order from the cumulative
    sum of the reordered log-decays (M = exp(-|C_{r(a)} - C_{r(b)}|), r the
    position of a token in the order), against the oracle's products."""
    rng = np.random.default_rng(940)
    B, H, L, d = 2, 1, 14, 4
    q, k, v, ll = _inputs(rng, B, H, L, d, 2)
    q, k = np.abs(q) + 0.25, np.abs(k) + 0.25
    orders = np.stack([rng.permutation(L), rng.permutation(L)])
    got = oracle_mod.full_reordered(q, k, v, ll, orders, 2, phi_kind=3)
    for b in range(B):
        M = np.zeros((L, L))
        for o in orders:
            rank = np.empty(L, dtype=int)
            rank[o] = np.arange(L)
            C = np.cumsum(ll[b, 0][o])
            Cr = C[rank]
            M += 0.5 * np.exp(-np.abs(Cr[:, None] - Cr[None, :]))
        A = (q[b, 0] @ k[b, 0].T) * M
        want = (A @ v[b, 0]) / A.sum(axis=1, keepdims=True)
        assert _rel(got[b, 0], want) < 1e-12


@pytest.mark.parametrize("mask_kind", MASKS)
def test_reordered_convex_hull(oracle_mod, mask_kind):
    rng = np.random.default_rng(950 + mask_kind)
    L = 15
    q, k, v, ll = _inputs(rng, 1, 2, L, 6, mask_kind)
    y = oracle_mod.full_reordered(q, k, v, ll, np.stack([rng.permutation(L), rng.permutation(L)]),
                                  mask_kind, phi_kind=1)
    assert np.all(y >= v.min(axis=2, keepdims=True) - 1e-12)
    assert np.all(y <= v.max(axis=2, keepdims=True) + 1e-12)


def test_reordered_rejects_non_permutations(oracle_mod):
    rng = np.random.default_rng(960)
    q, k, v, ll = _inputs(rng, 1, 1, 5, 2, 2)
    good = np.arange(5)
    for bad in (np.array([0, 1, 2, 3, 3]), np.array([0, 1, 2, 3, 5]), np.array([-1, 1, 2, 3, 4])):
        with pytest.raises(ValueError):
            oracle_mod.full_reordered(q, k, v, ll, np.stack([good, bad]), 2)


# ----------------------------------------- reordered full-form gradients --
def _fd_loss_reordered(o, q, k, v, ll, orders, dy, mask_kind, phi_kind):
    return float(np.sum(dy * o.full_reordered(q, k, v, ll, orders, mask_kind, phi_kind)))


@pytest.mark.parametrize("mask_kind", MASKS)
@pytest.mark.parametrize("phi_kind", (0, 3))
def test_full_bwd_reordered_matches_finite_differences(oracle_mod, mask_kind, phi_kind):
    """Every element of dq, dk, dv and dlog_lambda of the reordered full form
    against central differences of its forward oracle (float64)."""
    rng = np.random.default_rng(970 + 3 * mask_kind + phi_kind)
    L = 6
    q, k, v, ll = _inputs(rng, 1, 2, L, 4, mask_kind, lam_lo=0.5)
    if phi_kind == 3:
        q, k = np.abs(q) + 0.3, np.abs(k) + 0.3
    orders = np.stack([_non_involution(rng, L), _non_involution(rng, L)])
    dy = rng.standard_normal(q.shape)
    dq, dk, dv, dll = oracle_mod.full_bwd_reordered(q, k, v, ll, orders, dy, mask_kind, phi_kind)
    eps = 1e-6
    named = {"q": (q, dq), "k": (k, dk), "v": (v, dv)}
    if ll is not None:
        named["ll"] = (ll, dll)
    for name, (arr, grad) in named.items():
        for idx in np.ndindex(arr.shape):
            args = {"q": q, "k": k, "v": v, "ll": ll}
            a = arr.copy()
            a[idx] += eps
            args[name] = a
            fp = _fd_loss_reordered(oracle_mod, args["q"], args["k"], args["v"], args["ll"], orders, dy,
                                    mask_kind, phi_kind)
            a[idx] -= 2 * eps
            fm = _fd_loss_reordered(oracle_mod, args["q"], args["k"], args["v"], args["ll"], orders, dy,
                                    mask_kind, phi_kind)
            fd = (fp - fm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 2e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


@pytest.mark.parametrize("mask_kind", MASKS)
def test_full_bwd_reordered_one_order_twice(oracle_mod, mask_kind):
    """Both orders equal to pi: the gradients of the plain operator on the
    reordered sequence, put back in place (LIT: the plain gradients)."""
    rng = np.random.default_rng(980 + mask_kind)
    B, H, L, d = 2, 2, 9, 4
    q, k, v, ll = _inputs(rng, B, H, L, d, mask_kind)
    pi = _non_involution(rng, L)
    dy = rng.standard_normal(q.shape)
    got = oracle_mod.full_bwd_reordered(q, k, v, ll, np.stack([pi, pi]), dy, mask_kind)
    llp = ll[..., pi] if mask_kind == 2 else ll
    ref = oracle_mod.full_bwd(q[:, :, pi], k[:, :, pi], v[:, :, pi], llp, dy[:, :, pi], mask_kind)
    for n, (g, r) in enumerate(zip(got[:3], ref[:3])):
        back = np.empty_like(r)
        back[:, :, pi] = r
        assert _rel(g, back) < 1e-12, n
    if mask_kind == 2:
        back = np.empty_like(ref[3])
        back[..., pi] = ref[3]
        assert _rel(got[3], back) < 1e-12
    elif mask_kind == 1:
        assert _rel(got[3], ref[3]) < 1e-12
    else:
        assert got[3] is None
