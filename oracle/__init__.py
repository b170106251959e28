"""float64 CPU oracle for the LION bidirectional masked linear-attention operator.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never loads it, and this package imports nothing from the CUDA side.

The arithmetic lives in ``lion_oracle.c`` (plain C, float64, optional OpenMP
over heads).  This module only compiles it with gcc and marshals numpy arrays.

Forms (see the C file's header for the definitions and the page passages they
follow):

* :func:`full`  -- brute force ``Y = SCALE(QK^T (.) M) V`` with an explicit mask
  (rebuttal page, "Concern 1", Theorem 3.3 Eq 25).
* :func:`rnn`   -- forward and backward recurrences, diagonal removed once
  (rebuttal page, Theorem 3.3 Eq 20-24 and reply "1: Recurrence Form").
* :func:`chunk` -- chunkwise form ("LION Part IV - Results", "LION Chunk").
* :func:`full_reordered` -- the full form with the mask averaged over two
  traversal orders of the tokens (rebuttal page, "P2: Comparison against
  vision SSMs", item 1; the results page's reordered-patch models).
* :func:`rows`  -- brute force for a sample of rows of one head.
* :func:`mask`  -- the explicit mask of one head.
* :func:`phi`   -- the feature maps.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lion_oracle.c")
_LIB = os.path.join(_HERE, "liblion_oracle.so")

MASK_LIT, MASK_D, MASK_S = 0, 1, 2
PHI_DEFAULT, PHI_ELU1, PHI_SILU_L2, PHI_IDENTITY = 0, 1, 2, 3

_lib = None


def build(force: bool = False) -> str:
    """Compile ``lion_oracle.c`` into ``liblion_oracle.so`` (gcc, -O2, OpenMP if
    available).  Returns the library path."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        lib.oracle_phi.argtypes = [i, dp, ctypes.c_long, i, dp]
        lib.oracle_mask.argtypes = [i, dp, i, i, i, i, dp]
        form = [dp, dp, dp, dp, i, i, i, i, i, i]
        lib.oracle_lion_full.argtypes = form + [dp, i]
        lib.oracle_lion_rnn.argtypes = form + [dp, i]
        lib.oracle_lion_chunk.argtypes = form + [i, dp, i]
        lib.oracle_lion_rows.argtypes = form + [i, i, ctypes.POINTER(ctypes.c_int), i, dp]
        lib.oracle_row_kappa.argtypes = [dp, dp, dp, i, i, i, i, i, i, i, i, i, i, dp]
        lib.oracle_threads.argtypes = [i]
        lib.oracle_rnn_forward_half.argtypes = form + [dp, dp]
        lib.oracle_lion_full_bwd.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i, dp, dp, dp, dp, i]
        lib.oracle_lion_full_reordered.argtypes = [dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int),
                                                   i, i, i, i, i, i, dp, i]
        lib.oracle_lion_full_bwd_reordered.argtypes = [dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int), dp,
                                                       i, i, i, i, i, i, dp, dp, dp, dp, i]
        lib.oracle_lion_full_bwd_reordered.restype = ctypes.c_int
        for f in (lib.oracle_phi, lib.oracle_mask, lib.oracle_lion_full, lib.oracle_lion_rnn,
                  lib.oracle_lion_chunk, lib.oracle_lion_rows, lib.oracle_row_kappa,
                  lib.oracle_threads, lib.oracle_rnn_forward_half, lib.oracle_lion_full_bwd,
                  lib.oracle_lion_full_reordered):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _prep(q, k, v, log_lambda):
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [B, H, L, d] shape")
    return q, k, v, _f64(log_lambda)


def _check_ll(mask_kind, ll, B, H, L):
    if mask_kind == MASK_D and (ll is None or ll.shape != (H,)):
        raise ValueError("LION-D takes log_lambda of shape [H]")
    if mask_kind == MASK_S and (ll is None or ll.shape != (B, H, L)):
        raise ValueError("LION-S takes log_lambda of shape [B, H, L]")


def threads(n: int = 0) -> int:
    """OpenMP threads a call with ``threads=n`` uses (0 = all available)."""
    return _load().oracle_threads(n)


def phi(kind: int, x) -> np.ndarray:
    x = _f64(x)
    out = np.empty_like(x)
    d = x.shape[-1]
    rc = _load().oracle_phi(kind, _ptr(x), x.size // d, d, _ptr(out))
    if rc:
        raise ValueError(f"oracle_phi failed ({rc})")
    return out


def mask(mask_kind: int, log_lambda, L: int, b: int = 0, h: int = 0, H: int = 1) -> np.ndarray:
    ll = _f64(log_lambda)
    M = np.empty((L, L))
    rc = _load().oracle_mask(mask_kind, _ptr(ll), b, h, H, L, _ptr(M))
    if rc:
        raise ValueError(f"oracle_mask failed ({rc})")
    return M


def _run(fn, q, k, v, log_lambda, mask_kind, phi_kind, extra_before_y=(), threads=1):
    q, k, v, ll = _prep(q, k, v, log_lambda)
    B, H, L, d = q.shape
    _check_ll(mask_kind, ll, B, H, L)
    y = np.empty_like(q)
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(ll), B, H, L, d, mask_kind, phi_kind,
            *extra_before_y, _ptr(y), threads)
    if rc:
        raise ValueError(f"oracle call failed ({rc})")
    return y


def full(q, k, v, log_lambda, mask_kind, phi_kind=PHI_DEFAULT, threads=1):
    return _run(_load().oracle_lion_full, q, k, v, log_lambda, mask_kind, phi_kind, threads=threads)


def rnn(q, k, v, log_lambda, mask_kind, phi_kind=PHI_DEFAULT, threads=1):
    return _run(_load().oracle_lion_rnn, q, k, v, log_lambda, mask_kind, phi_kind, threads=threads)


def chunk(q, k, v, log_lambda, mask_kind, chunk, phi_kind=PHI_DEFAULT, threads=1):
    return _run(_load().oracle_lion_chunk, q, k, v, log_lambda, mask_kind, phi_kind,
                extra_before_y=(int(chunk),), threads=threads)


def full_reordered(q, k, v, log_lambda, orders, mask_kind, phi_kind=PHI_DEFAULT, threads=1):
    """Full form with the mask averaged over two traversal orders of the
    tokens: ``orders`` is [2][L] (each row a permutation; position t of order
    p holds token orders[p][t]), the same for every (b, h)."""
    q, k, v, ll = _prep(q, k, v, log_lambda)
    B, H, L, d = q.shape
    _check_ll(mask_kind, ll, B, H, L)
    o = np.ascontiguousarray(np.asarray(orders, dtype=np.int32))
    if o.shape != (2, L):
        raise ValueError("orders must be [2][L]")
    y = np.empty_like(q)
    rc = _load().oracle_lion_full_reordered(_ptr(q), _ptr(k), _ptr(v), _ptr(ll),
                                            o.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                            B, H, L, d, mask_kind, phi_kind, _ptr(y), threads)
    if rc:
        raise ValueError(f"oracle call failed ({rc})")
    return y


def full_bwd(q, k, v, log_lambda, dy, mask_kind, phi_kind=PHI_DEFAULT, threads=1):
    """Gradients of sum(dy * y) for the full form: ``(dq, dk, dv, dlog_lambda)``.
    ``dlog_lambda`` is None for LIT, [H] for D (summed over batch and
    positions), [B, H, L] for S (position 0 never enters the mask: 0)."""
    q, k, v, ll = _prep(q, k, v, log_lambda)
    B, H, L, d = q.shape
    _check_ll(mask_kind, ll, B, H, L)
    dy = _f64(dy)
    if dy.shape != q.shape:
        raise ValueError("dy must have the shape of q")
    dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    dll = None if mask_kind == MASK_LIT else np.empty((H,) if mask_kind == MASK_D else (B, H, L))
    rc = _load().oracle_lion_full_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(ll), _ptr(dy), B, H, L, d,
                                      mask_kind, phi_kind, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dll),
                                      threads)
    if rc:
        raise ValueError(f"oracle_lion_full_bwd failed ({rc})")
    return dq, dk, dv, dll


def full_bwd_reordered(q, k, v, log_lambda, orders, dy, mask_kind, phi_kind=PHI_DEFAULT, threads=1):
    """Gradients of sum(dy * y) for the reordered full form (``orders`` as in
    :func:`full_reordered`): ``(dq, dk, dv, dlog_lambda)`` shaped as
    :func:`full_bwd`'s."""
    q, k, v, ll = _prep(q, k, v, log_lambda)
    B, H, L, d = q.shape
    _check_ll(mask_kind, ll, B, H, L)
    dy = _f64(dy)
    if dy.shape != q.shape:
        raise ValueError("dy must have the shape of q")
    o = np.ascontiguousarray(np.asarray(orders, dtype=np.int32))
    if o.shape != (2, L):
        raise ValueError("orders must be [2][L]")
    dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    dll = None if mask_kind == MASK_LIT else np.empty((H,) if mask_kind == MASK_D else (B, H, L))
    rc = _load().oracle_lion_full_bwd_reordered(_ptr(q), _ptr(k), _ptr(v), _ptr(ll),
                                                o.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), _ptr(dy),
                                                B, H, L, d, mask_kind, phi_kind, _ptr(dq), _ptr(dk),
                                                _ptr(dv), _ptr(dll), threads)
    if rc:
        raise ValueError(f"oracle_lion_full_bwd_reordered failed ({rc})")
    return dq, dk, dv, dll


def rnn_forward_half(q, k, v, log_lambda, mask_kind, phi_kind=PHI_DEFAULT):
    """The forward recurrence alone: ``(yF [B,H,L,d], cF [B,H,L])`` with
    yF_i = phi(q_i)^T S^F_i and cF_i = phi(q_i)^T z^F_i."""
    q, k, v, ll = _prep(q, k, v, log_lambda)
    B, H, L, d = q.shape
    _check_ll(mask_kind, ll, B, H, L)
    yF = np.empty_like(q)
    cF = np.empty((B, H, L))
    rc = _load().oracle_rnn_forward_half(_ptr(q), _ptr(k), _ptr(v), _ptr(ll), B, H, L, d,
                                         mask_kind, phi_kind, _ptr(yF), _ptr(cF))
    if rc:
        raise ValueError(f"oracle_rnn_forward_half failed ({rc})")
    return yF, cF


def rows(q, k, v, log_lambda, mask_kind, b, h, row_idx, phi_kind=PHI_DEFAULT):
    """Brute-force outputs y[b, h, row_idx, :] (float64, [len(row_idx), d])."""
    q, k, v, ll = _prep(q, k, v, log_lambda)
    B, H, L, d = q.shape
    _check_ll(mask_kind, ll, B, H, L)
    r = np.ascontiguousarray(np.asarray(row_idx, dtype=np.int32))
    y = np.empty((r.size, d))
    rc = _load().oracle_lion_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(ll), B, H, L, d, mask_kind,
                                  phi_kind, b, h, r.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                  r.size, _ptr(y))
    if rc:
        raise ValueError(f"oracle_lion_rows failed ({rc})")
    return y


def row_kappa(q, k, log_lambda, mask_kind, b, h, i0, i1, phi_kind=PHI_DEFAULT):
    """Conditioning of rows [i0, i1) of head (b, h):
    kappa_i = sum_j M_ij (|phi(q_i)| . |phi(k_j)|) / |sum_j M_ij s_ij|: the
    componentwise condition number of the row sum under relative perturbations
    of the features (1 for non-negative features)."""
    q, k = _f64(q), _f64(k)
    ll = _f64(log_lambda)
    B, H, L, d = q.shape
    out = np.empty(i1 - i0)
    rc = _load().oracle_row_kappa(_ptr(q), _ptr(k), _ptr(ll), B, H, L, d, mask_kind, phi_kind,
                                  b, h, i0, i1, _ptr(out))
    if rc:
        raise ValueError(f"oracle_row_kappa failed ({rc})")
    return out
