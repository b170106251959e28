"""Python binding of liblion.so (the C ABI in ``include/lion.h``).

Argument marshalling only: every step of the operator runs in the CUDA
library.  Tensors are PyTorch CUDA tensors (PyTorch provides device memory and
streams); they are passed to the library as raw pointers.  If the library has
not been built the calls raise -- there is no other implementation to fall
back to.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblion.so")

# enums of include/lion.h
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_NO_MEMORY, ERR_TIMEOUT, ERR_RANGE = range(7)
MASK_LIT, MASK_D, MASK_S = 0, 1, 2
FORM_FULL, FORM_RNN, FORM_CHUNK = 0, 1, 2
DTYPE_BF16, DTYPE_FP32 = 0, 1
PHI_DEFAULT, PHI_ELU1, PHI_SILU_L2, PHI_IDENTITY = 0, 1, 2, 3
FULL_MAX_L = 8192

MASKS = {"lit": MASK_LIT, "d": MASK_D, "s": MASK_S}
FORMS = {"full": FORM_FULL, "rnn": FORM_RNN, "chunk": FORM_CHUNK}


class LionError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


class _Args(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("log_lambda", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("L", ctypes.c_int), ("d", ctypes.c_int),
        ("mask_kind", ctypes.c_int), ("form", ctypes.c_int), ("chunk", ctypes.c_int),
        ("dtype", ctypes.c_int), ("phi", ctypes.c_int),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("stream", ctypes.c_void_p), ("out_bf16", ctypes.c_int),
    ]


class _BwdArgs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("log_lambda", ctypes.c_void_p), ("dy", ctypes.c_void_p),
        ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("dlog_lambda", ctypes.c_void_p),
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("L", ctypes.c_int), ("d", ctypes.c_int),
        ("mask_kind", ctypes.c_int), ("dtype", ctypes.c_int), ("phi", ctypes.c_int),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("stream", ctypes.c_void_p),
    ]


class _ReorderArgs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("log_lambda", ctypes.c_void_p), ("order", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("L", ctypes.c_int), ("d", ctypes.c_int),
        ("mask_kind", ctypes.c_int), ("dtype", ctypes.c_int), ("phi", ctypes.c_int),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("stream", ctypes.c_void_p),
    ]


class _ReorderBwdArgs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("log_lambda", ctypes.c_void_p), ("order", ctypes.c_void_p), ("dy", ctypes.c_void_p),
        ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("dlog_lambda", ctypes.c_void_p),
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("L", ctypes.c_int), ("d", ctypes.c_int),
        ("mask_kind", ctypes.c_int), ("dtype", ctypes.c_int), ("phi", ctypes.c_int),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("stream", ctypes.c_void_p),
    ]


class _HostArgs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("log_lambda", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("L", ctypes.c_int), ("d", ctypes.c_int),
        ("mask_kind", ctypes.c_int), ("form", ctypes.c_int), ("chunk", ctypes.c_int),
        ("dtype", ctypes.c_int), ("phi", ctypes.c_int), ("slices", ctypes.c_int),
        ("stream", ctypes.c_void_p),
    ]


_lib = None

EXPORTS = ("lion_attn_fwd", "lion_attn_fwd_ex", "lion_attn_workspace_bytes", "lion_rnn_step",
           "lion_status_string", "lion_abi_version", "lion_sync_status",
           "lion_attn_fwd_rnn_noalloc", "lion_attn_bwd", "lion_attn_bwd_workspace_bytes",
           "lion_attn_fwd_causal", "lion_attn_fwd_reordered", "lion_attn_reordered_workspace_bytes",
           "lion_attn_fwd_host", "lion_attn_bwd_reordered", "lion_attn_reordered_bwd_workspace_bytes",
           "lion_attn_bwd_chunk", "lion_attn_bwd_chunk_workspace_bytes", "lion_debug_set_wait_cycles",
           "lion_debug_wait_timeout")
NOALLOC_MAX_HEAD_TOKENS = 1 << 20


def load(path: str = LIB_PATH):
    """Load liblion.so (raises if it is missing: build it with ``build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"liblion.so not found at {path}: build it with "
                           "bidirectional_masked_linear_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.lion_attn_fwd.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp]
    lib.lion_attn_fwd.restype = i
    lib.lion_attn_fwd_ex.argtypes = [ctypes.POINTER(_Args)]
    lib.lion_attn_fwd_ex.restype = i
    lib.lion_attn_workspace_bytes.argtypes = [i, i, i, i, i, i]
    lib.lion_attn_workspace_bytes.restype = ctypes.c_size_t
    lib.lion_rnn_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.lion_rnn_step.restype = i
    lib.lion_status_string.argtypes = [i]
    lib.lion_status_string.restype = ctypes.c_char_p
    lib.lion_attn_fwd_rnn_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, vp, vp]
    lib.lion_attn_fwd_rnn_noalloc.restype = i
    lib.lion_sync_status.argtypes = [vp]
    lib.lion_sync_status.restype = i
    lib.lion_abi_version.argtypes = []
    lib.lion_abi_version.restype = i
    lib.lion_attn_fwd_causal.argtypes = [ctypes.POINTER(_Args)]
    lib.lion_attn_fwd_causal.restype = i
    lib.lion_attn_bwd.argtypes = [ctypes.POINTER(_BwdArgs)]
    lib.lion_attn_bwd.restype = i
    lib.lion_attn_bwd_workspace_bytes.argtypes = [i, i, i, i]
    lib.lion_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.lion_debug_set_wait_cycles.argtypes = [ctypes.c_longlong]
    lib.lion_debug_set_wait_cycles.restype = i
    lib.lion_debug_wait_timeout.argtypes = [vp]
    lib.lion_debug_wait_timeout.restype = i
    lib.lion_attn_bwd_chunk.argtypes = [ctypes.POINTER(_BwdArgs)]
    lib.lion_attn_bwd_chunk.restype = i
    lib.lion_attn_bwd_chunk_workspace_bytes.argtypes = [i, i, i, i]
    lib.lion_attn_bwd_chunk_workspace_bytes.restype = ctypes.c_size_t
    lib.lion_attn_fwd_reordered.argtypes = [ctypes.POINTER(_ReorderArgs)]
    lib.lion_attn_fwd_reordered.restype = i
    lib.lion_attn_reordered_workspace_bytes.argtypes = [i, i, i, i]
    lib.lion_attn_reordered_workspace_bytes.restype = ctypes.c_size_t
    lib.lion_attn_fwd_host.argtypes = [ctypes.POINTER(_HostArgs)]
    lib.lion_attn_fwd_host.restype = i
    lib.lion_attn_bwd_reordered.argtypes = [ctypes.POINTER(_ReorderBwdArgs)]
    lib.lion_attn_bwd_reordered.restype = i
    lib.lion_attn_reordered_bwd_workspace_bytes.argtypes = [i, i, i, i]
    lib.lion_attn_reordered_bwd_workspace_bytes.restype = ctypes.c_size_t
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().lion_status_string(status).decode()


def _check(status: int):
    if status != OK:
        raise LionError(status, status_string(status))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_FP32
    raise TypeError(f"q, k, v must be bfloat16 or float32, got {t.dtype}")


def sync_status(stream=None) -> int:
    """Synchronise the stream and return the library's device status (OK;
    ERR_TIMEOUT if a kernel gave up on a bounded wait; ERR_INVALID_ARG if a
    traversal order given to attn_fwd_reordered was not a permutation;
    ERR_RANGE if a tensor-core kernel met a value past the fp16 range)."""
    return int(load().lion_sync_status(_stream_handle(stream)))


def workspace_bytes(B, H, L, d, form, chunk=64) -> int:
    return int(load().lion_attn_workspace_bytes(B, H, L, d, form, chunk))


def attn_fwd(q, k, v, log_lambda, mask_kind, form=FORM_CHUNK, chunk=64, out=None,
             phi=PHI_DEFAULT, workspace=None, stream=None, out_dtype=torch.float32):
    """Y = SCALE((phi(Q) phi(K)^T (.) M) V) for q, k, v of shape [B, H, L, d].

    ``log_lambda``: None (LIT), [H] (D) or [B, H, L] (S), float32, on the GPU.
    Returns ``out`` ([B, H, L, d], float32, or bfloat16 with ``out_dtype``:
    the fp32 result rounded to nearest even)."""
    lib = load()
    if isinstance(mask_kind, str):
        mask_kind = MASKS[mask_kind]
    if isinstance(form, str):
        form = FORMS[form]
    B, H, L, d = q.shape
    if out is None:
        out = torch.empty((B, H, L, d), dtype=out_dtype, device=q.device)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be float32 or bfloat16")
    out_bf16 = int(out.dtype == torch.bfloat16)
    dt = _dtype_code(q)
    if log_lambda is not None and log_lambda.dtype != torch.float32:
        raise TypeError("log_lambda must be float32")
    for t in (q, k, v, out) + ((log_lambda,) if log_lambda is not None else ()):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if q.dtype != k.dtype or q.dtype != v.dtype or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share dtype and shape")
    stream_h = _stream_handle(stream)
    if dt == DTYPE_BF16 and phi == PHI_DEFAULT and workspace is None and not out_bf16:
        st = lib.lion_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), B, H, L, d, mask_kind,
                               form, chunk, _ptr(out), stream_h)
    else:
        a = _Args(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(out), B, H, L, d, mask_kind,
                  form, chunk, dt, phi, _ptr(workspace),
                  0 if workspace is None else workspace.numel() * workspace.element_size(), stream_h,
                  out_bf16)
        st = lib.lion_attn_fwd_ex(ctypes.byref(a))
    _check(st)
    return out


def attn_fwd_rnn_noalloc(q, k, v, log_lambda, mask_kind, out=None, stream=None):
    """The recurrent form without any device allocation: the library's fixed
    scratch array holds the per-token normalisers (B*H*L <= 2^20)."""
    lib = load()
    if isinstance(mask_kind, str):
        mask_kind = MASKS[mask_kind]
    B, H, L, d = q.shape
    if out is None:
        out = torch.empty((B, H, L, d), dtype=torch.float32, device=q.device)
    if out.dtype != torch.float32 or out.shape != q.shape:
        raise TypeError("out must be float32 with the shape of q")
    if log_lambda is not None and log_lambda.dtype != torch.float32:
        raise TypeError("log_lambda must be float32")
    for t in (q, k, v, out) + ((log_lambda,) if log_lambda is not None else ()):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if q.dtype != k.dtype or q.dtype != v.dtype or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share dtype and shape")
    st = lib.lion_attn_fwd_rnn_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), B, H, L, d,
                                       mask_kind, _dtype_code(q), _ptr(out), _stream_handle(stream))
    _check(st)
    return out


def rnn_step(q, k, v, log_lambda, S, z, y_part, c_part, mask_kind, stream=None):
    """One token of one direction of the recurrent form for B*H heads, in place
    on the caller-owned state ``S`` [B,H,d,d] and ``z`` [B,H,d] (float32)."""
    lib = load()
    if isinstance(mask_kind, str):
        mask_kind = MASKS[mask_kind]
    B, H, d = q.shape
    st = lib.lion_rnn_step(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(S), _ptr(z),
                           _ptr(y_part), _ptr(c_part), B, H, d, mask_kind, _dtype_code(q),
                           _stream_handle(stream))
    _check(st)
    return y_part, c_part


def bwd_workspace_bytes(B, H, L, d, form=FORM_FULL) -> int:
    if form == FORM_CHUNK:
        return int(load().lion_attn_bwd_chunk_workspace_bytes(B, H, L, d))
    return int(load().lion_attn_bwd_workspace_bytes(B, H, L, d))


def attn_bwd(q, k, v, log_lambda, dy, mask_kind, phi=PHI_DEFAULT, workspace=None, stream=None, form=FORM_FULL):
    """Gradients of a loss through Y = SCALE((phi(Q) phi(K)^T (.) M) V), given
    ``dy`` = dLoss/dY ([B, H, L, d] float32).  Returns ``(dq, dk, dv,
    dlog_lambda)`` as float32 tensors; ``dlog_lambda`` is None for LIT, [H]
    for D and [B, H, L] for S.  ``form``: FORM_FULL (lion_attn_bwd, L <=
    FULL_MAX_L) or FORM_CHUNK (lion_attn_bwd_chunk, any L)."""
    lib = load()
    if isinstance(mask_kind, str):
        mask_kind = MASKS[mask_kind]
    B, H, L, d = q.shape
    dt = _dtype_code(q)
    for t in (q, k, v, dy) + ((log_lambda,) if log_lambda is not None else ()):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if dy.dtype != torch.float32 or dy.shape != q.shape:
        raise ValueError("dy must be float32 with the shape of q")
    dq = torch.empty((B, H, L, d), dtype=torch.float32, device=q.device)
    dk = torch.empty_like(dq)
    dv = torch.empty_like(dq)
    dll = None
    if mask_kind == MASK_D:
        dll = torch.empty((H,), dtype=torch.float32, device=q.device)
    elif mask_kind == MASK_S:
        dll = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    a = _BwdArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(dy), _ptr(dq), _ptr(dk), _ptr(dv),
                 _ptr(dll), B, H, L, d, mask_kind, dt, phi, _ptr(workspace),
                 0 if workspace is None else workspace.numel() * workspace.element_size(),
                 _stream_handle(stream))
    if isinstance(form, str):
        form = FORMS[form]
    if form not in (FORM_FULL, FORM_CHUNK):
        raise ValueError("the gradients run through the full or the chunkwise form")
    entry = lib.lion_attn_bwd_chunk if form == FORM_CHUNK else lib.lion_attn_bwd
    _check(entry(ctypes.byref(a)))
    return dq, dk, dv, dll


class LionAttention(torch.autograd.Function):
    """Y = SCALE((phi(Q) phi(K)^T (.) M) V) as a differentiable op: the
    forward runs the library's forward in the given form, the backward its
    gradient kernels (the forms agree, so the gradient is the same): the
    full form up to FULL_MAX_L tokens, the chunkwise form beyond."""

    @staticmethod
    def forward(ctx, q, k, v, log_lambda, mask_kind, form=FORM_CHUNK, chunk=128, phi=PHI_DEFAULT):
        ctx.save_for_backward(q, k, v, log_lambda)
        ctx.mask_kind, ctx.phi = mask_kind, phi
        return attn_fwd(q, k, v, log_lambda, mask_kind, form, chunk, phi=phi)

    @staticmethod
    def backward(ctx, dy):
        q, k, v, log_lambda = ctx.saved_tensors
        form = FORM_FULL if q.shape[2] <= FULL_MAX_L else FORM_CHUNK
        dq, dk, dv, dll = attn_bwd(q, k, v, log_lambda, dy.contiguous().float(), ctx.mask_kind, ctx.phi,
                                   form=form)
        return (dq.to(q.dtype), dk.to(k.dtype), dv.to(v.dtype),
                None if log_lambda is None else dll, None, None, None, None)


def attn_fwd_causal(q, k, v, log_lambda, mask_kind, form=FORM_CHUNK, chunk=64, out=None,
                    phi=PHI_DEFAULT, workspace=None, stream=None, out_dtype=torch.float32):
    """The forward half alone (a unidirectional model): y_i = sum_{j<=i}
    M_ij s_ij v_j / sum_{j<=i} M_ij s_ij, in any form."""
    lib = load()
    if isinstance(mask_kind, str):
        mask_kind = MASKS[mask_kind]
    if isinstance(form, str):
        form = FORMS[form]
    B, H, L, d = q.shape
    if out is None:
        out = torch.empty((B, H, L, d), dtype=out_dtype, device=q.device)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be float32 or bfloat16")
    for t in (q, k, v, out) + ((log_lambda,) if log_lambda is not None else ()):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    a = _Args(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(out), B, H, L, d, mask_kind,
              form, chunk, _dtype_code(q), phi, _ptr(workspace),
              0 if workspace is None else workspace.numel() * workspace.element_size(),
              _stream_handle(stream), int(out.dtype == torch.bfloat16))
    _check(lib.lion_attn_fwd_causal(ctypes.byref(a)))
    return out


def reordered_workspace_bytes(B, H, L, d) -> int:
    return int(load().lion_attn_reordered_workspace_bytes(B, H, L, d))


def attn_fwd_reordered(q, k, v, log_lambda, orders, mask_kind, out=None, phi=PHI_DEFAULT, workspace=None,
                       stream=None):
    """Full form with the mask averaged over two traversal orders of the
    tokens: ``orders`` is an int32 device tensor [2, L] (row p: the token at
    each position of traversal p), the same for every (b, h).  fp32 output."""
    lib = load()
    if isinstance(mask_kind, str):
        mask_kind = MASKS[mask_kind]
    B, H, L, d = q.shape
    if orders.dtype != torch.int32 or tuple(orders.shape) != (2, L):
        raise ValueError("orders must be int32 of shape [2, L]")
    if out is None:
        out = torch.empty((B, H, L, d), dtype=torch.float32, device=q.device)
    for t in (q, k, v, out, orders) + ((log_lambda,) if log_lambda is not None else ()):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    a = _ReorderArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(orders), _ptr(out), B, H, L, d,
                     mask_kind, _dtype_code(q), phi, _ptr(workspace),
                     0 if workspace is None else workspace.numel() * workspace.element_size(),
                     _stream_handle(stream))
    _check(lib.lion_attn_fwd_reordered(ctypes.byref(a)))
    return out


def attn_fwd_host(q, k, v, log_lambda, mask_kind, form=FORM_CHUNK, chunk=64, out=None, phi=PHI_DEFAULT,
                  slices=0, stream=None):
    """The operator on CPU tensors (page-locked for overlap): the library
    copies batch slices in, computes and copies them out on overlapping
    streams.  Returns the CPU float32 output, complete once ``stream`` (the
    current stream by default) is synchronised."""
    lib = load()
    if isinstance(mask_kind, str):
        mask_kind = MASKS[mask_kind]
    if isinstance(form, str):
        form = FORMS[form]
    B, H, L, d = q.shape
    if out is None:
        out = torch.empty((B, H, L, d), dtype=torch.float32, pin_memory=True)
    for t in (q, k, v, out) + ((log_lambda,) if log_lambda is not None else ()):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if t.is_cuda:
            raise ValueError("attn_fwd_host takes host tensors; use attn_fwd for device tensors")
    a = _HostArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(out), B, H, L, d, mask_kind, form, chunk,
                  _dtype_code(q), phi, slices, _stream_handle(stream))
    _check(lib.lion_attn_fwd_host(ctypes.byref(a)))
    return out


def reordered_bwd_workspace_bytes(B, H, L, d) -> int:
    return int(load().lion_attn_reordered_bwd_workspace_bytes(B, H, L, d))


def attn_bwd_reordered(q, k, v, log_lambda, orders, dy, mask_kind, phi=PHI_DEFAULT, workspace=None, stream=None):
    """Gradients through attn_fwd_reordered given ``dy`` ([B, H, L, d]
    float32): ``(dq, dk, dv, dlog_lambda)`` shaped as attn_bwd's."""
    lib = load()
    if isinstance(mask_kind, str):
        mask_kind = MASKS[mask_kind]
    B, H, L, d = q.shape
    if orders.dtype != torch.int32 or tuple(orders.shape) != (2, L):
        raise ValueError("orders must be int32 of shape [2, L]")
    if dy.dtype != torch.float32 or dy.shape != q.shape:
        raise ValueError("dy must be float32 with the shape of q")
    for t in (q, k, v, dy, orders) + ((log_lambda,) if log_lambda is not None else ()):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    dq = torch.empty((B, H, L, d), dtype=torch.float32, device=q.device)
    dk = torch.empty_like(dq)
    dv = torch.empty_like(dq)
    dll = None
    if mask_kind == MASK_D:
        dll = torch.empty((H,), dtype=torch.float32, device=q.device)
    elif mask_kind == MASK_S:
        dll = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    a = _ReorderBwdArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(orders), _ptr(dy), _ptr(dq), _ptr(dk),
                        _ptr(dv), _ptr(dll), B, H, L, d, mask_kind, _dtype_code(q), phi, _ptr(workspace),
                        0 if workspace is None else workspace.numel() * workspace.element_size(),
                        _stream_handle(stream))
    _check(lib.lion_attn_bwd_reordered(ctypes.byref(a)))
    return dq, dk, dv, dll


class LionReorderedAttention(torch.autograd.Function):
    """The full form with the mask averaged over two traversal orders as a
    differentiable op: forward by attn_fwd_reordered, backward by
    attn_bwd_reordered.  ``orders`` ([2, L] int32, on the GPU) gets no
    gradient."""

    @staticmethod
    def forward(ctx, q, k, v, log_lambda, orders, mask_kind, phi=PHI_DEFAULT):
        ctx.save_for_backward(q, k, v, log_lambda, orders)
        ctx.mask_kind, ctx.phi = mask_kind, phi
        return attn_fwd_reordered(q, k, v, log_lambda, orders, mask_kind, phi=phi)

    @staticmethod
    def backward(ctx, dy):
        q, k, v, log_lambda, orders = ctx.saved_tensors
        dq, dk, dv, dll = attn_bwd_reordered(q, k, v, log_lambda, orders, dy.contiguous().float(), ctx.mask_kind,
                                             ctx.phi)
        return (dq.to(q.dtype), dk.to(k.dtype), dv.to(v.dtype), None if log_lambda is None else dll, None, None,
                None)

