"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every entry point include/lion.h declares, and rejects bad arguments
with a status before launching anything."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lion.h")


@pytest.fixture(scope="module")
def lib():
    from bidirectional_masked_linear_gb300 import build, lion
    path = build.build()
    return lion.load(path)


def _declared():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(lion_[a-z0-9_]+)\s*\(", txt)))


def test_header_declares_the_abi():
    names = _declared()
    for want in ("lion_attn_fwd", "lion_attn_fwd_ex", "lion_rnn_step", "lion_status_string",
                 "lion_attn_workspace_bytes", "lion_attn_bwd", "lion_attn_bwd_workspace_bytes",
                 "lion_attn_fwd_causal", "lion_attn_fwd_reordered", "lion_attn_reordered_workspace_bytes",
                 "lion_attn_bwd_reordered", "lion_attn_reordered_bwd_workspace_bytes", "lion_attn_fwd_host",
                 "lion_attn_bwd_chunk", "lion_attn_bwd_chunk_workspace_bytes"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    from bidirectional_masked_linear_gb300 import lion
    out = subprocess.run(["nm", "-D", "--defined-only", lion.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\b[TW] (\w+)", out))
    for name in _declared():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings_and_version(lib):
    lib.lion_status_string.restype = ctypes.c_char_p
    assert lib.lion_status_string(0) == b"ok"
    assert b"invalid" in lib.lion_status_string(1)
    assert lib.lion_status_string(99) == b"unknown status"
    assert lib.lion_abi_version() == 2


def test_workspace_query(lib):
    from bidirectional_masked_linear_gb300 import lion
    # the full form: the tiled kernel's features (and LION-S prefix) at d = 64, 128; none below
    assert lion.workspace_bytes(2, 3, 10, 64, lion.FORM_FULL) >= 2 * (2 * 3 * 10 * 64) * 4
    assert lion.workspace_bytes(2, 3, 10, 16, lion.FORM_FULL) == 0
    assert lion.workspace_bytes(2, 3, 10, 64, lion.FORM_RNN) >= 2 * 3 * 10 * 4
    assert lion.workspace_bytes(0, 3, 10, 64, lion.FORM_RNN) == 0
    assert lion.workspace_bytes(1, 1, 10, 48, lion.FORM_RNN) == 0      # d unsupported


def test_bwd_workspace_query(lib):
    from bidirectional_masked_linear_gb300 import lion
    # phi(q), phi(k) and dnum (L*d floats each), four per-token floats, a double per head
    need = lion.bwd_workspace_bytes(2, 3, 10, 64)
    assert need >= 2 * 3 * 10 * (3 * 64 + 4) * 4 + 2 * 3 * 8
    assert lion.bwd_workspace_bytes(0, 3, 10, 64) == 0
    assert lion.bwd_workspace_bytes(1, 1, 10, 48) == 0


def test_reordered_workspace_query(lib):
    from bidirectional_masked_linear_gb300 import lion
    # phi(q), phi(k) (L*d floats each), two positions per token of the order,
    # two coordinates per head-token
    need = lion.reordered_workspace_bytes(2, 3, 10, 64)
    assert need >= 2 * 3 * 10 * (2 * 64 + 2) * 4 + 2 * 10 * 4
    assert lion.reordered_workspace_bytes(0, 3, 10, 64) == 0
    assert lion.reordered_workspace_bytes(1, 1, 10, 32) == 0    # d = 64 and 128 only


def test_reordered_bwd_workspace_query(lib):
    from bidirectional_masked_linear_gb300 import lion
    # phi(q), phi(k), dnum (L*d floats each); dden, the row shares (one float
    # per head-token each), coordinates and the row and column terms (two
    # each), two positions per token, a double per head
    need = lion.reordered_bwd_workspace_bytes(2, 3, 10, 64)
    assert need >= 2 * 3 * 10 * (3 * 64 + 8) * 4 + 2 * 10 * 4 + 2 * 3 * 8
    assert lion.reordered_bwd_workspace_bytes(0, 3, 10, 64) == 0
    assert lion.reordered_bwd_workspace_bytes(1, 1, 10, 16) == 0


def _reorder_bwd(lib, **kw):
    from bidirectional_masked_linear_gb300 import lion
    f = dict(q=4096, k=8192, v=12288, log_lambda=0, order=16384, dy=20480, dq=24576, dk=28672, dv=32768,
             dlog_lambda=0, B=1, H=1, L=8, d=64, mask_kind=0, dtype=0, phi=0, workspace=0, workspace_bytes=0,
             stream=0)
    f.update(kw)
    a = lion._ReorderBwdArgs(**f)
    lib.lion_attn_bwd_reordered.argtypes = [ctypes.POINTER(lion._ReorderBwdArgs)]
    return lib.lion_attn_bwd_reordered(ctypes.byref(a))


@pytest.mark.parametrize("kw", [
    dict(q=0), dict(k=0), dict(v=0), dict(order=0), dict(dy=0), dict(dq=0), dict(dk=0), dict(dv=0),
    dict(B=0), dict(H=0), dict(L=0), dict(d=48), dict(mask_kind=3), dict(dtype=2), dict(phi=4),
    dict(mask_kind=1, log_lambda=36864, dlog_lambda=0), dict(mask_kind=2, log_lambda=0, dlog_lambda=36864),
    dict(),   # pointers that are not device memory
])
def test_reordered_bwd_invalid_arguments_rejected_before_launch(lib, kw):
    assert _reorder_bwd(lib, **kw) == 1
    assert lib.lion_attn_bwd_reordered(None) == 1


def _reorder(lib, **kw):
    from bidirectional_masked_linear_gb300 import lion
    f = dict(q=4096, k=8192, v=12288, log_lambda=0, order=16384, out=20480, B=1, H=1, L=8, d=64,
             mask_kind=0, dtype=0, phi=0, workspace=0, workspace_bytes=0, stream=0)
    f.update(kw)
    a = lion._ReorderArgs(**f)
    return lib.lion_attn_fwd_reordered(ctypes.byref(a))


@pytest.mark.parametrize("kw", [
    dict(q=0), dict(k=0), dict(v=0), dict(out=0), dict(order=0), dict(order=16386),
    dict(B=0), dict(H=0), dict(L=0), dict(d=48), dict(mask_kind=3), dict(dtype=2), dict(phi=4),
    dict(mask_kind=1, log_lambda=0), dict(mask_kind=2, log_lambda=0),
    dict(),   # pointers that are not device memory
])
def test_reordered_invalid_arguments_rejected_before_launch(lib, kw):
    from bidirectional_masked_linear_gb300 import lion
    lib.lion_attn_fwd_reordered.argtypes = [ctypes.POINTER(lion._ReorderArgs)]
    assert _reorder(lib, **kw) == 1
    assert lib.lion_attn_fwd_reordered(None) == 1


def _host(lib, **kw):
    from bidirectional_masked_linear_gb300 import lion
    buf = (ctypes.c_char * 65536)()
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    f = dict(q=base, k=base + 4096, v=base + 8192, log_lambda=base + 12288, out=base + 16384, B=1, H=1, L=8,
             d=64, mask_kind=0, form=2, chunk=64, dtype=0, phi=0, slices=0, stream=0)
    f.update(kw)
    a = lion._HostArgs(**f)
    lib.lion_attn_fwd_host.argtypes = [ctypes.POINTER(lion._HostArgs)]
    return lib.lion_attn_fwd_host(ctypes.byref(a))


@pytest.mark.parametrize("kw", [
    dict(q=0), dict(k=0), dict(v=0), dict(out=0), dict(B=0), dict(H=0), dict(L=0), dict(d=48),
    dict(mask_kind=3), dict(form=3), dict(chunk=0), dict(dtype=2), dict(phi=4), dict(slices=-1),
    dict(mask_kind=2, log_lambda=0), dict(mask_kind=1, log_lambda=0),
])
def test_host_entry_invalid_arguments_rejected(lib, kw):
    assert _host(lib, **kw) == 1
    assert lib.lion_attn_fwd_host(None) == 1


def _bwd(lib, **kw):
    from bidirectional_masked_linear_gb300 import lion
    f = dict(q=4096, k=8192, v=12288, log_lambda=0, dy=16384, dq=20480, dk=24576, dv=28672,
             dlog_lambda=0, B=1, H=1, L=8, d=64, mask_kind=0, dtype=0, phi=0, workspace=0,
             workspace_bytes=0, stream=0)
    f.update(kw)
    a = lion._BwdArgs(**f)
    return lib.lion_attn_bwd(ctypes.byref(a))


@pytest.mark.parametrize("kw", [
    dict(q=0), dict(k=0), dict(v=0), dict(dy=0), dict(dq=0), dict(dk=0), dict(dv=0),
    dict(B=0), dict(H=0), dict(L=0), dict(d=48), dict(mask_kind=3), dict(dtype=2), dict(phi=4),
    dict(mask_kind=1, log_lambda=32768, dlog_lambda=0), dict(mask_kind=2, log_lambda=0, dlog_lambda=32768),
    dict(),   # pointers that are not device memory
])
def test_bwd_invalid_arguments_rejected_before_launch(lib, kw):
    from bidirectional_masked_linear_gb300 import lion
    lib.lion_attn_bwd.argtypes = [ctypes.POINTER(lion._BwdArgs)]
    assert _bwd(lib, **kw) == 1
    assert lib.lion_attn_bwd(None) == 1
    # the chunkwise gradients share the checks
    f = dict(q=4096, k=8192, v=12288, log_lambda=0, dy=16384, dq=20480, dk=24576, dv=28672,
             dlog_lambda=0, B=1, H=1, L=8, d=64, mask_kind=0, dtype=0, phi=0, workspace=0,
             workspace_bytes=0, stream=0)
    f.update(kw)
    assert lib.lion_attn_bwd_chunk(ctypes.byref(lion._BwdArgs(**f))) == 1
    assert lib.lion_attn_bwd_chunk(None) == 1


def test_bwd_chunk_workspace_query(lib):
    from bidirectional_masked_linear_gb300 import lion
    # per chunk of 64 tokens two (d+4)^2 states and its total; per token G
    # (d + 4 floats) and two terms; a double per head
    B, H, L, d = 2, 3, 200, 64
    need = lion.bwd_workspace_bytes(B, H, L, d, lion.FORM_CHUNK)
    N = (L + 63) // 64
    assert need >= B * H * (N * (2 * 68 * 68 + 1) * 4 + L * (68 + 2) * 4 + 8)
    assert lion.bwd_workspace_bytes(B, H, 100000, d, lion.FORM_CHUNK) > need
    assert lion.bwd_workspace_bytes(0, 3, 10, 64, lion.FORM_CHUNK) == 0
    assert lion.bwd_workspace_bytes(1, 1, 10, 48, lion.FORM_CHUNK) == 0
    # chunks of 32 at d = 128
    assert lion.bwd_workspace_bytes(1, 1, 64, 128, lion.FORM_CHUNK) >= 2 * (2 * 132 * 132) * 4


def _fwd(lib, q=1, k=1, v=1, ll=None, B=1, H=1, L=8, d=64, mask=0, form=2, chunk=64, out=1):
    vp = ctypes.c_void_p
    return lib.lion_attn_fwd(vp(q * 4096 if q else 0), vp(k * 8192 if k else 0),
                             vp(v * 12288 if v else 0), vp(ll), B, H, L, d, mask, form, chunk,
                             vp(out * 16384 if out else 0), vp(0))


@pytest.mark.parametrize("kw", [
    dict(q=0), dict(k=0), dict(v=0), dict(out=0),
    dict(B=0), dict(H=0), dict(L=0), dict(d=48), dict(d=0),
    dict(mask=3), dict(mask=-1), dict(form=3), dict(chunk=0),
    dict(mask=1, ll=None), dict(mask=2, ll=None),
])
def test_invalid_arguments_rejected_before_launch(lib, kw):
    # All of these fail host-side validation; no pointer is dereferenced.
    assert _fwd(lib, **kw) == 1


def test_host_pointers_rejected(lib):
    # Non-null but host-only memory (no GPU mapping): refused, never launched.
    buf = (ctypes.c_char * 65536)()
    base = ctypes.addressof(buf)
    base = (base + 255) // 256 * 256
    vp = ctypes.c_void_p
    st = lib.lion_attn_fwd(vp(base), vp(base), vp(base), None, 1, 1, 8, 16, 0, 2, 4,
                           vp(base), vp(0))
    assert st == 1


def test_misaligned_pointer_rejected(lib):
    vp = ctypes.c_void_p
    st = lib.lion_attn_fwd(vp(4096 + 2), vp(8192), vp(12288), None, 1, 1, 8, 64, 0, 2, 64,
                           vp(16384), vp(0))
    assert st == 1


def test_rnn_step_invalid(lib):
    vp = ctypes.c_void_p
    args = [vp(4096)] * 3 + [vp(0)] + [vp(8192)] * 4
    assert lib.lion_rnn_step(*args, 1, 1, 64, 0, 0, vp(0)) == 1      # not device memory
    assert lib.lion_rnn_step(vp(0), vp(0), vp(0), vp(0), vp(0), vp(0), vp(0), vp(0), 1, 1, 64, 0, 0,
                             vp(0)) == 1
    assert lib.lion_rnn_step(*args, 1, 1, 48, 0, 0, vp(0)) == 1
    assert lib.lion_rnn_step(*args, 1, 1, 64, 1, 0, vp(0)) == 1      # LION-D without decay
    assert lib.lion_rnn_step(*args, 1, 1, 64, 0, 7, vp(0)) == 1      # bad dtype


def test_product_path_has_no_cpu_fallback():
    """The binding only marshals arguments: it never imports the oracle and
    raises when the library is missing."""
    src = open(os.path.join(ROOT, "bidirectional_masked_linear_gb300", "lion.py")).read()
    assert "oracle" not in src
    from bidirectional_masked_linear_gb300 import lion
    saved = lion._lib
    try:
        lion._lib = None
        with pytest.raises(RuntimeError):
            lion.load("/nonexistent/liblion.so")
    finally:
        lion._lib = saved


def test_host_entry_slice_plan(tmp_path):
    """lion_attn_fwd_host's batch slicing (host_plan.h, compiled here with the
    host compiler): slices cover the batch in order, none is empty, there
    are min(S, B) of them, and with three or more slices the first and last
    are about half the others."""
    src = tmp_path / "plan.cpp"
    src.write_text(
        '#include <cstdio>\n#include "host_plan.h"\n'
        "int main() { int b[lion::kMaxSlices + 1];\n"
        "  for (int B = 1; B <= 300; ++B) for (int S = 1; S <= lion::kMaxSlices; ++S) {\n"
        "    int n = lion::slice_bounds(B, S, b); printf(\"%d %d %d\", B, S, n);\n"
        "    for (int s = 0; s <= n; ++s) printf(\" %d\", b[s]); printf(\"\\n\"); } }\n")
    exe = tmp_path / "plan"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", os.path.join(ROOT, "bidirectional_masked_linear_gb300", "csrc"),
                    str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    for line in filter(None, out):
        B, S, n, *bounds = map(int, line.split())
        assert n == min(S, B) and len(bounds) == n + 1
        assert bounds[0] == 0 and bounds[-1] == B
        sizes = [b - a for a, b in zip(bounds, bounds[1:])]
        assert min(sizes) >= 1
        if n >= 3 and B >= 2 * n:
            middle = sizes[1:-1]
            for edge in (sizes[0], sizes[-1]):
                assert edge <= min(middle) + 1 and edge >= max(middle) / 2 - 1, (B, S, sizes)


def test_header_is_plain_c(tmp_path):
    """include/lion.h compiles as C11 (no C++ in the ABI) and its structs
    have the field layout the Python binding declares."""
    from bidirectional_masked_linear_gb300 import lion
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    src = tmp_path / "abi.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "lion.h"\n'
        "int main(void) {\n"
        '  printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(lion_args), sizeof(lion_bwd_args),\n'
        "         sizeof(lion_reorder_args), sizeof(lion_reorder_bwd_args), sizeof(lion_host_args),\n"
        "         offsetof(lion_args, out_bf16));\n"
        "  return 0; }\n")
    exe = tmp_path / "abi"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), str(src), "-o", str(exe)],
                   check=True)
    sizes = list(map(int, subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()))
    want = [ctypes.sizeof(lion._Args), ctypes.sizeof(lion._BwdArgs), ctypes.sizeof(lion._ReorderArgs),
            ctypes.sizeof(lion._ReorderBwdArgs), ctypes.sizeof(lion._HostArgs), lion._Args.out_bf16.offset]
    assert sizes == want


def test_wait_bound_setter(lib):
    """The bound on device-side waits: negative values are refused, 0 restores
    the default; no launch is involved."""
    assert lib.lion_debug_set_wait_cycles(-1) == 1
    assert lib.lion_debug_set_wait_cycles(100000) == 0
    assert lib.lion_debug_set_wait_cycles(0) == 0
