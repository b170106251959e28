"""The allocation-free recurrent entry point (lion_attn_fwd_rnn_noalloc).

It exists for callers that cannot allocate device memory -- code inside a
framework that owns every byte through its own allocator, or a hot loop that
must not call cudaMalloc/cudaFree.  Its scratch is a fixed array of the
library.  Through the C ABI, two calls in a row must give exactly what the
regular recurrent form gives (the same kernel, whose scratch comes from the
stream-ordered allocator instead), and the result must match the float64
oracle; oversized problems are refused before anything launches.  This file
is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from bidirectional_masked_linear_gb300 import lion, synth
from parity import TOL_BF16, check_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bidirectional_masked_linear_gb300 import build
    return lion.load(build.build())


def _dev(inp):
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    ll = None if inp["log_lambda"] is None else inp["log_lambda"].cuda()
    return q, k, v, ll


@pytest.mark.parametrize("mask", ("lit", "d", "s"))
def test_noalloc_matches_rnn_form_twice(lib, mask):
    """Bit for bit the regular recurrent form, on two calls in a row (the
    second finds the first call's values in the shared scratch).  With 12
    heads of 300 tokens the regular form runs its two sweeps apart and combines them in a
    last launch, while this entry point runs them one after the other in
    each CTA: the two must still agree exactly."""
    inp = synth.make_inputs(3, 4, 300, 64, mask, "bf16", seed=77)
    q, k, v, ll = _dev(inp)
    ref = lion.attn_fwd(q, k, v, ll, inp["mask"], lion.FORM_RNN).cpu().numpy()
    vp = ctypes.c_void_p
    p = lambda t: vp(0) if t is None else vp(t.data_ptr())  # noqa: E731
    stream = vp(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        st = lib.lion_attn_fwd_rnn_noalloc(p(q), p(k), p(v), p(ll), 3, 4, 300, 64, inp["mask"],
                                           lion.DTYPE_BF16, p(out), stream)
        assert st == lion.OK
        torch.cuda.synchronize()
        y = out.cpu().numpy()
        assert np.array_equal(y, ref)


def test_noalloc_matches_oracle_through_the_binding(lib, oracle_mod):
    """LION-S at the ViT-T shape through lion.attn_fwd_rnn_noalloc, against
    the float64 oracle under the per-row bound of every parity test."""
    inp = synth.make_inputs(4, 3, 197, 64, "s", "bf16", seed=78)
    q, k, v, ll = _dev(inp)
    y = lion.attn_fwd_rnn_noalloc(q, k, v, ll, lion.MASK_S)
    torch.cuda.synchronize()
    q64, k64, v64, ll64 = (synth.as_f64(inp[x]) for x in ("q", "k", "v", "log_lambda"))
    ref = oracle_mod.full(q64, k64, v64, ll64, lion.MASK_S)
    check_rows(oracle_mod, y.cpu().numpy(), ref, TOL_BF16, q64, k64, ll64, lion.MASK_S)


def test_noalloc_binding_refuses_strided_tensors(lib):
    x = torch.zeros((1, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        lion.attn_fwd_rnn_noalloc(x.transpose(1, 2), x.transpose(1, 2), x.transpose(1, 2), None, lion.MASK_LIT)
    with pytest.raises(TypeError):
        lion.attn_fwd_rnn_noalloc(x, x, x, None, lion.MASK_LIT, out=torch.zeros_like(x))


def test_noalloc_refuses_oversized_problem(lib):
    x = torch.zeros((1, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((1, 1, 16, 64), dtype=torch.float32, device="cuda")
    vp = ctypes.c_void_p
    # claimed B*H*L one past the scratch capacity: refused before any launch
    L = lion.NOALLOC_MAX_HEAD_TOKENS + 1
    st = lib.lion_attn_fwd_rnn_noalloc(vp(x.data_ptr()), vp(x.data_ptr()), vp(x.data_ptr()), vp(0),
                                       1, 1, L, 64, 0, lion.DTYPE_BF16, vp(out.data_ptr()), vp(0))
    assert st == lion.ERR_UNSUPPORTED
