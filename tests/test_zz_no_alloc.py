"""The allocation-free recurrent entry point (lion_attn_fwd_rnn_noalloc).

It exists for callers that cannot allocate device memory -- code inside a
framework that owns every byte through its own allocator, or a hot loop that
must not call cudaMalloc/cudaFree.  Its scratch is a fixed array of the
library; this checks, through the C ABI, that two calls in a row give the
same answer as the regular recurrent form (which takes its workspace from the
stream-ordered allocator), and that oversized problems are refused before
anything launches.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from bidirectional_masked_linear_gb300 import lion, synth

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-3


def _rows(y, ref):
    return np.max(np.abs(y - ref), axis=-1) / np.max(np.abs(ref), axis=-1)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bidirectional_masked_linear_gb300 import build
    return lion.load(build.build())


@pytest.mark.parametrize("mask", ("lit", "d", "s"))
def test_noalloc_matches_rnn_form_twice(lib, mask):
    inp = synth.make_inputs(3, 4, 150, 64, mask, "bf16", seed=77)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    ll = None if inp["log_lambda"] is None else inp["log_lambda"].cuda()
    ref = lion.attn_fwd(q, k, v, ll, inp["mask"], lion.FORM_RNN).cpu().numpy()
    vp = ctypes.c_void_p
    p = lambda t: vp(0) if t is None else vp(t.data_ptr())  # noqa: E731
    stream = vp(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        st = lib.lion_attn_fwd_rnn_noalloc(p(q), p(k), p(v), p(ll), 3, 4, 150, 64, inp["mask"],
                                           lion.DTYPE_BF16, p(out), stream)
        assert st == lion.OK
        torch.cuda.synchronize()
        y = out.cpu().numpy()
        assert np.isfinite(y).all()
        assert np.max(_rows(y, ref)) < TOL_BF16


def test_noalloc_refuses_oversized_problem(lib):
    x = torch.zeros((1, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((1, 1, 16, 64), dtype=torch.float32, device="cuda")
    vp = ctypes.c_void_p
    # claimed B*H*L one past the scratch capacity: refused before any launch
    L = lion.NOALLOC_MAX_HEAD_TOKENS + 1
    st = lib.lion_attn_fwd_rnn_noalloc(vp(x.data_ptr()), vp(x.data_ptr()), vp(x.data_ptr()), vp(0),
                                       1, 1, L, 64, 0, lion.DTYPE_BF16, vp(out.data_ptr()), vp(0))
    assert st == lion.ERR_UNSUPPORTED
