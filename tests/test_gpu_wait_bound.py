"""The bound on device-side waits, exercised on the GPU without a hang.

The tensor-core kernels hand work between warps through mbarriers; every
wait is bounded (a launch parameter, lion_debug_set_wait_cycles), and a wait
that runs out records LION_ERR_TIMEOUT in the library's status word instead
of spinning.  lion_debug_wait_timeout runs that same wait, with nothing in
flight, on an mbarrier nothing arrives at: with a bound of 10^5 cycles it
gives up within microseconds, the status reports the timeout once, and the
library keeps working afterwards."""
import pytest
import torch

from bidirectional_masked_linear_gb300 import lion, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bidirectional_masked_linear_gb300 import build
    return lion.load(build.build())


def test_wait_that_nothing_completes_reports_a_timeout(lib):
    stream = torch.cuda.current_stream().cuda_stream
    assert lion.sync_status() == lion.OK
    assert lib.lion_debug_set_wait_cycles(100000) == lion.OK
    try:
        assert lib.lion_debug_wait_timeout(stream) == lion.OK
        assert lion.sync_status() == lion.ERR_TIMEOUT
        assert lion.sync_status() == lion.OK          # the flag was cleared
    finally:
        assert lib.lion_debug_set_wait_cycles(0) == lion.OK
    # the default bound is back, and a tensor-core call after the timeout is clean
    inp = synth.make_inputs(4, 3, 197, 64, "s", "bf16", seed=2100)
    g = {k: inp[k].cuda() for k in ("q", "k", "v", "log_lambda")}
    y = lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], lion.MASK_S, lion.FORM_CHUNK, 128)
    assert lion.sync_status() == lion.OK
    assert torch.isfinite(y).all()



@pytest.mark.parametrize("L,chunk", ((197, 128), (197, 64), (700, 128), (700, 64)))
def test_value_past_fp16_range_is_reported(lib, L, chunk):
    """The tensor-core chunk kernels compute on fp16 operands: a bf16 v of
    1e5 (past the fp16 maximum 65504) would become an infinity there.  The
    kernel that converts it raises LION_ERR_RANGE in the status word (the
    call itself returns OK, its output is not valid), and a later call with
    ordinary values is clean.  Every kernel kind: one launch for L <= 256,
    the pre-pass / segment scan / main pass above, chunks of 128 and 64."""
    inp = synth.make_inputs(2, 3, L, 64, "s", "bf16", seed=2110)
    g = {k: inp[k].cuda() for k in ("q", "k", "v", "log_lambda")}
    assert lion.sync_status() == lion.OK
    big = g["v"].clone()
    big[1, 2, L // 3, 5] = 1e5
    lion.attn_fwd(g["q"], g["k"], big, g["log_lambda"], lion.MASK_S, lion.FORM_CHUNK, chunk)
    assert lion.sync_status() == lion.ERR_RANGE
    y = lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], lion.MASK_S, lion.FORM_CHUNK, chunk)
    assert lion.sync_status() == lion.OK
    assert torch.isfinite(y).all()
