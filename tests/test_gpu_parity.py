"""GPU parity: the CUDA library (through its C ABI) against the float64 oracle
on the same seeded inputs, element by element, for every mask and form, at
small sizes (many tiles and ragged tails, edge cases) and at the full
workload sizes."""
import functools

import numpy as np
import pytest
import torch

from bidirectional_masked_linear_gb300 import lion, synth
from parity import STATS, TOL_BF16, TOL_FP32, check_rows, row_errors

pytestmark = pytest.mark.gpu

MASK_NAME = {0: "lit", 1: "d", 2: "s"}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bidirectional_masked_linear_gb300 import build
    lion.load(build.build())


def _cuda(inp):
    out = {}
    for key in ("q", "k", "v", "log_lambda"):
        t = inp[key]
        out[key] = None if t is None else t.cuda()
    return out


def run_gpu(inp, form, chunk=64, phi=0):
    g = _cuda(inp)
    y = lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], inp["mask"], form, chunk, phi=phi)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def f64(inp):
    return (synth.as_f64(inp["q"]), synth.as_f64(inp["k"]), synth.as_f64(inp["v"]),
            synth.as_f64(inp["log_lambda"]))


def check(oracle_mod, y, ref, inp, tol, phi=0, label=None):
    q, k, _, ll = f64(inp)
    return check_rows(oracle_mod, y, ref, tol, q, k, ll, inp["mask"], phi, label=label)


# --------------------------------------------------------------- tiny ---
def test_tiny_lion_d_fp32_all_forms(oracle_mod):
    """Tiny LION-D FP32 case (B=1, H=2, L=64, d=16, chunk 16): every form
    against the brute-force oracle at 1e-5."""
    inp = synth.workload_inputs("tiny_d_fp32", "d")
    q, k, v, ll = f64(inp)
    ref = oracle_mod.full(q, k, v, ll, 1)
    for form, chunk in ((lion.FORM_FULL, 16), (lion.FORM_RNN, 16), (lion.FORM_CHUNK, 16),
                        (lion.FORM_CHUNK, 5), (lion.FORM_CHUNK, 64)):
        y = run_gpu(inp, form, chunk)
        check(oracle_mod, y, ref, inp, TOL_FP32)


@pytest.mark.parametrize("mask", ("lit", "d", "s"))
@pytest.mark.parametrize("dtype,tol", (("fp32", TOL_FP32), ("bf16", TOL_BF16)))
def test_small_grid(oracle_mod, mask, dtype, tol):
    """Ragged lengths, every head dim, every form, several chunk lengths."""
    for L, d, chunks in ((1, 16, (1, 16)), (2, 32, (1, 3)), (17, 64, (4, 16, 64)),
                         (65, 128, (32, 64)), (130, 64, (16, 64, 128, 200)),
                         (197, 16, (32, 64, 128))):
        inp = synth.make_inputs(2, 3, L, d, mask, dtype, seed=L * 7 + d)
        q, k, v, ll = f64(inp)
        ref = oracle_mod.full(q, k, v, ll, inp["mask"])
        for form in (lion.FORM_FULL, lion.FORM_RNN):
            check(oracle_mod, run_gpu(inp, form), ref, inp, tol)
        for c in chunks:
            check(oracle_mod, run_gpu(inp, lion.FORM_CHUNK, c), ref, inp, tol)


@pytest.mark.parametrize("phi", (lion.PHI_ELU1, lion.PHI_SILU_L2, lion.PHI_IDENTITY))
def test_feature_map_override(oracle_mod, phi):
    inp = synth.make_inputs(1, 2, 70, 64, "s", "fp32", seed=5)
    q, k, v, ll = f64(inp)
    if phi == lion.PHI_IDENTITY:   # keep the row sums away from zero
        for key in ("q", "k"):
            inp[key] = inp[key].abs() + 0.1
        q, k, v, ll = f64(inp)
    ref = oracle_mod.full(q, k, v, ll, 2, phi)
    for form in (lion.FORM_FULL, lion.FORM_RNN, lion.FORM_CHUNK):
        check(oracle_mod, run_gpu(inp, form, 32, phi), ref, inp, TOL_FP32, phi)


@pytest.mark.parametrize("mask", ("lit", "d", "s"))
def test_many_heads_ragged_lengths(oracle_mod, mask):
    """More heads than SMs (each persistent CTA walks several heads) at every
    chunk count and ragged tail the tensor-core chunk path takes."""
    for L in (1, 5, 63, 64, 65, 128, 129, 200, 256):
        inp = synth.make_inputs(50, 7, L, 64, mask, "bf16", seed=300 + L)
        q, k, v, ll = f64(inp)
        ref = oracle_mod.full(q, k, v, ll, inp["mask"], threads=0)
        check(oracle_mod, run_gpu(inp, lion.FORM_CHUNK, 64), ref, inp, TOL_BF16)


@pytest.mark.parametrize("mask", ("lit", "d", "s"))
def test_chunk128_many_heads_ragged_lengths(oracle_mod, mask):
    """The 128-token-chunk tensor-core kernel: one and two chunks, ragged
    tails, padding rows inside a warp, more heads than SMs (every persistent
    CTA cycles its double-buffered head slots several times)."""
    for L in (1, 2, 31, 100, 127, 128, 129, 160, 197, 224, 225, 255, 256):
        inp = synth.make_inputs(40, 9, L, 64, mask, "bf16", seed=700 + L)
        q, k, v, ll = f64(inp)
        ref = oracle_mod.full(q, k, v, ll, inp["mask"], threads=0)
        check(oracle_mod, run_gpu(inp, lion.FORM_CHUNK, 128), ref, inp, TOL_BF16)


@pytest.mark.parametrize("phi", (lion.PHI_ELU1, lion.PHI_SILU_L2, lion.PHI_IDENTITY))
def test_chunk128_feature_maps(oracle_mod, phi):
    """Every feature map through the 128-token-chunk kernel (bf16)."""
    inp = synth.make_inputs(3, 4, 197, 64, "s", "bf16", seed=21)
    if phi == lion.PHI_IDENTITY:   # keep the row sums away from zero
        for key in ("q", "k"):
            inp[key] = (inp[key].float().abs() + 0.1).to(torch.bfloat16)
    q, k, v, ll = f64(inp)
    ref = oracle_mod.full(q, k, v, ll, 2, phi)
    check(oracle_mod, run_gpu(inp, lion.FORM_CHUNK, 128, phi), ref, inp, TOL_BF16, phi)


@pytest.mark.parametrize("scale", (1.5, 3.0))
def test_chunk128_steep_decay_exact_mask(oracle_mod, scale):
    """Decay ranges above 160 nats inside a 128-token chunk (log lambda around
    -scale per token): the kernel takes exp(-|p_i - p_j|) per element instead
    of the factorised mask; M underflows to 0 well inside the chunk."""
    inp = synth.make_inputs(2, 3, 230, 64, "s", "bf16", seed=int(31 * scale))
    inp["log_lambda"] = inp["log_lambda"] * (scale / 0.06)
    q, k, v, ll = f64(inp)
    ref = oracle_mod.full(q, k, v, ll, 2)
    check(oracle_mod, run_gpu(inp, lion.FORM_CHUNK, 128), ref, inp, TOL_BF16)


@pytest.mark.parametrize("mask", ("lit", "d", "s"))
def test_chunk128_long_sequences(oracle_mod, mask):
    """Sequences longer than 256 tokens at chunk 128: the pre-pass and segment
    scan, then the chunk-sequential main pass carrying the forward state,
    with ragged last chunks, blocks with one or two chunks, one or several
    segments per head and several heads per CTA.  With at least as many
    heads as SMs every head is one segment (40 x 9 and 2 x 80 here): no
    segment scan, zero entering states."""
    for B, H, L in ((1, 2, 257), (1, 2, 384), (1, 3, 700), (2, 1, 2000), (8, 5, 1000), (1, 6, 3000),
                    (40, 9, 300), (2, 80, 700)):
        inp = synth.make_inputs(B, H, L, 64, mask, "bf16", seed=900 + L + B)
        q, k, v, ll = f64(inp)
        ref = oracle_mod.rnn(q, k, v, ll, inp["mask"], threads=0)
        check(oracle_mod, run_gpu(inp, lion.FORM_CHUNK, 128), ref, inp, TOL_BF16)


# The long paths' later launches start before the earlier ones end
# (programmatic dependent launch) and wait for them only where they read their
# output.  Calls made back to back on one stream, with the workspace memory of
# one call reused by the next, must still give each call's own result: bit
# for bit the result of the same call made on its own.
@pytest.mark.gpu
@pytest.mark.parametrize("chunk", (64, 128))
def test_long_calls_back_to_back(chunk):
    shapes = ((1, 3, 3000), (2, 80, 700), (1, 2, 1500), (1, 6, 2000))   # several and one segment a head
    inps = [synth.make_inputs(B, H, L, 64, "s", "bf16", seed=1500 + i) for i, (B, H, L) in enumerate(shapes)]
    alone = [run_gpu(inp, lion.FORM_CHUNK, chunk) for inp in inps]
    devs = [_cuda(inp) for inp in inps]
    torch.cuda.synchronize()
    for rep in range(3):
        outs = [lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], "s", "chunk", chunk) for g in devs]
        torch.cuda.synchronize()
        assert lion.sync_status() == 0
        for i, (y, want) in enumerate(zip(outs, alone)):
            assert np.array_equal(y.cpu().numpy(), want), (chunk, rep, i)


@pytest.mark.parametrize("mask", ("lit", "d", "s"))
def test_long_sequences_blocks_and_segments(oracle_mod, mask):
    """Sequences longer than one 256-token block: the tensor-core path chains
    blocks (and, with few heads, segments of blocks across CTAs) through its
    pre-pass, segment scan and main pass."""
    for B, H, L in ((1, 2, 257), (1, 2, 700), (2, 1, 2000), (8, 5, 2000), (1, 6, 3000)):
        inp = synth.make_inputs(B, H, L, 64, mask, "bf16", seed=500 + L + B)
        q, k, v, ll = f64(inp)
        ref = oracle_mod.rnn(q, k, v, ll, inp["mask"], threads=0)
        check(oracle_mod, run_gpu(inp, lion.FORM_CHUNK, 64), ref, inp, TOL_BF16)


# ----------------------------------------------------- maximum lengths --
@pytest.mark.gpu
@pytest.mark.parametrize("mask", ("d", "s"))
def test_full_form_at_its_maximum_length(oracle_mod, mask):
    """L = LION_FULL_MAX_L through the full form, against the oracle's brute
    force on sampled rows (first, last, tile edges and random ones)."""
    L = lion.FULL_MAX_L
    inp = synth.make_inputs(1, 2, L, 64, mask, "bf16", seed=1500)
    y = run_gpu(inp, lion.FORM_FULL, 64)
    q, k, v, ll = f64(inp)
    rng = np.random.default_rng(1501)
    rows = np.unique(np.r_[0, 1, 31, 32, 63, 64, L // 2, L - 33, L - 2, L - 1, rng.integers(0, L, 22)])
    kind = 2 if inp["mask"] == lion.MASK_S else 1
    for h in range(2):
        ref = oracle_mod.rows(q, k, v, ll, inp["mask"], 0, h, rows)
        err = row_errors(y[0, h, rows], ref)
        for r, e in zip(rows, err):
            kap = oracle_mod.row_kappa(q, k, ll, inp["mask"], 0, h, int(r), int(r) + 1, kind)[0]
            assert e <= TOL_BF16 * max(1.0, kap), (h, int(r), e, kap)


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ("d", "s"))
def test_backward_at_its_maximum_length(mask):
    """Gradients at L = LION_FULL_MAX_L (the recompute build), checked by two
    identities that hold at any size: y is homogeneous of degree 1 in v, so
    sum_j dv_j . v_j = sum_i dy_i . y_i; and with identity features y_i does
    not change when q_i is scaled, so dq_i . q_i = 0 for every row."""
    L = lion.FULL_MAX_L
    inp = synth.make_inputs(1, 1, L, 64, mask, "fp32", seed=1510)
    for key in ("q", "k"):
        inp[key] = inp[key].abs() + 0.25
    g = _cuda(inp)
    dy = torch.randn((1, 1, L, 64), device="cuda", generator=torch.Generator(device="cuda").manual_seed(1511))
    dq, dk, dv, dll = lion.attn_bwd(g["q"], g["k"], g["v"], g["log_lambda"], dy, inp["mask"], 3)
    y = lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], inp["mask"], lion.FORM_FULL, 64, phi=3)
    torch.cuda.synchronize()
    v = g["v"].double()
    lhs = float((dv.double() * v).sum())
    rhs = float((dy.double() * y.double()).sum())
    scale = float((dv.double() * v).abs().sum() + (dy.double() * y.double()).abs().sum())
    assert abs(lhs - rhs) <= 1e-5 * scale, (lhs, rhs, scale)
    qd = g["q"].double()
    dot = (dq.double() * qd).sum(-1).abs()
    mag = (dq.double().abs() * qd.abs()).sum(-1)
    assert bool((dot <= 1e-4 * mag + 1e-30).all()), float((dot / mag).max())
    assert bool(torch.isfinite(dk).all()) and bool(torch.isfinite(dll).all())


# ----------------------------------------------------------- edge cases --
@pytest.mark.parametrize("mask", ("d", "s"))
def test_vanishing_decay_is_identity(oracle_mod, mask):
    """log lambda = -1e4: M = I and y_i = v_i."""
    inp = synth.make_inputs(1, 2, 100, 64, mask, "bf16", seed=9)
    inp["log_lambda"] = torch.full_like(inp["log_lambda"], -1e4)
    v = synth.as_f64(inp["v"])
    for form, c in ((lion.FORM_FULL, 64), (lion.FORM_RNN, 64), (lion.FORM_CHUNK, 64),
                    (lion.FORM_CHUNK, 128), (lion.FORM_CHUNK, 7)):
        e = row_errors(run_gpu(inp, form, c), v)
        assert np.max(e) < TOL_BF16


def test_unit_decay_equals_lit():
    inp = synth.make_inputs(2, 2, 150, 64, "d", "bf16", seed=10)
    inp["log_lambda"] = torch.zeros_like(inp["log_lambda"])
    lit = dict(inp, log_lambda=None, mask=0)
    for form in (lion.FORM_FULL, lion.FORM_RNN, lion.FORM_CHUNK):
        a = run_gpu(inp, form, 64)
        b = run_gpu(lit, form, 64)
        assert np.max(row_errors(a, b)) < TOL_BF16


@pytest.mark.parametrize("mask", ("lit", "d", "s"))
def test_gpu_forms_agree(oracle_mod, mask):
    """The GPU forms (full, RNN, chunk 32 / 64 / 128) agree with each other
    under the same per-row bound as against the oracle (Theorem 3.3: the
    forms are equal): every row of every pair within tol * max(1, kappa_i),
    and every form within that bound of the float64 oracle."""
    inp = synth.make_inputs(4, 3, 197, 64, mask, "bf16", seed=11)
    ys = {"full": run_gpu(inp, lion.FORM_FULL), "rnn": run_gpu(inp, lion.FORM_RNN)}
    for c in (32, 64, 128):
        ys[f"chunk{c}"] = run_gpu(inp, lion.FORM_CHUNK, c)
    q, k, v, ll = f64(inp)
    ref = oracle_mod.full(q, k, v, ll, inp["mask"])
    names = list(ys)
    for a in names:
        check(oracle_mod, ys[a], ref, inp, TOL_BF16, label=f"forms {mask}: {a} vs oracle")
    for n, a in enumerate(names):
        for b in names[n + 1:]:
            check(oracle_mod, ys[a], ys[b], inp, TOL_BF16, label=f"forms {mask}: {a} vs {b}")


def test_device_status_clean_after_calls():
    inp = _cuda(synth.make_inputs(2, 2, 197, 64, "s", "bf16", seed=3))
    lion.attn_fwd(inp["q"], inp["k"], inp["v"], inp["log_lambda"], 2, lion.FORM_CHUNK, 64)
    assert lion.sync_status() == lion.OK


def test_errors_on_gpu():
    inp = _cuda(synth.make_inputs(1, 1, 16, 64, "lit", "bf16"))
    with pytest.raises(lion.LionError) as ei:
        lion.attn_fwd(inp["q"], inp["k"], inp["v"], None, 0, lion.FORM_CHUNK, 0)
    assert ei.value.status == lion.ERR_INVALID_ARG
    big = torch.empty((1, 1, lion.FULL_MAX_L + 1, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lion.LionError) as ei:
        lion.attn_fwd(big, big, big, None, 0, lion.FORM_FULL)
    assert ei.value.status == lion.ERR_UNSUPPORTED
    host = torch.zeros((1, 1, 16, 64), dtype=torch.bfloat16)        # host memory
    with pytest.raises(lion.LionError):
        lion.attn_fwd(host, host, host, None, 0, lion.FORM_CHUNK,
                      out=torch.empty((1, 1, 16, 64), device="cuda"))
    # the decode step's state moves as 16-byte rows: a state 4 bytes off is refused
    x = torch.zeros((1, 1, 64), dtype=torch.bfloat16, device="cuda")
    S = torch.zeros(64 * 64 + 1, device="cuda")[1:].view(1, 1, 64, 64)
    z, yp, cp = (torch.zeros(s_, device="cuda") for s_ in ((1, 1, 64), (1, 1, 64), (1, 1)))
    with pytest.raises(lion.LionError) as ei:
        lion.rnn_step(x, x, x, None, S, z, yp, cp, lion.MASK_LIT)
    assert ei.value.status == lion.ERR_INVALID_ARG


@pytest.mark.parametrize("dtype", ("bf16", "fp32"))
def test_rnn_caller_workspace(oracle_mod, dtype):
    """The recurrent form with a caller workspace of lion_attn_workspace_bytes
    (the features of every token computed once by a first launch) gives the
    bits of the call whose workspace the library allocates, and matches the
    oracle; a workspace holding only c^F (B*H*L floats) is refused."""
    B, H, L, d = 2, 3, 301, 64
    inp = synth.make_inputs(B, H, L, d, "s", dtype, seed=41)
    g = _cuda(inp)
    need = lion.workspace_bytes(B, H, L, d, lion.FORM_RNN)
    assert need > 4 * B * H * L
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")    # NaN-patterned scratch
    y0 = lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], 2, lion.FORM_RNN)
    y1 = lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], 2, lion.FORM_RNN, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    tol = TOL_FP32 if dtype == "fp32" else TOL_BF16
    q, k, v, ll = f64(inp)
    check(oracle_mod, y1.cpu().numpy(), oracle_mod.full(q, k, v, ll, 2, threads=0), inp, tol,
          label=f"rnn caller workspace {dtype}")
    small = torch.empty((4 * B * H * L,), dtype=torch.uint8, device="cuda")
    with pytest.raises(lion.LionError) as ei:
        lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], 2, lion.FORM_RNN, workspace=small)
    assert ei.value.status == lion.ERR_INVALID_ARG


@pytest.mark.parametrize("d,B,H", ((16, 8, 20), (32, 8, 10)))
def test_rnn_split_sweeps_equal_fused_sweeps(d, B, H):
    """With few heads (under two column CTAs an SM) the recurrent form runs
    its two sweeps at once in separate CTAs and combines them in a last
    launch; with many, each CTA runs them one after the other.  A batch row
    computed alone (split sweeps) gives the bits it gets inside the whole
    batch (fused sweeps).  At d >= 64 the same head count also sets how many
    lanes share a state column, and with it the order of the column sums, so
    there the allocation-free entry point (fused sweeps, same lanes) is the
    comparison."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert B * H * (d // 8) >= 2 * sms > H * (d // 8)
    inp = synth.make_inputs(B, H, 300, d, "s", "bf16", seed=91)
    g = _cuda(inp)
    y_all = lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], 2, lion.FORM_RNN)
    for b in (0, B - 1):
        one = {x: g[x][b:b + 1].contiguous() for x in ("q", "k", "v", "log_lambda")}
        y_one = lion.attn_fwd(one["q"], one["k"], one["v"], one["log_lambda"], 2, lion.FORM_RNN)
        torch.cuda.synchronize()
        assert torch.equal(y_one, y_all[b:b + 1])


@pytest.mark.parametrize("d", (16, 32, 64, 128))
def test_rnn_step_matches_rnn_form(oracle_mod, d):
    """Feeding tokens one at a time through lion_rnn_step, forward and then
    backward (with lambda of the next token), and combining with the diagonal
    removed once reproduces the operator, at every head dim."""
    B, H, L = 2, 3, 24
    inp = synth.make_inputs(B, H, L, d, "s", "bf16", seed=12 + d)
    q, k, v = inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda()
    ll = inp["log_lambda"].cuda()
    yF = torch.empty((B, H, L, d), device="cuda")
    cF = torch.empty((B, H, L), device="cuda")
    yB = torch.empty_like(yF)
    cB = torch.empty_like(cF)
    for direction in (0, 1):
        S = torch.zeros((B, H, d, d), device="cuda")
        z = torch.zeros((B, H, d), device="cuda")
        order = range(L) if direction == 0 else range(L - 1, -1, -1)
        for i in order:
            if direction == 0:
                lam = ll[:, :, i].contiguous()
            else:
                lam = ll[:, :, i + 1].contiguous() if i + 1 < L else torch.full((B, H), -1e4, device="cuda")
            yp = torch.empty((B, H, d), device="cuda")
            cp = torch.empty((B, H), device="cuda")
            lion.rnn_step(q[:, :, i].contiguous(), k[:, :, i].contiguous(), v[:, :, i].contiguous(),
                          lam, S, z, yp, cp, lion.MASK_S)
            (yF if direction == 0 else yB)[:, :, i] = yp
            (cF if direction == 0 else cB)[:, :, i] = cp
    torch.cuda.synchronize()
    fq = torch.nn.functional.normalize(torch.nn.functional.silu(q.double()), dim=-1, eps=1e-12)
    fk = torch.nn.functional.normalize(torch.nn.functional.silu(k.double()), dim=-1, eps=1e-12)
    sii = (fq * fk).sum(-1)
    y = (yF.double() + yB.double() - sii[..., None] * v.double()) / (cF.double() + cB.double() - sii)[..., None]
    qq, kk, vv, lll = f64(inp)
    ref = oracle_mod.full(qq, kk, vv, lll, 2)
    check(oracle_mod, y.cpu().numpy(), ref, inp, TOL_BF16, label=f"rnn_step d={d}")


def test_rnn_step_in_a_cuda_graph():
    """A decode loop of lion_rnn_step calls captured into a CUDA graph and
    replayed gives the bits of the same calls launched one by one."""
    B, H, d, T = 4, 3, 64, 6
    g = torch.Generator(device="cuda").manual_seed(77)
    q, k, v = (torch.randn((T, B, H, d), device="cuda", generator=g).to(torch.bfloat16) for _ in range(3))
    ll = torch.nn.functional.logsigmoid(torch.randn((T, B, H), device="cuda", generator=g) + 3.0)

    def run(S, z, ys, cs):
        for t in range(T):
            lion.rnn_step(q[t], k[t], v[t], ll[t], S, z, ys[t], cs[t], lion.MASK_S,
                          stream=torch.cuda.current_stream())

    fresh = lambda: (torch.zeros((B, H, d, d), device="cuda"), torch.zeros((B, H, d), device="cuda"),
                     torch.zeros((T, B, H, d), device="cuda"), torch.zeros((T, B, H), device="cuda"))
    S0, z0, y0, c0 = fresh()
    run(S0, z0, y0, c0)
    S1, z1, y1, c1 = fresh()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="relaxed"):
        run(S1, z1, y1, c1)
    S1.zero_()
    z1.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in ((S0, S1), (z0, z1), (y0, y1), (c0, c1)):
        assert torch.equal(a, b)


# ----------------------------------------------------- full workloads ----
@functools.lru_cache(maxsize=None)
def _workload(name, mask):
    return synth.workload_inputs(name, mask)


@functools.lru_cache(maxsize=None)
def _reference(name, mask):
    import oracle
    inp = _workload(name, mask)
    q, k, v, ll = f64(inp)
    if synth.WORKLOADS[name].L > 1024:
        return oracle.rnn(q, k, v, ll, inp["mask"], threads=0)
    return oracle.full(q, k, v, ll, inp["mask"], threads=0)


FULL_CASES = [
    ("vit_t_s", "s", lion.FORM_CHUNK, 64),
    ("vit_b", "lit", lion.FORM_CHUNK, 32), ("vit_b", "lit", lion.FORM_CHUNK, 64),
    ("vit_b", "lit", lion.FORM_CHUNK, 128), ("vit_b", "lit", lion.FORM_FULL, 64),
    ("vit_b", "d", lion.FORM_CHUNK, 32), ("vit_b", "d", lion.FORM_CHUNK, 64),
    ("vit_b", "d", lion.FORM_CHUNK, 128), ("vit_b", "d", lion.FORM_FULL, 64),
    ("vit_b", "s", lion.FORM_CHUNK, 32), ("vit_b", "s", lion.FORM_CHUNK, 64),
    ("vit_b", "s", lion.FORM_CHUNK, 128), ("vit_b", "s", lion.FORM_FULL, 64),
    ("bert_large", "d", lion.FORM_CHUNK, 64), ("bert_large", "d", lion.FORM_CHUNK, 128),
    ("bert_large", "s", lion.FORM_CHUNK, 64), ("bert_large", "s", lion.FORM_CHUNK, 128),
    ("hires_2496", "d", lion.FORM_CHUNK, 64), ("hires_2496", "d", lion.FORM_CHUNK, 128),
    ("hires_2496", "d", lion.FORM_RNN, 64),
    ("hires_2496", "s", lion.FORM_CHUNK, 64), ("hires_2496", "s", lion.FORM_CHUNK, 128),
    ("hires_2496", "s", lion.FORM_RNN, 64),
    ("lra_4096", "s", lion.FORM_CHUNK, 128), ("lra_4096", "d", lion.FORM_CHUNK, 128),
    ("lra_4096", "s", lion.FORM_CHUNK, 64), ("lra_4096", "s", lion.FORM_RNN, 64),
]


@pytest.mark.parametrize("name,mask,form,chunk", FULL_CASES)
def test_full_workload(oracle_mod, name, mask, form, chunk):
    """Every output row of the workload against the float64 oracle.  Rows
    whose plain error exceeds tol need the conditioning factor kappa_i; with
    elu+1 features kappa = 1, so LIT and LION-D must have none, and with SiLU
    features at most 1% of the rows may lean on it.  The counts, the largest
    kappa used and the worst error as a fraction of its bound are printed at
    the end of the run."""
    inp = _workload(name, mask)
    ref = _reference(name, mask)
    y = run_gpu(inp, form, chunk)
    form_name = {lion.FORM_FULL: "full", lion.FORM_RNN: "rnn", lion.FORM_CHUNK: f"chunk{chunk}"}[form]
    st = check(oracle_mod, y, ref, inp, TOL_BF16, label=f"workload {name} {mask} {form_name}")
    if mask in ("lit", "d"):
        assert st["kappa_rows"] == 0, st
    else:
        assert st["kappa_rows"] <= 0.01 * st["rows"], st


# ------------------------------------------------------------- backward ---
# Gradients through the full form (the training path, rebuttal page reply
# "Concern 1", Theorem 3.3 Eq 25) against the float64 oracle's gradients,
# which finite differences of the forward pin.  The GPU path computes in
# fp32; each gradient tensor is compared relative to its largest entry.
TOL_BWD = 2e-4


def _bwd_check(oracle_mod, B, H, L, d, mask, dtype, phi=0, seed=0, positive=False):
    inp = synth.make_inputs(B, H, L, d, mask, dtype, seed=seed)
    if positive:   # identity features need row sums away from zero
        for key in ("q", "k"):
            inp[key] = (inp[key].float().abs() + 0.25).to(inp[key].dtype)
    q64, k64, v64, ll64 = f64(inp)
    dy = np.random.default_rng(seed + 1).standard_normal((B, H, L, d)).astype(np.float32)
    ref = oracle_mod.full_bwd(q64, k64, v64, ll64, dy.astype(np.float64), inp["mask"], phi)
    g = _cuda(inp)
    got = lion.attn_bwd(g["q"], g["k"], g["v"], g["log_lambda"], torch.from_numpy(dy).cuda(),
                        inp["mask"], phi)
    torch.cuda.synchronize()
    _grad_rows(ref, got, f"bwd {MASK_NAME[inp['mask']]} {dtype} ({B},{H},{L},{d}) phi {phi}")
    return got


def _grad_rows(ref, got, label, tol=TOL_BWD, tol_dll=None):
    """Per row (one token's d gradient entries of dq, dk, dv; one entry of
    dlog_lambda) the error relative to that row's own scale, with a floor of
    1e-3 of the tensor's largest entry for rows whose gradient cancels to
    near zero.  The scale of a dq, dk or dv row is its largest entry.  LION-S's
    dlog_lambda_u is the suffix sum over m >= u of dLoss/dP_m (the derivative
    by the prefix of the decays), so its scale is the sum of the magnitudes
    of those terms, sum_{m>=u} |dlog_lambda_m - dlog_lambda_{m+1}| (which is
    at least |dlog_lambda_u|): the componentwise bound of a sum.  LION-D's
    [H] vector is compared entry by entry.  A tensor whose exact value is 0
    (dq and dk at L = 1) is measured against the case's other gradients."""
    scale = max(float(np.abs(r).max()) for r in ref if r is not None)
    worst = {}
    for name, r, x in zip(("dq", "dk", "dv", "dlog_lambda"), ref, got):
        if r is None:
            assert x is None
            continue
        x = x.cpu().numpy().astype(np.float64)
        assert x.shape == r.shape, name
        rr = r.reshape(-1, r.shape[-1]) if name != "dlog_lambda" else r.reshape(-1, 1)
        xx = x.reshape(rr.shape)
        floor = 1e-3 * max(float(np.abs(rr).max()), 1e-2 * scale)
        den = np.maximum(np.abs(rr).max(axis=1), floor)
        if name == "dlog_lambda" and r.ndim == 3:
            terms = np.abs(r - np.concatenate([r[..., 1:], np.zeros_like(r[..., :1])], axis=-1))
            suffix = np.flip(np.cumsum(np.flip(terms, -1), -1), -1)
            den = np.maximum(suffix.reshape(-1), floor)
        err = np.abs(xx - rr).max(axis=1) / den
        worst[name] = float(err.max())
        lim = tol_dll if (name == "dlog_lambda" and tol_dll is not None) else tol
        assert worst[name] <= lim, (label, name, worst[name], int(np.argmax(err)))
    STATS.append((label, {f"worst {k} row err": v for k, v in worst.items()}))


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ("lit", "d", "s"))
@pytest.mark.parametrize("dtype", ("bf16", "fp32"))
def test_backward_matches_oracle(oracle_mod, mask, dtype):
    for n, (B, H, L, d) in enumerate(((1, 2, 64, 16), (2, 3, 197, 64), (1, 2, 33, 32), (1, 1, 300, 128),
                                      (1, 2, 515, 64), (2, 1, 7, 64), (1, 1, 1100, 64))):
        _bwd_check(oracle_mod, B, H, L, d, mask, dtype, seed=700 + 10 * n)


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ("lit", "d", "s"))
def test_backward_single_token(mask):
    """L = 1: y = v whatever q and k are, so dv = dy and dq = dk = 0 up to the
    fp32 rounding of v - y; the decay never enters (dlog_lambda = 0)."""
    inp = synth.make_inputs(3, 2, 1, 64, mask, "bf16", seed=760)
    g = _cuda(inp)
    dy = torch.randn(3, 2, 1, 64, device="cuda")
    dq, dk, dv, dll = lion.attn_bwd(g["q"], g["k"], g["v"], g["log_lambda"], dy, inp["mask"])
    scale = float(dy.abs().max())
    assert float((dv - dy).abs().max()) <= 1e-5 * scale
    assert float(dq.abs().max()) <= 1e-3 * scale and float(dk.abs().max()) <= 1e-3 * scale
    if dll is not None:
        assert float(dll.abs().max()) == 0.0


@pytest.mark.gpu
@pytest.mark.parametrize("mask,phi,positive", (("lit", 2, False), ("d", 2, False), ("s", 1, False),
                                               ("s", 3, True), ("lit", 3, True)))
def test_backward_feature_maps(oracle_mod, mask, phi, positive):
    _bwd_check(oracle_mod, 2, 2, 150, 64, mask, "bf16", phi=phi, seed=800, positive=positive)


@pytest.mark.gpu
def test_backward_steep_decay(oracle_mod):
    """Fast-decaying LION-S (log lambda scaled by 40): most of M underflows.
    elu+1 features keep the row sums (here about s_ii) away from zero, so the
    case measures the mask, not a near-zero denominator's conditioning."""
    inp = synth.make_inputs(2, 2, 120, 64, "s", "bf16", seed=810)
    inp["log_lambda"] = inp["log_lambda"] * 40.0
    q64, k64, v64, ll64 = f64(inp)
    dy = np.random.default_rng(811).standard_normal(q64.shape).astype(np.float32)
    ref = oracle_mod.full_bwd(q64, k64, v64, ll64, dy.astype(np.float64), inp["mask"], 1)
    g = _cuda(inp)
    got = lion.attn_bwd(g["q"], g["k"], g["v"], g["log_lambda"], torch.from_numpy(dy).cuda(), inp["mask"], 1)
    _grad_rows(ref, got, "bwd steep-decay s")


@pytest.mark.gpu
def test_autograd_function_uses_the_backward():
    """LionAttention: forward by the chunk form, backward by attn_bwd."""
    inp = synth.make_inputs(2, 3, 197, 64, "s", "bf16", seed=820)
    g = _cuda(inp)
    q = g["q"].clone().requires_grad_(True)
    k = g["k"].clone().requires_grad_(True)
    v = g["v"].clone().requires_grad_(True)
    ll = g["log_lambda"].clone().requires_grad_(True)
    y = lion.LionAttention.apply(q, k, v, ll, lion.MASK_S, lion.FORM_CHUNK, 128)
    dy = torch.randn_like(y)
    y.backward(dy)
    dq, dk, dv, dll = lion.attn_bwd(g["q"], g["k"], g["v"], g["log_lambda"], dy, lion.MASK_S)
    assert torch.equal(q.grad, dq.to(q.dtype)) and torch.equal(k.grad, dk.to(k.dtype))
    assert torch.equal(v.grad, dv.to(v.dtype)) and torch.equal(ll.grad, dll)


# --------------------------------------------------------- causal (f3) ---
# The forward half alone, y_i = sum_{j<=i} M_ij s_ij v_j / sum_{j<=i} M_ij s_ij
# (rebuttal page reply "1: Recurrence Form"; the unidirectional LION-S of reply
# "Q5"), against the oracle's forward recurrence (pinned to the causal Linear
# Transformer at lambda = 1).  fp32 arithmetic on the CUDA cores.
TOL_CAUSAL = 1e-4


def _causal_check(oracle_mod, inp, form, chunk, phi=0):
    q, k, v, ll = f64(inp)
    B, H, L, d = q.shape
    yF, cF = oracle_mod.rnn_forward_half(q, k, v, ll, inp["mask"], phi)
    ref = yF / cF[..., None]
    g = _cuda(inp)
    y = lion.attn_fwd_causal(g["q"], g["k"], g["v"], g["log_lambda"], inp["mask"], form, chunk, phi=phi)
    y = y.cpu().numpy().astype(np.float64)
    kind = phi or (2 if inp["mask"] == lion.MASK_S else 1)
    err = row_errors(y, ref)
    for b in range(B):
        for h in range(H):
            M = np.tril(oracle_mod.mask(inp["mask"], ll, L, b, h, H))
            fq, fk = oracle_mod.phi(kind, q[b, h]), oracle_mod.phi(kind, k[b, h])
            den = (M * (fq @ fk.T)).sum(1)
            kap = (M * (np.abs(fq) @ np.abs(fk).T)).sum(1) / np.abs(den)
            bad = err[b, h] > TOL_CAUSAL * np.maximum(1.0, kap)
            assert not bad.any(), (form, chunk, b, h, np.argwhere(bad)[:3], err[b, h][bad][:3])


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ("lit", "d", "s"))
@pytest.mark.parametrize("dtype", ("bf16", "fp32"))
def test_causal_matches_forward_half(oracle_mod, mask, dtype):
    for n, (B, H, L, d) in enumerate(((1, 2, 64, 16), (2, 3, 197, 64), (1, 2, 300, 32), (1, 1, 77, 128))):
        inp = synth.make_inputs(B, H, L, d, mask, dtype, seed=900 + 10 * n)
        for form, chunk in ((lion.FORM_FULL, 0), (lion.FORM_RNN, 0), (lion.FORM_CHUNK, 16),
                            (lion.FORM_CHUNK, 64), (lion.FORM_CHUNK, 100)):
            _causal_check(oracle_mod, inp, form, max(chunk, 1))


@pytest.mark.gpu
def test_causal_feature_maps_and_single_token(oracle_mod):
    inp = synth.make_inputs(2, 2, 130, 64, "lit", "bf16", seed=950)
    _causal_check(oracle_mod, inp, lion.FORM_CHUNK, 64, phi=2)
    inp = synth.make_inputs(2, 2, 130, 64, "s", "bf16", seed=951)
    _causal_check(oracle_mod, inp, lion.FORM_RNN, 1, phi=1)
    # L = 1: y_0 = v_0
    inp = synth.make_inputs(3, 2, 1, 64, "s", "bf16", seed=952)
    g = _cuda(inp)
    for form in (lion.FORM_FULL, lion.FORM_RNN, lion.FORM_CHUNK):
        y = lion.attn_fwd_causal(g["q"], g["k"], g["v"], g["log_lambda"], inp["mask"], form, 8)
        assert torch.allclose(y, g["v"].float(), rtol=1e-5, atol=1e-6)   # (s v) / s, rounded


# ------------------------------------------------- patch reordering (f2) --
# The full form with the mask averaged over two traversal orders of the tokens
# (rebuttal page, reply "P2: Comparison against vision SSMs", item 1; results
# page "LION Part IV - Results", the reordered-patch models), against the
# oracle's brute force (pinned by the one-order, reversal and cumulative-sum
# cases).  fp32 arithmetic on the CUDA cores; rows are measured against the
# averaged mask's conditioning like every other SiLU case.
TOL_REORDER = 1e-4


def _vit_grid_orders(side=14):
    """Class token first, then the patch grid row by row, or column by column."""
    rows = np.arange(1 + side * side)
    cols = np.concatenate([[0], 1 + np.arange(side * side).reshape(side, side).T.ravel()])
    return np.stack([rows, cols]).astype(np.int32)


def _avg_mask(oracle_mod, mask, ll, orders, b, h, H, L):
    M = np.zeros((L, L))
    for o in orders:
        llo = ll[:, :, o] if mask == lion.MASK_S else ll
        M[np.ix_(o, o)] += 0.5 * oracle_mod.mask(mask, llo, L, b, h, H)
    return M


def _reorder_check(oracle_mod, inp, orders, phi=0):
    q, k, v, ll = f64(inp)
    B, H, L, d = q.shape
    ref = oracle_mod.full_reordered(q, k, v, ll, orders, inp["mask"], phi)
    g = _cuda(inp)
    o = torch.from_numpy(np.ascontiguousarray(orders, dtype=np.int32)).cuda()
    y = lion.attn_fwd_reordered(g["q"], g["k"], g["v"], g["log_lambda"], o, inp["mask"], phi=phi)
    assert lion.sync_status() == lion.OK
    y = y.cpu().numpy().astype(np.float64)
    kind = phi or (2 if inp["mask"] == lion.MASK_S else 1)
    err = row_errors(y, ref)
    for b in range(B):
        for h in range(H):
            M = _avg_mask(oracle_mod, inp["mask"], ll, orders, b, h, H, L)
            fq, fk = oracle_mod.phi(kind, q[b, h]), oracle_mod.phi(kind, k[b, h])
            den = (M * (fq @ fk.T)).sum(1)
            kap = (M * (np.abs(fq) @ np.abs(fk).T)).sum(1) / np.abs(den)
            bad = err[b, h] > TOL_REORDER * np.maximum(1.0, kap)
            assert not bad.any(), (b, h, np.argwhere(bad)[:3], err[b, h][bad][:3])


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ("lit", "d", "s"))
@pytest.mark.parametrize("dtype", ("bf16", "fp32"))
def test_reordered_matches_oracle(oracle_mod, mask, dtype):
    rng = np.random.default_rng(1200)
    inp = synth.make_inputs(2, 3, 197, 64, mask, dtype, seed=1201)
    _reorder_check(oracle_mod, inp, _vit_grid_orders())
    for n, (B, H, L, d) in enumerate(((1, 2, 300, 128), (2, 2, 7, 64), (1, 1, 1, 64), (1, 2, 515, 64))):
        inp = synth.make_inputs(B, H, L, d, mask, dtype, seed=1210 + 10 * n)
        _reorder_check(oracle_mod, inp, np.stack([rng.permutation(L), rng.permutation(L)]))


@pytest.mark.gpu
@pytest.mark.parametrize("mask,phi", (("s", 1), ("d", 2), ("lit", 3)))
def test_reordered_feature_maps(oracle_mod, mask, phi):
    rng = np.random.default_rng(1250)
    inp = synth.make_inputs(2, 2, 150, 64, mask, "bf16", seed=1251)
    if phi == 3:   # identity features need row sums away from zero
        for key in ("q", "k"):
            inp[key] = (inp[key].float().abs() + 0.25).to(inp[key].dtype)
    _reorder_check(oracle_mod, inp, np.stack([rng.permutation(150), rng.permutation(150)]), phi=phi)


@pytest.mark.gpu
def test_reordered_invalid_orders_are_reported():
    """A row that is not a permutation: the call returns OK, the kernels keep
    every index in range, and the next status query says INVALID_ARG (then
    the flag is clear)."""
    inp = synth.make_inputs(1, 2, 40, 64, "s", "bf16", seed=1260)
    g = _cuda(inp)
    good = np.arange(40)
    for bad in (np.r_[np.arange(39), 5], np.r_[np.arange(39), 45], np.r_[-1, np.arange(1, 40)]):
        o = torch.from_numpy(np.stack([good, bad]).astype(np.int32)).cuda()
        lion.attn_fwd_reordered(g["q"], g["k"], g["v"], g["log_lambda"], o, lion.MASK_S)
        assert lion.sync_status() == lion.ERR_INVALID_ARG
        assert lion.sync_status() == lion.OK
    with pytest.raises(lion.LionError):
        q32 = torch.zeros((1, 1, 8, 32), dtype=torch.bfloat16, device="cuda")
        lion.attn_fwd_reordered(q32, q32, q32, None, torch.zeros((2, 8), dtype=torch.int32, device="cuda"),
                                lion.MASK_LIT)


def _reorder_bwd_check(oracle_mod, inp, orders, seed, phi=0):
    q64, k64, v64, ll64 = f64(inp)
    dy = np.random.default_rng(seed).standard_normal(q64.shape).astype(np.float32)
    ref = oracle_mod.full_bwd_reordered(q64, k64, v64, ll64, orders, dy.astype(np.float64), inp["mask"], phi)
    g = _cuda(inp)
    o = torch.from_numpy(np.ascontiguousarray(orders, dtype=np.int32)).cuda()
    got = lion.attn_bwd_reordered(g["q"], g["k"], g["v"], g["log_lambda"], o, torch.from_numpy(dy).cuda(),
                                  inp["mask"], phi)
    assert lion.sync_status() == lion.OK
    _grad_rows(ref, got, f"reordered bwd {MASK_NAME[inp['mask']]} {tuple(q64.shape)} phi {phi}")


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ("lit", "d", "s"))
@pytest.mark.parametrize("dtype", ("bf16", "fp32"))
def test_reordered_backward_matches_oracle(oracle_mod, mask, dtype):
    """Gradients through the reordered full form against the oracle's (pinned
    by finite differences), for ViT-grid and random orders."""
    rng = np.random.default_rng(1600)
    inp = synth.make_inputs(2, 3, 197, 64, mask, dtype, seed=1601)
    _reorder_bwd_check(oracle_mod, inp, _vit_grid_orders(), 1602)
    for n, (B, H, L, d) in enumerate(((1, 2, 150, 64), (1, 1, 130, 128), (2, 1, 7, 64))):
        inp = synth.make_inputs(B, H, L, d, mask, dtype, seed=1610 + 10 * n)
        _reorder_bwd_check(oracle_mod, inp, np.stack([rng.permutation(L), rng.permutation(L)]), 1611 + 10 * n)
    # L = 1: y = v, so dv = dy and dq = dk = 0 up to the fp32 rounding of v - y
    inp = synth.make_inputs(3, 2, 1, 64, mask, dtype, seed=1640)
    g = _cuda(inp)
    dy = torch.randn(3, 2, 1, 64, device="cuda")
    o = torch.zeros((2, 1), dtype=torch.int32, device="cuda")
    dq, dk, dv, dll = lion.attn_bwd_reordered(g["q"], g["k"], g["v"], g["log_lambda"], o, dy, inp["mask"])
    scale = float(dy.abs().max())
    assert float((dv - dy).abs().max()) <= 1e-5 * scale
    assert float(dq.abs().max()) <= 1e-3 * scale and float(dk.abs().max()) <= 1e-3 * scale
    if dll is not None:
        assert float(dll.abs().max()) == 0.0


@pytest.mark.gpu
def test_reordered_backward_long_sequence(oracle_mod):
    """L = 1100: above the stored-tile limit, the columns pass recomputes the
    scores."""
    rng = np.random.default_rng(1670)
    inp = synth.make_inputs(1, 1, 1100, 64, "s", "bf16", seed=1671)
    _reorder_bwd_check(oracle_mod, inp, np.stack([rng.permutation(1100), rng.permutation(1100)]), 1672)


@pytest.mark.gpu
def test_reordered_backward_feature_map_and_invalid_orders(oracle_mod):
    rng = np.random.default_rng(1650)
    inp = synth.make_inputs(2, 2, 120, 64, "s", "bf16", seed=1651)
    _reorder_bwd_check(oracle_mod, inp, np.stack([rng.permutation(120), rng.permutation(120)]), 1652, phi=1)
    g = _cuda(inp)
    bad = torch.from_numpy(np.stack([np.arange(120), np.r_[np.arange(119), 7]]).astype(np.int32)).cuda()
    lion.attn_bwd_reordered(g["q"], g["k"], g["v"], g["log_lambda"], bad, torch.zeros((2, 2, 120, 64), device="cuda"),
                            lion.MASK_S)
    assert lion.sync_status() == lion.ERR_INVALID_ARG
    assert lion.sync_status() == lion.OK


@pytest.mark.gpu
def test_reordered_autograd_function_uses_the_reordered_backward():
    inp = synth.make_inputs(2, 3, 197, 64, "s", "bf16", seed=1660)
    g = _cuda(inp)
    o = torch.from_numpy(_vit_grid_orders()).cuda()
    q = g["q"].clone().requires_grad_(True)
    k = g["k"].clone().requires_grad_(True)
    v = g["v"].clone().requires_grad_(True)
    ll = g["log_lambda"].clone().requires_grad_(True)
    y = lion.LionReorderedAttention.apply(q, k, v, ll, o, lion.MASK_S)
    dy = torch.randn_like(y)
    y.backward(dy)
    dq, dk, dv, dll = lion.attn_bwd_reordered(g["q"], g["k"], g["v"], g["log_lambda"], o, dy, lion.MASK_S)
    assert torch.equal(q.grad, dq.to(q.dtype)) and torch.equal(k.grad, dk.to(k.dtype))
    assert torch.equal(v.grad, dv.to(v.dtype)) and torch.equal(ll.grad, dll)


# ------------------------------------------------- host-buffer entry -----
# lion_attn_fwd_host runs the same kernels on slices of the batch copied in
# and out by the library: its output equals the device entry point's bit for
# bit, whatever the slicing.
@pytest.mark.gpu
@pytest.mark.parametrize("mask", ("lit", "d", "s"))
def test_host_entry_matches_device_entry(mask):
    for B, H, L, chunk, form, dtype in ((5, 3, 197, 128, "chunk", "bf16"), (3, 2, 300, 128, "chunk", "bf16"),
                                        (4, 2, 64, 64, "full", "fp32"), (2, 2, 77, 16, "rnn", "fp32")):
        inp = synth.make_inputs(B, H, L, 64, mask, dtype, seed=1300 + L)
        g = _cuda(inp)
        want = lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], inp["mask"], form, chunk).cpu()
        host = {k: (None if inp[k] is None else inp[k].contiguous().pin_memory()) for k in ("q", "k", "v", "log_lambda")}
        for slices in (0, 1, 2, 3, B):
            got = lion.attn_fwd_host(host["q"], host["k"], host["v"], host["log_lambda"], inp["mask"], form, chunk,
                                     slices=slices)
            torch.cuda.synchronize()
            assert torch.equal(got, want), (B, L, form, slices)
    # pageable host memory is accepted (copied synchronously); device memory is refused
    inp = synth.make_inputs(2, 2, 50, 64, mask, "bf16", seed=1390)
    g = _cuda(inp)
    want = lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], inp["mask"], "chunk", 64).cpu()
    got = lion.attn_fwd_host(inp["q"], inp["k"], inp["v"], inp["log_lambda"], inp["mask"], "chunk", 64,
                             out=torch.empty_like(want))
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    with pytest.raises(ValueError):
        lion.attn_fwd_host(g["q"], g["k"], g["v"], g["log_lambda"], inp["mask"], "chunk", 64)


# Consecutive calls on two caller streams in turn (how a serving loop issues
# batches, and how bench.py times the end-to-end path): the calls share the
# library's copy streams, and one call's copies in overlap the previous call's
# compute and copies out.  Each batch's output must still be its own, bit for
# bit the device entry point's.
@pytest.mark.gpu
def test_host_entry_on_two_streams_in_turn():
    B, H, L = 6, 3, 197
    batches = [synth.make_inputs(B, H, L, 64, "s", "bf16", seed=1400 + i) for i in range(4)]
    wants = []
    for inp in batches:
        g = _cuda(inp)
        wants.append(lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], inp["mask"], "chunk", 128).cpu())
    hosts = [{k: inp[k].contiguous().pin_memory() for k in ("q", "k", "v", "log_lambda")} for inp in batches]
    outs = [torch.empty((B, H, L, 64), dtype=torch.float32).pin_memory() for _ in batches]
    streams = [torch.cuda.current_stream(), torch.cuda.Stream()]
    for rep in range(3):
        for o in outs:
            o.fill_(float("nan"))
        for i, (h, o) in enumerate(zip(hosts, outs)):
            lion.attn_fwd_host(h["q"], h["k"], h["v"], h["log_lambda"], "s", "chunk", 128, out=o,
                               slices=1 if rep == 0 else rep + 1, stream=streams[i % 2])
        torch.cuda.synchronize()
        for i, (o, want) in enumerate(zip(outs, wants)):
            assert torch.equal(o, want), (rep, i)


# --------------------------------------------------- bfloat16 output -----
# out_bf16: the chunk-128 kernels store y as bfloat16 themselves; the other
# paths round an fp32 temporary.  Either way each value must be the fp32
# result rounded to nearest even, bit for bit.
@pytest.mark.gpu
@pytest.mark.parametrize("mask", ("lit", "d", "s"))
def test_bf16_output_is_the_rounded_fp32_output(mask):
    for B, H, L, form, chunk, dtype in ((3, 4, 197, "chunk", 128, "bf16"),   # chunk-128, L <= 256
                                        (2, 2, 700, "chunk", 128, "bf16"),   # chunk-128, long
                                        (2, 2, 150, "chunk", 64, "bf16"),    # chunk-64, rounded after
                                        (2, 2, 90, "full", 1, "fp32"), (2, 2, 90, "rnn", 1, "fp32")):
        inp = synth.make_inputs(B, H, L, 64, mask, dtype, seed=1400 + L)
        g = _cuda(inp)
        y32 = lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], inp["mask"], form, chunk)
        y16 = lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], inp["mask"], form, chunk,
                            out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert y16.dtype == torch.bfloat16
        assert torch.equal(y16, y32.to(torch.bfloat16)), (B, L, form, chunk)
    inp = synth.make_inputs(2, 2, 100, 64, mask, "bf16", seed=1450)
    g = _cuda(inp)
    y32 = lion.attn_fwd_causal(g["q"], g["k"], g["v"], g["log_lambda"], inp["mask"], "chunk", 32)
    y16 = lion.attn_fwd_causal(g["q"], g["k"], g["v"], g["log_lambda"], inp["mask"], "chunk", 32,
                               out_dtype=torch.bfloat16)
    assert torch.equal(y16, y32.to(torch.bfloat16))

