"""GPU parity of the chunkwise gradients (lion_attn_bwd_chunk) against the
float64 oracle's gradients, which central finite differences of the forward
pin (test_oracle_pins.py), and, at the high-resolution length the oracle's
quadratic gradients cannot reach, against identities that hold at any size:
Euler's identity in v, the scale invariances of identity features, and
directional derivatives of the fp32 forward.  The gradients are the full
form's (rebuttal page, reply "Concern 1", Theorem 3.3 Eq 25); the chunkwise
route mirrors the forward's scans ("LION Part IV - Results", "LION Chunk")."""
import numpy as np
import pytest
import torch

from bidirectional_masked_linear_gb300 import lion, synth
from test_gpu_parity import MASK_NAME, TOL_BWD, _cuda, _grad_rows, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bidirectional_masked_linear_gb300 import build
    lion.load(build.build())


def _chunk_check(oracle_mod, inp, seed, phi=0):
    q64, k64, v64, ll64 = f64(inp)
    dy = np.random.default_rng(seed).standard_normal(q64.shape).astype(np.float32)
    ref = oracle_mod.full_bwd(q64, k64, v64, ll64, dy.astype(np.float64), inp["mask"], phi, threads=0)
    g = _cuda(inp)
    got = lion.attn_bwd(g["q"], g["k"], g["v"], g["log_lambda"], torch.from_numpy(dy).cuda(), inp["mask"], phi,
                        form=lion.FORM_CHUNK)
    torch.cuda.synchronize()
    B, H, L, d = q64.shape
    _grad_rows(ref, got, f"bwd chunk {MASK_NAME[inp['mask']]} {inp['q'].dtype} ({B},{H},{L},{d}) phi {phi}")
    return got


@pytest.mark.parametrize("mask", ("lit", "d", "s"))
@pytest.mark.parametrize("dtype", ("bf16", "fp32"))
def test_bwd_chunk_matches_oracle(oracle_mod, mask, dtype):
    """Every head dim (chunks of 64 tokens; 32 at d = 128), one token, one
    chunk, exact chunk multiples, ragged last chunks and many chunks."""
    for n, (B, H, L, d) in enumerate(((1, 2, 64, 16), (2, 3, 197, 64), (1, 2, 33, 32), (1, 1, 300, 128),
                                      (1, 2, 515, 64), (2, 1, 7, 64), (1, 2, 128, 64),
                                      (1, 1, 129, 128), (1, 1, 2048, 64))):
        inp = synth.make_inputs(B, H, L, d, mask, dtype, seed=1900 + 10 * n)
        _chunk_check(oracle_mod, inp, 1901 + 10 * n)


@pytest.mark.parametrize("mask", ("lit", "d", "s"))
def test_bwd_chunk_single_token(mask):
    """L = 1: y = v whatever q and k are, so dv = dy and dq = dk = 0 up to the
    fp32 rounding of v - y; the decay never enters (dlog_lambda = 0)."""
    inp = synth.make_inputs(3, 2, 1, 64, mask, "bf16", seed=1940)
    g = _cuda(inp)
    dy = torch.randn(3, 2, 1, 64, generator=torch.Generator().manual_seed(1941)).cuda()
    dq, dk, dv, dll = lion.attn_bwd(g["q"], g["k"], g["v"], g["log_lambda"], dy, inp["mask"], form=lion.FORM_CHUNK)
    scale = float(dy.abs().max())
    assert float((dv - dy).abs().max()) <= 1e-5 * scale
    assert float(dq.abs().max()) <= 1e-3 * scale and float(dk.abs().max()) <= 1e-3 * scale
    if dll is not None:
        assert float(dll.abs().max()) == 0.0


@pytest.mark.parametrize("mask,phi,positive", (("lit", 2, False), ("d", 2, False), ("s", 1, False),
                                               ("s", 3, True), ("d", 3, True)))
def test_bwd_chunk_feature_maps(oracle_mod, mask, phi, positive):
    inp = synth.make_inputs(2, 2, 150, 64, mask, "bf16", seed=1950)
    if positive:   # identity features need row sums away from zero
        for key in ("q", "k"):
            inp[key] = (inp[key].float().abs() + 0.25).to(inp[key].dtype)
    _chunk_check(oracle_mod, inp, 1951, phi)


def test_bwd_chunk_steep_decay(oracle_mod):
    """log lambda scaled by 40: most of M underflows, inside chunks and across
    them (the carried states decay to zero within a chunk).  The inputs of the
    full-form gradients' steep-decay case, held to the same bound: y_i is
    then close to v_i and dA_ii = dy_i . (v_i - y_i) / den_i cancels, which
    both routes compute the same way."""
    inp = synth.make_inputs(2, 2, 120, 64, "s", "bf16", seed=810)
    inp["log_lambda"] = inp["log_lambda"] * 40.0
    q64, k64, v64, ll64 = f64(inp)
    dy = np.random.default_rng(811).standard_normal(q64.shape).astype(np.float32)
    ref = oracle_mod.full_bwd(q64, k64, v64, ll64, dy.astype(np.float64), inp["mask"], 1)
    g = _cuda(inp)
    got = lion.attn_bwd(g["q"], g["k"], g["v"], g["log_lambda"], torch.from_numpy(dy).cuda(), inp["mask"], 1,
                        form=lion.FORM_CHUNK)
    # the full form lands at 1.9e-4 of a row on these inputs, the chunkwise
    # route (another summation order for y_i, hence for v_i - y_i) at 2.7e-4
    _grad_rows(ref, got, "bwd chunk steep-decay s", tol=5e-4)


@pytest.mark.parametrize("mask", ("d", "s"))
def test_bwd_chunk_matches_full_form_gradients_at_8192(mask):
    """At the full form's maximum length both gradient routes run on the GPU
    in fp32: they agree row by row.  elu+1 features keep every row sum away
    from zero, so that the comparison measures the two routes and not the
    rounding that an ill-conditioned row (SiLU features, a row sum that
    cancels) amplifies differently in each."""
    inp = synth.make_inputs(1, 2, lion.FULL_MAX_L, 64, mask, "bf16", seed=1970)
    g = _cuda(inp)
    dy = torch.randn(inp["q"].shape, generator=torch.Generator().manual_seed(1971)).cuda()
    full = lion.attn_bwd(g["q"], g["k"], g["v"], g["log_lambda"], dy, inp["mask"], lion.PHI_ELU1)
    chunk = lion.attn_bwd(g["q"], g["k"], g["v"], g["log_lambda"], dy, inp["mask"], lion.PHI_ELU1,
                          form=lion.FORM_CHUNK)
    ref = tuple(None if x is None else x.double().cpu().numpy() for x in full)
    # LION-D's dlog_lambda_h = sum_m m dLoss/dP_m over 8192 positions: its
    # terms cancel (they sum to zero without the weights m), and the two
    # routes' fp32 per-token terms differ by 1e-6 of each, about 2e-4 of it
    _grad_rows(ref, chunk, f"bwd chunk vs full {mask} (1,2,8192,64)", tol_dll=1e-3)


def _fp32_inputs(B, H, L, mask, seed, phi_identity=False):
    inp = synth.make_inputs(B, H, L, 64, mask, "fp32", seed=seed)
    if phi_identity:
        for key in ("q", "k"):
            inp[key] = inp[key].abs() + 0.25
    return _cuda(inp), inp["mask"]


def _loss(g, mask, dy, phi):
    """sum(dy * y) in float64 from the fp32 recurrent forward."""
    y = lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], mask, lion.FORM_RNN, phi=phi)
    return float((y.double() * dy.double()).sum())


HIRES_L = synth.WORKLOADS["hires_2496"].L


def test_bwd_chunk_high_resolution_identities():
    """L = 24,337 (the 2496-pixel image): Euler's identity in v (y is linear in
    v, so sum v . dv = sum dy . y per head), and with identity features the
    scale invariances (y is unchanged by scaling one q_i, or every k_j:
    q_i . dq_i = 0 per row, sum_j k_j . dk_j = 0 per head)."""
    for mask, phi in (("s", lion.PHI_DEFAULT), ("d", lion.PHI_DEFAULT), ("s", lion.PHI_IDENTITY)):
        g, mk = _fp32_inputs(1, 2, HIRES_L, mask, 1980, phi_identity=phi == lion.PHI_IDENTITY)
        dy = torch.randn(g["q"].shape, generator=torch.Generator().manual_seed(1981)).cuda()
        dq, dk, dv, dll = lion.attn_bwd(g["q"], g["k"], g["v"], g["log_lambda"], dy, mk, phi, form=lion.FORM_CHUNK)
        y = lion.attn_fwd(g["q"], g["k"], g["v"], g["log_lambda"], mk, lion.FORM_RNN, phi=phi)
        torch.cuda.synchronize()
        assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
        lhs = (g["v"].double() * dv.double()).sum(dim=(2, 3))
        rhs = (dy.double() * y.double()).sum(dim=(2, 3))
        scale = (g["v"].double() * dv.double()).abs().sum(dim=(2, 3))
        assert float(((lhs - rhs).abs() / scale).max()) < 1e-5, (mask, phi)
        if phi == lion.PHI_IDENTITY:
            qd = (g["q"].double() * dq.double()).sum(-1)
            qs = (g["q"].double().norm(dim=-1) * dq.double().norm(dim=-1))
            assert float((qd.abs() / qs.clamp_min(1e-30)).max()) < 1e-3, mask
            kd = (g["k"].double() * dk.double()).sum(dim=(2, 3))
            ks = (g["k"].double() * dk.double()).abs().sum(dim=(2, 3))
            assert float((kd.abs() / ks).max()) < 1e-4, mask


@pytest.mark.parametrize("mask", ("d", "s"))
def test_bwd_chunk_high_resolution_directional_derivatives(mask):
    """L = 24,337: for a random direction of each input, the central
    difference of sum(dy . y) through the fp32 forward equals the gradient's
    directional derivative.  elu+1 features keep every row sum away from zero
    (with SiLU features a row whose sum nearly cancels makes the loss too
    curved for a finite step), and log lambda moves by a relative step
    (l (1 +- eps n), n ~ N(0, 1)) so that every decay stays below 1."""
    phi = lion.PHI_ELU1
    g, mk = _fp32_inputs(1, 2, HIRES_L, mask, 1990)
    dy = torch.randn(g["q"].shape, generator=torch.Generator().manual_seed(1991)).cuda()
    grads = dict(zip(("q", "k", "v", "log_lambda"),
                     lion.attn_bwd(g["q"], g["k"], g["v"], g["log_lambda"], dy, mk, phi, form=lion.FORM_CHUNK)))
    gen = torch.Generator().manual_seed(1992)

    def central(key, delta, eps):
        gp, gm = dict(g), dict(g)
        gp[key] = (g[key] + eps * delta).contiguous()
        gm[key] = (g[key] - eps * delta).contiguous()
        return (_loss(gp, mk, dy, phi) - _loss(gm, mk, dy, phi)) / (2 * eps)

    for key in ("q", "k", "v", "log_lambda"):
        delta = torch.randn(g[key].shape, generator=gen).cuda()
        if key == "log_lambda":
            # a relative step of every decay; the loss is steep along it, so a
            # larger step with Richardson's combination, (4 f(e) - f(2e)) / 3,
            # which removes the e^2 term, keeps the fp32 forward's rounding small
            delta = delta * g[key]
            fd = (4 * central(key, delta, 0.05) - central(key, delta, 0.1)) / 3
        else:
            fd = central(key, delta, 1e-2)
        an = float((grads[key].double() * delta.double()).sum())
        # LION-D's one decay per head: dlog_lambda_h = sum_m m dLoss/dP_m, whose
        # terms sum to zero without the weights m, so the fp32 per-token terms'
        # rounding (1e-6 of each) leaves about 1e-3 of the total at this length
        tol = 5e-3 if (key, mask) == ("log_lambda", "d") else 1e-3
        assert abs(fd - an) <= tol * abs(an) + 1e-2, (mask, key, fd, an)


def test_bwd_chunk_autograd_beyond_the_full_form():
    """LionAttention takes the chunkwise gradients past FULL_MAX_L."""
    g, mk = _fp32_inputs(1, 1, lion.FULL_MAX_L + 100, "s", 1995)
    q = g["q"].clone().requires_grad_(True)
    y = lion.LionAttention.apply(q, g["k"], g["v"], g["log_lambda"], mk, lion.FORM_CHUNK, 64)
    dy = torch.randn(y.shape, generator=torch.Generator().manual_seed(1996)).cuda()
    y.backward(dy)
    dq, _, _, _ = lion.attn_bwd(g["q"], g["k"], g["v"], g["log_lambda"], dy, mk, form=lion.FORM_CHUNK)
    assert torch.equal(q.grad, dq)
    assert float(dq.abs().max()) > 0 and TOL_BWD > 0
