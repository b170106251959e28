#!/usr/bin/env python
"""Throughput of the LION chunkwise forward operator on GB300.

One step = one call of the operator (feature map, log-decay prefix,
intra-chunk attention, chunk states, scans, combine/normalise) over one batch
of synthetic inputs already resident in HBM.  Default workload: ViT-B
(B=64, H=12, L=197, d=64), LION-S, chunk 128 (two chunks per head).  The
L=24,337 high-resolution workload is measured in the same run at chunk 128
(the pre-pass and the main pass of the long-sequence tensor-core path; the
main pass chains the segments itself) and reported under ``secondary``; every other workload, mask, form and
chunk length of the scope's configurations gets a line under ``configs``.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bidirectional_masked_linear_gb300 import lion, synth  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20      # > 129 MB L2
HIRES_CHUNK = 128               # chunk of the long-sequence tensor-core path
# fp32 arithmetic peak of the CUDA cores, from unit counts and the clock:
# 152 SMs x 128 fp32 lanes x 2 flop (FMA) x 2.07 GHz
FP32_ALU_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the dominant
# kernel, per unit (head) from one ncu capture, keyed by the SHA-256 of that
# kernel's sources at the time of the capture.  A key that no longer matches
# the sources reports null: the counters describe another kernel.  Keys are
# (chunk, sequence longer than 256 tokens): the long chunk-128 path has its
# own main pass.
_CSRC = "bidirectional_masked_linear_gb300/csrc/"
_COMMON = (_CSRC + "c128_common.cuh", _CSRC + "tc_ptx.cuh")
# the kernels one call launches, per (chunk, sequence longer than 256 tokens),
# with the sources each kernel is built from
_CALL_KERNELS = {
    (128, False): {"lion_chunk128_tc_kernel": (_CSRC + "lion_c128.cu",) + _COMMON},
    (128, True): {"lion_chunk128_pre_kernel": (_CSRC + "lion_c128P.cu",) + _COMMON,
                  "lion_chunk128_long_kernel": (_CSRC + "lion_c128L.cu",) + _COMMON},
}
# (kernel, sources sha, workload, mask, chunk) -> DRAM bytes per head (read +
# write) of one launch, from one ncu capture of that kernel
TRAFFIC_PER_HEAD = {
    # ViT-B shape at B = 128 (1536 heads), LION-S: 117.5 MB read + 35.9 MB written
    ("lion_chunk128_tc_kernel", "5dd15b36b1d88a0130d751da3af2ef9cc4b7e06423483cb1ffe51fca1118ae0c",
     "vit_b", "s", 128): (117484288 + 35912448) / 1536,
    # L = 24,337 (B = 2, H = 12, 24 heads), LION-S, the two launches of a call
    ("lion_chunk128_pre_kernel", "d8fc821aac36c539e362804654aebf24bd9d6d12636b2681774f8785d1d68d67",
     "hires_2496", "s", 128): (152046592 + 22330624) / 24,
    ("lion_chunk128_long_kernel", "90361246639db1e489f6cb005845a359cd6356e849622cdadd27fb782e4cfa79",
     "hires_2496", "s", 128): (270046208 + 110145536) / 24,
}


def _sources_sha(files):
    import hashlib
    h = hashlib.sha256()
    for rel in files:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_bytes(w, mask, chunk):
    """DRAM traffic of one whole call (every kernel it launches), with each
    kernel's bytes; None when a kernel has no capture at its current sources."""
    kernels = _CALL_KERNELS.get((chunk, w.L > 256))
    if not kernels:
        return None, None
    per = {}
    for name, files in kernels.items():
        b = TRAFFIC_PER_HEAD.get((name, _sources_sha(files), w.name, mask, chunk))
        if b is None:
            return None, None
        per[name] = b * w.B * w.H
    return sum(per.values()), per


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            hbm = next((float(v) for k, v in d.items() if "hbm" in k.lower() and
                        isinstance(v, (int, float))), None)
            bf16 = d.get("bf16_tflops")
            if hbm:
                return hbm, float(bf16) if bf16 else FALLBACK_BF16_TFLOPS, "measured"
        except (OSError, ValueError):
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def algorithmic_bytes(w, mask: str, out_bytes: int = 4) -> int:
    """Bytes the operator must move per call: q, k, v read once, y (fp32, or
    bf16 with out_bytes = 2) written once, plus the decays (per token for
    LION-S, per head for D)."""
    el = 2 if w.dtype == "bf16" else 4
    n = w.B * w.H * w.L * w.d
    b = 3 * n * el + out_bytes * n
    if mask == "s":
        b += 4 * w.B * w.H * w.L
    elif mask == "d":
        b += 4 * w.H
    return b


def _sm_count() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152


def long_segments(w, sms: int) -> int:
    """Segments a head's 256-token blocks are cut into on the long chunk
    paths: enough that B*H*segments fills the SMs, one when the heads alone
    do."""
    nbl = (w.L + 255) // 256
    bh = w.B * w.H
    nseg = min(nbl, max(1, sms // bh)) if nbl > 1 and bh < sms else 1
    segb = (nbl + nseg - 1) // nseg
    return (nbl + segb - 1) // segb


def kernels_per_call(form: str, chunk: int, w, mask: str = "s", sms: int = 152) -> int:
    """Kernel launches one operator call makes: the tensor-core chunk paths
    (bf16, d=64, chunk 64 or 128) take one launch up to 256 tokens; beyond,
    chunk 128 two (pre-pass, main pass, which chains the segments itself)
    and chunk 64 three (pre-pass, segment scan, main pass), two when every
    head is one segment; the recurrent form two with its workspace
    (the features of every token, then the column CTAs), three when the
    column CTAs (d / 8 a head) number under two an SM and L >= 256, so that
    the two sweeps run in separate CTAs and a last launch combines them; the
    full form at
    d = 64 and 128 two (the features, the tiled pass), three for LION-S (its
    prefix first); every other path one."""
    tc = form == "chunk" and chunk in (64, 128) and w.d == 64 and w.dtype == "bf16"
    if form == "rnn":
        return 3 if w.B * w.H * (w.d // 8) < 2 * sms and w.L >= 256 else 2
    if form == "full" and w.d in (64, 128):
        return 3 if mask == "s" else 2
    if tc and w.L > 256:
        return 2 if chunk == 128 or long_segments(w, sms) == 1 else 3
    return 1


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}", "--format=csv,noheader",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1].split()[0]))
                smax.append(float(parts[2].split()[0]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist, ws, rank, local
    return None, 1, 0, 0


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def _max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _build_once(dist, rank):
    """Rank 0 compiles the library (if anything is stale) while the others
    wait for its outcome in the process group's key-value store; a failed
    build ends every rank with the same error instead of leaving the others
    in a collective."""
    from bidirectional_masked_linear_gb300 import build
    if dist is None:
        build.build()
        return
    store = dist.distributed_c10d._get_default_store()
    if rank == 0:
        try:
            build.build()
            store.set("lion_build", "ok")
        except Exception as e:  # noqa: BLE001 -- reported to every rank
            store.set("lion_build", "failed: " + str(e).splitlines()[0][:200])
            raise
    else:
        store.wait(["lion_build"])
        outcome = store.get("lion_build").decode()
        if outcome != "ok":
            raise SystemExit(f"rank {rank}: library build on rank 0 {outcome}")


def time_device(call, steps, warmup, flush, stream):
    """Per-step CUDA-event durations (ms) of `call` on `stream`, L2 flushed
    before every step (outside the events)."""
    for _ in range(warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def _workload(name, batch=0):
    w = synth.WORKLOADS[name]
    if batch:
        import dataclasses
        w = dataclasses.replace(w, B=batch)
    return w


def measure(name, mask, chunk, form, steps, warmup, flush, batch=0, out_dtype=torch.float32):
    w = _workload(name, batch)
    inp = synth.make_inputs(w.B, w.H, w.L, w.d, mask, w.dtype, w.seed, w.lam)
    dev = {k: (None if inp[k] is None else inp[k].cuda()) for k in ("q", "k", "v", "log_lambda")}
    out = torch.empty((w.B, w.H, w.L, w.d), dtype=out_dtype, device="cuda")
    fcode = lion.FORMS[form]
    wsb = lion.workspace_bytes(w.B, w.H, w.L, w.d, fcode, chunk)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        lion.attn_fwd(dev["q"], dev["k"], dev["v"], dev["log_lambda"], inp["mask"], fcode, chunk,
                      out=out, workspace=ws)

    times = time_device(call, steps, warmup, flush, stream)
    return w, inp, times, (dev, out, ws, call)


def measure_e2e(w, inp, mask, chunk, form, steps, warmup):
    """Same metric end to end through the library's host-buffer entry point
    (lion_attn_fwd_host): pinned host inputs, the library's copies in, the
    operator and the copies out, all inside the timed region.  The calls go
    out as a serving loop would issue consecutive batches: on two caller
    streams in turn, each into its own pinned output buffer, one call per
    batch (no slicing), so that one batch's copies in overlap the previous
    batch's compute and copies out."""
    fcode = lion.FORMS[form]
    host = {k: (None if inp[k] is None else inp[k].pin_memory()) for k in ("q", "k", "v", "log_lambda")}
    outs = [torch.empty((w.B, w.H, w.L, w.d), dtype=torch.float32).pin_memory() for _ in range(2)]
    main = torch.cuda.current_stream()
    streams = [main, torch.cuda.Stream()]
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = outs[0].numel() * outs[0].element_size()

    def step(k):
        lion.attn_fwd_host(host["q"], host["k"], host["v"], host["log_lambda"], inp["mask"], fcode, chunk,
                           out=outs[k % 2], slices=1, stream=streams[k % 2])

    for k in range(warmup):
        step(k)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(main)
    streams[1].wait_event(a)
    for k in range(steps):
        step(k)
    main.wait_stream(streams[1])
    b.record(main)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return ms, h2d, d2h


def bwd_flops(w) -> int:
    """Algorithmic flops of the gradients through the full form per call: the
    six L x L x d products they need (S = phi(Q) phi(K)^T, the recomputed
    A V, G V^T, dS phi(K), dS^T phi(Q), A^T G), 2 L^2 d flops each, per head."""
    return 12 * w.B * w.H * w.L * w.L * w.d


def bwd_chunk_flops(w) -> int:
    """Algorithmic flops of the chunkwise gradients per call, chunks of C
    tokens: per chunk six C x C x d products (scores, A [V|1], dA, (M.dA)
    phi(K), (M.dA)^T phi(Q), A^T G) and twelve C x d x d state products (two
    summaries and two applications each of the phi(k) [v;1]^T and phi(q) G^T
    states, forward and backward), 2 flops a multiply-add: 12 L C d + 24 L d^2
    per head."""
    C = 32 if w.d >= 128 else 64
    return w.B * w.H * w.L * (12 * C * w.d + 24 * w.d * w.d)


def bwd_launches(mask, d) -> int:
    """Kernels one lion_attn_bwd call launches: phi, rows and columns passes;
    the dl pass for LION-D and LION-S; the batch sum for LION-D; the prefix of
    log-lambda for LION-S when d >= 64 (the register-tiled passes)."""
    return 3 + (mask != "lit") + (mask == "d") + (mask == "s" and d >= 64)


def measure_bwd(w, mask, steps, warmup, flush, chunkwise=False):
    """CUDA-event time of one gradient call (lion_attn_bwd, or
    lion_attn_bwd_chunk with `chunkwise`, all its kernels) through the C entry
    point with preallocated outputs and workspace."""
    import ctypes
    inp = synth.make_inputs(w.B, w.H, w.L, w.d, mask, w.dtype, w.seed, w.lam)
    dev = {k: (None if inp[k] is None else inp[k].cuda()) for k in ("q", "k", "v", "log_lambda")}
    dy = torch.randn((w.B, w.H, w.L, w.d), dtype=torch.float32, device="cuda")
    grads = [torch.empty_like(dy) for _ in range(3)]
    dll = None
    if inp["mask"] == lion.MASK_D:
        dll = torch.empty((w.H,), dtype=torch.float32, device="cuda")
    elif inp["mask"] == lion.MASK_S:
        dll = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device="cuda")
    wsb = lion.bwd_workspace_bytes(w.B, w.H, w.L, w.d, lion.FORM_CHUNK if chunkwise else lion.FORM_FULL)
    wsp = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    p = lambda t: None if t is None else t.data_ptr()
    a = lion._BwdArgs(p(dev["q"]), p(dev["k"]), p(dev["v"]), p(dev["log_lambda"]), p(dy),
                      p(grads[0]), p(grads[1]), p(grads[2]), p(dll), w.B, w.H, w.L, w.d,
                      inp["mask"], lion.DTYPE_BF16 if w.dtype == "bf16" else lion.DTYPE_FP32,
                      lion.PHI_DEFAULT, wsp.data_ptr(), wsb, stream.cuda_stream)
    lib = lion.load()

    entry = lib.lion_attn_bwd_chunk if chunkwise else lib.lion_attn_bwd

    def call():
        st = entry(ctypes.byref(a))
        if st:
            raise RuntimeError(f"gradient call failed ({st})")

    return time_device(call, steps, warmup, flush, stream)


def reorder_flops(w) -> int:
    """Algorithmic flops of the full form per call: phi(Q) phi(K)^T and the
    masked product with V, 2 L^2 d flops each, per head."""
    return 4 * w.B * w.H * w.L * w.L * w.d


def reorder_launches(mask) -> int:
    """Kernels one lion_attn_fwd_reordered call launches: the order check,
    phi and the full form; LION-S adds the prefix along each order."""
    return 3 + (mask == "s")


def vit_grid_orders(L):
    """Two traversals of a ViT token sequence (class token first, then a
    square patch grid): the patches row by row, and column by column.  Any
    permutation costs the same; these stand in for the pages' two orders."""
    side = int(round((L - 1) ** 0.5))
    if side * side != L - 1:
        rows = torch.arange(L, dtype=torch.int32)
        return torch.stack([rows, rows.flip(0)])
    rows = torch.arange(L, dtype=torch.int32)
    cols = torch.cat([torch.zeros(1, dtype=torch.int32),
                      1 + torch.arange(side * side, dtype=torch.int32).reshape(side, side).t().reshape(-1)])
    return torch.stack([rows, cols])


def measure_reordered(w, mask, steps, warmup, flush):
    """CUDA-event time of one lion_attn_fwd_reordered call through the C
    entry point with a preallocated output and workspace."""
    import ctypes
    inp = synth.make_inputs(w.B, w.H, w.L, w.d, mask, w.dtype, w.seed, w.lam)
    dev = {k: (None if inp[k] is None else inp[k].cuda()) for k in ("q", "k", "v", "log_lambda")}
    orders = vit_grid_orders(w.L).cuda()
    out = torch.empty((w.B, w.H, w.L, w.d), dtype=torch.float32, device="cuda")
    wsb = lion.reordered_workspace_bytes(w.B, w.H, w.L, w.d)
    wsp = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    p = lambda t: None if t is None else t.data_ptr()
    a = lion._ReorderArgs(p(dev["q"]), p(dev["k"]), p(dev["v"]), p(dev["log_lambda"]), orders.data_ptr(),
                          out.data_ptr(), w.B, w.H, w.L, w.d, inp["mask"],
                          lion.DTYPE_BF16 if w.dtype == "bf16" else lion.DTYPE_FP32, lion.PHI_DEFAULT,
                          wsp.data_ptr(), wsb, stream.cuda_stream)
    lib = lion.load()

    def call():
        st = lib.lion_attn_fwd_reordered(ctypes.byref(a))
        if st:
            raise RuntimeError(f"lion_attn_fwd_reordered failed ({st})")

    t = time_device(call, steps, warmup, flush, stream)
    if lion.sync_status() != lion.OK:
        raise RuntimeError("traversal order rejected on the device")
    return t


def measure_reordered_bwd(w, mask, steps, warmup, flush):
    """CUDA-event time of one lion_attn_bwd_reordered call (the same orders as
    measure_reordered) with preallocated gradients and workspace."""
    inp = synth.make_inputs(w.B, w.H, w.L, w.d, mask, w.dtype, w.seed, w.lam)
    dev = {k: (None if inp[k] is None else inp[k].cuda()) for k in ("q", "k", "v", "log_lambda")}
    orders = vit_grid_orders(w.L).cuda()
    dy = torch.randn((w.B, w.H, w.L, w.d), dtype=torch.float32, device="cuda")
    ws = torch.empty(lion.reordered_bwd_workspace_bytes(w.B, w.H, w.L, w.d), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        lion.attn_bwd_reordered(dev["q"], dev["k"], dev["v"], dev["log_lambda"], orders, dy, inp["mask"],
                                workspace=ws)

    t = time_device(call, steps, warmup, flush, stream)
    if lion.sync_status() != lion.OK:
        raise RuntimeError("traversal order rejected on the device")
    return t


def stream_bytes(B, H, d, in_bytes=2) -> int:
    """Bytes one decode step must move: the fp32 state S (d x d) and z read
    and written, the token's q, k, v and log-lambda read, y_part and c_part
    written, per head."""
    return B * H * (2 * (d * d + d) * 4 + 3 * d * in_bytes + 4 + d * 4 + 4)


def measure_causal(w, mask, form, chunk, steps, warmup, flush):
    """The forward half alone (lion_attn_fwd_causal) on the workload's
    inputs, with its workspace passed in; CUDA events, L2 flushed."""
    inp = synth.make_inputs(w.B, w.H, w.L, w.d, mask, w.dtype, w.seed, w.lam)
    dev = {k: (None if inp[k] is None else inp[k].cuda()) for k in ("q", "k", "v", "log_lambda")}
    out = torch.empty((w.B, w.H, w.L, w.d), dtype=torch.float32, device="cuda")
    fcode = lion.FORMS[form]
    wsb = lion.workspace_bytes(w.B, w.H, w.L, w.d, fcode, max(chunk, 1))
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        lion.attn_fwd_causal(dev["q"], dev["k"], dev["v"], dev["log_lambda"], inp["mask"], fcode, max(chunk, 1),
                             out=out, workspace=ws)

    return time_device(call, steps, warmup, flush, stream)


def measure_stream(B, H, d, mask, steps, warmup):
    """Decode: `steps` consecutive lion_rnn_step calls (one direction, one
    token each for B*H heads), every step's inputs resident in HBM before
    the timed region.  A decode loop is launch-bound when driven call by call
    from the host, so the steps are captured once into a CUDA graph and the
    graph is replayed; CUDA events around the replays.  Returns the ms per
    step of the replay and of the same steps launched one by one."""
    import ctypes
    T = steps + warmup
    g = torch.Generator(device="cuda").manual_seed(1234)
    q = torch.randn((T, B, H, d), device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn((T, B, H, d), device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn((T, B, H, d), device="cuda", generator=g).to(torch.bfloat16)
    mk = lion.MASKS[mask]
    ll = None
    if mk == lion.MASK_S:
        ll = torch.nn.functional.logsigmoid(torch.randn((T, B, H), device="cuda", generator=g) + 3.0)
    elif mk == lion.MASK_D:
        ll = torch.log(torch.rand((H,), device="cuda", generator=g) * 0.099 + 0.9).expand(T, H).contiguous()
    S = torch.zeros((B, H, d, d), device="cuda")
    z = torch.zeros((B, H, d), device="cuda")
    y = torch.empty((B, H, d), device="cuda")
    c = torch.empty((B, H), device="cuda")
    lib = lion.load()
    vp = ctypes.c_void_p

    def step(t):
        stream = torch.cuda.current_stream()
        st = lib.lion_rnn_step(vp(q[t].data_ptr()), vp(k[t].data_ptr()), vp(v[t].data_ptr()),
                               vp(None if ll is None else ll[t].data_ptr()), vp(S.data_ptr()),
                               vp(z.data_ptr()), vp(y.data_ptr()), vp(c.data_ptr()), B, H, d, mk,
                               lion.DTYPE_BF16, vp(stream.cuda_stream))
        if st:
            raise RuntimeError(f"lion_rnn_step failed ({st})")

    def timed(fn, reps):
        stream = torch.cuda.current_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    for t in range(warmup):
        step(t)
    torch.cuda.synchronize()
    eager = timed(lambda: [step(t) for t in range(warmup, T)], 1) / steps
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="relaxed"):
        for t in range(warmup, T):
            step(t)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    return timed(graph.replay, 5) / steps, eager


def _oracle_sample(name, mask, budget_s, threads):
    """tokens/s of the float64 oracle on a bounded sample of a workload: batch
    rows (all H heads each) in order, wrapping round to the first row, until
    `budget_s` of wall time is spent (at least one row).  The form is the one
    the scope's measurement plan names: the brute force for the ViT-length
    workloads (up to 256 tokens), the recurrent form for the longer ones
    (BERT-large, L = 24,337, LRA: the brute force is O(L^2) in memory and
    time)."""
    import oracle
    w = synth.WORKLOADS[name]
    inp = synth.workload_inputs(name, mask)
    q, k, v, ll = (synth.as_f64(inp[x]) for x in ("q", "k", "v", "log_lambda"))
    fn, form = (oracle.full, "brute-force full form") if w.L <= 256 else (oracle.rnn, "recurrent form")
    oracle.threads(threads)
    cores = oracle.threads(threads)
    rows, t0 = 0, time.perf_counter()
    while rows == 0 or (time.perf_counter() - t0) < budget_s:
        b = rows % w.B
        sl = slice(b, b + 1)
        lls = None if ll is None else (ll if mask == "d" else ll[sl])
        fn(q[sl], k[sl], v[sl], lls, inp["mask"], threads=threads)
        rows += 1
    dt = time.perf_counter() - t0
    par = "OpenMP over heads" if cores > 1 else "one thread"
    return {"value": rows * w.L / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows} batch rows of {w.B} (wrapping; {rows * w.H} heads x L={w.L}), "
                      f"float64 {form}, {par}, {dt:.1f} s"}


def cpu_baseline(name, mask, budget_s=10.0):
    """The float64 oracle as it stands, on all host cores and on one, each on
    a bounded sample of the workload (see _oracle_sample)."""
    res = _oracle_sample(name, mask, budget_s, 0)
    res["single_thread"] = _oracle_sample(name, mask, budget_s / 2, 1)
    return res


def run_reference(args, dist, ws, rank):
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    budget = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    res = []
    for i in range(args.warmup + args.steps):
        r = _oracle_sample(args.workload, args.mask, budget, 0)
        if i >= args.warmup:
            res.append(r)
    val = statistics.median(r["value"] for r in res)
    ms = w.B * w.L / val * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(args, w),
            "cpu_baseline": dict(res[-1], value=val),
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


METRIC = "LION attn fwd tokens/s (chunkwise form)"

# Every workload / mask / form / chunk of the scope's configurations that is
# not the headline, each timed for its own line: (workload, mask, form, chunk)
CONFIG_LINES = [
    ("tiny_d_fp32", "d", "chunk", 16), ("tiny_d_fp32", "d", "full", 16), ("tiny_d_fp32", "d", "rnn", 16),
    ("vit_t_s", "s", "chunk", 64),
] + [("vit_b", m, "chunk", c) for m in ("lit", "d", "s") for c in (32, 64, 128)] + [
    ("vit_b", m, f, 0) for m in ("lit", "d", "s") for f in ("full", "rnn")] + [
    ("bert_large", m, "chunk", c) for m in ("d", "s") for c in (64, 128)] + [
    ("hires_2496", m, "chunk", c) for m in ("d", "s") for c in (64, 128)] + [
    ("hires_2496", m, "rnn", 0) for m in ("d", "s")] + [
    ("lra_4096", "s", "chunk", 64), ("lra_4096", "d", "chunk", 128), ("lra_4096", "s", "rnn", 0),
]


def full_flops(w) -> int:
    """Algorithmic flops of the full form per call: phi(Q) phi(K)^T and the
    masked product with [V | 1], 2 L^2 d flops each, per head."""
    return 4 * w.B * w.H * w.L * w.L * w.d


def rnn_flops(w) -> int:
    """Algorithmic flops of the recurrent form per call: both sweeps update the
    d x (d + 1) state (S and z) and apply it to phi(q), a multiply-add per
    element each: 2 * 2 * 2 d (d + 1) per token and head."""
    return 8 * w.B * w.H * w.L * w.d * (w.d + 1)


def measure_config(c, flush, hbm_peak, steps=20, warmup=3):
    """One line of ``configs``: CUDA-event time of one call, tokens/s, and the
    fraction of the roofline that bounds the path: HBM bytes for the chunk
    form, the fp32 CUDA-core peak for the full form (O(L^2 d) arithmetic on
    16 + 4 bytes a token) and for the recurrent form (O(d^2) arithmetic a
    token, sequential along the tokens)."""
    name, mask, form, chunk = c
    w, _, t, _k = measure(name, mask, chunk or 64, form, steps, warmup, flush)
    ms = statistics.mean(t)
    line = {"workload": f"{w.name} B={w.B} H={w.H} L={w.L} d={w.d}", "mask": mask, "form": form,
            "chunk": chunk if form == "chunk" else None, "input_dtype": w.dtype,
            "value": w.B * w.L / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
            "launches_per_call": kernels_per_call(form, chunk, w, mask, _sm_count()),
            "path": path_name(form, chunk, w)}
    b = algorithmic_bytes(w, mask)
    hbm = {"bound": "hbm", "achieved": b / (ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
           "frac": b / (ms * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": b}
    if form in ("full", "rnn"):
        fl = full_flops(w) if form == "full" else rnn_flops(w)
        line["roofline"] = {"bound": "alu", "achieved": fl / (ms * 1e-3) / 1e12, "peak": FP32_ALU_PEAK_TFLOPS,
                            "unit": "TFLOP/s", "frac": fl / (ms * 1e-3) / 1e12 / FP32_ALU_PEAK_TFLOPS,
                            "algorithmic_flops": fl}
        # the same bytes the chunk form's roofline counts, for comparison
        line["hbm"] = hbm
    else:
        line["roofline"] = hbm
    return line


def path_name(form, chunk, w) -> str:
    tc = form == "chunk" and w.d == 64 and w.dtype == "bf16"
    if tc and chunk in (64, 128):
        passes = ""
        if w.L > 256:
            passes = (" (pre-pass, main pass)" if chunk == 128 else
                      " (pre-pass, main pass; one segment a head)" if long_segments(w, _sm_count()) == 1
                      else " (pre-pass, segment scan, main pass)")
        return f"tcgen05 chunk-{chunk}" + passes
    if form == "full" and w.d in (64, 128):
        return "full form, fp32 CUDA cores, register-tiled"
    if form == "chunk" and chunk <= 64:
        return "chunk form, fp32 CUDA cores, register-tiled"
    return {"full": "full form, fp32 CUDA cores", "rnn": "recurrent form, fp32 CUDA cores",
            "chunk": "chunk form, fp32 CUDA cores"}[form]


def _config(args, w):
    return {"workload": f"{w.name} B={w.B} H={w.H} L={w.L} d={w.d}", "mask": args.mask,
            "form": args.form, "chunk": args.chunk, "input_dtype": w.dtype, "out_dtype": "f32",
            "global_batch": w.B, "seq_len": w.L, "parallelism": f"replicas x{args.gpus}",
            "l2": "flushed before every timed step (256 MiB write)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--workload", default="vit_b", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--mask", default="s", choices=("lit", "d", "s"))
    ap.add_argument("--chunk", type=int, default=128)
    ap.add_argument("--form", default="chunk", choices=("chunk", "full", "rnn"))
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-streaming", action="store_true")
    ap.add_argument("--no-reordered", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (profiling captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    dist, ws, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, dist, ws, rank)
        if dist is not None:
            dist.destroy_process_group()
        return

    torch.cuda.set_device(local)
    from bidirectional_masked_linear_gb300 import build
    _build_once(dist, rank)
    lion.load(build.LIB)
    hbm_peak, bf16_peak, peak_src = _peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    _barrier(dist)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        t_wall = time.perf_counter()
        w, inp, times, _keep = measure(args.workload, args.mask, args.chunk, args.form,
                                       args.steps, args.warmup, flush, args.batch)
        t_wall = time.perf_counter() - t_wall
    torch.cuda.synchronize()
    _barrier(dist)
    clocks = clk.summary()
    ms = statistics.mean(times)
    ms_all = _max_over_ranks(dist, ms)
    tokens = w.B * w.L
    value = ws * tokens / (ms_all * 1e-3)
    abytes = algorithmic_bytes(w, args.mask)
    achieved = abytes / (ms * 1e-3) / 1e9
    e2e = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h = measure_e2e(w, inp, args.mask, args.chunk, args.form, 50, 5)
        e2e_ms = _max_over_ranks(dist, e2e_ms)
        e2e = {"value": ws * tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "api": "lion_attn_fwd_host (pinned host buffers), one call per batch on two caller streams in "
                      "turn, each into its own pinned output buffer, so that a batch's copies in overlap the "
                      "previous batch's compute and copies out"}

    secondary = None
    if not args.no_secondary and args.workload != "hires_2496":
        w2, _, t2, _k2 = measure("hires_2496", args.mask if args.mask != "lit" else "s", HIRES_CHUNK,
                                 "chunk", 50, 3, flush)
        ms2 = statistics.mean(t2)
        b2 = algorithmic_bytes(w2, args.mask if args.mask != "lit" else "s")
        tr2, tr2k = traffic_bytes(w2, args.mask if args.mask != "lit" else "s", HIRES_CHUNK)
        secondary = {"workload": f"{w2.name} B={w2.B} H={w2.H} L={w2.L} d={w2.d}", "chunk": HIRES_CHUNK,
                     "value": w2.B * w2.L / (ms2 * 1e-3), "unit": "tokens/s", "ms_per_step": ms2,
                     "launches_per_call": kernels_per_call("chunk", HIRES_CHUNK, w2, "s", _sm_count()),
                     "roofline": {"bound": "hbm", "achieved": b2 / (ms2 * 1e-3) / 1e9,
                                  "peak": hbm_peak, "unit": "GB/s",
                                  "frac": b2 / (ms2 * 1e-3) / 1e9 / hbm_peak,
                                  "algorithmic_bytes": b2,
                                  "traffic": tr2, "traffic_per_kernel": tr2k,
                                  "note": "achieved and traffic cover the whole call: pre-pass and main "
                                          "pass (which chains the segments itself)"}}
        del _k2

    lra = None
    if not args.no_secondary and args.workload != "lra_4096":
        w3, _, t3, _k3 = measure("lra_4096", args.mask if args.mask != "lit" else "s", 128, "chunk", 50, 3, flush)
        ms3 = statistics.mean(t3)
        b3 = algorithmic_bytes(w3, args.mask if args.mask != "lit" else "s")
        lra = {"workload": f"{w3.name} B={w3.B} H={w3.H} L={w3.L} d={w3.d}", "chunk": 128,
               "value": w3.B * w3.L / (ms3 * 1e-3), "unit": "tokens/s", "ms_per_step": ms3,
               "roofline": {"bound": "hbm", "achieved": b3 / (ms3 * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                            "frac": b3 / (ms3 * 1e-3) / 1e9 / hbm_peak}}
        del _k3

    bf16_out = None
    if not args.no_secondary and args.form == "chunk" and args.chunk == 128 and w.dtype == "bf16":
        w4, _, t4, _k4 = measure(args.workload, args.mask, 128, "chunk", 50, 3, flush, args.batch,
                                 out_dtype=torch.bfloat16)
        ms4 = statistics.mean(t4)
        b4 = algorithmic_bytes(w4, args.mask, out_bytes=2)
        bf16_out = {"workload": _config(args, w)["workload"], "out_dtype": "bf16 (the fp32 result rounded to nearest even)",
                    "value": w4.B * w4.L / (ms4 * 1e-3), "unit": "tokens/s", "ms_per_step": ms4,
                    "roofline": {"bound": "hbm", "achieved": b4 / (ms4 * 1e-3) / 1e9, "peak": hbm_peak,
                                 "unit": "GB/s", "frac": b4 / (ms4 * 1e-3) / 1e9 / hbm_peak,
                                 "algorithmic_bytes": b4}}
        del _k4

    backward = None
    if not args.no_backward and w.L <= lion.FULL_MAX_L:
        tb = measure_bwd(w, args.mask, 20, 3, flush)
        msb = statistics.mean(tb)
        fl = bwd_flops(w)
        backward = {"form": "full", "value": w.B * w.L / (msb * 1e-3), "unit": "tokens/s", "ms_per_call": msb,
                    "launches_per_call": bwd_launches(args.mask, w.d),
                    "roofline": {"bound": "alu", "achieved": fl / (msb * 1e-3) / 1e12,
                                 "peak": FP32_ALU_PEAK_TFLOPS, "unit": "TFLOP/s",
                                 "frac": fl / (msb * 1e-3) / 1e12 / FP32_ALU_PEAK_TFLOPS,
                                 "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 flop x 2.07 GHz",
                                 "algorithmic_flops": fl}}

    if not args.no_backward:
        chunk_lines = []
        for wb in (w, synth.WORKLOADS["hires_2496"]):
            mb = args.mask if args.mask != "lit" or wb is w else "s"
            tc = measure_bwd(wb, mb, 10 if wb.L > 4096 else 20, 3, flush, chunkwise=True)
            msc = statistics.mean(tc)
            flc = bwd_chunk_flops(wb)
            chunk_lines.append({
                "form": "chunk", "workload": f"{wb.name} B={wb.B} H={wb.H} L={wb.L} d={wb.d}", "mask": mb,
                "value": wb.B * wb.L / (msc * 1e-3), "unit": "tokens/s", "ms_per_call": msc,
                "launches_per_call": 5 + (mb != "lit") + (mb == "d"),
                "roofline": {"bound": "alu", "achieved": flc / (msc * 1e-3) / 1e12, "peak": FP32_ALU_PEAK_TFLOPS,
                             "unit": "TFLOP/s", "frac": flc / (msc * 1e-3) / 1e12 / FP32_ALU_PEAK_TFLOPS,
                             "algorithmic_flops": flc}})
        backward = dict(backward or {}, chunkwise=chunk_lines)

    reordered = None
    if not args.no_reordered and w.L <= lion.FULL_MAX_L and w.d in (64, 128):
        tr = measure_reordered(w, args.mask, 20, 3, flush)
        msr = statistics.mean(tr)
        flr = reorder_flops(w)
        reordered = {"form": "full, mask averaged over two traversal orders",
                     "orders": "class token, then the patch grid by rows / by columns",
                     "value": w.B * w.L / (msr * 1e-3), "unit": "tokens/s", "ms_per_call": msr,
                     "launches_per_call": reorder_launches(args.mask),
                     "roofline": {"bound": "alu", "achieved": flr / (msr * 1e-3) / 1e12,
                                  "peak": FP32_ALU_PEAK_TFLOPS, "unit": "TFLOP/s",
                                  "frac": flr / (msr * 1e-3) / 1e12 / FP32_ALU_PEAK_TFLOPS,
                                  "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 flop x 2.07 GHz",
                                  "algorithmic_flops": flr}}
        trb = measure_reordered_bwd(w, args.mask, 10, 3, flush)
        msrb = statistics.mean(trb)
        flb = bwd_flops(w)
        reordered["backward"] = {"ms_per_call": msrb, "value": w.B * w.L / (msrb * 1e-3), "unit": "tokens/s",
                                 "roofline": {"bound": "alu", "achieved": flb / (msrb * 1e-3) / 1e12,
                                              "peak": FP32_ALU_PEAK_TFLOPS, "unit": "TFLOP/s",
                                              "frac": flb / (msrb * 1e-3) / 1e12 / FP32_ALU_PEAK_TFLOPS,
                                              "algorithmic_flops": flb}}

    causal = None
    if not args.no_streaming:
        causal = []
        for cform, cchunk in (("full", 0), ("chunk", 64), ("rnn", 0)):
            tc = measure_causal(w, args.mask, cform, cchunk, 20, 3, flush)
            msc = statistics.mean(tc)
            causal.append({"workload": f"{w.name} B={w.B} H={w.H} L={w.L} d={w.d}", "mask": args.mask,
                           "form": cform, "chunk": cchunk or None, "value": w.B * w.L / (msc * 1e-3),
                           "unit": "tokens/s", "ms_per_call": msc,
                           "path": "lion_attn_fwd_causal (the forward half), fp32 CUDA cores"})

    streaming = None
    if not args.no_streaming:
        ms_s, ms_eager = measure_stream(w.B, w.H, w.d, args.mask, 200, 10)
        sb = stream_bytes(w.B, w.H, w.d)
        streaming = {"workload": f"decode B={w.B} H={w.H} d={w.d}, lion_rnn_step (one direction), "
                                 "200 steps captured in a CUDA graph and replayed, inputs resident",
                     "value": w.B / (ms_s * 1e-3), "unit": "tokens/s", "us_per_step": ms_s * 1e3,
                     "us_per_step_launched_one_by_one": ms_eager * 1e3,
                     "roofline": {"bound": "hbm", "achieved": sb / (ms_s * 1e-3) / 1e9, "peak": hbm_peak,
                                  "unit": "GB/s", "frac": sb / (ms_s * 1e-3) / 1e9 / hbm_peak,
                                  "bytes_per_step": sb,
                                  "note": "the fp32 states (B*H*d*d*4 bytes) stay in the 129 MB L2 between steps"}}

    configs = None
    if not args.no_configs:
        configs = [measure_config(c, flush, hbm_peak) for c in CONFIG_LINES
                   if (c[0], c[1], c[2], c[3]) != (args.workload, args.mask, args.form, args.chunk)]

    cpu = None
    if rank == 0 and ws >= 1 and not args.no_cpu_baseline and ws == 1:
        cpu = cpu_baseline(args.workload, args.mask)
        if secondary is not None:
            # the long workload's baseline: the recurrent-form oracle
            secondary["cpu_baseline"] = cpu_baseline("hires_2496", args.mask if args.mask != "lit" else "s",
                                                     budget_s=5.0)
        for c in configs or []:
            # BERT-large's baseline (the recurrent-form oracle), beside its LION-S chunk-128 line
            if c["workload"].startswith("bert_large ") and c["mask"] == "s" and c.get("chunk") == 128:
                c["cpu_baseline"] = cpu_baseline("bert_large", "s", budget_s=2.0)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_all,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": _config(args, w),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak,
                         "traffic": traffic_bytes(w, args.mask, args.chunk)[0] if args.form == "chunk" else None,
                         "peak_source": peak_src, "algorithmic_bytes": abytes},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps * kernels_per_call(args.form, args.chunk, w, args.mask, _sm_count()),
            "clocks": clocks,
            "wall_s_timed_region": t_wall,
            "secondary": secondary,
            "lra": lra,
            "bf16_out": bf16_out,
            "backward": backward,
            "reordered": reordered,
            "causal": causal,
            "streaming": streaming,
            "configs": configs,
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
