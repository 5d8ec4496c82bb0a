#!/usr/bin/env python
"""Benchmark of the block-sparse attention forward hot path on GB300.

A step is one pass of the whole path over one batch: bsa_build_mask (static
spec evaluation or mean-pooled top-k selection, CSR + bitmap emit) followed by
bsa_forward (tile ordering + the tcgen05 block-sparse FlashAttention kernel). For a
static mask the tile ordering is planned once after the warm-up (bsa_forward_plan),
as the mask itself is pre-generated once.

Reported metric: effective TFLOP/s, counting only active block pairs
(4 * block^2 * d FLOPs per active pair per head), plus ms per forward call and
its fraction of the measured dense bf16 tensor peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Timing: W warm-up steps, a short clock-settling phase, then exactly K timed
steps, each replayed from CUDA graphs and bracketed by CUDA events on the
launching stream; L2 is flushed (256 MB write) before every timed step.
The end-to-end figure copies each step's inputs in from pinned host memory and its
outputs out inside the timed region, overlapped by chunks of heads on three streams.
--impl reference times the CPU oracle (test infrastructure, double precision)
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from block_sparse_attention_mean_gb300 import workloads as wl  # noqa: E402

DEFAULT_WORKLOAD = "long_topk"
FLUSH_BYTES = 256 << 20
FP32_FMA_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12  # CUDA-core fp32 peak of the GB300 (nominal clock)
NOMINAL_BF16_TFLOPS = 2250.0  # GB300 dense bf16 tensor peak, nominal (context beside the measured one)
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "fwd_tc_traffic.txt")
FWD_SOURCE = os.path.join(ROOT, "block_sparse_attention_mean_gb300", "csrc", "fwd_tc.cu")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-chunks", type=int, default=0,
                    help="end-to-end: heads in this many chunks, copy-in / compute / copy-out overlapped "
                         "(0: about 128 MB of copies per chunk)")
    ap.add_argument("--tokens", type=float, default=0.0,
                    help="time the token-sparse forward (bsa_forward_tokens) at this token density instead: "
                         "groups of 128 queries and K = floor(density * N) tokens per group, both seeded random")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--residual", action="store_true",
                    help="time bsa_forward_residual (residual compensation) with R captured at warm-up")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def effective_flops(w, nnz: int) -> float:
    return float(nnz) * 4.0 * w.block * w.block * w.d


def max_over_ranks(x: float, device) -> float:
    """Largest value of x across the ranks of the default process group (x itself
    without one). Every rank replicates the workload, so the slowest rank's time
    is the job's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, world: int, steps: int, total_ms: float) -> float:
    """Whole-job effective TFLOP/s: the work of every rank over the slowest rank's time."""
    return flops_per_step * world * steps / (total_ms * 1e-3) / 1e12


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def traffic_from_profile():
    """dram bytes per forward launch from the committed ncu summary, or None when the
    kernel source changed after that capture."""
    try:
        fields = {}
        with open(PROFILE_TRAFFIC) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        sha = hashlib.sha256(open(FWD_SOURCE, "rb").read()).hexdigest()
        if fields.get("fwd_tc.cu sha256") != sha:
            return None
        return float(fields["dram_bytes_per_launch_scaled"])
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.tmp.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def gpu_index_for(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v for v in vis.split(",") if v.strip()]
    if local_rank < len(ids) and ids[local_rank].strip().isdigit():
        return int(ids[local_rank])
    return local_rank


# ---------------------------------------------------------------- CPU oracle timing


def oracle_head_mask(w, inp, head: int):
    """uint8 [nQB, nKB] block mask of one (b, h) head from the oracle alone."""
    import oracle
    if w.mask == wl.TOPK:
        q = inp["q"].reshape(w.B * w.H, w.N, w.d)[head:head + 1]
        k = inp["k"].reshape(w.B * w.H, w.N, w.d)[head:head + 1]
        return oracle.select_mask(q, k, w.block, w.density)[0]
    if w.mask == wl.BAND:
        return oracle.band_mask(w.nQB, w.n_text_blocks, w.band, w.anchors)
    if w.mask == wl.CUBOID:
        return oracle.cuboid_mask(w.n_text_blocks, w.grid)
    return inp["mask"].reshape(w.B * w.H, w.nQB, w.nKB)[head]


def oracle_nnz(w, inp) -> int:
    """Active block pairs of the whole workload, counted on the oracle's masks of every head."""
    return int(sum(int(oracle_head_mask(w, inp, h).sum()) for h in range(w.B * w.H)))


def time_oracle(w, inp, budget_s: float, seed: int = 0):
    """Time the oracle on one head and extrapolate to the workload.

    One seeded (b, h) head is timed: its mask (the oracle's selector or static
    evaluator) and its attention, on all of its query rows when that fits about
    `budget_s` seconds, else on a seeded sample of them scaled linearly to all rows.
    The head's time is then scaled by B*H (every head does the same work).
    Returns (seconds for the full workload, sample description, cores)."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(seed)
    BH = w.B * w.H
    h = int(rng.integers(BH))
    q = inp["q"].reshape(BH, w.N, w.d)[h:h + 1]
    k = inp["k"].reshape(BH, w.N, w.d)[h:h + 1]
    v = inp["v"].reshape(BH, w.N, w.d)[h:h + 1]
    t0 = time.perf_counter()
    mask = oracle_head_mask(w, inp, h)[None]
    t_mask = time.perf_counter() - t0
    probe = np.sort(rng.choice(w.N, size=min(256, w.N), replace=False))
    t0 = time.perf_counter()
    oracle.attention(q, k, v, mask, w.block, rows=probe)
    per_row = (time.perf_counter() - t0) / probe.size
    n = int(min(w.N, max(probe.size, budget_s / max(per_row, 1e-9))))
    rows = np.sort(rng.choice(w.N, size=n, replace=False)) if n < w.N else np.arange(w.N, dtype=np.int64)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, mask, w.block, rows=rows)
    t_rows = time.perf_counter() - t0
    head_s = t_mask + t_rows * w.N / n
    cores = os.cpu_count() or 1
    sample = (f"extrapolated: one head (b*H+h = {h}) timed, its mask plus attention on {n} of its {w.N} "
              f"query rows (seeded{', scaled linearly to all rows' if n < w.N else ''}), then x{BH} heads; "
              f"OpenMP over rows on {cores} cores")
    return head_s * BH, sample, cores


# ---------------------------------------------------------------- our arm


def run_ours(args, world, rank, local):
    import torch
    import torch.distributed as dist

    from block_sparse_attention_mean_gb300 import binding as bb
    from block_sparse_attention_mean_gb300 import build as bbuild

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    bbuild.build()
    bb.load()
    w = wl.WORKLOADS[args.workload]
    inp = wl.make_inputs(w)
    dev = torch.device("cuda", local)

    def upload(name):
        if w.dtype == "bf16":
            return torch.from_numpy(inp[name + "_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(inp[name]).to(dev)

    q, k, v = upload("q"), upload("k"), upload("v")
    dt = bb.BF16 if w.dtype == "bf16" else bb.FP32
    B, H, N, d, bs = w.B, w.H, w.N, w.d, w.block
    nB = N // bs
    W = (nB + 31) // 32
    spec = None
    mask_dev = None
    if w.mask == wl.BAND:
        spec = bb.band_spec(w.n_text_blocks, w.band, list(w.anchors))
    elif w.mask == wl.CUBOID:
        spec = bb.cuboid_spec(w.n_text_blocks, w.grid)
    elif w.mask == wl.EXPLICIT:
        mask_dev = torch.from_numpy(wl.pack_bitmap_words(inp["mask"]).reshape(-1)).to(dev)
        spec = bb.explicit_spec(mask_dev)
    cap = bb.bsa_mask_nnz(B, H, N, bs, w.density, spec)
    row_ptr = torch.empty(B * H * nB + 1, dtype=torch.int32, device=dev)
    col_idx = torch.empty(cap, dtype=torch.int32, device=dev)
    bitmap = torch.empty(B * H * nB * W, dtype=torch.int32, device=dev)
    ws_m = bb.workspace(0, B, H, N, d, bs, dev)
    ws_f = bb.workspace(1, B, H, N, d, bs, dev)
    O = torch.empty_like(q)
    LSE = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    qk_in = (None, None) if spec is not None else (q, k)

    def build_call(s):
        bb.bsa_build_mask(qk_in[0], qk_in[1], dt, B, H, N, d, bs, w.density, spec, row_ptr, col_idx, cap,
                          bitmap, ws_m, ws_m.numel(), s)

    R = None
    if args.residual:
        # anchor step, outside the timed region: dense output (every block active) and sparse
        # output of this workload, R = O_dense - O_sparse
        ones = np.ones((B, H, nB, nB), dtype=np.uint8)
        full_dev = torch.from_numpy(wl.pack_bitmap_words(ones).reshape(-1)).to(dev)
        full_spec = bb.explicit_spec(full_dev)
        cap_full = bb.bsa_mask_nnz(B, H, N, bs, 0.0, full_spec)
        rp_f = torch.empty(B * H * nB + 1, dtype=torch.int32, device=dev)
        ci_f = torch.empty(cap_full, dtype=torch.int32, device=dev)
        bm_f = torch.empty(B * H * nB * W, dtype=torch.int32, device=dev)
        bb.bsa_build_mask(None, None, dt, B, H, N, d, bs, 0.0, full_spec, rp_f, ci_f, cap_full, bm_f, ws_m,
                          ws_m.numel(), None)
        O_dense = torch.empty_like(q)
        bb.bsa_forward(q, k, v, dt, B, H, N, d, bs, rp_f, ci_f, bm_f, 0, 0.0, O_dense, LSE, ws_f, ws_f.numel(), None)
        bb.bsa_build_mask(qk_in[0], qk_in[1], dt, B, H, N, d, bs, w.density, spec, row_ptr, col_idx, cap,
                          bitmap, ws_m, ws_m.numel(), None)
        bb.bsa_forward(q, k, v, dt, B, H, N, d, bs, row_ptr, col_idx, bitmap, w.index_mode, 0.0, O, LSE, ws_f,
                       ws_f.numel(), None)
        R = bb.residual_capture(O_dense, O)
        torch.cuda.synchronize()
        del O_dense, rp_f, ci_f, bm_f, full_dev

    # a static mask is pre-generated once ([P1] section 5.3), and so is the forward's work list
    # over it (bsa_forward_plan, after the warm-up): the timed forwards reuse it
    planned = spec is not None and dt == bb.BF16
    fwd_mode = [w.index_mode]

    def fwd_call(s):
        if R is None:
            bb.bsa_forward(q, k, v, dt, B, H, N, d, bs, row_ptr, col_idx, bitmap, fwd_mode[0], 0.0, O, LSE, ws_f,
                           ws_f.numel(), s)
        else:
            bb.bsa_forward_residual(q, k, v, dt, B, H, N, d, bs, row_ptr, col_idx, bitmap, fwd_mode[0], 0.0, R, O,
                                    LSE, ws_f, ws_f.numel(), s)

    # kernels of one step: the build (pooling, scoring, selection for a dynamic mask; pattern and
    # copy for a shared static pattern; rows, scan and emit for a per-head bitmap), then the
    # forward (work list or plan gate, and the forward kernel; one CUDA-core kernel for fp32)
    if spec is None:
        build_launches = 3
    elif spec.kind != bb.STATIC_EXPLICIT or spec.broadcast_bh:
        build_launches = 2
    else:
        build_launches = 3
    launches_per_step = build_launches + (1 if dt == bb.FP32 else 2)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            build_call(stream)
            fwd_call(stream)
        if planned:
            bb.bsa_forward_plan(dt, B, H, N, d, bs, row_ptr, col_idx, bitmap, w.index_mode, ws_f, ws_f.numel(),
                                stream)
            fwd_mode[0] = w.index_mode | bb.INDEX_PLANNED
            fwd_call(stream)
    for ws in (ws_m, ws_f):
        code = bb.bsa_check_device_error(ws, stream)
        if code != 0:
            raise bb.BsaError(code, "warm-up")
    nnz = int(row_ptr[-1].item())
    if not torch.isfinite(LSE[LSE > -float("inf")]).all():
        raise RuntimeError("non-finite LSE after warm-up")

    # CUDA graphs of the two calls (falls back to eager launches if capture fails)
    graphs = None
    try:
        g_build, g_fwd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_build, stream=stream):
            build_call(torch.cuda.current_stream())
        with torch.cuda.graph(g_fwd, stream=stream):
            fwd_call(torch.cuda.current_stream())
        graphs = (g_build, g_fwd)
    except Exception as exc:  # noqa: BLE001
        print(f"# graph capture failed ({exc}); timing eager launches", file=sys.stderr)

    def step():
        if graphs:
            graphs[0].replay()
            graphs[1].replay()
        else:
            build_call(stream)
            fwd_call(stream)

    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sampler = ClockSampler(gpu_index_for(local))
    sampler.start()
    with torch.cuda.stream(stream):
        t_end = time.perf_counter() + 1.5  # let clocks settle under load
        while time.perf_counter() < t_end:
            for _ in range(20):
                flush.zero_()
                step()
            stream.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            if graphs:
                graphs[0].replay()
                ev[i][1].record(stream)
                graphs[1].replay()
            else:
                build_call(stream)
                ev[i][1].record(stream)
                fwd_call(stream)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        if world > 1:
            dist.barrier()
    clocks = sampler.stop()
    code = bb.bsa_check_device_error(ws_f, stream) or bb.bsa_check_device_error(ws_m, stream)
    if code != 0:
        raise bb.BsaError(code, "timed steps")
    step_ms = [e[0].elapsed_time(e[2]) for e in ev]
    fwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
    build_ms = [e[0].elapsed_time(e[1]) for e in ev]
    total_ms = max_over_ranks(sum(step_ms), dev)
    flops = effective_flops(w, nnz)
    ms_per_step = total_ms / args.steps
    value = job_throughput(flops, world, args.steps, total_ms)

    # end to end through the C ABI from pinned host buffers. Heads are independent, so the step
    # runs in chunks of heads on three streams: chunk c + 1 is copied in while chunk c is
    # computed (mask build + forward, the same calls on the chunk's heads) and chunk c - 1 is
    # copied out. Copies in and out share the host link (about 210 GB/s each way on this machine).
    e2e = None
    if args.e2e_steps > 0:
        BHt = B * H
        moved = sum(t.numel() * t.element_size() for t in (q, k, v, O, LSE))
        # about 128 MB per chunk (more chunks cost more than they overlap on small steps: dynamic_topk
        # in 4 chunks took 1.39 ms against 1.20 ms in one)
        C = args.e2e_chunks if args.e2e_chunks > 0 else max(1, moved // (128 << 20))
        while C > 1 and BHt % C != 0:
            C -= 1  # whole heads per chunk
        if spec is not None and spec.kind == bb.STATIC_EXPLICIT:
            C = 1  # a per-head explicit bitmap is not split by head here
        hc = BHt // C
        # chunks of hc heads; without a shared plan the last chunk is split into single heads, so
        # that the compute and copy-out left after the last copy-in are one head's
        spans = [(c * hc, (c + 1) * hc) for c in range(C)]
        if not planned and C > 1 and hc > 1:
            spans = spans[:-1] + [(h, h + 1) for h in range((C - 1) * hc, C * hc)]
        hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
        hO = torch.empty(O.shape, dtype=O.dtype).pin_memory()
        hL = torch.empty(LSE.shape, dtype=LSE.dtype).pin_memory()
        flat = lambda t: t.reshape(BHt, N, -1) if t.dim() == 4 else t.reshape(BHt, N)  # noqa: E731
        dq, dk, dv, dO, dL = flat(q), flat(k), flat(v), flat(O), flat(LSE)
        sq, sk, sv, sO, sL = flat(hq), flat(hk), flat(hv), flat(hO), flat(hL)
        cap_c = bb.bsa_mask_nnz(1, hc, N, bs, w.density, spec)
        rp_c = torch.empty(hc * nB + 1, dtype=torch.int32, device=dev)
        ci_c = torch.empty(max(cap_c, 1), dtype=torch.int32, device=dev)
        bm_c = torch.empty(hc * nB * W, dtype=torch.int32, device=dev)
        wsm_c = bb.workspace(0, 1, hc, N, d, bs, dev)
        wsf_c = bb.workspace(1, 1, hc, N, d, bs, dev)
        s_in, s_cmp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
        mode_c = w.index_mode
        if planned:  # a static mask is the same for every head: one plan serves every chunk
            bb.bsa_build_mask(None, None, dt, 1, hc, N, d, bs, w.density, spec, rp_c, ci_c, cap_c, bm_c, wsm_c,
                              wsm_c.numel(), s_cmp)
            bb.bsa_forward_plan(dt, 1, hc, N, d, bs, rp_c, ci_c, bm_c, w.index_mode, wsf_c, wsf_c.numel(), s_cmp)
            mode_c |= bb.INDEX_PLANNED

        def chunk_compute(h0, h1, st):
            sl, nh = slice(h0, h1), h1 - h0
            qc, kc, vc = dq[sl], dk[sl], dv[sl]
            bb.bsa_build_mask(None if spec is not None else qc, None if spec is not None else kc, dt, 1, nh, N, d,
                              bs, w.density, spec, rp_c, ci_c, cap_c, bm_c, wsm_c, wsm_c.numel(), st)
            if R is None:
                bb.bsa_forward(qc, kc, vc, dt, 1, nh, N, d, bs, rp_c, ci_c, bm_c, mode_c, 0.0, dO[sl], dL[sl],
                               wsf_c, wsf_c.numel(), st)
            else:
                bb.bsa_forward_residual(qc, kc, vc, dt, 1, nh, N, d, bs, rp_c, ci_c, bm_c, mode_c, 0.0,
                                        R.reshape(BHt, N, d)[sl], dO[sl], dL[sl], wsf_c, wsf_c.numel(), st)

        e2e_ms = []
        for i in range(args.e2e_steps + 2):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_in)
            for h0, h1 in spans:
                sl = slice(h0, h1)
                with torch.cuda.stream(s_in):
                    dq[sl].copy_(sq[sl], non_blocking=True)
                    dk[sl].copy_(sk[sl], non_blocking=True)
                    dv[sl].copy_(sv[sl], non_blocking=True)
                    ev_in = torch.cuda.Event()
                    ev_in.record(s_in)
                s_cmp.wait_event(ev_in)
                chunk_compute(h0, h1, s_cmp)
                ev_c = torch.cuda.Event()
                ev_c.record(s_cmp)
                s_out.wait_event(ev_c)
                with torch.cuda.stream(s_out):
                    sO[sl].copy_(dO[sl], non_blocking=True)
                    sL[sl].copy_(dL[sl], non_blocking=True)
            e1.record(s_out)
            e1.synchronize()
            if i >= 2:
                e2e_ms.append(e0.elapsed_time(e1))
        for ws in (wsm_c, wsf_c):
            code = bb.bsa_check_device_error(ws, s_cmp)
            if code != 0:
                raise bb.BsaError(code, "end-to-end steps")
        # heads are independent, so the chunked calls give the unchunked step's outputs: bit for bit
        # when no query tile is split, else to rounding (a chunk of fewer heads can split its longest
        # tiles differently, and split tiles merge their partial sums in another order)
        torch.cuda.synchronize()
        build_call(stream)
        fwd_call(stream)
        torch.cuda.synchronize()
        O_ref, L_ref = O.cpu(), LSE.cpu()
        e2e_exact = torch.equal(hO, O_ref) and torch.equal(hL, L_ref)
        if not e2e_exact:
            o_err = (hO.float() - O_ref.float()).abs().max().item()
            fin = torch.isfinite(L_ref)
            l_err = (hL[fin] - L_ref[fin]).abs().max().item() if fin.any() else 0.0
            if not (o_err <= 2e-2 and l_err <= 1e-3 and torch.equal(torch.isfinite(hL), fin)):
                raise RuntimeError(f"end-to-end outputs differ from the unchunked step's (O {o_err}, LSE {l_err})")
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
        d2h = hO.numel() * hO.element_size() + hL.numel() * hL.element_size()
        e2e_mean = max_over_ranks(sum(e2e_ms) / len(e2e_ms), dev)
        e2e = {"value": round(job_throughput(flops, world, 1, e2e_mean), 3), "unit": "TFLOP/s",
               "ms_per_step": round(e2e_mean, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "pipeline": f"{len(spans)} chunks of {'/'.join(str(b - a) for a, b in spans)} heads: copy-in, mask build + "
                           "forward, copy-out on three streams",
               "outputs": "equal to the unchunked step's" if e2e_exact else "within rounding of the unchunked step's"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peaks, peak_kind = measured_peaks()
    fwd_mean = sum(fwd_ms) / len(fwd_ms)
    achieved = flops / (fwd_mean * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        full_s, sample, cores = time_oracle(w, inp, budget_s=10.0)
        cpu = {"value": round(flops / full_s / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": sample, "ms_per_call_extrapolated": round(full_s * 1e3, 1)}
    line = {
        "metric": "block-sparse attn fwd effective TFLOP/s (active blocks only, 4*bs^2*d per pair)",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded generator; no dataset or weights)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "block": w.block,
                   "mask": w.mask, "density": w.density if w.mask == wl.TOPK else None,
                   "active_block_pairs": nnz, "block_density": round(nnz / (w.B * w.H * nB * nB), 5),
                   "index_mode": "bitmap" if w.index_mode else "csr",
                   "l2": "flushed (256 MB write) before every timed step", "cuda_graphs": bool(graphs),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "residual": "O_sparse + R (R captured at warm-up)" if R is not None else None,
                   "work_list": "planned once with the static mask (bsa_forward_plan)" if planned
                   else "built in every forward call"},
        "fwd_ms_per_call": round(fwd_mean, 5), "build_mask_ms": round(sum(build_ms) / len(build_ms), 5),
        "fwd_tflops": round(achieved, 2), "pct_of_bf16_peak": round(100 * achieved / peak, 2),
        "pct_of_nominal_bf16_peak": round(100 * achieved / NOMINAL_BF16_TFLOPS, 2),
        "wall_s_timed_loop": round(wall, 4),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic_from_profile() if R is None else None,
                     "kernel": "fwd_tc_kernel" + ("" if planned else " (+ tile_order_kernel in the same bracket)"),
                     "peak_source": f"{peak_kind} bf16_tflops (burst); the target of 60% is read against it",
                     "nominal_peak": NOMINAL_BF16_TFLOPS,
                     "frac_of_nominal": round(achieved / NOMINAL_BF16_TFLOPS, 4)},
        "e2e": e2e, "gpu_launches": launches_per_step * args.steps, "clocks": clocks, "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------- reference arm (CPU oracle)


def run_reference(args, world, rank):
    if rank != 0:
        return
    w = wl.WORKLOADS[args.workload]
    inp = wl.make_inputs(w)
    nnz = oracle_nnz(w, inp)  # the oracle's own masks, every head
    flops = effective_flops(w, nnz)
    for i in range(max(args.warmup, 0)):
        time_oracle(w, inp, budget_s=0.5, seed=i)
    totals = []
    sample = cores = None
    for i in range(args.steps):
        full_s, sample, cores = time_oracle(w, inp, budget_s=1.0, seed=100 + i)
        totals.append(full_s)
    ms = 1e3 * sum(totals) / len(totals)
    value = flops / (ms * 1e-3) / 1e12
    line = {"impl": "reference",
            "metric": "block-sparse attn fwd effective TFLOP/s (active blocks only, 4*bs^2*d per pair)",
            "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator)",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "block": w.block,
                       "active_block_pairs": nnz},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_tokens(args):
    """Token-sparse forward on one GPU: the workload's Q, K, V, seeded random query groups and
    token sets (the timing does not depend on which tokens are chosen), L2 flushed before every
    call, CUDA events on the launching stream."""
    import torch

    from block_sparse_attention_mean_gb300 import binding as bb
    from block_sparse_attention_mean_gb300 import build as bbuild

    bbuild.build()
    bb.load()
    w = wl.WORKLOADS[args.workload]
    inp = wl.make_inputs(w)
    dev = torch.device("cuda", 0)
    up = (lambda n: torch.from_numpy(inp[n + "_bits"].view(np.int16)).to(dev).view(torch.bfloat16)) \
        if w.dtype == "bf16" else (lambda n: torch.from_numpy(inp[n]).to(dev))
    q, k, v = up("q"), up("k"), up("v")
    BH, N, d, C = w.B * w.H, w.N, w.d, 128
    K = max(1, int(np.floor(args.tokens * N)))
    rng = np.random.default_rng(w.seed)
    perm = torch.from_numpy(np.stack([rng.permutation(N) for _ in range(BH)]).astype(np.int32)).to(dev)
    toks = torch.from_numpy(np.stack([np.sort(rng.choice(N, size=(K,), replace=False))
                                      for _ in range(BH * (N // C))]).reshape(BH, N // C, K).astype(np.int32)).to(dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    O = torch.empty_like(q)
    L = torch.empty((w.B, w.H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def call():
        bb.bsa_forward_tokens(q, k, v, bb.BF16 if w.dtype == "bf16" else bb.FP32, w.B, w.H, N, d, perm, toks, K,
                              0.0, O, L, ws, ws.numel(), stream)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            call()
        code = bb.bsa_check_device_error(ws, stream)
        if code != 0:
            raise bb.BsaError(code, "token forward warm-up")
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    flops = 4.0 * BH * N * K * d  # every query row against its group's K tokens

    # the anchor-step stages of the token path, once each after a warm-up: the query groups
    # and the exact token selection (with the dense LSE of a full-index forward)
    def timed(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            fn()
            torch.cuda.synchronize()
            flush.zero_()
            e0.record(stream)
            out = fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return out, e0.elapsed_time(e1)

    gperm, group_ms = timed(lambda: bb.query_groups(q, stream=stream))
    # the dense logsumexp (every block active) by the LSE-only forward; the block size of an
    # all-active index does not change the result, and 128-key steps run the QK^T MMAs at N = 128
    nb = -(-N // 128)
    ones = np.ones((w.B, w.H, nb, nb), dtype=np.uint8)
    full = bb.build_mask(None, None, 128, spec=bb.explicit_spec(
        torch.from_numpy(wl.pack_bitmap_words(ones).reshape(-1)).to(dev)), shape=(w.B, w.H, N, d))
    lse, lse_ms = timed(lambda: bb.forward_lse(q, k, full, stream=stream))
    del full
    _, select_ms = timed(lambda: bb.select_tokens(q, k, gperm, lse, args.tokens, stream=stream))
    tflops = flops / (ms * 1e-3) / 1e12
    peaks, peak_kind = measured_peaks()
    line = {"metric": "token-sparse attn fwd effective TFLOP/s (4*K*d per query row)", "value": round(tflops, 3),
            "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "dtype": "bf16" if w.dtype == "bf16" else "f32",
            "data": "synthetic (seeded Q, K, V; seeded random groups and token sets)",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": N, "d": d, "group": C, "tokens_per_group": K,
                       "l2": "flushed (256 MB write) before every timed call"},
            "anchor_step_ms": {"query_groups": round(group_ms, 3), "dense_lse": round(lse_ms, 3),
                               "select_tokens": round(select_ms, 3)},
            "roofline": ({"bound": "tensor", "achieved": round(tflops, 3), "peak": float(peaks["bf16_tflops"]),
                          "unit": "TFLOP/s", "frac": round(tflops / float(peaks["bf16_tflops"]), 4),
                          "kernel": "fwd_tc_kernel in token mode (Q rows by TMA gather, K and V rows by cp.async)",
                          "peak_source": f"{peak_kind} bf16_tflops (burst)"} if w.dtype == "bf16" else
                         # fp32 inputs run on CUDA cores: bounded by the fp32 FMA pipe
                         {"bound": "alu", "achieved": round(tflops, 3), "peak": FP32_FMA_TFLOPS,
                          "unit": "TFLOP/s", "frac": round(tflops / FP32_FMA_TFLOPS, 4),
                          "kernel": "fwd_tokens_kernel (CUDA cores)",
                          "peak_source": "derived: 152 SMs x 128 fp32 FMA lanes x 2 FLOP x 2.07 GHz"})}
    print(json.dumps(line))


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.tokens > 0.0:
        run_tokens(args)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
