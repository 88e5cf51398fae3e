"""Benchmark of the causal linear-attention hot path on GB300.

One step = one pass of every hot-path row on synthetic inputs resident in
HBM.  The headline line (``value``) is the BASED Taylor prefill,
B=8, H=16, N=4096, d'=16, d_v=64, bf16 in / fp32 state, in tokens/s (B*N per
step).  The same run also times, under ``paths``:
  based_prefill_decay  the headline workload with a fixed per-head decay
  taylor_fp32_small    Taylor linear attention fp32, B=1, H=2, N=256 (latency)
  gdn_prefill       Gated DeltaNet prefill B=4, H=16, N=16384, d=128
  gdn_prefill_long  Gated DeltaNet prefill B=1, H=16, N=1,048,576, d=128
  gated_prefill     scalar-gate (A_t = alpha_t I) prefill on the gdn_prefill inputs
  decode_gdn        1000 decode steps, 256 seqs x 16 heads, 128x128 state
  decode_taylor     1000 decode steps, 256 seqs x 16 heads, 273x64 state + z
  decode_swa        1000 sliding-window softmax decode steps, 256 seqs x 16 heads, window 64
  notebank_write    NoteBank write side: scores of 192 channels (d_k 256) over 16K tokens + note addresses
  notebank_route    NoteBank routing of one 64-token question over 4092 notes x 192 channels
each with its own rate and roofline.

Timing: W untimed warm-up steps, then K steps; each launch is bracketed by
CUDA events on its own stream and an L2 flush (a 512 MiB write, outside the
events) separates timed steps.  Multi-GPU (torchrun): each rank runs its own
copy of the workload (weak scaling, no collective on the data path); the
per-rank times are max-reduced.  ``--impl reference`` times the fp64 CPU
oracle (the only reference there is for this method) on the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synthetic  # noqa: E402

L2_FLUSH_BYTES = 512 << 20
HEADLINE = "based_prefill"
METRIC = "prefill & decode tokens/s on 1 GB300; % of tensor-core / HBM roofline (ncu)"

# Algorithmic HBM bytes per token-head (inputs read once, outputs written once):
#  Taylor prefill  q,k (2*16*2 B) + v (64*2 B) + y (64*2 B)                    = 320 B
#  GDN prefill     q,k,v (3*128*2 B) + o (128*2 B) + alpha,beta (2*4 B)        = 1032 B
#  GDN decode      state read+write 2*128*128*4 + q,k,v,o 4*128*2 + alpha,beta = 132,104 B
#  Taylor decode   (s,z) read+write 2*(273*64+273)*4 + q,k 2*16*2 + v,y 2*64*2  = 142,248 B
# plus, for prefill, the final fp32 state written once per (b,h).
BYTES_PER_TOKEN_HEAD = {"taylor_prefill": 320, "gdn_prefill": 1032,
                        "gdn_decode": 2 * 128 * 128 * 4 + 4 * 128 * 2 + 8,
                        "taylor_decode": 2 * (273 * 64 + 273) * 4 + 2 * 16 * 2 + 2 * 64 * 2,
                        # window 64, d 64, bf16: the full window's keys and values read, the new
                        # token's k, v written into the ring, q, k, v read, o written
                        "swa_decode": 2 * 64 * 64 * 2 + 2 * 64 * 2 + 3 * 64 * 2 + 64 * 2}
SWA_WINDOW, SWA_D = 64, 64
# fp32 FMA rate of the CUDA cores (no tensor cores): 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz (the maximum SM
# clock); the peak the routing kernel's cosines are measured against
FP32_ALU_TFLOPS = round(152 * 128 * 2 * 2.07e9 / 1e12, 1)
STATE_BYTES = {"taylor": (273 * 64 + 273) * 4, "gdn": 128 * 128 * 4}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def _code_only(text):
    """C++/CUDA source without comments or trailing blanks: what a compiler sees, so that a change of a
    comment does not count as a change of the kernel (no kernel here has "//" or "/*" in a literal)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_sources_sha(files):
    """Hash of the code (comments left out) of a kernel's source files."""
    h = hashlib.sha256()
    for f in files:
        path = os.path.join(ROOT, "linear_attention_recurrence_chunked_gb300", "csrc", f)
        h.update(_code_only(open(path, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


# Dense contractions per chunk and head that the chunked form of each method needs (multiply-adds x 2),
# the "intra-chunk GEMM" work the tensor cores run:
#  GDN (C = 64, d_k = d_v = 128): [K;Q] K^T, W = T diag(beta gamma) K, U~ = T diag(beta) V, P U (5 of
#      2*64*64*128) and W S0^T, Q S0^T, the state update U^T K (3 of 2*64*128*128); the triangular inverse
#      T (its two 64-level products run as tf32 MMAs, the rest on the CUDA cores) is not counted.
#  scalar gate (same chunk): Q K^T, P (beta V) and Q S0^T, the update (no W, no U~, no inverse).
#  BASED (C = 128, d' = 16, the 153-wide compact feature basis, d_v = 64 plus the normaliser column):
#      Q K^T 2*128*128*16, readout phi(Q) [S | z] 2*128*153*65, intra-chunk P [V | 1] 2*128*128*65,
#      update phi(K)^T [V | 1] 2*153*128*65.
_SMALL, _BIG = 2 * 64 * 64 * 128, 2 * 64 * 128 * 128
GDN_CHUNK_FLOPS = {"gdn": 5 * _SMALL + 3 * _BIG, "gated": 2 * _SMALL + 2 * _BIG}
TAYLOR_CHUNK_FLOPS = 2 * 128 * 128 * 16 + 2 * 128 * 153 * 65 + 2 * 128 * 128 * 65 + 2 * 153 * 128 * 65


def ncu_entry(key):
    """The committed ncu summary of a kernel, if its sources are unchanged since it was taken; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(key)
    if not d or d.get("source_sha") != kernel_sources_sha(d.get("sources", [])):
        return None
    return d


def tensor_fraction(flops_per_launch, ms_per_launch, pk, key):
    """Intra-chunk GEMM FLOPs per launch / event time, against the measured sustained dense bf16 rate; the
    tensor-pipe activity ncu measured for the same kernel (percent of elapsed cycles) beside it."""
    ach = flops_per_launch / (ms_per_launch * 1e-3) / 1e12
    peak = pk.get("bf16_tflops_sustained") or pk["bf16_tflops"]
    e = ncu_entry(key) or {}
    return {"bound": "tensor", "flops_per_launch": int(flops_per_launch), "achieved": round(ach, 1),
            "peak": peak, "unit": "TFLOP/s", "frac": round(ach / peak, 4),
            "ncu_tensor_pipe_pct": e.get("tensor_pipe_pct")}


def ncu_traffic(key):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    sources are unchanged since it was taken; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(key)
    if not d:
        return None
    if d.get("source_sha") != kernel_sources_sha(d.get("sources", [])):
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during timing."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[4:8]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        loaded = [x for x in sm if x > 0.5 * (max(sm) if sm else 0)]
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm


class Timer:
    """Per-launch CUDA-event timing on one stream, L2 flushed between launches."""

    def __init__(self, stream, flush_buf):
        self.stream = stream
        self.flush_buf = flush_buf
        self.events = []

    def run(self, fn, flush=True):
        with torch.cuda.stream(self.stream):
            if flush:
                self.flush_buf.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(self.stream)
            fn()
            b.record(self.stream)
        self.events.append((a, b))

    def total_ms(self):
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in self.events)

    def reset(self):
        self.events = []


def rank_seed_offset(rank: int) -> int:
    """Each rank runs its own replica of the workload on its own seeded inputs
    (independent problems: weak scaling, no collective on the data path)."""
    return 1000 * int(rank)


def max_over_ranks(x: float, ws: int) -> float:
    """Slowest rank's time (the job is done when the last replica is)."""
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, ws: int, max_seconds: float) -> float:
    """Units all ranks processed divided by the slowest rank's time."""
    return ws * units_per_rank / max_seconds


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def roofline(bytes_per_launch, ms_per_launch, peak_gbs, traffic):
    ach = bytes_per_launch / (ms_per_launch * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": peak_gbs, "unit": "GB/s",
            "frac": round(ach / peak_gbs, 4), "traffic": traffic,
            "algorithmic_bytes": int(bytes_per_launch)}


def gpu_arm(args, ws, rank, local):
    import linear_attention_recurrence_chunked_gb300 as la
    from linear_attention_recurrence_chunked_gb300 import _build

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _build.build()
    la.load_library()
    pk = peaks()
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    seed_off = rank_seed_offset(rank)
    launches = 0

    # --- headline: BASED prefill --------------------------------------------
    w = synthetic.WORKLOADS[HEADLINE]
    x = synthetic.workload_inputs(HEADLINE, device=dev, seed=w.seed + seed_off)
    q, k, v = x["q"], x["k"], x["v"]
    y = torch.empty((w.B, w.H, w.N, 64), dtype=torch.bfloat16, device=dev)
    s = torch.empty((w.B, w.H, la.TAYLOR_D, 64), dtype=torch.float32, device=dev)
    z = torch.empty((w.B, w.H, la.TAYLOR_D), dtype=torch.float32, device=dev)

    def based_step():
        la.la_based_prefill(q, k, v, y=y, s_out=s, z_out=z, stream=stream)

    timer = Timer(stream, flush)
    for _ in range(args.warmup):
        timer.run(based_step)
    timer.reset()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(ws)
    for _ in range(args.steps):
        timer.run(based_step)
    ms_total = timer.total_ms()
    barrier(ws)
    launches += args.steps * KERNELS_PER_CALL["based_prefill"]
    ms_total = max_over_ranks(ms_total, ws)
    ms_step = ms_total / args.steps
    tokens = w.B * w.N
    value = whole_job_rate(tokens * args.steps, ws, ms_total * 1e-3)
    bytes_launch = BYTES_PER_TOKEN_HEAD["taylor_prefill"] * w.B * w.H * w.N + STATE_BYTES["taylor"] * w.B * w.H
    roof = roofline(bytes_launch, ms_step, pk["hbm_gbs"], ncu_traffic("taylor_prefill"))
    roof["peak_source"] = pk["source"]
    tensor = tensor_fraction(TAYLOR_CHUNK_FLOPS * w.B * w.H * ((w.N + 127) // 128), ms_step, pk, "taylor_prefill")

    # --- e2e through the C ABI with host buffers ----------------------------
    # Every step copies its inputs in from pinned host memory and its results (y and the final state)
    # back out.  Steps are pipelined over two device buffer sets, as a serving loop would run them:
    # step i's inputs go in on one copy stream while step i-1 computes and step i-2's results go out
    # on the other; the whole K-step region is timed, L2 still flushed before each kernel.  (More
    # copy streams per direction do not help: the host link, ~160 GB/s per direction here, is the
    # limit.)
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    hy, hs, hz = (torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (y, s, z))
    bufs = [(q, k, v, y, s, z), tuple(torch.empty_like(t) for t in (q, k, v, y, s, z))]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_run(n):
        ev_comp, ev_out = [None, None], [None, None]
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for i in range(n):
            bq, bk, bv, by, bs, bz = bufs[i % 2]
            with torch.cuda.stream(s_in):
                if ev_comp[i % 2] is not None:
                    s_in.wait_event(ev_comp[i % 2])  # step i-2's kernel has read this set's inputs
                bq.copy_(hq, non_blocking=True)
                bk.copy_(hk, non_blocking=True)
                bv.copy_(hv, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            with torch.cuda.stream(stream):
                stream.wait_event(ev_in)
                if ev_out[i % 2] is not None:
                    stream.wait_event(ev_out[i % 2])  # step i-2's results are out of this set
                flush.zero_()
                la.la_based_prefill(bq, bk, bv, y=by, s_out=bs, z_out=bz, stream=stream)
                ev_comp[i % 2] = torch.cuda.Event()
                ev_comp[i % 2].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i % 2])
                hy.copy_(by, non_blocking=True)
                hs.copy_(bs, non_blocking=True)
                hz.copy_(bz, non_blocking=True)
                ev_out[i % 2] = torch.cuda.Event()
                ev_out[i % 2].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        stop.record(stream)
        return start, stop

    e2e_run(args.warmup)
    torch.cuda.synchronize()
    barrier(ws)
    start, stop = e2e_run(args.steps)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(start.elapsed_time(stop), ws)
    barrier(ws)
    launches += args.steps * KERNELS_PER_CALL["based_prefill"]
    e2e = {"value": whole_job_rate(tokens * args.steps, ws, e2e_ms * 1e-3), "unit": "tokens/s",
           "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in (hq, hk, hv))),
           "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in (hy, hs, hz)))}
    del hq, hk, hv, hy, hs, hz

    paths = {}
    if not args.headline_only:
        paths, extra_launches = other_paths(args, la, dev, stream, flush, pk, seed_off, ws)
        launches += extra_launches
    clk = clocks.stop()

    line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.description, "B": w.B, "H": w.H, "N": w.N, "d_feat": 16, "d_v": 64,
                       "tokens_per_step": tokens, "seed": w.seed, "l2": "flushed between timed steps (512 MiB write)",
                       "parallelism": f"replicas{ws}" if ws > 1 else "single"},
            "roofline": roof, "tensor": tensor, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
            "paths": paths}
    return line


KERNELS_PER_CALL = {"based_prefill": 1, "gdn_prefill": 2, "decode": 1}


PATH_NAMES = ("based_prefill_decay", "taylor_fp32_small", "gdn_prefill", "gdn_prefill_long", "gated_prefill", "decode_gdn", "decode_taylor",
              "decode_swa", "notebank_write", "notebank_route")

# NoteBank sizes (NoteBank App. C: GDN backbone with J = 192 layer-head channels of d_k = 256, write chunks of
# 512 tokens, 16-dimensional addresses, about 4092 stored notes; the question length is a synthetic choice)
NB_L, NB_H, NB_D, NB_N, NB_CHUNK, NB_WINDOW = 24, 8, 256, 16384, 512, 48
NB_NOTES, NB_NOTE_LEN, NB_Q, NB_R = 4092, 64, 64, 2


def decay_rates(H):
    """Fixed per-head retention for the decayed BASED path: lambda_h = 1 - 2^-(5 + h mod 8), a spread from a
    32-token to a 4096-token memory (the pages give no values)."""
    return torch.tensor([1.0 - 2.0 ** -(5 + h % 8) for h in range(H)], dtype=torch.float32)


def other_paths(args, la, dev, stream, flush, pk, seed_off, ws, only=None):
    out = {}
    launches = 0
    steps = max(1, args.steps)
    if only is None or only == "based_prefill_decay":
        # the headline workload with a fixed per-head decay (a separate instantiation of the kernel)
        w = synthetic.WORKLOADS[HEADLINE]
        x = synthetic.workload_inputs(HEADLINE, device=dev, seed=w.seed + seed_off)
        lam = decay_rates(w.H).to(dev)
        y = torch.empty((w.B, w.H, w.N, 64), dtype=torch.bfloat16, device=dev)
        s = torch.empty((w.B, w.H, la.TAYLOR_D, 64), dtype=torch.float32, device=dev)
        z = torch.empty((w.B, w.H, la.TAYLOR_D), dtype=torch.float32, device=dev)

        def dstep():
            la.la_based_prefill(x["q"], x["k"], x["v"], y=y, s_out=s, z_out=z, stream=stream, decay=lam)

        t = Timer(stream, flush)
        for _ in range(args.warmup):
            t.run(dstep)
        t.reset()
        barrier(ws)
        for _ in range(steps):
            t.run(dstep)
        ms = max_over_ranks(t.total_ms(), ws) / steps
        launches += steps * KERNELS_PER_CALL["based_prefill"]
        byts = BYTES_PER_TOKEN_HEAD["taylor_prefill"] * w.B * w.H * w.N + STATE_BYTES["taylor"] * w.B * w.H
        out["based_prefill_decay"] = {"workload": w.description + ", per-head decay 1 - 2^-(5 + h mod 8)",
                                      "tokens_per_s": round(whole_job_rate(w.B * w.N, ws, ms * 1e-3), 1),
                                      "ms": round(ms, 4),
                                      "roofline": roofline(byts, ms, pk["hbm_gbs"], ncu_traffic("based_prefill_decay")),
                                      "tensor": tensor_fraction(TAYLOR_CHUNK_FLOPS * w.B * w.H * ((w.N + 127) // 128),
                                                                ms, pk, "based_prefill_decay")}
        del x, y, s, z
        torch.cuda.empty_cache()
    if only is None or only == "taylor_fp32_small":
        # the small fp32 configuration (B=1, H=2, N=256): two CTAs, so a latency figure, not a roofline one
        w = synthetic.WORKLOADS["taylor_fp32_small"]
        x = synthetic.workload_inputs(w.name, device=dev, seed=w.seed + seed_off)
        y = torch.empty((w.B, w.H, w.N, 64), dtype=torch.float32, device=dev)
        s = torch.empty((w.B, w.H, la.TAYLOR_D, 64), dtype=torch.float32, device=dev)
        z = torch.empty((w.B, w.H, la.TAYLOR_D), dtype=torch.float32, device=dev)
        wsf = torch.empty(max(1, la.la_based_prefill_workspace_size(x["q"], x["k"], x["v"], y)), dtype=torch.uint8,
                          device=dev)

        def fstep():
            la.la_based_prefill(x["q"], x["k"], x["v"], y=y, s_out=s, z_out=z, workspace=wsf, stream=stream)

        t = Timer(stream, flush)
        for _ in range(args.warmup):
            t.run(fstep)
        t.reset()
        barrier(ws)
        for _ in range(steps):
            t.run(fstep)
        ms = max_over_ranks(t.total_ms(), ws) / steps
        launches += steps * KERNELS_PER_CALL["based_prefill"]
        byts = sum(a.numel() * a.element_size() for a in (x["q"], x["k"], x["v"], y, s, z))
        out["taylor_fp32_small"] = {"workload": w.description, "tokens_per_s": round(whole_job_rate(w.B * w.N, ws,
                                                                                                 ms * 1e-3), 1),
                                    "ms": round(ms, 4),
                                    "roofline": roofline(byts, ms, pk["hbm_gbs"], ncu_traffic("taylor_fp32_small"))}
        del x, y, s, z, wsf
    for name in ("gdn_prefill", "gdn_prefill_long", "gated_prefill"):
        if only is not None and name != only:
            continue
        # the scalar gate (A_t = alpha_t I) runs on the GDN workload's inputs
        w = synthetic.WORKLOADS["gdn_prefill" if name == "gated_prefill" else name]
        prefill = la.la_gated_prefill if name == "gated_prefill" else la.la_gdn_prefill
        reps = max(1, min(steps, args.long_steps)) if name == "gdn_prefill_long" else steps
        N = getattr(args, "tokens", None) if only == name and getattr(args, "tokens", None) else w.N
        x = synthetic.workload_inputs(w.name, device=dev, seed=w.seed + seed_off, N=N)
        o = torch.empty((w.B, w.H, N, 128), dtype=torch.bfloat16, device=dev)
        S = torch.empty((w.B, w.H, 128, 128), dtype=torch.float32, device=dev)
        ws_t = torch.empty(max(1, la.la_gdn_prefill_workspace_size(x["q"], x["k"], x["v"], x["alpha"], x["beta"])),
                           dtype=torch.uint8, device=dev)

        def step():
            prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], o=o, S_out=S, workspace=ws_t, stream=stream)

        t = Timer(stream, flush)
        for _ in range(min(args.warmup, 3) if name == "gdn_prefill_long" else args.warmup):
            t.run(step)
        t.reset()
        barrier(ws)
        for _ in range(reps):
            t.run(step)
        ms = max_over_ranks(t.total_ms(), ws) / reps
        # one launch when the (b,h) pairs leave at least 16 SMs for forming the records beside the scan
        # (one CTA per SM); else the chunk-parallel inversion kernel, then the scan; sequences split
        # into segments run the scan as three kernels (maps, combine, outputs) after the inversion
        segments = la.la_gdn_prefill_workspace_size_min(x["q"], x["k"], x["v"], x["alpha"], x["beta"]) > 0
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        per_call = 4 if segments else (1 if w.B * w.H + 16 <= sms else KERNELS_PER_CALL["gdn_prefill"])
        launches += reps * per_call
        byts = BYTES_PER_TOKEN_HEAD["gdn_prefill"] * w.B * w.H * N + STATE_BYTES["gdn"] * w.B * w.H
        r = roofline(byts, ms, pk["hbm_gbs"], ncu_traffic(name) if N == w.N else None)
        desc = w.description.replace("Gated DeltaNet", "Scalar-gate") if name == "gated_prefill" else w.description
        if N != w.N:
            desc = desc.replace(f"N={w.N}", f"N={N}")
        nch = w.B * w.H * ((N + 63) // 64)
        out[name] = {"workload": desc, "tokens_per_s": round(whole_job_rate(w.B * N, ws, ms * 1e-3), 1),
                     "ms": round(ms, 4), "roofline": r,
                     "tensor": tensor_fraction(GDN_CHUNK_FLOPS["gated" if name == "gated_prefill" else "gdn"] * nch,
                                               ms, pk, name)}
        del x, o, S, ws_t
        torch.cuda.empty_cache()

    w = synthetic.WORKLOADS["decode"]
    S_, H_, n_steps = w.B, w.H, w.N
    if only is not None:
        n_steps = max(1, args.steps)
    for variant in ("gdn", "taylor"):
        if only is not None and f"decode_{variant}" != only:
            continue
        n_inputs = 16  # distinct per-step inputs, cycled (each step still reads its own q, k, v)
        xs = [synthetic.decode_step_inputs(S_, H_, i, seed=w.seed + seed_off, device=dev)[variant]
              for i in range(n_inputs)]
        if variant == "gdn":
            state = torch.zeros((S_, H_, 128, 128), device=dev)
            z = None
        else:
            state = torch.zeros((S_, H_, la.TAYLOR_D, 64), device=dev)
            z = torch.zeros((S_, H_, la.TAYLOR_D), device=dev)
        outb = torch.empty((S_, H_, 128 if variant == "gdn" else 64), dtype=torch.bfloat16, device=dev)

        def run_steps(count):
            for i in range(count):
                xi = xs[i % n_inputs]
                if variant == "gdn":
                    la.la_decode_step(la.LA_VARIANT_GDN, xi["q"], xi["k"], xi["v"], state, alpha=xi["alpha"],
                                      beta=xi["beta"], out=outb, stream=stream)
                else:
                    la.la_decode_step(la.LA_VARIANT_TAYLOR, xi["q"], xi["k"], xi["v"], state, z=z, out=outb,
                                      stream=stream)

        t = Timer(stream, flush)
        t.run(lambda: run_steps(min(n_steps, 50) if only is None else max(1, args.warmup)))  # warm-up
        t.reset()
        barrier(ws)
        t.run(lambda: run_steps(n_steps))  # the state (>L2) is streamed every step
        ms = max_over_ranks(t.total_ms(), ws)
        launches += n_steps * KERNELS_PER_CALL["decode"]
        per_step = ms / n_steps
        key = f"{variant}_decode"
        byts = BYTES_PER_TOKEN_HEAD[key] * S_ * H_
        r = roofline(byts, per_step, pk["hbm_gbs"], ncu_traffic(key))
        out[f"decode_{variant}"] = {"workload": f"{variant} decode {S_} seqs x {H_} heads x {n_steps} steps",
                                    "tokens_per_s": round(whole_job_rate(S_, ws, per_step * 1e-3), 1),
                                    "ms_per_step": round(per_step, 5), "roofline": r}
        del xs, state, z, outb
        torch.cuda.empty_cache()
    if only is None or only == "decode_swa":
        # sliding-window softmax decode (the window layers of BASED), window 64, head dim 64;
        # every sequence starts with a full window, positions precomputed per step
        S_, H_ = w.B, w.H
        n_steps = w.N if only is None else max(1, args.steps)
        g = torch.Generator(device="cpu").manual_seed(w.seed + 7 + seed_off)
        n_inputs = 16
        xs = [tuple((torch.randn((S_, H_, SWA_D), generator=g) * SWA_D ** -0.25).to(torch.bfloat16).to(dev)
                    for _ in range(3)) for _ in range(n_inputs)]
        kc = (torch.randn((S_, H_, SWA_WINDOW, SWA_D), generator=g) * SWA_D ** -0.25).to(torch.bfloat16).to(dev)
        vc = torch.randn((S_, H_, SWA_WINDOW, SWA_D), generator=g).to(torch.bfloat16).to(dev)
        total = n_steps + 64
        pos = (SWA_WINDOW + torch.arange(total, dtype=torch.int64)).view(total, 1).repeat(1, S_).to(dev)
        outb = torch.empty((S_, H_, SWA_D), dtype=torch.bfloat16, device=dev)

        def run_swa(count, first):
            for i in range(count):
                qx, kx, vx = xs[i % n_inputs]
                la.la_swa_decode_step(qx, kx, vx, kc, vc, pos[first + i], out=outb, stream=stream)

        t = Timer(stream, flush)
        t.run(lambda: run_swa(min(n_steps, 50) if only is None else max(1, args.warmup), 0))  # warm-up
        t.reset()
        barrier(ws)
        t.run(lambda: run_swa(n_steps, 0))
        ms = max_over_ranks(t.total_ms(), ws)
        launches += n_steps
        per_step = ms / n_steps
        byts = BYTES_PER_TOKEN_HEAD["swa_decode"] * S_ * H_
        r = roofline(byts, per_step, pk["hbm_gbs"], ncu_traffic("swa_decode"))
        out["decode_swa"] = {"workload": f"sliding-window softmax decode {S_} seqs x {H_} heads, window "
                                         f"{SWA_WINDOW}, d {SWA_D}, {n_steps} steps (ring caches "
                                         f"{2 * S_ * H_ * SWA_WINDOW * SWA_D * 2 >> 20} MiB, L2-resident)",
                             "tokens_per_s": round(whole_job_rate(S_, ws, per_step * 1e-3), 1),
                             "ms_per_step": round(per_step, 5), "roofline": r}
        del xs, kc, vc, pos, outb
        torch.cuda.empty_cache()
    if only is None or only in ("notebank_write", "notebank_route"):
        nb, nb_launches = notebank_paths(args, la, dev, stream, flush, pk, seed_off, ws, only)
        out.update(nb)
        launches += nb_launches
    return out, launches


def notebank_paths(args, la, dev, stream, flush, pk, seed_off, ws, only):
    """NoteBank's write side on one 16K-token document (scores of all 192 channels, then the addresses of
    two notes per 512-token chunk) and its routing of one question over 4092 stored notes."""
    out, launches = {}, 0
    steps = max(1, args.steps)
    g = torch.Generator(device="cpu").manual_seed(11 + seed_off)
    J = NB_L * NB_H
    if only is None or only == "notebank_write":
        k = torch.randn((NB_L, NB_H, NB_N, NB_D), generator=g).to(torch.bfloat16).to(dev)
        q = torch.randn((NB_L, NB_H, NB_N, NB_D), generator=g).to(torch.bfloat16).to(dev)
        coords = torch.stack([torch.randperm(NB_D, generator=g)[:16] for _ in range(J)]).view(NB_L, NB_H, 16)
        coords = coords.to(torch.int32).to(dev)
        n_notes = 2 * (NB_N // NB_CHUNK)
        starts = torch.arange(n_notes, dtype=torch.int64) * (NB_CHUNK // 2)
        spans = torch.stack([starts, torch.full_like(starts, NB_NOTE_LEN)], dim=1).to(dev)

        def wstep():
            d_ch, _, _ = la.la_notebank_scores(k, chunk=NB_CHUNK, window=NB_WINDOW, stream=stream)
            la.la_notebank_address(d_ch, q, coords, spans, stream=stream)

        t = Timer(stream, flush)
        for _ in range(args.warmup):
            t.run(wstep)
        t.reset()
        barrier(ws)
        for _ in range(steps):
            t.run(wstep)
        ms = max_over_ranks(t.total_ms(), ws) / steps
        launches += 3 * steps  # chunk scores, token scores, addresses
        # algorithmic bytes: every key read once, d_ch written and read once, d_mean and w written,
        # and per (note, channel) the span's scores and 16 query coordinates
        byts = J * NB_N * (NB_D * 2 + 4 + 4) + NB_N * 8 + n_notes * J * (NB_NOTE_LEN * 4 + 16 * 2 * 2 + 4)
        out["notebank_write"] = {"workload": f"NoteBank write side: {J} channels ({NB_L} layers x {NB_H} heads), "
                                             f"d_k {NB_D}, {NB_N} tokens, chunks of {NB_CHUNK}, "
                                             f"{n_notes} note addresses",
                                 "tokens_per_s": round(whole_job_rate(NB_N, ws, ms * 1e-3), 1),
                                 "ms": round(ms, 4),
                                 "roofline": roofline(byts, ms, pk["hbm_gbs"], ncu_traffic("notebank_write"))}
        del k, q
        torch.cuda.empty_cache()
    if only is None or only == "notebank_route":
        rho = torch.randn((NB_NOTES, J, 16), generator=g).to(torch.bfloat16).to(dev)
        u = torch.randn((J, NB_Q, 16), generator=g).to(torch.bfloat16).to(dev)
        positions = (torch.arange(NB_NOTES, dtype=torch.int64) * 32).to(dev)

        def rstep():
            la.la_notebank_route(rho, u, NB_R, positions=positions, stream=stream)

        t = Timer(stream, flush)
        for _ in range(args.warmup):
            t.run(rstep)
        t.reset()
        barrier(ws)
        for _ in range(steps):
            t.run(rstep)
        ms = max_over_ranks(t.total_ms(), ws) / steps
        launches += 2 * steps
        flops = 2.0 * NB_NOTES * J * NB_Q * 16
        out["notebank_route"] = {"workload": f"NoteBank routing: {NB_NOTES} notes x {J} channels x 16-dim addresses, "
                                             f"{NB_Q}-token question, R = {NB_R}",
                                 "questions_per_s": round(whole_job_rate(1, ws, ms * 1e-3), 1),
                                 "ms": round(ms, 4),
                                 "roofline": {"bound": "alu", "achieved": round(flops / (ms * 1e-3) / 1e12, 3),
                                              "peak": FP32_ALU_TFLOPS,
                                              "frac": round(flops / (ms * 1e-3) / 1e12 / FP32_ALU_TFLOPS, 4),
                                              "unit": "TFLOP/s fp32 (cosines)", "traffic": ncu_traffic("notebank_route"),
                                              "peak_source": "152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz"}}
        del rho, u
        torch.cuda.empty_cache()
    return out, launches


# ---------------------------------------------------------------------------
# CPU oracle arm (cpu_baseline and --impl reference)


def oracle_taylor_sample(heads=128):
    """Oracle on a bounded sample of the headline workload: `heads` of its
    128 (batch, head) pairs over the full N=4096 tokens (seeded on the CPU;
    the default is the whole workload, about a second of host time)."""
    w = synthetic.WORKLOADS[HEADLINE]
    B = max(1, heads // w.H)
    return synthetic.taylor_inputs(B, w.H, w.N, dtype=w.dtype, seed=w.seed), B * w.N


def time_oracle_once(inp):
    import oracle
    t0 = time.perf_counter()
    oracle.taylor(*(synthetic.to_oracle(inp[n]) for n in ("q", "k", "v")))
    return time.perf_counter() - t0


def cpu_baseline():
    import oracle
    oracle.build()
    inp, tokens = oracle_taylor_sample()
    dt = time_oracle_once(inp)
    return {"value": round(tokens / dt, 1), "unit": "tokens/s", "cores": oracle.default_threads(), "kind": "oracle",
            "sample": f"fp64 C oracle on the whole headline workload (8 sequences x 16 heads x 4096 tokens, "
                      f"CPU-seeded inputs); {dt:.2f} s wall"}


def _timed(fn):
    t0 = time.perf_counter()
    fn()
    return time.perf_counter() - t0


def path_cpu_baselines(paths):
    """The oracle, as it stands, timed on a bounded sample of each secondary path's workload (a few
    heads, channels or sequences of it; about a second to a few seconds each), in the path's own
    unit: a token counts once for all of its heads, so a sample of h of H heads over n tokens is
    n * h / H tokens.  Adds "cpu_baseline" to every path present in `paths`."""
    import oracle
    oracle.build()
    cores = oracle.default_threads()
    wb, wg, wl, wd = (synthetic.WORKLOADS[n] for n in ("based_prefill", "gdn_prefill", "gdn_prefill_long", "decode"))

    def put(name, units, dt, unit, sample):
        if name in paths:
            paths[name]["cpu_baseline"] = {"value": round(units / dt, 2), "unit": unit, "cores": cores,
                                           "kind": "oracle", "sample": f"{sample}; {dt:.2f} s wall"}

    if "taylor_fp32_small" in paths:
        w = synthetic.WORKLOADS["taylor_fp32_small"]
        x = synthetic.workload_inputs(w.name)
        dt = _timed(lambda: oracle.taylor(*(synthetic.to_oracle(x[n]) for n in ("q", "k", "v"))))
        put("taylor_fp32_small", w.B * w.N, dt, "tokens/s", "fp64 C oracle on the whole workload")
    if "based_prefill_decay" in paths:
        x = synthetic.taylor_inputs(1, wb.H, wb.N, dtype=wb.dtype, seed=wb.seed)
        lam = decay_rates(wb.H).double().numpy()
        dt = _timed(lambda: oracle.taylor(*(synthetic.to_oracle(x[n]) for n in ("q", "k", "v")), decay=lam))
        put("based_prefill_decay", wb.N, dt, "tokens/s", f"fp64 C oracle, 1 sequence x {wb.H} heads x {wb.N} tokens")
    for name, w, heads, n in (("gdn_prefill", wg, 2, wg.N), ("gated_prefill", wg, 2, wg.N),
                              ("gdn_prefill_long", wl, 1, 65536)):
        if name not in paths:
            continue
        x = synthetic.gdn_inputs(1, heads, n, dtype=w.dtype, seed=w.seed)
        fn = oracle.gated if name == "gated_prefill" else oracle.gdn
        dt = _timed(lambda: fn(*(synthetic.to_oracle(x[m]) for m in ("q", "k", "v")), x["alpha"].numpy(),
                               x["beta"].numpy()))
        put(name, n * heads / w.H, dt, "tokens/s", f"fp64 C oracle, {heads} of the {w.H} heads x {n} tokens")
    seqs, steps = 128, 16  # decode: 128 of the 256 sequences (all 16 heads), 16 consecutive steps
    if "decode_gdn" in paths:
        x = synthetic.gdn_inputs(seqs, wd.H, steps, dtype=torch.bfloat16, seed=wd.seed)
        dt = _timed(lambda: oracle.gdn(*(synthetic.to_oracle(x[m]) for m in ("q", "k", "v")), x["alpha"].numpy(),
                                       x["beta"].numpy()))
        put("decode_gdn", seqs * steps, dt, "tokens/s", f"fp64 C oracle, {seqs} sequences x {wd.H} heads x {steps} steps")
    if "decode_taylor" in paths:
        x = synthetic.taylor_inputs(seqs, wd.H, steps, dtype=torch.bfloat16, seed=wd.seed)
        dt = _timed(lambda: oracle.taylor(*(synthetic.to_oracle(x[m]) for m in ("q", "k", "v"))))
        put("decode_taylor", seqs * steps, dt, "tokens/s",
            f"fp64 C oracle, {seqs} sequences x {wd.H} heads x {steps} steps")
    if "decode_swa" in paths:
        g = torch.Generator().manual_seed(wd.seed)
        n_seq, heads = 64, wd.H  # 64 sequences x 16 heads, one step at position 64 with a full window
        qh, kh = ((torch.randn((n_seq, heads, SWA_WINDOW + 1, SWA_D), generator=g) * SWA_D ** -0.25)
                  .to(torch.bfloat16) for _ in range(2))
        vh = torch.randn((n_seq, heads, SWA_WINDOW + 1, SWA_D), generator=g).to(torch.bfloat16)
        dt = _timed(lambda: oracle.swa(*(synthetic.to_oracle(t) for t in (qh, kh, vh)), SWA_WINDOW,
                                       SWA_D ** -0.5, t_samples=[SWA_WINDOW]))
        put("decode_swa", n_seq, dt, "tokens/s", f"numpy oracle, {n_seq} sequences x {heads} heads, one step")
    if "notebank_write" in paths:
        g = torch.Generator().manual_seed(11)
        k = torch.randn((1, NB_H, NB_N, NB_D), generator=g).to(torch.bfloat16)
        q = torch.randn((1, NB_H, NB_N, NB_D), generator=g).to(torch.bfloat16)
        coords = np.stack([np.random.default_rng(h).permutation(NB_D)[:16] for h in range(NB_H)]).reshape(1, NB_H, 16)
        n_notes = 2 * (NB_N // NB_CHUNK)
        spans = np.stack([np.arange(n_notes) * (NB_CHUNK // 2), np.full(n_notes, NB_NOTE_LEN)], axis=1)

        def nb_write():
            r = oracle.notebank_scores(synthetic.to_oracle(k), chunk=NB_CHUNK, window=NB_WINDOW)
            oracle.notebank_address(r["d_ch"], synthetic.to_oracle(q), coords, spans)

        dt = _timed(nb_write)
        put("notebank_write", NB_N / NB_L, dt, "tokens/s",
            f"numpy oracle, 1 of the {NB_L} layers ({NB_H} channels) x {NB_N} tokens, {n_notes} note addresses")
    if "notebank_route" in paths:
        g = torch.Generator().manual_seed(12)
        J = NB_L * NB_H
        rho = torch.randn((NB_NOTES, J, 16), generator=g).to(torch.bfloat16).float().numpy()
        u = torch.randn((J, NB_Q, 16), generator=g).to(torch.bfloat16).float().numpy()
        dt = _timed(lambda: oracle.notebank_route(rho, u, NB_R))
        put("notebank_route", 1, dt, "questions/s",
            f"numpy oracle, all {NB_NOTES} notes x {J} channels, one {NB_Q}-token question")


def reference_arm(args, ws, rank):
    import oracle
    if rank != 0:
        return None
    oracle.build()
    inp, tokens = oracle_taylor_sample()
    for _ in range(args.warmup):
        time_oracle_once(inp)
    total = sum(time_oracle_once(inp) for _ in range(args.steps))
    value = tokens * args.steps / total
    w = synthetic.WORKLOADS[HEADLINE]
    cores = oracle.default_threads()
    return {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.description, "B": w.B, "H": w.H, "N": w.N, "d_feat": 16, "d_v": 64,
                       "tokens_per_step": tokens, "sample": "all 128 heads, all 4096 tokens"},
            "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": "fp64 C oracle on 8 sequences x 16 heads x 4096 tokens per step"},
            "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--long-steps", type=int, default=3, help="timed passes of the 1M-token prefill")
    ap.add_argument("--headline-only", action="store_true", help="skip the secondary paths")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=PATH_NAMES, default=None,
                    help="time one secondary path alone (K timed launches or decode steps), for profiling")
    ap.add_argument("--tokens", type=int, default=None,
                    help="with --only and a GDN prefill path: N tokens per sequence instead of the workload's "
                         "(smaller profiling captures of the same launch configuration)")
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    ws, rank, local = dist_env()
    if args.impl == "reference":
        line = reference_arm(args, ws, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if args.only is not None:
        import linear_attention_recurrence_chunked_gb300 as la
        from linear_attention_recurrence_chunked_gb300 import _build
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        _build.build()
        la.load_library()
        stream = torch.cuda.Stream(device=dev)
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        paths, launches = other_paths(args, la, dev, stream, flush, peaks(), rank_seed_offset(rank), ws, only=args.only)
        if rank == 0:
            print(json.dumps({"only": args.only, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
                              "gpu_launches": launches, **paths[args.only]}), flush=True)
        return
    line = gpu_arm(args, ws, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline and ws == 1:
            line["cpu_baseline"] = cpu_baseline()
            path_cpu_baselines(line["paths"])
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
