#!/usr/bin/env python
"""Throughput of the Gated DeltaNet core on one GB300 (or N, weak scaling).

Headline ("step" = one pass of the whole hot path over one batch): one fused
decode step of the batched-decode workload (B=128, Hk=16, Hv=32, Dk=Dv=128,
K=4: conv window + conv + SiLU + q/k norm + gates + recurrence on a 256 MiB
f32 state), carried step after step.  value = state GB/s (state bytes read +
written per step / device time per step).  The JSON line also carries the
roofline of the decode kernel (all algorithmic bytes / kernel time vs the
measured HBM copy peak), the end-to-end rate through the public API with
host buffers, the prefill tokens/s of the single-sequence and ragged prefill
workloads, and the CPU oracle's rate on a bounded sample.

--impl reference runs the reference arm: the CPU oracle, timed on this
host's cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from gated_deltanet_linear_04_gb300 import workloads as wl  # noqa: E402

METRIC = "GDN decode state GB/s (% HBM peak) and prefill tokens/s on 1 GB300"
HEADLINE = "decode_b128"


# ---------------------------------------------------------------------------
# byte / flop accounting (algorithmic, per unit)
# ---------------------------------------------------------------------------
def decode_bytes(d: wl.Dims) -> dict:
    state = d.B * d.Hv * d.Dv * d.Dk * 4
    conv_state = d.B * (d.K - 1) * d.C * 2
    return {
        "state_rw": 2 * state,
        "conv_state_rw": 2 * conv_state,
        "qkv": d.B * d.C * 2,
        "ab": 2 * d.B * d.Hv * 2,
        "y": d.B * d.Hv * d.Dv * 2,
        "params": d.C * d.K * 2 + 2 * d.Hv * 4,
    }


def recurrence_flops_per_token(d: wl.Dims) -> int:
    # decay (1), kv dot (2), update (2), output dot (2) per state element
    return 7 * d.Dk * d.Dv * d.Hv


def chunk_mma_flops(d: wl.Dims, C: int = 64) -> int:
    """Tensor-core flops of one chunk of one head in the chunked form:
    [K;Q]K^T (2C x C x Dk), U = T diag(beta) V (C x C x Dv), W = T diag(beta
    gamma) K (C x C x Dk), D = U - W S0^T and the S0 part of Y (C x Dv x Dk
    each), the state update D^T P (Dv x Dk x C) and the intra-chunk part of Y
    (C x C x Dv), 2 flops per multiply-add."""
    return 6 * C * C * d.Dk + 4 * C * C * d.Dv + 6 * C * d.Dv * d.Dk


def backward_chunk_mma_flops(d: wl.Dims, C: int = 64) -> int:
    """Tensor-core flops of one chunk of one head in the chunked backward,
    2 flops per multiply-add: the chunked forward that keeps the chunk states
    (chunk_mma_flops); the chain images (K K^T again 2C x C x Dk, Wb = T^T F K
    C x C x Dk, dY^T P and its product with T Dv x C x C each, Cq = dY^T
    gamma Q Dv x Dk x C); the chain (G Wb^T and the state-gradient update, Dv
    x C x Dk each); gradients I ([K;Q] K^T, S0 [gamma K; gamma Q]^T Dv x 2C x
    Dk, [dY; dZ] D^T 2C x C x Dv); gradients II (S0^T [dY; dZ]^T Dk x 2C x
    Dv, G^T D^T Dk x C x Dv, K^T [dPM; H + H^T]^T Dk x 2C x C, Q^T dPM Dk x C
    x C)."""
    own = 16 * C * C * d.Dk + 8 * C * C * d.Dv + 16 * C * d.Dv * d.Dk
    return chunk_mma_flops(d, C) + own


def active_chunks(mask, T: int, B: int, C: int = 64) -> int:
    """Chunks of C steps holding at least one valid step (the chunked kernels
    skip the others)."""
    n = (T + C - 1) // C
    if mask is None:
        return B * n
    m = mask.reshape(B, T)
    pad = n * C - T
    if pad:
        m = torch.nn.functional.pad(m, (0, pad))
    return int((m.reshape(B, n, C) != 0).any(dim=2).sum().item())


# tf32 : bf16 dense tensor rate on GB300 (1.1 vs 2.25 PFLOP/s nominal)
TF32_PER_BF16 = 1.1 / 2.25

# FP32 pipe of GB300: 152 SMs x 128 FP32 lanes, one fused multiply-add
# (2 flops) per lane and clock
GB300_SMS = 152
FP32_LANES_PER_SM = 128


def fp32_peak_tflops(sm_mhz: float) -> float:
    return GB300_SMS * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12


def conv_bytes(d: wl.Dims, n_valid: int) -> int:
    """Algorithmic bytes of one conv_update call: every valid token's qkv row
    read and its q, k, v rows written (bf16), the taps, and the conv_state read
    and written; padded tokens' zero outputs are written too (B*T*C*2 out)."""
    return n_valid * d.C * 2 + d.B * d.T * d.C * 2 + d.C * d.K * 2 + 2 * d.B * (d.K - 1) * d.C * 2


# ---------------------------------------------------------------------------
# environment: peaks, clocks, ranks
# ---------------------------------------------------------------------------
def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "sm_max_mhz": float(j.get("sm_max_mhz", 2070.0)), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms; keeps the
    samples that fall inside [start, stop]."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.12)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self) -> dict:
        rows = [l for (t, l) in self.lines if self.t0 is not None and self.t0 - 0.06 <= t <= (self.t1 or t) + 0.06]
        if not rows:
            rows = [l for (_, l) in self.lines]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [x.strip() for x in r.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2]))
                mx.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def source_hash(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "gated_deltanet_linear_04_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(profile: str, src_files) -> float | None:
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (its 'source_hash' line matches)."""
    p = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m_h = re.search(r"source_hash:\s*([0-9a-f]+)", txt)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m_h or not m_b or m_h.group(1) != source_hash(*src_files):
        return None
    return float(m_b.group(1))


# ---------------------------------------------------------------------------
# CPU oracle leg (bounded sample)
# ---------------------------------------------------------------------------
def oracle_decode_rate(w: wl.Workload, budget_s: float) -> dict:
    import oracle
    oracle.build_oracle()
    d = w.dims
    inp = wl.workload_inputs(w)
    cw = wl.bf16_bits(inp["conv_w"])
    A_log, dt = inp["A_log"].numpy(), inp["dt_bias"].numpy()
    cs = wl.bf16_bits(inp["conv_state"])
    st = inp["state"].numpy().astype(np.float64)
    threads = os.cpu_count() or 1
    steps, t_used = 0, 0.0
    while t_used < budget_s and steps < w.steps:
        s_in = wl.decode_step_inputs(w, steps)
        sb = [{k: wl.bf16_bits(s_in[k]) for k in ("qkv", "a", "b")}]
        t0 = time.perf_counter()
        _, st, cs = oracle.decode(d, sb, cw, A_log, dt, cs, st, threads=threads)
        t_used += time.perf_counter() - t0
        steps += 1
    by = decode_bytes(d)
    return {"steps": steps, "seconds": t_used, "state_gbs": by["state_rw"] * steps / t_used / 1e9,
            "tokens_per_s": d.B * steps / t_used, "cores": threads}


def oracle_decode_steps(w: wl.Workload, steps: int, warmup: int, budget_s: float) -> dict:
    """The reference arm: `warmup` untimed and `steps` timed carried decode
    steps of the workload through the oracle, each step on the first `rows`
    batch rows (all heads of each), `rows` sized from a first calibration
    step so that the whole run takes about `budget_s` seconds."""
    import oracle
    oracle.build_oracle()
    d = w.dims
    inp = wl.workload_inputs(w)
    cw = wl.bf16_bits(inp["conv_w"])
    A_log, dt = inp["A_log"].numpy(), inp["dt_bias"].numpy()
    cs_all = wl.bf16_bits(inp["conv_state"])
    st_all = inp["state"].numpy().astype(np.float64)
    threads = os.cpu_count() or 1

    def one_step(step, nb, cs, st):
        s_in = wl.decode_step_inputs(w, step)
        sb = [{k: wl.bf16_bits(s_in[k])[:nb] for k in ("qkv", "a", "b")}]
        t0 = time.perf_counter()
        _, st, cs = oracle.decode(d.with_(B=nb), sb, cw, A_log, dt, cs, st, threads=threads)
        return time.perf_counter() - t0, cs, st

    nb0 = min(d.B, threads)
    t_cal, _, _ = one_step(0, nb0, cs_all[:nb0], st_all[:nb0])
    per_row = t_cal / nb0
    rows = int(max(1, min(d.B, budget_s / max(1, steps + warmup) / per_row)))
    cs, st = cs_all[:rows], st_all[:rows]
    for i in range(warmup):
        _, cs, st = one_step(i, rows, cs, st)
    t_used = 0.0
    for i in range(warmup, warmup + steps):
        t, cs, st = one_step(i, rows, cs, st)
        t_used += t
    state_rw = 2 * rows * d.Hv * d.Dv * d.Dk * 4
    return {"steps": steps, "warmup": warmup, "rows": rows, "seconds": t_used,
            "state_gbs": state_rw * steps / t_used / 1e9, "cores": threads}


def oracle_prefill_rate(w: wl.Workload, heads_per_row: int = 0, vec: bool = False, budget_s: float = 0.0) -> dict:
    """The oracle over whole heads of a prefill workload: every batch row, at
    the workload's full T and row lengths, `heads_per_row` v-heads of it,
    drawn with the workload's distributions (the dims reduced to those heads:
    one k-head shared by them; all Hv heads = the workload itself, its own
    seeded inputs).  The heads run in parallel, one per core.  Without
    `heads_per_row`, a first run with one head per core sizes a second, timed
    run to about `budget_s` seconds (at most the whole workload).  With `vec`,
    the recurrence with one decay factor per key channel over the same shapes
    (gates drawn like the vectorized benchmark's).  Returns tokens/s of the
    whole workload: valid head-steps done / Hv / seconds."""
    d = w.dims
    cores = os.cpu_count() or 1
    if not heads_per_row:
        n0 = min(d.Hv, max(1, cores // d.B))
        first = oracle_prefill_rate(w, n0, vec)
        if budget_s <= 0:
            return first
        n_h = min(d.Hv, max(n0, int(n0 * budget_s / max(first["seconds"], 1e-3)) // n0 * n0))
        return first if n_h == n0 else oracle_prefill_rate(w, n_h, vec)
    import oracle
    oracle.build_oracle()
    n_h = heads_per_row
    ds = d if n_h == d.Hv else d.with_(Hk=1, Hv=n_h)
    seed = 1000 + w.index
    p = wl.make_params(ds, seed)
    a = wl.make_activations(ds, seed + 7919)
    st = wl.make_states(ds, seed + 15485863, w.conv_state, w.state)
    lens = wl.workload_lengths(w) if w.ragged else torch.full((d.B,), d.T, dtype=torch.int64)
    mask = wl.right_padded_mask(lens, d.T).numpy() if w.ragged else None
    pairs = [(b, hv) for b in range(ds.B) for hv in range(ds.Hv)]
    threads = min(cores, len(pairs))
    s0 = st["state"].numpy().astype(np.float64)
    if not vec:
        bits = {k: wl.bf16_bits(v) for k, v in (("qkv", a["qkv"]), ("a", a["a"]), ("b", a["b"]),
                                                 ("conv_w", p["conv_w"]), ("conv_state", st["conv_state"]))}
        t0 = time.perf_counter()
        oracle.layer_core(ds, bits["qkv"], bits["conv_w"], bits["a"], bits["b"], p["A_log"].numpy(),
                          p["dt_bias"].numpy(), bits["conv_state"], s0, mask, pairs, threads)
        sec = time.perf_counter() - t0
        what = "full core (conv, gates, recurrence)"
    else:
        gen = torch.Generator().manual_seed(6000 + w.index)
        q = torch.randn((ds.B, ds.T, ds.Hk, ds.Dk), generator=gen)
        k = torch.randn((ds.B, ds.T, ds.Hk, ds.Dk), generator=gen)
        q = (q / q.norm(dim=-1, keepdim=True) / ds.Dk ** 0.5).to(torch.bfloat16)
        k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
        v = torch.randn((ds.B, ds.T, ds.Hv, ds.Dv), generator=gen).to(torch.bfloat16)
        gv = torch.exp(-torch.rand((ds.B, ds.T, ds.Hv, ds.Dk), generator=gen) * 0.5).double().numpy()
        beta = torch.sigmoid(torch.randn((ds.B, ds.T, ds.Hv), generator=gen)).double().numpy()
        t0 = time.perf_counter()
        oracle.recurrence_vec(ds, wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), gv, beta, s0, mask, threads)
        sec = time.perf_counter() - t0
        what = "recurrence with per-channel decay"
    head_steps = int(lens.sum().item()) * n_h
    return {"value": round(head_steps / d.Hv / sec, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "seconds": round(sec, 3),
            "sample": "%d of %d v-heads per row, all %d rows at T=%d (%d valid head-steps), f64 oracle %s" % (
                n_h, d.Hv, d.B, d.T, head_steps, what)}


def oracle_decode_b1_rate(w: wl.Workload, budget_s: float) -> dict:
    """The oracle over the single-sequence decode workload's first carried
    steps (all heads), as many as fit the time budget."""
    import oracle
    oracle.build_oracle()
    d = w.dims
    inp = wl.workload_inputs(w)
    cw = wl.bf16_bits(inp["conv_w"])
    A_log, dt = inp["A_log"].numpy(), inp["dt_bias"].numpy()
    cs = wl.bf16_bits(inp["conv_state"])
    st = inp["state"].numpy().astype(np.float64)
    threads = min(os.cpu_count() or 1, d.B * d.Hv)
    steps, t_used = 0, 0.0
    while t_used < budget_s and steps < w.steps:
        s_in = wl.decode_step_inputs(w, steps)
        sb = [{k: wl.bf16_bits(s_in[k]) for k in ("qkv", "a", "b")}]
        t0 = time.perf_counter()
        _, st, cs = oracle.decode(d, sb, cw, A_log, dt, cs, st, threads=threads)
        t_used += time.perf_counter() - t0
        steps += 1
    return {"value": round(d.B * steps / t_used, 2), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "seconds": round(t_used, 3),
            "sample": "first %d of %d carried decode steps (all %d heads), f64 oracle" % (steps, w.steps,
                                                                                         d.B * d.Hv)}


# ---------------------------------------------------------------------------
# GPU legs
# ---------------------------------------------------------------------------
def bench_decode(gdn, w: wl.Workload, steps: int, warmup: int, dev, sampler) -> dict:
    d = w.dims
    d1 = d.with_(T=1)
    inp = wl.workload_inputs(w)
    n_in = min(w.steps, steps + warmup)
    step_in = [wl.decode_step_inputs(w, i) for i in range(n_in)]
    qkv_h = torch.stack([s["qkv"][:, 0] for s in step_in]).pin_memory()   # [n, B, C]
    a_h = torch.stack([s["a"][:, 0] for s in step_in]).pin_memory()
    b_h = torch.stack([s["b"][:, 0] for s in step_in]).pin_memory()
    qkv, a, b = qkv_h.to(dev), a_h.to(dev), b_h.to(dev)
    conv_w, A_log, dt_bias = inp["conv_w"].to(dev), inp["A_log"].to(dev), inp["dt_bias"].to(dev)
    conv_state = inp["conv_state"].to(dev)
    state = inp["state"].to(dev)
    y = torch.empty((d.B, d.Hv, d.Dv), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        j = i % n_in
        gdn.gdn_recurrent_decode(d1, qkv[j], conv_w, conv_state, a[j], b[j], A_log, dt_bias, state, None, y, stream)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    # the K timed steps, as a serving loop runs them: captured once as one CUDA
    # graph (K decode launches joined by programmatic edges, each reading the
    # state the one before wrote) and replayed.  The same K steps launched one
    # by one from the host are timed too (ms_eager): they pay the first
    # launch's start-up latency inside the timed region.
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for i in range(steps):
                j = (warmup + i) % n_in
                gdn.gdn_recurrent_decode(d1, qkv[j], conv_w, conv_state, a[j], b[j], A_log, dt_bias, state, None, y,
                                         side)
    stream.wait_stream(side)
    graph.replay()                      # untimed: uploads the graph
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    sampler.mark_start()
    ev[0].record(stream)
    for i in range(steps):
        step(warmup + i)
    ev[1].record(stream)
    torch.cuda.synchronize()
    ev[2].record(stream)
    graph.replay()
    ev[3].record(stream)
    torch.cuda.synchronize()
    sampler.mark_stop()
    ms_eager = ev[0].elapsed_time(ev[1]) / steps
    ms = ev[2].elapsed_time(ev[3]) / steps
    if gdn.gdn_device_status() != gdn.GDN_OK:
        raise RuntimeError("device error word set during the decode benchmark")
    del graph

    # end to end through the C ABI with host buffers: every step's inputs are
    # copied in from pinned host memory and its y copied back out inside
    # gdn_recurrent_decode_host_steps, which double-buffers them in a device
    # staging area on its own copy streams, so step i+1's inputs travel while
    # step i computes, as a serving loop would.
    staging = torch.empty(gdn.gdn_decode_host_staging_size(d1), dtype=torch.uint8, device=dev)
    y_h = torch.empty((n_in, d.B, d.Hv, d.Dv), dtype=torch.bfloat16).pin_memory()

    def e2e_run(first, n):
        done = 0
        while done < n:
            j = (first + done) % n_in
            m = min(n - done, n_in - j)
            gdn.gdn_recurrent_decode_host_steps(d1, m, qkv_h[j:j + m], a_h[j:j + m], b_h[j:j + m], y_h[j:j + m],
                                                conv_w, conv_state, A_log, dt_bias, state, None, staging, stream)
            done += m

    e2e_run(0, warmup)
    torch.cuda.synchronize()
    # five full runs, the median reported: the host-memory copies of this path
    # now and then stall for tens of milliseconds on a shared host (seen with
    # and without the clock sampler running), which the device-resident loop
    # never sees
    runs = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_wall = time.perf_counter()
        e0.record(stream)
        e2e_run(warmup, steps)
        e1.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        runs.append(max(e0.elapsed_time(e1), t_wall * 1e3) / steps)
    if gdn.gdn_device_status() != gdn.GDN_OK:
        raise RuntimeError("device error word set during the end-to-end decode benchmark")
    e2e_ms = statistics.median(runs)
    per_step = (d.B * d1.C, d.B * d.Hv, d.B * d.Hv * d.Dv)
    return {"ms": ms, "ms_eager": ms_eager, "e2e_ms": e2e_ms, "e2e_runs_ms": runs,
            "h2d": per_step[0] * 2 + 2 * per_step[1] * 2, "d2h": per_step[2] * 2}


def bench_decode_small(gdn, w: wl.Workload, dev, reps: int = 3) -> dict:
    """Single-sequence decode: the workload's carried steps (1024), launched
    back to back and as one captured CUDA graph (launch overhead removed).
    The 2 MiB state stays in L2, so its GB/s is not an HBM-roofline figure."""
    d = w.dims
    d1 = d.with_(T=1)
    inp = wl.workload_inputs(w)
    steps = [wl.decode_step_inputs(w, i) for i in range(w.steps)]
    qkv = torch.stack([x["qkv"][:, 0] for x in steps]).to(dev)
    a = torch.stack([x["a"][:, 0] for x in steps]).to(dev)
    b = torch.stack([x["b"][:, 0] for x in steps]).to(dev)
    conv_w, A_log, dt_bias = inp["conv_w"].to(dev), inp["A_log"].to(dev), inp["dt_bias"].to(dev)
    cs0, st0 = inp["conv_state"].to(dev), inp["state"].to(dev)
    cs, st = cs0.clone(), st0.clone()
    y = torch.empty((w.steps, d.B, d.Hv, d.Dv), dtype=torch.bfloat16, device=dev)

    def run(stream):
        for i in range(w.steps):
            gdn.gdn_recurrent_decode(d1, qkv[i], conv_w, cs, a[i], b[i], A_log, dt_bias, st, None, y[i], stream)

    stream = torch.cuda.current_stream()
    run(stream)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    t_eager = []
    for _ in range(reps):
        cs.copy_(cs0); st.copy_(st0)
        ev[0].record(stream); run(stream); ev[1].record(stream)
        torch.cuda.synchronize()
        t_eager.append(ev[0].elapsed_time(ev[1]))
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            run(torch.cuda.current_stream())
    stream.wait_stream(side)
    t_graph = []
    for _ in range(reps):
        cs.copy_(cs0); st.copy_(st0)
        ev[0].record(stream); g.replay(); ev[1].record(stream)
        torch.cuda.synchronize()
        t_graph.append(ev[0].elapsed_time(ev[1]))
    if gdn.gdn_device_status() != gdn.GDN_OK:
        raise RuntimeError("device error word set during the single-sequence decode benchmark")
    by = sum(decode_bytes(d).values())
    us_e, us_g = min(t_eager) * 1e3 / w.steps, min(t_graph) * 1e3 / w.steps
    return {"workload": w.name, "steps": w.steps, "us_per_step_eager": round(us_e, 3),
            "us_per_step_graph": round(us_g, 3), "tokens_per_s_graph": round(d.B / (us_g / 1e6), 1),
            "gbs_graph_l2_resident": round(by / (us_g / 1e6) / 1e9, 1)}


def bench_backward(gdn, w: wl.Workload, dev, peaks, chunk: int = 0, iters: int = 3) -> dict:
    """The backward pass of the recurrence over one workload call (gradients of
    y and of the final state with respect to q, k, v, g, beta and the initial
    state), from device-generated inputs of the workload's shapes; chunk = 0
    the sequential form, 64 the chunked form on the tensor cores (its roofline:
    the MMA flops of the whole call, forward included, against the tf32 rate)."""
    d = w.dims
    gen = torch.Generator(device=dev)
    gen.manual_seed(5000 + w.index)
    q = torch.randn((d.B, d.T, d.Hk, d.Dk), generator=gen, device=dev)
    k = torch.randn((d.B, d.T, d.Hk, d.Dk), generator=gen, device=dev)
    q = (q / q.norm(dim=-1, keepdim=True) / d.Dk ** 0.5).to(torch.bfloat16)
    k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    v = torch.randn((d.B, d.T, d.Hv, d.Dv), generator=gen, device=dev).to(torch.bfloat16)
    g = torch.exp(-torch.rand((d.B, d.T, d.Hv), generator=gen, device=dev) * 0.5)
    beta = torch.sigmoid(torch.randn((d.B, d.T, d.Hv), generator=gen, device=dev))
    s0 = torch.randn((d.B, d.Hv, d.Dv, d.Dk), generator=gen, device=dev) * 0.05
    dy = (torch.randn((d.B, d.T, d.Hv, d.Dv), generator=gen, device=dev) * 0.1).to(torch.bfloat16)
    mask = None
    n_valid = d.B * d.T
    if w.ragged:
        lens = wl.workload_lengths(w)
        mask = wl.right_padded_mask(lens, d.T).to(dev)
        n_valid = int(lens.sum())
    outs = [torch.empty((d.B, d.T, d.Hk, d.Dk), device=dev), torch.empty((d.B, d.T, d.Hk, d.Dk), device=dev),
            torch.empty((d.B, d.T, d.Hv, d.Dv), device=dev), torch.empty((d.B, d.T, d.Hv), device=dev),
            torch.empty((d.B, d.T, d.Hv), device=dev), torch.empty((d.B, d.Hv, d.Dv, d.Dk), device=dev)]
    size_fn = gdn.gdn_prefill_backward_chunked_workspace_size if chunk else gdn.gdn_prefill_backward_workspace_size
    call = gdn.gdn_prefill_backward_chunked if chunk else gdn.gdn_prefill_backward
    ws = torch.empty(size_fn(d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def once():
        call(d, q, k, v, g, beta, s0, mask, dy, None, *outs, ws, stream)

    once()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        once()
    e1.record(stream)
    torch.cuda.synchronize()
    if gdn.gdn_device_status() != gdn.GDN_OK:
        raise RuntimeError("device error word set during the backward benchmark")
    ms = e0.elapsed_time(e1) / iters
    res = {"workload": w.name, "chunk": chunk, "ms": round(ms, 4), "tokens": n_valid,
           "tokens_per_s": round(n_valid / (ms / 1e3), 1), "workspace_mb": round(ws.numel() / 2 ** 20, 1)}
    if chunk:
        n_ch = active_chunks(mask, d.T, d.B) * d.Hv
        fl = backward_chunk_mma_flops(d) * n_ch
        tflops = fl / (ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"] * TF32_PER_BF16
        res["roofline"] = {"bound": "tensor", "achieved": round(tflops, 2), "peak": round(peak, 1),
                           "unit": "TFLOP/s", "frac": round(tflops / peak, 4), "traffic": None,
                           "algorithmic_flops": fl, "units": n_ch, "unit_name": "chunk of 64 steps x head",
                           "flops_per_unit": backward_chunk_mma_flops(d),
                           "kernel": "the whole chunked backward call (forward with chunk records, chain images, "
                                     "reverse chain, two gradient passes)",
                           "peak_source": peaks["source"] + " bf16 x nominal tf32/bf16 (1.1/2.25)"}
    return res


def bench_decode_gated(gdn, w: wl.Workload, dev, iters: int = 200) -> dict:
    """One decode step of the batched-decode workload with the layer's gated
    RMS norm: the gated entry point vs decode followed by the separate norm
    kernel (the state is carried across the steps either way)."""
    d = w.dims.with_(T=1)
    gen = torch.Generator(device=dev)
    gen.manual_seed(4000 + w.index)
    qkv = torch.randn((d.B, d.C), generator=gen, device=dev).to(torch.bfloat16)
    a = torch.randn((d.B, d.Hv), generator=gen, device=dev).to(torch.bfloat16)
    b = torch.randn((d.B, d.Hv), generator=gen, device=dev).to(torch.bfloat16)
    conv_w = (torch.randn((d.C, d.K), generator=gen, device=dev) * 0.5).to(torch.bfloat16)
    A_log = torch.log(torch.empty(d.Hv, device=dev).uniform_(1.0, 16.0, generator=gen))
    dt_bias = torch.randn(d.Hv, generator=gen, device=dev) * 0.5
    cs = torch.randn((d.B, d.K - 1, d.C), generator=gen, device=dev).to(torch.bfloat16)
    st = torch.randn((d.B, d.Hv, d.Dv, d.Dk), generator=gen, device=dev) * 0.05
    z = torch.randn((d.B, d.Hv, d.Dv), generator=gen, device=dev).to(torch.bfloat16)
    norm_w = torch.empty(d.Dv, device=dev).uniform_(0.5, 1.5, generator=gen)
    y = torch.empty((d.B, d.Hv, d.Dv), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(y)
    stream = torch.cuda.current_stream()

    def step(fused):
        if fused:
            gdn.gdn_recurrent_decode_gated(d, qkv, conv_w, cs, a, b, A_log, dt_bias, st, None, z, norm_w, 1e-6,
                                           out, stream)
        else:
            gdn.gdn_recurrent_decode(d, qkv, conv_w, cs, a, b, A_log, dt_bias, st, None, y, stream)
            gdn.gdn_rmsnorm_gated(d, y, z, norm_w, 1e-6, out, stream)

    us = {}
    for fused in (True, False):
        for _ in range(3):
            step(fused)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            step(fused)
        e1.record(stream)
        torch.cuda.synchronize()
        us[fused] = e0.elapsed_time(e1) / iters * 1e3
    if gdn.gdn_device_status() != gdn.GDN_OK:
        raise RuntimeError("device error word set during the gated decode benchmark")
    state_rw = 2 * d.B * d.Hv * d.Dv * d.Dk * 4
    return {"workload": w.name, "us_per_step_gdn_recurrent_decode_gated": round(us[True], 2),
            "us_per_step_decode_then_norm": round(us[False], 2),
            "state_gbs_gated": round(state_rw / (us[True] / 1e6) / 1e9, 1)}


def bench_decode_window(gdn, w: wl.Workload, dev, T: int = 4, iters: int = 20) -> dict:
    """Speculative-verify window: T tokens per row of the batched-decode
    workload in one fused kernel, all T committed (the state is streamed once
    per window instead of once per token)."""
    d = w.dims.with_(T=T)
    gen = torch.Generator(device=dev)
    gen.manual_seed(3000 + w.index)
    qkv = torch.randn((d.B, T, d.C), generator=gen, device=dev).to(torch.bfloat16)
    a = torch.randn((d.B, T, d.Hv), generator=gen, device=dev).to(torch.bfloat16)
    b = torch.randn((d.B, T, d.Hv), generator=gen, device=dev).to(torch.bfloat16)
    conv_w = (torch.randn((d.C, d.K), generator=gen, device=dev) * 0.5).to(torch.bfloat16)
    A_log = torch.log(torch.empty(d.Hv, device=dev).uniform_(1.0, 16.0, generator=gen))
    dt_bias = torch.randn(d.Hv, generator=gen, device=dev) * 0.5
    cs = torch.randn((d.B, d.K - 1, d.C), generator=gen, device=dev).to(torch.bfloat16)
    st = torch.randn((d.B, d.Hv, d.Dv, d.Dk), generator=gen, device=dev) * 0.05
    y = torch.empty((d.B, T, d.Hv, d.Dv), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        gdn.gdn_decode_window(d, qkv, conv_w, cs, a, b, A_log, dt_bias, st, None, y, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        gdn.gdn_decode_window(d, qkv, conv_w, cs, a, b, A_log, dt_bias, st, None, y, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    if gdn.gdn_device_status() != gdn.GDN_OK:
        raise RuntimeError("device error word set during the decode-window benchmark")
    ms = e0.elapsed_time(e1) / iters
    state_rw = 2 * d.B * d.Hv * d.Dv * d.Dk * 4
    return {"workload": w.name, "window": T, "us_per_window": round(ms * 1e3, 2),
            "tokens_per_s": round(d.B * T / (ms / 1e3), 1), "state_gbs": round(state_rw / (ms / 1e3) / 1e9, 1)}


def bench_rmsnorm_gated(gdn, w: wl.Workload, dev, iters: int = 5) -> dict:
    """The RMSNormGated output over a whole prefill output (B*T*Hv rows of Dv):
    HBM-bound, 6 bytes per element (y and z in, out)."""
    d = w.dims
    gen = torch.Generator(device=dev)
    gen.manual_seed(2000 + w.index)
    y = (torch.randn((d.B, d.T, d.Hv, d.Dv), generator=gen, device=dev) * 0.1).to(torch.bfloat16)
    z = torch.randn((d.B, d.T, d.Hv, d.Dv), generator=gen, device=dev).to(torch.bfloat16)
    nw = torch.empty(d.Dv, device=dev).uniform_(0.5, 1.5, generator=gen)
    out = torch.empty_like(y)
    stream = torch.cuda.current_stream()
    gdn.gdn_rmsnorm_gated(d, y, z, nw, 1e-6, out, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        gdn.gdn_rmsnorm_gated(d, y, z, nw, 1e-6, out, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / iters
    nbytes = 3 * y.numel() * 2 + d.Dv * 4
    del y, z, out
    return {"workload": w.name, "ms": round(ms, 4), "bytes": nbytes, "gbs": round(nbytes / (ms / 1e3) / 1e9, 1)}


def bench_prefill(gdn, w: wl.Workload, dev, iters: int, chunk: int, peaks: dict = None) -> dict:
    """Full core (conv + gates + recurrence) over one workload call."""
    d = w.dims
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + w.index)
    qkv = torch.randn((d.B, d.T, d.C), generator=gen, device=dev).to(torch.bfloat16)
    conv_w = (torch.randn((d.C, d.K), generator=gen, device=dev) * 0.5).to(torch.bfloat16)
    a = torch.randn((d.B, d.T, d.Hv), generator=gen, device=dev).to(torch.bfloat16)
    b = torch.randn((d.B, d.T, d.Hv), generator=gen, device=dev).to(torch.bfloat16)
    A_log = torch.log(torch.empty(d.Hv, device=dev).uniform_(1.0, 16.0, generator=gen))
    dt_bias = torch.randn(d.Hv, generator=gen, device=dev) * 0.5
    state0 = (torch.randn((d.B, d.Hv, d.Dv, d.Dk), generator=gen, device=dev) * 0.05 if w.state == "normal"
              else torch.zeros((d.B, d.Hv, d.Dv, d.Dk), device=dev))
    mask = None
    n_valid = d.B * d.T
    if w.ragged:
        lens = wl.workload_lengths(w)
        mask = wl.right_padded_mask(lens, d.T).to(dev)
        n_valid = int(lens.sum())
    conv_state = torch.zeros((d.B, d.K - 1, d.C), dtype=torch.bfloat16, device=dev)
    q = torch.empty((d.B, d.T, d.Hk, d.Dk), dtype=torch.bfloat16, device=dev)
    k = torch.empty_like(q)
    v = torch.empty((d.B, d.T, d.Hv, d.Dv), dtype=torch.bfloat16, device=dev)
    g = torch.empty((d.B, d.T, d.Hv), dtype=torch.float32, device=dev)
    beta = torch.empty_like(g)
    y = torch.empty((d.B, d.T, d.Hv, d.Dv), dtype=torch.bfloat16, device=dev)
    s_out = torch.empty_like(state0)
    nws = gdn.gdn_prefill_workspace_size(d, chunk)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    # events around each part of each call; the calls are queued back to back
    # and read after one synchronisation, so the host's per-call work (argument
    # checks, tensor-map encoding) overlaps the previous call's kernels instead
    # of sitting inside the measured intervals
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(iters)]

    def once(ev=None):
        if ev:
            ev[0].record(stream)
        gdn.gdn_conv_update(d, qkv, conv_w, conv_state, mask, q, k, v, stream)
        if ev:
            ev[3].record(stream)
        gdn.gdn_gating(d, a, b, A_log, dt_bias, g, beta, stream)
        if ev:
            ev[1].record(stream)
        gdn.gdn_prefill(d, q, k, v, g, beta, state0, s_out, mask, y, chunk, ws if nws else None, stream)
        if ev:
            ev[2].record(stream)

    once()
    torch.cuda.synchronize()
    for ev in evs:
        once(ev)
    torch.cuda.synchronize()
    t_tot = sum(ev[0].elapsed_time(ev[2]) for ev in evs)
    t_rec = sum(ev[1].elapsed_time(ev[2]) for ev in evs)
    t_conv = sum(ev[0].elapsed_time(ev[3]) for ev in evs)
    if gdn.gdn_device_status() != gdn.GDN_OK:
        raise RuntimeError("device error word set during the prefill benchmark")
    ms, ms_rec, ms_conv = t_tot / iters, t_rec / iters, t_conv / iters
    flops = recurrence_flops_per_token(d) * n_valid

    # the layer's gated RMS norm on top of the recurrence: the gated entry
    # point (the norm in the chunked kernel's epilogue when the heads fill the
    # GPU) vs the recurrence followed by the separate norm kernel
    z = (torch.randn((d.B, d.T, d.Hv, d.Dv), generator=gen, device=dev)).to(torch.bfloat16)
    norm_w = torch.empty(d.Dv, device=dev).uniform_(0.5, 1.5, generator=gen)
    out = torch.empty_like(y)

    def gated(fused):
        if fused:
            gdn.gdn_prefill_gated(d, q, k, v, g, beta, state0, s_out, mask, z, norm_w, 1e-6, out, chunk,
                                  ws if nws else None, stream)
        else:
            gdn.gdn_prefill(d, q, k, v, g, beta, state0, s_out, mask, y, chunk, ws if nws else None, stream)
            gdn.gdn_rmsnorm_gated(d, y, z, norm_w, 1e-6, out, stream)

    t_g = {}
    ev = evs[0]
    for fused in (True, False):
        gated(fused)
        torch.cuda.synchronize()
        ev[0].record(stream)
        for _ in range(iters):
            gated(fused)
        ev[1].record(stream)
        torch.cuda.synchronize()
        t_g[fused] = ev[0].elapsed_time(ev[1]) / iters
    if gdn.gdn_device_status() != gdn.GDN_OK:
        raise RuntimeError("device error word set during the gated prefill benchmark")
    res = {"workload": w.name, "chunk": chunk, "ms": round(ms, 4), "recurrence_ms": round(ms_rec, 4),
           "conv_ms": round(ms_conv, 4), "tokens": n_valid, "tokens_per_s": n_valid / (ms / 1e3),
           "recurrence_tflops": flops / (ms_rec / 1e3) / 1e12,
           "recurrence_gated_norm_ms": {"gdn_prefill_gated": round(t_g[True], 4),
                                        "prefill_then_norm": round(t_g[False], 4)}}
    peaks = peaks or load_peaks()
    if chunk == 64:
        # tensor-core work of the chunked form over the chunks it computes,
        # against the tf32 rate (measured bf16 peak x the nominal tf32 ratio)
        n_ch = active_chunks(mask, d.T, d.B) * d.Hv
        tflops = chunk_mma_flops(d) * n_ch / (ms_rec / 1e3) / 1e12
        peak = peaks["bf16_tflops"] * TF32_PER_BF16
        res["roofline"] = {"bound": "tensor", "achieved": round(tflops, 2), "peak": round(peak, 1),
                           "unit": "TFLOP/s", "frac": round(tflops / peak, 4), "traffic": None,
                           "algorithmic_flops": chunk_mma_flops(d) * n_ch, "units": n_ch,
                           "unit_name": "chunk of 64 steps x head", "flops_per_unit": chunk_mma_flops(d),
                           "kernel": "the chunked recurrence launch (tcgen05 kind::tf32 and kind::f16 products)",
                           "peak_source": peaks["source"] + " bf16 x nominal tf32/bf16 (1.1/2.25)"}
    else:
        # the sequential form: 7 Dk Dv flops per head-step on the FP32 pipe
        tfl = flops / (ms_rec / 1e3) / 1e12
        peak = fp32_peak_tflops(peaks["sm_max_mhz"])
        res["roofline"] = {"bound": "alu", "achieved": round(tfl, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                           "frac": round(tfl / peak, 4), "traffic": None, "algorithmic_flops": flops,
                           "units": n_valid * d.Hv, "unit_name": "head-step",
                           "flops_per_unit": 7 * d.Dk * d.Dv, "kernel": "prefill_seq_kernel",
                           "peak_source": "152 SMs x 128 FP32 lanes x 2 flops x %.0f MHz" % peaks["sm_max_mhz"]}
    cb = conv_bytes(d, n_valid)
    res["conv_roofline"] = {"bound": "hbm", "achieved": round(cb / (ms_conv / 1e3) / 1e9, 1),
                            "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": round(cb / (ms_conv / 1e3) / 1e9 / peaks["hbm_gbs"], 4), "traffic": None,
                            "algorithmic_bytes": cb, "kernel": "conv_update_kernel + conv_state_kernel",
                            "peak_source": peaks["source"]}
    return res


def bench_prefill_vec(gdn, w: wl.Workload, dev, iters: int = 3, peaks: dict = None) -> dict:
    """The recurrence with one decay factor per key channel (g [B, T, Hv, Dk])
    over a prefill workload's shapes, sequential form, from device-drawn
    inputs: q/k unit-norm-scaled like the conv output, g in (e^-0.5, 1)."""
    d = w.dims
    gen = torch.Generator(device=dev)
    gen.manual_seed(6000 + w.index)
    q = torch.randn((d.B, d.T, d.Hk, d.Dk), generator=gen, device=dev)
    k = torch.randn((d.B, d.T, d.Hk, d.Dk), generator=gen, device=dev)
    q = (q / q.norm(dim=-1, keepdim=True) / d.Dk ** 0.5).to(torch.bfloat16)
    k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    v = torch.randn((d.B, d.T, d.Hv, d.Dv), generator=gen, device=dev).to(torch.bfloat16)
    gv = torch.exp(-torch.rand((d.B, d.T, d.Hv, d.Dk), generator=gen, device=dev) * 0.5)
    beta = torch.sigmoid(torch.randn((d.B, d.T, d.Hv), generator=gen, device=dev))
    s0 = (torch.randn((d.B, d.Hv, d.Dv, d.Dk), generator=gen, device=dev) * 0.05 if w.state == "normal"
          else torch.zeros((d.B, d.Hv, d.Dv, d.Dk), device=dev))
    mask, n_valid = None, d.B * d.T
    if w.ragged:
        lens = wl.workload_lengths(w)
        mask = wl.right_padded_mask(lens, d.T).to(dev)
        n_valid = int(lens.sum())
    y = torch.empty((d.B, d.T, d.Hv, d.Dv), dtype=torch.bfloat16, device=dev)
    s_out = torch.empty_like(s0)
    stream = torch.cuda.current_stream()
    gdn.gdn_prefill_vec(d, q, k, v, gv, beta, s0, s_out, mask, y, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        gdn.gdn_prefill_vec(d, q, k, v, gv, beta, s0, s_out, mask, y, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    if gdn.gdn_device_status() != gdn.GDN_OK:
        raise RuntimeError("device error word set during the vectorized-gating benchmark")
    ms = e0.elapsed_time(e1) / iters
    peaks = peaks or load_peaks()
    flops = recurrence_flops_per_token(d) * n_valid
    tfl = flops / (ms / 1e3) / 1e12
    peak = fp32_peak_tflops(peaks["sm_max_mhz"])
    return {"workload": w.name, "ms": round(ms, 4), "tokens": n_valid, "tokens_per_s": round(n_valid / (ms / 1e3), 1),
            "roofline": {"bound": "alu", "achieved": round(tfl, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                         "frac": round(tfl / peak, 4), "traffic": None, "algorithmic_flops": flops,
                         "units": n_valid * d.Hv, "unit_name": "head-step", "flops_per_unit": 7 * d.Dk * d.Dv,
                         "kernel": "prefill_seq_kernel (per-channel decay)",
                         "peak_source": "152 SMs x 128 FP32 lanes x 2 flops x %.0f MHz" % peaks["sm_max_mhz"]}}


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2048)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--no-prefill", action="store_true", help="only the headline decode (no other sections)")
    ap.add_argument("--parts", default="decode_b1,rmsnorm,window,decode_gated,prefill,prefill_vec,backward",
                    help="comma-separated sections to run after the headline decode")
    ap.add_argument("--backward-workloads", default="prefill_t8192,prefill_ragged",
                    help="workloads of the backward section (a subset keeps an ncu capture small)")
    ap.add_argument("--prefill-workloads", default="prefill_t8192,prefill_ragged",
                    help="workloads of the prefill section (a subset keeps an ncu capture small)")
    ap.add_argument("--backward-t", type=int, default=0,
                    help="run the backward workloads at this sequence length instead (small profiling captures)")
    ap.add_argument("--backward-chunks", default="0,64", help="backward forms to time: 0 sequential, 64 chunked")
    ap.add_argument("--prefill-t", type=int, default=0,
                    help="run the prefill section at this T instead of the workload's (profiling captures of a "
                         "small case only; the benchmark figures use the workloads' own T)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--ref-budget-s", type=float, default=90.0,
                    help="reference arm: about this many seconds for all warm-up and timed oracle steps")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    ws, rank, local = dist_env()
    w = wl.WORKLOADS[HEADLINE]
    d = w.dims
    by = decode_bytes(d)
    alg_bytes = sum(by.values())

    if args.impl == "reference":
        if ws > 1:
            torch.distributed.init_process_group("gloo")
            if rank != 0:
                torch.distributed.destroy_process_group()
                return
        r = oracle_decode_steps(w, args.steps, args.warmup, args.ref_budget_s)
        ms = r["seconds"] / r["steps"] * 1e3
        line = {"impl": "reference", "metric": METRIC, "value": round(r["state_gbs"], 4), "unit": "GB/s",
                "n_gpus": args.gpus, "steps": r["steps"], "warmup": r["warmup"], "ms_per_step": round(ms, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": w.name, "B": d.B, "Hk": d.Hk, "Hv": d.Hv,
                                                "Dk": d.Dk, "Dv": d.Dv, "K": d.K},
                "cpu_baseline": {"value": round(r["state_gbs"], 4), "unit": "GB/s", "cores": r["cores"],
                                 "kind": "oracle",
                                 "sample": "%d timed carried decode steps after %d untimed ones, each on the "
                                           "first %d of the %d batch rows (all %d heads of each row)" % (
                                     r["steps"], r["warmup"], r["rows"], d.B, d.Hv)},
                "e2e": {"value": round(r["state_gbs"], 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        if ws > 1:
            torch.distributed.destroy_process_group()
        return

    from gated_deltanet_linear_04_gb300 import gdn
    gdn.lib()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)

    peaks = load_peaks()
    with ClockSampler(local) as sampler:
        barrier(ws)
        res = bench_decode(gdn, w, args.steps, args.warmup, dev, sampler)
    ms = max_over_ranks(res["ms"], ws)
    ms_eager = max_over_ranks(res["ms_eager"], ws)
    e2e_ms = max_over_ranks(res["e2e_ms"], ws)
    clocks = sampler.summary()

    small_decode = None
    gated_norm = None
    window = None
    decode_gated = None
    prefill = []
    parts = set() if args.no_prefill else set(args.parts.split(","))
    if "decode_b1" in parts:
        small_decode = bench_decode_small(gdn, wl.WORKLOADS["decode_b1"], dev)
        if rank == 0 and not args.no_cpu:
            small_decode["cpu_baseline"] = oracle_decode_b1_rate(wl.WORKLOADS["decode_b1"], args.cpu_budget_s / 4)
    if "rmsnorm" in parts:
        gated_norm = bench_rmsnorm_gated(gdn, wl.WORKLOADS["prefill_ragged"], dev)
    if "window" in parts:
        window = bench_decode_window(gdn, w, dev)
    if "decode_gated" in parts:
        decode_gated = bench_decode_gated(gdn, w, dev)
    backward = None
    if "backward" in parts:
        backward = []
        for name in args.backward_workloads.split(","):
            w_b = wl.WORKLOADS[name]
            if args.backward_t > 0:
                w_b = wl.Workload(w_b.name + "_t%d" % args.backward_t, w_b.index, w_b.dims.with_(T=args.backward_t),
                                  w_b.steps, w_b.conv_state, w_b.state, w_b.ragged, min(w_b.len_lo, args.backward_t),
                                  min(w_b.len_hi, args.backward_t))
            for chunk in [int(x) for x in args.backward_chunks.split(",")]:
                backward.append(bench_backward(gdn, w_b, dev, peaks, chunk))
    prefill_vec = None
    if "prefill_vec" in parts:
        prefill_vec = bench_prefill_vec(gdn, wl.WORKLOADS["prefill_t8192"], dev, 3, peaks)
        if rank == 0 and not args.no_cpu:
            prefill_vec["cpu_baseline"] = oracle_prefill_rate(wl.WORKLOADS["prefill_t8192"], vec=True,
                                                              budget_s=args.cpu_budget_s / 2)
    if "prefill" in parts:
        for name in args.prefill_workloads.split(","):
            entries = []
            w_p = wl.WORKLOADS[name]
            if args.prefill_t > 0:
                w_p = wl.Workload(w_p.name + "_t%d" % args.prefill_t, w_p.index, w_p.dims.with_(T=args.prefill_t),
                                  w_p.steps, w_p.conv_state, w_p.state, w_p.ragged, min(w_p.len_lo, args.prefill_t),
                                  min(w_p.len_hi, args.prefill_t))
            for chunk in (0, 64):
                try:
                    entries.append(bench_prefill(gdn, w_p, dev, 3, chunk, peaks))
                except gdn.GdnError as e:
                    if e.status != gdn.GDN_ERR_UNSUPPORTED:
                        raise
                    entries.append({"workload": name, "chunk": chunk, "unavailable": "chunked form not built"})
            if rank == 0 and not args.no_cpu:
                # the oracle on a bounded sample of the same workload, once per
                # workload: the same figure stands beside both forms
                cb = oracle_prefill_rate(w_p, budget_s=args.cpu_budget_s)
                for e_ in entries:
                    e_["cpu_baseline"] = cb
            prefill.extend(entries)

    cpu = None
    if rank == 0 and not args.no_cpu:
        r = oracle_decode_rate(w, args.cpu_budget_s)
        cpu = {"value": round(r["state_gbs"], 4), "unit": "GB/s", "cores": r["cores"], "kind": "oracle",
               "sample": "first %d carried decode steps of %s (all %d heads), f64 C+numpy oracle" % (
                   r["steps"], w.name, d.B * d.Hv)}

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return
    value = by["state_rw"] * ws / (ms / 1e3) / 1e9
    achieved = alg_bytes / (ms / 1e3) / 1e9
    traffic = profiled_traffic("decode_b128_ncu.md", ["decode.cu", "common.cuh"])
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": d.B, "T": 1, "Hk": d.Hk, "Hv": d.Hv, "Dk": d.Dk, "Dv": d.Dv,
                   "K": d.K, "carried_steps": args.steps, "distinct_step_inputs": min(w.steps, args.steps +
                                                                                    args.warmup),
                   "l2": "inputs larger than L2 (512 MiB of state read+written per step)",
                   "launch": "the K steps as one captured CUDA graph, replayed once",
                   "parallelism": "replicas" if ws > 1 else "single"},
        "tokens_per_s": round(d.B * ws / (ms / 1e3), 1),
        "ms_per_step_eager": round(ms_eager, 5),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                     "algorithmic_bytes": alg_bytes, "kernel": "gdn::decode_kernel<128, false>",
                     "peak_source": peaks["source"]},
        "e2e": {"value": round(by["state_rw"] * ws / (e2e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "statistic": "median of 5 runs",
                "runs": [round(by["state_rw"] / (r / 1e3) / 1e9, 1) for r in res["e2e_runs_ms"]]},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "prefill": prefill,
        "prefill_vec": prefill_vec,
        "decode_b1": small_decode,
        "rmsnorm_gated": gated_norm,
        "decode_window": window,
        "decode_gated_norm": decode_gated,
        "backward": backward,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
