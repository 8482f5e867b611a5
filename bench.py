"""Absorbed-MLA decode benchmark: latent-cache GB/s, % of HBM peak, queries/s.

One step = one full decode (plan, query absorption, split-KV attend, merge +
up-projection) over one batch whose latent cache is resident in HBM.  The
default workload is the DeepSeek-V3 attention shape: 128 heads, 64 rows,
8192 cached tokens each, bf16 cache in 64-token pages behind a random page
table (603,979,776 cache bytes per step, larger than the 129 MB L2, so no
flush is needed between steps).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--fmt FORMAT] [--q-len T] [--h16-kernel mma|cuda_cores]

Other workloads (--workload): the V2-Lite batch and the ragged / quantized V3
decodes, several query tokens per row (v2lite_mtp, v3_mtp), the unabsorbed
prefill (v2lite_prefill, v3_prefill), the output projection (v2lite_oproj,
v3_oproj) and the fused cache producer (v3_project_prefill, v3_project_decode).

--impl reference times the fp64 CPU oracle on this host's cores on a bounded
sample of the same workload (the only place the bench runs the oracle, with
the cpu_baseline leg of the default arm).
Under torchrun (N > 1) every rank decodes its own replica batch (weak
scaling, no collective on the data path); rank 0 prints.
"""

from __future__ import annotations

import argparse
import csv
import dataclasses
import hashlib
import io
import json
import math
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "absorbed-MLA decode latent-cache GB/s (% HBM peak) and queries/s, 1 GB300"
BYTES_PER_TOKEN = {"bf16": 1152, "int8": 624, "int4": 400, "int8_token": 624, "int4_sym": 400, "int4_pe4": 400}
DESCR = {
    "v2lite_batch": "V2-Lite shape decode: H=16, B=32, seqlen 4096, contiguous bf16 latent cache",
    "v3_paged": "DeepSeek-V3 shape decode: H=128, B=64, seqlen 8192, paged bf16 latent cache "
                "(page 64, seeded random page table)",
    "v3_ragged": "DeepSeek-V3 shape ragged decode: H=128, B=128, lognormal seqlens (median 4096, clip 256..32768), "
                 "paged",
    "v3_quant": "DeepSeek-V3 shape decode over a quantized cache: H=128, B=64, seqlen 32768, paged",
    "v2lite_mtp": "V2-Lite shape, 8 causal query tokens per row: H=16, B=32, seqlen 4096, contiguous bf16 cache",
    "v3_mtp": "DeepSeek-V3 shape, 2 causal query tokens per row: H=128, B=64, seqlen 8192, paged bf16 cache",
}


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def source_digest(text: str) -> str:
    """sha256 of a CUDA source with its comments and whitespace removed, so that
    the digest changes with the code and not with its comments (no string
    literal in the hashed source holds a comment marker)."""
    code = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    code = re.sub(r"//[^\n]*", " ", code)
    code = re.sub(r"\s+", " ", code).strip()
    return hashlib.sha256(code.encode()).hexdigest()


def kernel_traffic(kind: str, fmt: str, workload: str, cache_bytes: int):
    """DRAM bytes per launch of the attend kernel from the committed ncu summary,
    or None when missing, taken on a different kernel source (code, not
    comments: see source_digest) or on another workload or size."""
    path = os.path.join(ROOT, "profiles", "attend_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        src = os.path.join(ROOT, "mla_absorbed_latent_gb300", "csrc", d["source"])
        with open(src, encoding="utf-8") as f:
            h = source_digest(f.read())
        if h != d["source_digest"] or d.get("kind") != kind or d.get("fmt", "bf16") != fmt:
            return None
        if d.get("workload_name") != workload or int(d.get("cache_bytes", -1)) != int(cache_bytes):
            return None
        return int(d["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in csv.reader(io.StringIO(out)):
            if len(row) < 9:
                continue
            try:
                sm.append(float(row[1]))
                mx.append(float(row[2]))
            except ValueError:
                continue
            for n, v in zip(names, row[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ----------------------------------------------------------------------------

def oracle_time(prob, budget_s: float, max_rows: int | None = None, outputs: dict | None = None):
    """Time the fp64 absorbed oracle over successive rows until budget_s of oracle
    work; returns (cache bytes processed, seconds, rows).  With `outputs`, each
    row's oracle output [H, 128] is stored there under its row index."""
    import oracle as O
    Wuk, Wuv = O.split_wkv_b(synth.bf16_bits_to_f32(prob.wkv), prob.H)
    qn = synth.bf16_bits_to_f32(prob.q_nope)
    qp = synth.bf16_bits_to_f32(prob.q_pe)
    done_bytes, spent, rows = 0, 0.0, 0
    bpt = BYTES_PER_TOKEN[prob.fmt]
    for b in range(prob.B):
        c, p = prob.sequence(b)
        C, P = O.dequantized_tokens(prob.fmt, synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p))
        t0 = time.perf_counter()
        out, _, _ = O.absorbed_decode(qn[b], qp[b], C, P, Wuk, Wuv, prob.scale)
        spent += time.perf_counter() - t0
        if outputs is not None:
            outputs[b] = out
        done_bytes += int(prob.seqlens[b]) * bpt
        rows += 1
        if spent >= budget_s or (max_rows is not None and rows >= max_rows):
            break
    return done_bytes, spent, rows


def oracle_time_q(prob, T, qn, qp, budget_s: float, max_rows: int | None = None, outputs: dict | None = None):
    """oracle_time for T causal query tokens per row (absorbed_attend_causal);
    outputs[b] = out [T, H, 128]."""
    import oracle as O
    Wuk, Wuv = O.split_wkv_b(synth.bf16_bits_to_f32(prob.wkv), prob.H)
    done_bytes, spent, rows = 0, 0.0, 0
    bpt = BYTES_PER_TOKEN[prob.fmt]
    for b in range(prob.B):
        c, p = prob.sequence(b)
        C, P = O.dequantized_tokens(prob.fmt, synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p))
        t0 = time.perf_counter()
        out, _ = O.absorbed_attend_causal(synth.bf16_bits_to_f32(qn[b]), synth.bf16_bits_to_f32(qp[b]), C, P, Wuk, Wuv,
                                          prob.scale)
        spent += time.perf_counter() - t0
        if outputs is not None:
            outputs[b] = out
        done_bytes += int(prob.seqlens[b]) * bpt
        rows += 1
        if spent >= budget_s or (max_rows is not None and rows >= max_rows):
            break
    return done_bytes, spent, rows


def parity_stats(got: dict, ref: dict):
    """Agreement of the timed decode's output rows with the oracle's rows (both
    {row: [H, 128] array}): largest absolute error, worst per-head relative RMS
    error, and whether every element is within 2e-2 + 1e-2 |ref| and every head
    within 1e-2 relative RMS (the parity tests' tolerance)."""
    rows = sorted(set(got) & set(ref))
    if not rows:
        return None
    max_abs, worst_rel, ok = 0.0, 0.0, True
    for b in rows:
        g = np.asarray(got[b], np.float64)
        r = np.asarray(ref[b], np.float64)
        err = np.abs(g - r)
        max_abs = max(max_abs, float(err.max()))
        ok = ok and bool(np.all(err <= 2e-2 + 1e-2 * np.abs(r))) and bool(np.all(np.isfinite(g)))
        nref = np.linalg.norm(r, axis=-1)
        live = nref > 0
        if live.any():
            rel = np.linalg.norm(g - r, axis=-1)[live] / nref[live]
            worst_rel = max(worst_rel, float(rel.max()))
    ok = ok and worst_rel <= 1e-2
    return {"rows": len(rows), "max_abs_err": max_abs, "worst_head_rel_rms": worst_rel, "within_tolerance": ok}


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise max of a list of floats over the ranks of the default process
    group (the values unchanged without one): each rank's timings, so the job is
    timed by its slowest rank."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def job_throughput(bytes_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank decodes its own replica batch (weak scaling), so
    the job moves world x the per-rank cache bytes in the slowest rank's time."""
    return bytes_per_rank * world / (ms_per_step * 1e-3) / 1e9


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------
# arms
# ----------------------------------------------------------------------------

def run_reference(args, wl, fmt):
    rank = _env_int("RANK", 0)
    if rank != 0:
        return 0
    from synth.device import problem_from_workload
    prob = problem_from_workload(wl, fmt)
    T = q_len_of(args, wl)
    if T is not None:
        qn, qp = synth.gen_queries_multi(prob.H, T, prob.seqlens, prob.seed)
        one = lambda: oracle_time_q(prob, T, qn, qp, 0.0, max_rows=1)  # noqa: E731
    else:
        one = lambda: oracle_time(prob, 0.0, max_rows=1)  # noqa: E731
    # warm-up: one row, untimed
    for _ in range(args.warmup):
        one()
    total_bytes, total_s = 0, 0.0
    for _ in range(args.steps):
        nbytes, s, _rows = one()   # one row per step
        total_bytes += nbytes
        total_s += s
    gbs = total_bytes / total_s / 1e9
    bpq = int(prob.seqlens[0]) * BYTES_PER_TOKEN[fmt]
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {DESCR.get(wl.name, '')}", "cache_fmt": fmt,
                   "sample": "one batch row (all heads, full sequence) per step"},
        "queries_per_s": gbs * 1e9 / bpq * (T or 1),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": host_cores(), "kind": "oracle",
                         "sample": f"{args.steps} rows of {wl.name}, one per step, fp64 numpy absorbed oracle"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


SCRUB_BELOW = 512 * 2 ** 20   # cache streams under this are timed with an L2 scrub between steps
SCRUB_BYTES = 256 * 2 ** 20   # > the 129 MB L2


def timed_steps(step, steps, stream, scrub_buf=None):
    """Mean ms of `steps` steps on `stream`: back to back between two events, or,
    with scrub_buf, each step alone between its own events after writing
    scrub_buf (a buffer larger than L2), so no step finds the cache in L2."""
    import torch
    if scrub_buf is None:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for k in range(steps):
        scrub_buf.zero_()
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    return float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))


def l2_note(cache_bytes, scrub):
    if scrub:
        return (f"{SCRUB_BYTES >> 20} MB L2 scrub before every timed step (cache stream {cache_bytes / 1e6:.0f} MB, "
                f"near the 129 MB L2); each step timed alone")
    return "inputs larger than L2 (cache stream per step > 129 MB), no flush"


def q_len_of(args, wl):
    """Query tokens per row when the step runs through mla_decode_q (None: the
    single-query chain)."""
    if args.q_len is not None:
        return args.q_len
    return wl.q_len if wl.q_len > 1 else None


E2E_PIPELINE_BYTES = 1 << 20  # a step's copies from which the end-to-end loop overlaps them with the neighbours


def e2e_loop(torch, stream, steps, h_in, dev_in, h_out, dev_out, run):
    """(ms per step, how the copies ran) of the end-to-end loop through the
    public call.  Every step copies its inputs from pinned host memory and its
    result back; with at least E2E_PIPELINE_BYTES of copies per step they run on
    copy streams overlapping the neighbouring steps (pipelined_e2e), else in
    line on the compute stream (measured on GB300: overlapping 5 MB per step
    raises the v3_paged figure by 18 %, overlapping 0.3 MB lowers the v2lite one,
    the cross-stream events costing more than the copies they hide)."""
    nbytes = sum(t.numel() * t.element_size() for t in h_in) + h_out.numel() * h_out.element_size()
    if nbytes >= E2E_PIPELINE_BYTES:
        return (pipelined_e2e(torch, stream, steps, h_in, dev_in, h_out, dev_out, run),
                "every step: its query from pinned host memory in and its output to pinned host memory out, on copy "
                "streams with double-buffered device tensors (overlapping the neighbouring steps)")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        for h, d in zip(h_in, dev_in[0]):
            d.copy_(h, non_blocking=True)
        run(dev_in[0], dev_out[0])
        h_out.copy_(dev_out[0], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    return (e0.elapsed_time(e1) / steps,
            "every step: its query from pinned host memory in and its output to pinned host memory out, in line on "
            "the compute stream (under 1 MB of copies per step)")


def pipelined_e2e(torch, stream, steps, h_in, dev_in, h_out, dev_out, run):
    """ms per step of a serving loop through the public call: every step copies
    its inputs from pinned host memory and its result back to pinned host
    memory.  The copies run on their own streams (host-to-device, device-to-host)
    with the device buffers doubled, so step k+1's inputs arrive and step k's
    result leaves while the GPU computes (a step's own copies never overlap its
    call).  h_in: pinned host inputs; dev_in: two lists of device inputs (one per
    buffer); dev_out: two device results; run(inputs, result) enqueues one call
    on `stream`."""
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    h2d.wait_stream(stream)
    d2h.wait_stream(stream)

    def load(k):
        i = k % 2
        with torch.cuda.stream(h2d):
            if k >= 2:
                h2d.wait_event(ev_done[i])  # the call of step k - 2 has read buffer i
            for h, d in zip(h_in, dev_in[i]):
                d.copy_(h, non_blocking=True)
            ev_in[i].record(h2d)

    load(0)
    for k in range(steps):
        i = k % 2
        if k + 1 < steps:
            load(k + 1)
        stream.wait_event(ev_in[i])
        if k >= 2:
            stream.wait_event(ev_out[i])  # step k - 2's result has been read back
        run(dev_in[i], dev_out[i])
        ev_done[i].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev_done[i])
            h_out.copy_(dev_out[i], non_blocking=True)
            ev_out[i].record(d2h)
    stream.wait_stream(h2d)
    stream.wait_stream(d2h)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_ours_q(args, wl, fmt, T):
    """One step = one mla_decode_q call: T causal query tokens per row."""
    import torch
    torch.cuda.set_device(_env_int("LOCAL_RANK", 0))
    import mla_absorbed_latent_gb300 as mla
    from synth.device import DeviceDecode, bits_to_device, problem_from_workload
    prob = problem_from_workload(wl, fmt)
    dev = DeviceDecode(prob)
    H, B = prob.H, prob.B
    qn, qp = synth.gen_queries_multi(H, T, prob.seqlens, prob.seed)
    d_qn, d_qp = bits_to_device(qn), bits_to_device(qp)
    ws_bytes = mla.mla_decode_q_workspace_bytes(B, H, T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    cache_bytes = int(np.sum(prob.seqlens)) * BYTES_PER_TOKEN[fmt]

    def step():
        mla.mla_decode_q(d_qn, d_qp, dev.W_UK, dev.W_UV, H, T, dev.cache, dev.page_table, prob.max_pages,
                         dev.seqlens, B, prob.scale, ws, ws_bytes, out, None, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, info = mla.mla_get_device_status()
    if st != mla.MLA_OK:
        raise RuntimeError(f"device status after warm-up: {mla.mla_status_string(st)} ({info})")
    scrub = cache_bytes < SCRUB_BELOW
    scrub_buf = torch.empty(SCRUB_BYTES, dtype=torch.uint8, device="cuda") if scrub else None
    clocks = ClockSampler(torch.cuda.current_device())
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ms_step = timed_steps(step, args.steps, stream, scrub_buf)
    clock_info = clocks.stop()
    # each call alone (events between the calls; scrubbed when the step is)
    call_ms = timed_steps(step, args.steps, stream, scrub_buf) if not scrub else ms_step
    st, info = mla.mla_get_device_status()
    if st != mla.MLA_OK:
        raise RuntimeError(f"device status after timing: {mla.mla_status_string(st)} ({info})")

    h_qn, h_qp = d_qn.cpu().pin_memory(), d_qp.cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))

    def call_q(ins, res):
        mla.mla_decode_q(ins[0], ins[1], dev.W_UK, dev.W_UV, H, T, dev.cache, dev.page_table, prob.max_pages,
                         dev.seqlens, B, prob.scale, ws, ws_bytes, res, None, stream)

    e2e_ms, e2e_copies = e2e_loop(torch, stream, e2e_steps, [h_qn, h_qp],
                                  [[d_qn, d_qp], [torch.empty_like(d_qn), torch.empty_like(d_qp)]], h_out,
                                  [out, torch.empty_like(out)], call_q)

    cpu, parity = None, None
    if not args.no_cpu_baseline:
        ref_rows = {}
        nbytes, secs, rows = oracle_time_q(prob, T, qn, qp, args.cpu_seconds, outputs=ref_rows)
        cpu = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"{rows} of {B} rows of {wl.name} ({T} queries x {H} heads, full sequences), fp64 numpy "
                         f"causal absorbed oracle, {secs:.1f} s"}
        try:
            got = synth.bf16_bits_to_f32(h_out.view(torch.int16).numpy().view(np.uint16))
            parity = parity_stats({b: got[b] for b in ref_rows}, ref_rows)
        except Exception as exc:
            parity = {"error": repr(exc), "within_tolerance": False}

    hbm, tf_burst, tf_sus, peak_src = load_peaks()
    flops_tok = 2 * H * T * (576 + 512)  # useful work: T queries of H heads per cached token
    ai = flops_tok / BYTES_PER_TOKEN[fmt]
    ridge = tf_burst * 1e12 / (hbm * 1e9)
    gbs = cache_bytes / (call_ms * 1e-3) / 1e9
    tflops = cache_bytes / BYTES_PER_TOKEN[fmt] * flops_tok / (call_ms * 1e-3) / 1e12
    if ai < ridge:
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "traffic": None,
                "peak_source": peak_src, "tensor_tflops": tflops, "arith_intensity": ai}
    else:
        roof = {"bound": "tensor", "achieved": tflops, "peak": tf_burst, "unit": "TFLOP/s", "frac": tflops / tf_burst,
                "traffic": None, "peak_source": peak_src + " (bf16, burst)", "hbm_gbs": gbs, "arith_intensity": ai}
    roof["timed"] = "the whole mla_decode_q call (plan, q-absorb, attend, merge): a lower bound of the attend kernel's"
    G = 128 // H
    line = {
        "metric": METRIC, "value": cache_bytes / (ms_step * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {DESCR.get(wl.name, '')}", "H": H, "B": B, "q_len": T,
                   "seqlen": int(prob.seqlens.max()), "cache_fmt": fmt, "cache_bytes_per_step": cache_bytes,
                   "l2": l2_note(cache_bytes, scrub),
                   "passes_over_cache": -(-T // G),
                   "attend_kernel": f"tcgen05, {min(T, G)} of {G} token lanes per pass in use"},
        "queries_per_s": B * T / (ms_step * 1e-3),
        "roofline": roof,
        "call_ms": call_ms,
        "cpu_baseline": cpu,
        "parity": parity,
        "e2e": {"value": cache_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h_qn.numel() * 2 + h_qp.numel() * 2, "d2h_bytes_per_step": h_out.numel() * 2,
                "copies": e2e_copies},
        "gpu_launches": 5 * args.steps,  # plan, q-absorb, attend, merge, exact-recompute check
        "clocks": clock_info,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, wl, fmt):
    import torch
    import torch.distributed as dist
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local = _env_int("LOCAL_RANK", 0)
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    import mla_absorbed_latent_gb300 as mla
    from synth.device import DeviceDecode, problem_from_workload

    prob = problem_from_workload(wl, fmt)
    dev = DeviceDecode(prob)
    H, B = prob.H, prob.B
    stream = torch.cuda.current_stream()
    cache_bytes = int(np.sum(prob.seqlens)) * BYTES_PER_TOKEN[fmt]
    if H == 16:
        mla.mla_decode_select_kernel(16, {"mma": mla.MLA_KERNEL_MMA,
                                          "cuda_cores": mla.MLA_KERNEL_CUDA_CORES}[args.h16_kernel])
    kind = mla.mla_decode_kernel_kind(H) if fmt == "bf16" else mla.MLA_KERNEL_TCGEN05
    kind_name = {mla.MLA_KERNEL_TCGEN05: "tcgen05", mla.MLA_KERNEL_MMA: "mma.sync",
                 mla.MLA_KERNEL_CUDA_CORES: "cuda-core"}[kind]

    def step(ev=None):
        # ev: 5 events bracketing plan | absorb_q | attend | combine (the step-wise
        # calls); without events the step is one mla_decode call (the same kernels)
        p = prob
        if ev is None:
            dev.decode(stream)
            return
        if ev is not None:
            ev[0].record(stream)
        mla.mla_decode_plan(H, fmt, dev.seqlens, B, p.max_pages, dev.workspace, dev.ws_bytes, stream)
        if ev is not None:
            ev[1].record(stream)
        mla.mla_decode_absorb_q(dev.q_nope, dev.q_pe, dev.W_UK, H, B, dev.workspace, dev.ws_bytes, stream)
        if ev is not None:
            ev[2].record(stream)
        mla.mla_decode_attend(H, dev.cache, dev.page_table, p.max_pages, dev.seqlens, B, p.scale, dev.workspace,
                              dev.ws_bytes, stream)
        if ev is not None:
            ev[3].record(stream)
        mla.mla_decode_combine(dev.W_UV, H, B, dev.workspace, dev.ws_bytes, dev.out, None, stream)
        if ev is not None:
            ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, info = mla.mla_get_device_status()
    if st != mla.MLA_OK:
        raise RuntimeError(f"device status after warm-up: {mla.mla_status_string(st)} ({info})")

    attend_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    scrub = cache_bytes < SCRUB_BELOW
    scrub_buf = torch.empty(SCRUB_BYTES, dtype=torch.uint8, device="cuda") if scrub else None
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    # no events between the launches of a step: consecutive kernels overlap their prologues
    elapsed_ms = timed_steps(step, args.steps, stream, scrub_buf) * args.steps
    clock_info = clocks.stop() if clocks else None
    # per-stage times (and the attend time of the roofline) from a second run of
    # the same steps with events between the launches
    for k in range(args.steps):
        if scrub_buf is not None:
            scrub_buf.zero_()
        step(attend_ev[k])
    torch.cuda.synchronize()
    attend_ms = float(np.mean([e[2].elapsed_time(e[3]) for e in attend_ev]))
    stage_ms = {name: float(np.mean([e[k].elapsed_time(e[k + 1]) for e in attend_ev]))
                for k, name in enumerate(("plan", "absorb_q", "attend", "combine"))}
    if world > 1:
        elapsed_ms, attend_ms = max_over_ranks([elapsed_ms, attend_ms], dist, device="cuda")
        dist.barrier()
    st, info = mla.mla_get_device_status()
    if st != mla.MLA_OK:
        raise RuntimeError(f"device status after timing: {mla.mla_status_string(st)} ({info})")

    # end to end through the public call: pinned host query in, host result out
    h_qn = dev.q_nope.cpu().pin_memory()
    h_qp = dev.q_pe.cpu().pin_memory()
    h_out = torch.empty(dev.out.shape, dtype=dev.out.dtype).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    p_ = dev.prob

    def call(ins, res):
        mla.mla_decode(ins[0], ins[1], dev.W_UK, dev.W_UV, p_.H, dev.cache, dev.page_table, p_.max_pages,
                       dev.seqlens, p_.B, p_.scale, dev.workspace, dev.ws_bytes, res, stream)

    e2e_ms, e2e_copies = e2e_loop(torch, stream, e2e_steps, [h_qn, h_qp],
                                  [[dev.q_nope, dev.q_pe], [torch.empty_like(dev.q_nope), torch.empty_like(dev.q_pe)]],
                                  h_out, [dev.out, torch.empty_like(dev.out)], call)
    h2d = h_qn.numel() * 2 + h_qp.numel() * 2
    d2h = h_out.numel() * 2

    # CPU oracle on the host cores (rank 0, one GPU only), bounded sample
    cpu, parity = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ref_rows = {}
        nbytes, secs, rows = oracle_time(prob, args.cpu_seconds, outputs=ref_rows)
        cpu = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"{rows} of {B} rows of {wl.name} (all {H} heads, full sequences), fp64 numpy absorbed "
                         f"oracle, {secs:.1f} s"}
        try:  # the same rows of the last timed end-to-end decode against the oracle
            got = synth.bf16_bits_to_f32(h_out.view(torch.int16).numpy().view(np.uint16))
            parity = parity_stats({b: got[b] for b in ref_rows}, ref_rows)
        except Exception as exc:  # a broken comparison is reported, not taken for a skipped one
            parity = {"error": repr(exc), "within_tolerance": False}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    hbm, tf_burst, tf_sus, peak_src = load_peaks()
    ms_step = elapsed_ms / args.steps
    total_bytes = cache_bytes * world
    value = job_throughput(cache_bytes, world, ms_step)
    attend_gbs = cache_bytes / (attend_ms * 1e-3) / 1e9
    flops_tok = 2 * H * (576 + 512)
    traffic = kernel_traffic(kind_name, fmt, wl.name, cache_bytes)
    if kind == mla.MLA_KERNEL_MMA:
        # 16 heads: 30 FLOP per cache byte, far below any tensor ridge; the cache stream binds
        tflops = cache_bytes / BYTES_PER_TOKEN[fmt] * flops_tok / (attend_ms * 1e-3) / 1e12
        roof = {"bound": "hbm", "achieved": attend_gbs, "peak": hbm, "unit": "GB/s", "frac": attend_gbs / hbm,
                "traffic": traffic, "peak_source": peak_src, "tensor_tflops": tflops,
                "arith_intensity": flops_tok / BYTES_PER_TOKEN[fmt]}
    elif kind == mla.MLA_KERNEL_TCGEN05:
        tflops = cache_bytes / BYTES_PER_TOKEN[fmt] * flops_tok / (attend_ms * 1e-3) / 1e12
        ai = flops_tok / BYTES_PER_TOKEN[fmt]            # FLOP per cache byte
        ridge = tf_burst * 1e12 / (hbm * 1e9)
        if ai < ridge:  # bf16 pages (AI ~242): the cache stream binds
            roof = {"bound": "hbm", "achieved": attend_gbs, "peak": hbm, "unit": "GB/s", "frac": attend_gbs / hbm,
                    "traffic": traffic, "peak_source": peak_src, "tensor_tflops": tflops,
                    "tensor_frac": tflops / tf_burst, "arith_intensity": ai}
        else:  # quantized pages: the bf16 MMAs on the dequantized tiles bind
            roof = {"bound": "tensor", "achieved": tflops, "peak": tf_burst, "unit": "TFLOP/s",
                    "frac": tflops / tf_burst, "traffic": traffic, "peak_source": peak_src + " (bf16, burst)",
                    "hbm_gbs": attend_gbs, "hbm_frac": attend_gbs / hbm, "arith_intensity": ai}
    else:
        # CUDA-core kernel: fp32 FMA bound; peak = SMs x 128 FMA/clk x 2 FLOP x max SM clock
        props = torch.cuda.get_device_properties(torch.cuda.current_device())
        sm_max = (clock_info or {}).get("sm_max_mhz", 2070.0)
        alu_peak = props.multi_processor_count * 128 * 2 * sm_max * 1e6 / 1e12
        achieved = cache_bytes / BYTES_PER_TOKEN[fmt] * flops_tok / (attend_ms * 1e-3) / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
                "frac": achieved / alu_peak, "traffic": traffic, "peak_source": "derived: SMs*128 FMA*2*max clock",
                "hbm_gbs": attend_gbs, "hbm_frac": attend_gbs / hbm}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {DESCR.get(wl.name, '')}", "H": H, "B": B,
                   "seqlen": int(prob.seqlens.max()), "cache_fmt": fmt, "cache_bytes_per_step": cache_bytes,
                   "l2": l2_note(cache_bytes, scrub),
                   "parallelism": f"replicas x{world} (batch-sharded, no collective)",
                   "attend_kernel": kind_name},
        "pct_hbm_peak": 100.0 * value / (hbm * world),
        "queries_per_s": B * world / (ms_step * 1e-3),
        "roofline": roof,
        "attend_ms": attend_ms,
        "stage_ms": stage_ms,  # mean per-stage times of one step, from events recorded between its launches
        "cpu_baseline": cpu,
        "parity": parity,  # the oracle rows of cpu_baseline against the timed decode's output
        "e2e": {"value": total_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "copies": e2e_copies},
        # plan, absorb_q, attend, combine (merge + up-projection) and, after the tcgen05 kernel, the exact-recompute check
        "gpu_launches": (5 if kind == mla.MLA_KERNEL_TCGEN05 else 4) * args.steps,
        "clocks": clock_info,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------
# the cache producer (down-projection + RMSNorm + RoPE + page write), a second workload
# ----------------------------------------------------------------------------
PROJECT_METRIC = "fused cache producer (kv down-projection, RMSNorm, RoPE, page write) tokens/s, 1 GB300"
PROJECT = {
    # name: (hidden, B, T, description)
    "v3_project_prefill": (7168, 16, 2048, "DeepSeek-V3 width (hidden 7168): 16 rows x 2048 new tokens "
                                           "(a 32,768-token prefill chunk) into a paged pool"),
    "v3_project_decode": (7168, 64, 1, "DeepSeek-V3 width (hidden 7168): one new token for each of 64 rows "
                                       "(the decode-time append)"),
}
PROJECT_EPS, PROJECT_THETA = 1e-6, 10000.0


def _project_problem(name, fmt):
    hidden, B, T, _ = PROJECT[name]
    seed = 40
    w, g = synth.gen_project_weights(hidden, seed)
    x = np.stack([synth.gen_hidden(hidden, seed, b, T) for b in range(B)])
    pos0 = np.full(B, 8192 - T, dtype=np.int32) if T < 64 else np.zeros(B, dtype=np.int32)
    table, num_pages = synth.make_page_table(pos0 + T, seed, True)
    return hidden, B, T, w, g, x, pos0, table, num_pages


def project_oracle_time(name, fmt, budget_s):
    """fp64 oracle producer over successive tokens until budget_s of oracle work;
    returns (tokens, seconds)."""
    import oracle as O
    hidden, B, T, w, g, x, pos0, _, _ = _project_problem(name, fmt)
    wf, gf = synth.bf16_bits_to_f32(w), synth.bf16_bits_to_f32(g)
    done, spent = 0, 0.0
    for b in range(B):
        for t0 in range(0, T, 64):
            xs = synth.bf16_bits_to_f32(x[b, t0:t0 + 64])
            t1 = time.perf_counter()
            O.project_latent(xs, wf, gf, pos0[b] + np.arange(t0, t0 + len(xs)), PROJECT_EPS, PROJECT_THETA)
            spent += time.perf_counter() - t1
            done += len(xs)
            if spent >= budget_s:
                return done, spent
    return done, spent


def project_work(ntok: int, hidden: int, fmt: str):
    """Algorithmic FLOPs and bytes of one producer call: the projection (2 x 576 x
    hidden per token); the weight once, the inputs and the page writes."""
    flops = 2.0 * ntok * 576 * hidden
    nbytes = 576 * hidden * 2 + ntok * hidden * 2 + ntok * BYTES_PER_TOKEN[fmt]
    return flops, nbytes


def project_roofline(flops: float, nbytes: int, ms: float, peaks):
    """The binding roofline of a producer call: the tensor peak when its FLOP per
    byte is above the ridge of the measured peaks, else the HBM copy bandwidth."""
    hbm, tf_burst, _tf_sus, peak_src = peaks
    tflops = flops / (ms * 1e-3) / 1e12
    gbs = nbytes / (ms * 1e-3) / 1e9
    if flops / nbytes > tf_burst * 1e12 / (hbm * 1e9):
        return {"bound": "tensor", "achieved": tflops, "peak": tf_burst, "unit": "TFLOP/s", "frac": tflops / tf_burst,
                "traffic": None, "peak_source": peak_src + " (bf16, burst)", "hbm_gbs": gbs}
    return {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "traffic": None,
            "peak_source": peak_src, "tensor_tflops": tflops}


def run_project(args, name, fmt):
    import torch
    torch.cuda.set_device(_env_int("LOCAL_RANK", 0))
    import mla_absorbed_latent_gb300 as mla
    from synth.device import bits_to_device
    hidden, B, T, w, g, x, pos0, table, num_pages = _project_problem(name, fmt)
    ntok = B * T
    dev_x, dev_w, dev_g = bits_to_device(x), bits_to_device(w), bits_to_device(g)
    pool = torch.zeros(num_pages * mla.mla_cache_page_bytes(fmt), dtype=torch.uint8, device="cuda")
    cache = mla.cache_struct(fmt, num_pages, pool)
    pt = torch.from_numpy(table).cuda()
    pos = torch.from_numpy(pos0).cuda()
    ksplit = args.k_splits
    ws_bytes = mla.mla_cache_project_workspace_bytes(B, T, hidden, ksplit)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")  # > L2: scrubbed between steps

    def call(xin=dev_x, latent=None):
        mla.mla_cache_project_append(cache, xin, hidden, dev_w, dev_g, PROJECT_EPS, PROJECT_THETA, pt,
                                     table.shape[1], pos, B, T, latent, ksplit, ws, ws_bytes, stream)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    st, info = mla.mla_get_device_status()
    if st != mla.MLA_OK:
        raise RuntimeError(f"device status after warm-up: {mla.mla_status_string(st)} ({info})")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device())
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for k in range(args.steps):
        flush.zero_()
        ev[k][0].record(stream)
        call()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    st, info = mla.mla_get_device_status()
    if st != mla.MLA_OK:
        raise RuntimeError(f"device status after timing: {mla.mla_status_string(st)} ({info})")
    ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))

    # end to end: x from pinned host memory in, the bf16 payload out, every step
    h_x = dev_x.cpu().pin_memory()
    lat = torch.empty((B, T, 576), dtype=torch.bfloat16, device="cuda")
    h_lat = torch.empty(lat.shape, dtype=lat.dtype).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(args.steps, 10))
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(e2e_steps):
        dev_x.copy_(h_x, non_blocking=True)
        call(latent=lat)
        h_lat.copy_(lat, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    cpu = None
    if not args.no_cpu_baseline:
        n, secs = project_oracle_time(name, fmt, min(args.cpu_seconds, 10.0))
        cpu = {"value": n / secs, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"{n} of {ntok} tokens of {name}, fp64 numpy oracle producer, {secs:.1f} s"}

    flops, nbytes = project_work(ntok, hidden, fmt)
    roof = project_roofline(flops, nbytes, ms, load_peaks())
    line = {
        "metric": PROJECT_METRIC, "value": ntok / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{name}: {PROJECT[name][3]}", "hidden": hidden, "B": B, "T": T, "cache_fmt": fmt,
                   "k_splits": ksplit or "auto", "k_split_workspace_bytes": ws_bytes, "l2": "256 MB scrub between timed steps",
                   "algorithmic_bytes": nbytes, "flops": flops},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": ntok / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h_x.numel() * 2,
                "d2h_bytes_per_step": h_lat.numel() * 2},
        "gpu_launches": (2 if ws_bytes > 0 else 1) * args.steps,  # the projection (and the finishing kernel of a split)
        "clocks": clock_info,
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------
# the unabsorbed causal prefill (expanded keys and values), a third workload
# ----------------------------------------------------------------------------
PREFILL_METRIC = "unabsorbed causal MLA prefill query tokens/s (expansion + attention), 1 GB300"
PREFILL = {
    # name: (H, B, n = T, seed, description)
    "v2lite_prefill": (16, 4, 4096, 60, "V2-Lite shape: H=16, 4 rows x a 4096-token causal prefill, paged bf16 cache"),
    "v3_prefill": (128, 1, 8192, 61, "DeepSeek-V3 shape: H=128, one 8192-token causal prefill, paged bf16 cache"),
}


def prefill_work(H, B, n, T):
    """Algorithmic FLOPs of one prefill call: the expansion (2 x 256 x 512 per
    cached token and head) and the causal attention (2 x (192 + 128) per visible
    (query, key) pair and head)."""
    pairs = B * sum(n - T + t + 1 for t in range(T))
    return 2.0 * B * n * H * 256 * 512 + 2.0 * H * (192 + 128) * pairs


def run_prefill(args, name):
    import torch
    torch.cuda.set_device(_env_int("LOCAL_RANK", 0))
    import mla_absorbed_latent_gb300 as mla
    from synth.device import DeviceDecode, bits_to_device, make_problem
    H, B, n, seed, desc = PREFILL[name]
    T = n
    prob = make_problem(H, [n] * B, seed)
    dev = DeviceDecode(prob)
    qn, qp = synth.gen_queries_multi(H, T, prob.seqlens, seed)
    d_qn, d_qp = bits_to_device(qn), bits_to_device(qp)
    ws_bytes = mla.mla_prefill_workspace_bytes(B, H, prob.max_pages)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        mla.mla_prefill(d_qn, d_qp, dev.wkv, H, T, dev.cache, dev.page_table, prob.max_pages, dev.seqlens, B,
                        prob.scale, ws, ws_bytes, out, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, info = mla.mla_get_device_status()
    if st != mla.MLA_OK:
        raise RuntimeError(f"device status after warm-up: {mla.mla_status_string(st)} ({info})")
    clocks = ClockSampler(torch.cuda.current_device())
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ms = timed_steps(step, args.steps, stream, None)  # the workspace (expanded K/V) is far larger than L2
    clock_info = clocks.stop()
    # the same queries through the absorbed multi-query decode, for comparison
    wq = mla.mla_decode_q_workspace_bytes(B, H, T)
    wsq = torch.empty(wq, dtype=torch.uint8, device="cuda")
    outq = torch.empty_like(out)

    def step_abs():
        mla.mla_decode_q(d_qn, d_qp, dev.W_UK, dev.W_UV, H, T, dev.cache, dev.page_table, prob.max_pages, dev.seqlens,
                         B, prob.scale, wsq, wq, outq, None, stream)

    step_abs()
    torch.cuda.synchronize()
    ms_abs = timed_steps(step_abs, max(1, min(args.steps, 3)), stream, None)
    st, info = mla.mla_get_device_status()
    if st != mla.MLA_OK:
        raise RuntimeError(f"device status after timing: {mla.mla_status_string(st)} ({info})")

    h_qn, h_qp = d_qn.cpu().pin_memory(), d_qp.cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(args.steps, 10))
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(e2e_steps):
        d_qn.copy_(h_qn, non_blocking=True)
        d_qp.copy_(h_qp, non_blocking=True)
        step()
        h_out.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    cpu, parity = None, None
    if not args.no_cpu_baseline:
        # the oracle's expand-then-attend path on a bounded sample: the last few
        # queries of row 0 (every head, full causal views)
        import oracle as O
        Wuk, Wuv = O.split_wkv_b(synth.bf16_bits_to_f32(prob.wkv), H)
        c, p = prob.sequence(0)
        C, P = synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p)
        k = 16
        t_start = time.perf_counter()
        ref = O.naive_attend_causal(synth.bf16_bits_to_f32(qn[0, T - k:]), synth.bf16_bits_to_f32(qp[0, T - k:]),
                                    C, P, Wuk, Wuv, prob.scale, q_pos=np.arange(n - k, n))
        secs = time.perf_counter() - t_start
        cpu = {"value": k / secs, "unit": "query tokens/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"the last {k} of {T} queries of row 0 of {name} (all {H} heads, full causal views), fp64 "
                         f"numpy expand-then-attend oracle, {secs:.1f} s"}
        got = synth.bf16_bits_to_f32(h_out.view(torch.int16).numpy().view(np.uint16))[0, T - k:]
        parity = parity_stats({0: got}, {0: ref})

    flops = prefill_work(H, B, n, T)
    hbm, tf_burst, _tf_sus, peak_src = load_peaks()
    tflops = flops / (ms * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": tflops, "peak": tf_burst, "unit": "TFLOP/s", "frac": tflops / tf_burst,
            "traffic": None, "peak_source": peak_src + " (bf16, burst)",
            "timed": "the whole mla_prefill call (expansion and attention kernels)"}
    line = {
        "metric": PREFILL_METRIC, "value": B * T / (ms * 1e-3), "unit": "query tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{name}: {desc}", "H": H, "B": B, "seqlen": n, "q_len": T, "cache_fmt": "bf16",
                   "flops": flops, "l2": "expanded keys/values larger than L2, no flush"},
        "roofline": roof,
        "absorbed_ms": ms_abs,  # the same causal queries through mla_decode_q
        "cpu_baseline": cpu,
        "parity": parity,
        "e2e": {"value": B * T / (e2e_ms * 1e-3), "unit": "query tokens/s",
                "h2d_bytes_per_step": h_qn.numel() * 2 + h_qp.numel() * 2, "d2h_bytes_per_step": h_out.numel() * 2},
        "gpu_launches": 2 * args.steps,  # expansion, attention
        "clocks": clock_info,
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------
# the output projection after the value up-projection (y = o Wo^T)
# ----------------------------------------------------------------------------
OPROJ_METRIC = "MLA output projection (o Wo^T) weight-stream GB/s (% HBM peak), 1 GB300"
OPROJ = {
    # name: (H, R rows, hidden, description)
    "v3_oproj": (128, 64, 7168, "DeepSeek-V3 shape: 64 decode rows x (128 heads x 128) -> hidden 7168"),
    "v2lite_oproj": (16, 32, 2048, "V2-Lite shape: 32 decode rows x (16 heads x 128) -> hidden 2048"),
}


def run_oproj(args, name):
    import torch
    torch.cuda.set_device(_env_int("LOCAL_RANK", 0))
    import mla_absorbed_latent_gb300 as mla
    from synth.device import bits_to_device
    H, R, hidden, desc = OPROJ[name]
    rng = np.random.default_rng(130)
    o_bits = synth.f32_to_bf16_bits(rng.standard_normal((R, H, 128)).astype(np.float32))
    wo = synth.gen_out_weights(H, hidden, seed=131)
    d_o, d_w = bits_to_device(o_bits), bits_to_device(wo)
    y = torch.empty((R, hidden), dtype=torch.bfloat16, device="cuda")
    ws_bytes = mla.mla_output_projection_workspace_bytes(R, H, hidden)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    w_bytes = hidden * H * 128 * 2
    scrub = torch.empty(SCRUB_BYTES, dtype=torch.uint8, device="cuda") if w_bytes < SCRUB_BELOW else None

    def step():
        mla.mla_output_projection(d_o, d_w, R, H, hidden, y, ws, ws_bytes, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    ms = timed_steps(step, args.steps, stream, scrub)
    clock_info = clocks.stop()
    st, info = mla.mla_get_device_status()
    if st != mla.MLA_OK:
        raise RuntimeError(f"device status after timing: {mla.mla_status_string(st)} ({info})")
    h_o = d_o.cpu().pin_memory()
    h_y = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(5):
        d_o.copy_(h_o, non_blocking=True)
        step()
        h_y.copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / 5
    cpu, parity = None, None
    if not args.no_cpu_baseline:
        import oracle as O
        t0 = time.perf_counter()
        ref = O.output_projection(synth.bf16_bits_to_f32(o_bits), synth.bf16_bits_to_f32(wo))
        secs = time.perf_counter() - t0
        cpu = {"value": w_bytes / secs / 1e9, "unit": "GB/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"the whole {name} projection, fp64 numpy oracle, {secs:.2f} s"}
        got = synth.bf16_bits_to_f32(h_y.view(torch.int16).numpy().view(np.uint16))
        parity = parity_stats({0: got}, {0: ref})
    hbm, *_rest = load_peaks()
    gbs = w_bytes / (ms * 1e-3) / 1e9
    line = {
        "metric": OPROJ_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{name}: {desc}", "H": H, "R": R, "hidden": hidden, "weight_bytes": w_bytes,
                   "k_splits": "by size", "l2": l2_note(w_bytes, scrub is not None)},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "traffic": None,
                     "peak_source": load_peaks()[3], "algorithmic_bytes": "the weight (hidden x H*128 bf16)"},
        "cpu_baseline": cpu,
        "parity": parity,
        "e2e": {"value": w_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h_o.numel() * 2,
                "d2h_bytes_per_step": h_y.numel() * 2},
        "gpu_launches": args.steps,
        "clocks": clock_info,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="v3_paged",
                    choices=sorted(DESCR) + sorted(PROJECT) + sorted(PREFILL) + sorted(OPROJ))
    ap.add_argument("--fmt", default=None, choices=sorted(BYTES_PER_TOKEN))
    ap.add_argument("--seqlen", type=int, default=None,
                    help="override every row's length (a smaller case of the workload's shape, e.g. for ncu)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--k-splits", type=int, default=0,
                    help="producer workloads: CTA pairs per 128-token tile over the hidden dimension (0 = by size)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--h16-kernel", choices=["mma", "cuda_cores"], default="mma",
                    help="attend kernel of the 16-head decode workloads (the warp-level MMA kernel, or the "
                         "CUDA-core baseline)")
    ap.add_argument("--q-len", type=int, default=None,
                    help="query tokens per row through mla_decode_q (default: the workload's; 1 runs the single-"
                         "query step of an H=16 workload on the tensor cores)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload in OPROJ:
        if args.impl == "reference":
            return 0 if _env_int("RANK", 0) != 0 else print(json.dumps(
                {"impl": "reference", "unavailable": "the output projection has no separate reference arm; its oracle "
                 "timing is the cpu_baseline of the default arm"})) or 0
        return run_oproj(args, args.workload)
    if args.workload in PREFILL:
        if args.impl == "reference":
            if _env_int("RANK", 0) != 0:
                return 0
            import oracle as O
            H, B, n, seed, desc = PREFILL[args.workload]
            from synth.device import make_problem
            prob = make_problem(H, [n] * B, seed)
            qn, qp = synth.gen_queries_multi(H, n, prob.seqlens, seed)
            Wuk, Wuv = O.split_wkv_b(synth.bf16_bits_to_f32(prob.wkv), H)
            c, p = prob.sequence(0)
            k = 16
            t0 = time.perf_counter()
            O.naive_attend_causal(synth.bf16_bits_to_f32(qn[0, n - k:]), synth.bf16_bits_to_f32(qp[0, n - k:]),
                                  synth.bf16_bits_to_f32(c), synth.bf16_bits_to_f32(p), Wuk, Wuv, prob.scale,
                                  q_pos=np.arange(n - k, n))
            v = k / (time.perf_counter() - t0)
            print(json.dumps({"impl": "reference", "metric": PREFILL_METRIC, "value": v, "unit": "query tokens/s",
                              "n_gpus": args.gpus, "steps": 1, "warmup": 0, "higher_is_better": True, "dtype": "f64",
                              "data": "synthetic", "config": {"workload": args.workload},
                              "cpu_baseline": {"value": v, "unit": "query tokens/s", "cores": host_cores(),
                                               "kind": "oracle", "sample": f"the last {k} queries of row 0"},
                              "e2e": {"value": v, "unit": "query tokens/s", "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 0}}), flush=True)
            return 0
        return run_prefill(args, args.workload)
    if args.workload in PROJECT:
        fmt = args.fmt or "bf16"
        if args.impl == "reference":
            if _env_int("RANK", 0) != 0:
                return 0
            n, secs = project_oracle_time(args.workload, fmt, 10.0)
            print(json.dumps({"impl": "reference", "metric": PROJECT_METRIC, "value": n / secs, "unit": "tokens/s",
                              "n_gpus": args.gpus, "steps": 1, "warmup": 0, "higher_is_better": True,
                              "dtype": "f64", "data": "synthetic", "config": {"workload": args.workload},
                              "cpu_baseline": {"value": n / secs, "unit": "tokens/s", "cores": host_cores(),
                                               "kind": "oracle", "sample": f"{n} tokens"},
                              "e2e": {"value": n / secs, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 0}}), flush=True)
            return 0
        return run_project(args, args.workload, fmt)
    wl = synth.get_workload(args.workload)
    if args.seqlen is not None:
        if wl.ragged or args.seqlen < 1:
            raise SystemExit("--seqlen needs a uniform-length workload and a positive length")
        wl = dataclasses.replace(wl, seqlen=args.seqlen)
    fmt = args.fmt or wl.fmts[0]
    if args.impl == "reference":
        return run_reference(args, wl, fmt)
    T = q_len_of(args, wl)
    if T is not None:
        if _env_int("WORLD_SIZE", 1) > 1:
            raise SystemExit("the multi-query workloads run on one GPU")
        return run_ours_q(args, wl, fmt, T)
    return run_ours(args, wl, fmt)


if __name__ == "__main__":
    sys.exit(main())
