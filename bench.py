#!/usr/bin/env python
"""Benchmark of the GQA attention hot path on GB300.

One step = one generate call's attention work for one layer of the Qwen3-4B
geometry (32 q / 8 kv heads, head_dim 128) at batch 4: cache reset, prefill of
four 2048-token prompts (K1 fused norm/RoPE/append + K2 tcgen05 causal
attention) and 128 decode steps (K3, one fused launch each), all through the
C ABI.  Inputs are synthetic (seeded N(0,1) bf16, see configs.py) and resident
in HBM; L2 is flushed (a 256 MiB read) between steps, outside the timed events.

Prints one JSON line.  `--impl reference` times the fp64 CPU oracle instead
(single-threaded, a bounded sample of the same step, extrapolated).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/step & HBM GB/s; prefill-attn TFLOP/s; fraction of GB300 roofline"
UNIT = "µs/step"
STEP_DEF = ("reset + prefill of 4 x 2048-token prompts + 128 decode steps, one attention layer "
            "(32 q / 8 kv heads, head_dim 128, cache capacity 2176)")


# ---------------------------------------------------------------- helpers
class L2Flush:
    """Evicts L2 by READING a 256 MiB buffer (twice the 129 MB L2) that nothing
    else touches: earlier dirty lines are written back during the flush, outside
    the timed events, and the next timed kernel finds L2 full of clean lines
    (a flush that writes its buffer would leave L2 dirty, so the next kernel's
    misses would pay for those write-backs)."""

    def __init__(self):
        import torch
        self.buf = torch.ones(256 << 20, dtype=torch.uint8, device="cuda")
        self.sink = torch.empty((), dtype=torch.int64, device="cuda")

    def zero_(self):
        import torch
        torch.sum(self.buf, dim=0, dtype=torch.int64, out=self.sink)
        return self


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def git_rev():
    try:
        rev = subprocess.run(["git", "rev-parse", "--short", "HEAD"], cwd=ROOT, capture_output=True,
                             text=True).stdout.strip()
        dirty = subprocess.run(["git", "status", "--porcelain"], cwd=ROOT, capture_output=True,
                               text=True).stdout.strip() != ""
        return rev or None, dirty
    except OSError:
        return None, None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "reasons": parts[5:9],
                             "power": float(parts[3]) if parts[3] not in ("[N/A]", "") else None})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        active = sorted({names[i] for r in rows for i, v in enumerate(r["reasons"])
                         if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": active,
                "samples": len(rows)}


# ---------------------------------------------------------------- oracle sample
class OracleStepModel:
    """Times the oracle's two parts separately and extrapolates one full step."""

    def __init__(self, w, inp, frac_rows):
        import numpy as np
        from gqa_attention_preallocated_qa_gb300.inputs import bf16_bits_to_f64 as F
        from oracle import oracle
        self.w, self.frac = w, frac_rows
        self.o = oracle
        g = oracle.Geometry(w.B, w.Hq, w.Hkv, w.D, w.cap, w.theta, w.eps)
        self.lay = oracle.OracleLayer(g)
        self.q, self.k, self.v, self.wq, self.wk = (F(a) for a in (inp.q, inp.k, inp.v, inp.wq,
                                                                    inp.wk))
        self.lay.prefill_transform(w.prompt_lens, self.q, self.k, self.v, self.wq, self.wk)
        self.lens0 = self.lay.lens.copy()
        self.cu = np.concatenate([[0], np.cumsum(w.prompt_lens)])
        # strided rows starting mid-stride: their mean key count is the prompt's mean
        self.rows = [(b, i) for b in range(w.B)
                     for i in range(frac_rows // 2, w.prompt_lens[b], frac_rows)]
        self.d = tuple(F(a) for a in (inp.dq[0], inp.dk[0], inp.dv[0]))
        self.desc = (f"every {frac_rows}th prompt row (from row {frac_rows // 2}) of each sequence (norm + RoPE + causal "
                     f"attention, all heads) scaled x{frac_rows}, plus one full decode step "
                     f"(all 4 x 32 heads over 2049 keys) scaled x{w.steps}")

    def sample(self):
        w, o, lay = self.w, self.o, self.lay
        t0 = time.perf_counter()
        for b, i in self.rows:
            t = self.cu[b] + i
            for h in range(w.Hq):
                lay.prefill_row(b, h, i, o.rope(o.rmsnorm(self.q[t, h], self.wq, w.eps), i, w.theta))
            for h in range(w.Hkv):
                o.rope(o.rmsnorm(self.k[t, h], self.wk, w.eps), i, w.theta)
        t1 = time.perf_counter()
        lay.lens[...] = self.lens0
        lay.decode(*self.d, self.wq, self.wk)
        t2 = time.perf_counter()
        return (t1 - t0) * self.frac + (t2 - t1) * w.steps, t2 - t0  # (extrapolated s, spent s)


# ---------------------------------------------------------------- distributed
def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, ws: int) -> float:
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def job_us_per_step(total_ms: float, steps: int, ws: int):
    """Whole-job µs per step of work and the slowest rank's ms per step.  Each
    of the ws ranks runs `steps` steps of its own (weak scaling), so the job
    does ws * steps steps in the slowest rank's time."""
    total_ms_max = reduce_max(total_ms, ws)
    ms_per_step = total_ms_max / steps
    return ms_per_step * 1e3 / ws, ms_per_step


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import numpy as np
    import torch

    from gqa_attention_preallocated_qa_gb300 import binding as qa
    from gqa_attention_preallocated_qa_gb300.configs import QWEN3_4B_B4 as w

    ws, rank, local = dist_info()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    pk = peaks()
    inp = w.inputs()

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

    q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    dq, dk, dv = dev(inp.dq), dev(inp.dk), dev(inp.dv)
    out = torch.empty_like(q)
    dout = torch.empty((w.steps, w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    flush = L2Flush()
    h = qa.qa_cache_alloc(1, w.B, w.Hq, w.Hkv, w.D, w.cap, w.theta, w.eps)
    lib = qa.lib
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    lens_arr = qa._i32(w.prompt_lens)
    P = {n: t.data_ptr() for n, t in dict(q=q, k=k, v=v, wq=wq, wk=wk, out=out).items()}
    dq_p = [dq[s].data_ptr() for s in range(w.steps)]
    dk_p = [dk[s].data_ptr() for s in range(w.steps)]
    dv_p = [dv[s].data_ptr() for s in range(w.steps)]
    do_p = [dout[s].data_ptr() for s in range(w.steps)]

    def step(evs=None):
        if evs:
            evs[0].record(stream)
        st = lib.qa_cache_reset(h, sh)
        if evs:
            evs[1].record(stream)
        st |= lib.qa_prefill(h, 0, w.B, lens_arr, P["q"], P["k"], P["v"], P["wq"], P["wk"],
                             P["out"], sh)
        if evs:
            evs[2].record(stream)
        for s in range(w.steps):
            st |= lib.qa_decode_step(h, 0, w.B, dq_p[s], dk_p[s], dv_p[s], P["wq"], P["wk"],
                                     do_p[s], sh)
        if evs:
            evs[3].record(stream)
        if st:
            raise RuntimeError(f"qa call failed with status {st}")

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    err = qa.qa_get_device_error(h)
    if err[0]:
        raise RuntimeError(f"device error after warm-up: {err}")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    stats0 = qa.qa_stats(h)
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.zero_()
            step(events[i])
        torch.cuda.synchronize()
    barrier(ws)
    stats1 = qa.qa_stats(h)
    launches = sum(stats1[n] - stats0[n] for n in stats1)
    err = qa.qa_get_device_error(h)
    if err[0]:
        raise RuntimeError(f"device error in the timed region: {err}")

    step_ms = [e[0].elapsed_time(e[3]) for e in events]
    pre_ms = [e[1].elapsed_time(e[2]) for e in events]
    dec_ms = [e[2].elapsed_time(e[3]) for e in events]
    total_ms = sum(step_ms)
    job_us, ms_per_step = job_us_per_step(total_ms, args.steps, ws)

    # algorithmic work
    flops = w.causal_flops()
    L0 = w.prompt_lens[0]
    dec_bytes = sum(w.B * w.Hkv * (L0 + s + 1) * w.D * 2 * 2 for s in range(w.steps))
    pre_us = statistics.mean(pre_ms) * 1e3
    dec_us_per_step = statistics.mean(dec_ms) * 1e3 / w.steps
    pre_tflops = flops / (pre_us * 1e-6) / 1e12
    dec_gbs = dec_bytes / w.steps / (dec_us_per_step * 1e-6) / 1e9
    dec_share = sum(dec_ms) / total_ms

    # K1 and K2 alone (the two halves of a prefill call), L2 flushed before each
    k1_us, k2_us = time_prefill_halves(args, qa, h, w, P, lens_arr, flush, stream)
    k1_bytes = w.T * (w.Hq + 2 * w.Hkv) * w.D * 2 * 2  # each row read once, written once
    k1_gbs = k1_bytes / (k1_us * 1e-6) / 1e9
    k2_tflops = flops / (k2_us * 1e-6) / 1e12

    # e2e through the public API with host buffers (pinned), copies inside the timed region
    e2e = run_e2e(args, qa, h, w, inp, stream)
    qa.qa_cache_free(h)

    # the decode sweep: every step reads its K/V from HBM (layers cycled)
    with ClockSampler(local) as sweep_clocks:
        sweep, isolated = decode_sweep(args, pk, args.sweep_steps)
    cold = next(p for p in sweep if (p["B"], p["L"]) == (4, 2048))

    roof_cold = {"bound": "hbm", "kernel": "k3_decode_kernel<128,4>",
                 "workload": "decode step, B=4, cache length 2048 (+ growth), HBM-cold: "
                             f"{cold['layers']} layer caches cycled, {cold['steps']} steps",
                 "achieved": cold["hbm_gbs"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                 "frac": cold["frac_of_measured_hbm"],
                 "traffic": traffic_for("k3_decode", cold["kv_bytes_per_step"]),
                 "traffic_regime": "cold launch, nothing of the cache in L2 (ncu)",
                 "per_launch_bytes": cold["kv_bytes_per_step"],
                 "duration": "events around the whole loop / steps (launch gaps included)"}
    roof_iso = {"bound": "hbm", "kernel": "k3_decode_kernel<128,4>",
                "workload": "one isolated decode step, B=4, L=2048, HBM-cold",
                "achieved": isolated["hbm_gbs"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": isolated["frac_of_measured_hbm"], "traffic": None,
                "per_launch_bytes": isolated["kv_bytes_per_step"],
                "duration": isolated["how"]}
    roof_l2 = {"bound": "hbm", "kernel": "k3_decode_kernel<128,4>",
               "workload": "decode steps of the generate call above, one layer: its 35.7 MB "
                           "cache stays in the 129 MB L2 (L2-resident, not an HBM figure)",
               "achieved": round(dec_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
               "frac": round(dec_gbs / pk["hbm_gbs"], 4), "traffic": None,
               "per_launch_bytes": round(dec_bytes / w.steps),
               "duration": "decode span / 128 launches (includes inter-launch gaps)"}
    roof_k1 = {"bound": "hbm", "kernel": "k1t_norm_rope_append_kernel<128> (token-tiled)",
               "workload": "qa_prefill_transform, B=4 x 2048 prompt rows",
               "achieved": round(k1_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
               "frac": round(k1_gbs / pk["hbm_gbs"], 4),
               "traffic": traffic_for("k1_norm", k1_bytes), "per_launch_bytes": k1_bytes,
               "duration": "mean over 40 launches, L2 flushed before each"}
    roof_k2 = {"bound": "tensor", "kernel": "k2c_prefill_kernel (CTA pairs, cta_group::2)",
               "workload": "qa_prefill_attend, B=4 x 2048 causal",
               "achieved": round(k2_tflops, 1), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
               "frac": round(k2_tflops / pk["bf16_tflops"], 4),
               "traffic": traffic_for("k2_prefill", None), "per_launch_flops": flops,
               "duration": "mean over 40 launches, L2 flushed before each"}
    roof_pre = {"bound": "tensor", "kernel": "k1t_norm_rope_append_kernel<128> + k2c_prefill_kernel",
                "workload": "qa_prefill call (K1 + K2), B=4 x 2048",
                "achieved": round(pre_tflops, 1), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(pre_tflops / pk["bf16_tflops"], 4), "traffic": None,
                "per_launch_flops": flops, "duration": "prefill call (K1 + K2) span"}
    rev, dirty = git_rev()
    line = {
        "metric": METRIC, "value": round(job_us, 2), "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "qwen3_4b_b4_p2048_d128", "step": STEP_DEF, "batch": w.B,
                   "prompt": w.prompt_lens[0], "decode_steps": w.steps, "layers": 1,
                   "l2": "flushed between steps (a 256 MiB read, outside the timed events)",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "components": {
            "decode_attn_us_per_step": round(dec_us_per_step, 3),
            "decode_hbm_gbs": round(dec_gbs, 1),
            "decode_frac_of_measured_hbm": round(dec_gbs / pk["hbm_gbs"], 4),
            "prefill_attn_us": round(pre_us, 2),
            "prefill_attn_tflops": round(pre_tflops, 1),
            "prefill_frac_of_measured_bf16": round(pre_tflops / pk["bf16_tflops"], 4),
            "decode_l2_resident": "the single-layer decode figures above: the layer's 35.7 MB "
                                  "cache stays in L2 (see decode_sweep for HBM-cold steps)",
            "k1_append_us": round(k1_us, 2), "k1_append_hbm_gbs": round(k1_gbs, 1),
            "k1_frac_of_measured_hbm": round(k1_gbs / pk["hbm_gbs"], 4),
            "k2_prefill_attn_us": round(k2_us, 2), "k2_prefill_attn_tflops": round(k2_tflops, 1),
            "k2_frac_of_measured_bf16": round(k2_tflops / pk["bf16_tflops"], 4),
            "decode_time_share": round(dec_share, 4),
            "step_ms_p50": round(statistics.median(step_ms), 4),
            "step_ms_spread": round((max(step_ms) - min(step_ms)) / statistics.median(step_ms), 4),
            "decode_sweep": sweep,
            "decode_sweep_clocks": sweep_clocks.summary(),
            "decode_isolated": isolated,
            "peaks": pk["source"],
        },
        "roofline": roof_cold,
        "roofline_all": [roof_cold, roof_iso, roof_l2, roof_k1, roof_k2, roof_pre],
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks.summary(),
        "git": {"rev": rev, "dirty": dirty},
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        model = OracleStepModel(w, inp, frac_rows=64)
        ests, spent = [], 0.0
        while spent < args.cpu_budget:
            est, sp = model.sample()
            ests.append(est)
            spent += sp
        line["cpu_baseline"] = {"value": round(statistics.median(ests) * 1e6, 1), "unit": UNIT,
                                "cores": 1, "kind": "oracle",
                                "sample": model.desc + f"; {len(ests)} samples, {spent:.1f} s",
                                "host_cpus": os.cpu_count()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def time_prefill_halves(args, qa, h, w, P, lens_arr, flush, stream, reps=40):
    """Mean µs of K1 alone (qa_prefill_transform) and of K2 alone
    (qa_prefill_attend over the rows K1 just appended), each launch after an
    L2 flush, on the generate call's prompt.  A mean, not a median: event
    timestamps come in steps of about a microsecond, and the launches start at
    random phases of that step, so the mean resolves what one sample cannot."""
    import torch
    lib = qa.lib
    sh = stream.cuda_stream
    qp = torch.empty((w.T, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    out2 = torch.empty_like(qp)
    t1, t2 = [], []
    for i in range(reps + 3):
        lib.qa_cache_reset(h, sh)
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        st = lib.qa_prefill_transform(h, 0, w.B, lens_arr, P["q"], P["k"], P["v"], P["wq"],
                                      P["wk"], qp.data_ptr(), sh)
        b.record(stream)
        flush.zero_()
        c, d = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c.record(stream)
        st |= lib.qa_prefill_attend(h, 0, w.B, lens_arr, qp.data_ptr(), out2.data_ptr(), sh)
        d.record(stream)
        torch.cuda.synchronize()
        if st:
            raise RuntimeError(f"prefill halves failed with status {st}")
        if i >= 3:
            t1.append(a.elapsed_time(b) * 1e3)
            t2.append(c.elapsed_time(d) * 1e3)
    if qa.qa_get_device_error(h)[0]:
        raise RuntimeError("device error while timing the prefill halves")
    return statistics.mean(t1), statistics.mean(t2)


def run_e2e(args, qa, h, w, inp, stream):
    """Same step through the public API with HOST buffers: every step copies its
    inputs (prompt q/k/v, norm weights, the 128 decode tokens' q/k/v) from
    pinned host memory to the device and reads its results (prefill output and
    the 128 decode outputs) back, all inside the timed events.  As a caller
    would, the step overlaps copies with compute: the prompt goes up one
    sequence at a time on an upload stream and each sequence is prefilled (a
    chunked qa_prefill call for that sequence alone) as soon as its rows have
    arrived, the decode tokens' inputs follow, and the prefill output comes
    back on a download stream while the decode steps run; all streams join
    before the step's end event."""
    import numpy as np
    import torch
    lib = qa.lib
    sh = stream.cuda_stream
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

    def flat(*arrays):
        return np.concatenate([np.ascontiguousarray(a).reshape(-1) for a in arrays])

    parts = (inp.q, inp.k, inp.v, inp.wq, inp.wk, inp.dq, inp.dk, inp.dv)
    host_in = torch.from_numpy(flat(*parts).view(np.int16)).view(torch.bfloat16).pin_memory()
    dev_in = torch.empty_like(host_in, device="cuda")
    sizes = [a.size for a in parts]
    offs = [int(o) for o in np.concatenate([[0], np.cumsum(sizes)])]
    ptr = [dev_in.data_ptr() + 2 * o for o in offs[:-1]]
    q_p, k_p, v_p, wq_p, wk_p, dq_p, dk_p, dv_p = ptr
    step_q, step_kv = w.B * w.Hq * w.D * 2, w.B * w.Hkv * w.D * 2
    T = w.T
    n_out_pre = T * w.Hq * w.D
    dev_out = torch.empty(n_out_pre + w.steps * w.B * w.Hq * w.D, dtype=torch.bfloat16,
                          device="cuda")
    host_out = torch.empty(dev_out.shape, dtype=torch.bfloat16).pin_memory()
    out_p = dev_out.data_ptr()
    dout_p = out_p + n_out_pre * 2
    cu = [0]
    for L in w.prompt_lens:
        cu.append(cu[-1] + L)
    qrow, kvrow = w.Hq * w.D, w.Hkv * w.D  # elements per token
    lens_one = []
    for b in range(w.B):
        lens_one.append(qa._i32([w.prompt_lens[i] if i == b else 0 for i in range(w.B)]))
    flush = L2Flush()

    def copy_rows(dst, src, base, row, a, b):
        dst[base + a * row:base + b * row].copy_(src[base + a * row:base + b * row], non_blocking=True)

    def step():
        up.wait_stream(stream)  # nothing of this step starts before the step's start event
        down.wait_stream(stream)
        arrived = []
        with torch.cuda.stream(up):
            copy_rows(dev_in, host_in, offs[3], 1, 0, offs[5] - offs[3])  # norm weights
            for b in range(w.B):
                a, e = cu[b], cu[b + 1]
                copy_rows(dev_in, host_in, offs[0], qrow, a, e)
                copy_rows(dev_in, host_in, offs[1], kvrow, a, e)
                copy_rows(dev_in, host_in, offs[2], kvrow, a, e)
                ev = torch.cuda.Event()
                ev.record(up)
                arrived.append(ev)
            dev_in[offs[5]:].copy_(host_in[offs[5]:], non_blocking=True)  # decode tokens
            dec_in = torch.cuda.Event()
            dec_in.record(up)
        st = lib.qa_cache_reset(h, sh)
        for b in range(w.B):
            a = cu[b]
            stream.wait_event(arrived[b])
            st |= lib.qa_prefill(h, 0, w.B, lens_one[b], q_p + 2 * a * qrow, k_p + 2 * a * kvrow,
                                 v_p + 2 * a * kvrow, wq_p, wk_p, out_p + 2 * a * qrow, sh)
        # the prefill output goes down once the uploads are done (the two directions
        # share the link's bandwidth), while the decode steps run
        done = torch.cuda.Event()
        done.record(stream)
        with torch.cuda.stream(down):
            down.wait_event(done)
            host_out[:n_out_pre].copy_(dev_out[:n_out_pre], non_blocking=True)
        stream.wait_event(dec_in)
        for s in range(w.steps):
            st |= lib.qa_decode_step(h, 0, w.B, dq_p + s * step_q, dk_p + s * step_kv,
                                     dv_p + s * step_kv, wq_p, wk_p, dout_p + s * step_q, sh)
        host_out[n_out_pre:].copy_(dev_out[n_out_pre:], non_blocking=True)
        stream.wait_stream(up)
        stream.wait_stream(down)  # every prefill output is back before the step's end event
        if st:
            raise RuntimeError(f"qa call failed with status {st}")

    for _ in range(3):
        step()
    n = max(3, min(args.steps, args.e2e_steps))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    torch.cuda.synchronize()
    for i in range(n):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in evs) / n
    return {"value": round(ms * 1e3, 2), "unit": UNIT, "h2d_bytes_per_step": host_in.numel() * 2,
            "d2h_bytes_per_step": host_out.numel() * 2, "steps": n, "host_buffers": "pinned",
            "copies": "prompt up one sequence at a time, each prefilled as it arrives; prefill "
                      "output down during the decode steps"}


def kernel_source_digest(kernel: str) -> str:
    """sha256 (first 16 hex digits) over the kernel's source file and the
    headers of its own that it includes, with comments and whitespace removed (a
    comment edit does not change the kernel the counters were taken on)."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "gqa_attention_preallocated_qa_gb300", "csrc")
    src = {"k3_decode": "k3_decode_splitkv.cu", "k3_multi": "k3_decode_splitkv.cu",
           "k2_prefill": "k2_prefill_tcgen05.cu", "k1_norm": "k1_norm_rope_append.cu"}[kernel]
    h = hashlib.sha256()
    extra = ("k2_items.h",) if kernel == "k2_prefill" else ()
    for name in (src, "qa_device.cuh", "qa_internal.h") + extra:
        with open(os.path.join(csrc, name)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)  # block comments
        text = re.sub(r"//[^\n]*", " ", text)                # line comments
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, algorithmic_bytes):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else null)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            d = json.load(fh)[kernel]
        if d.get("source_sha256_16") != kernel_source_digest(kernel):
            return None
        return d["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------- decode sweep
def host_ahead(launches: int, us_per_launch: float = 6.0):
    """Put the device behind the host: a GPU sleep long enough for the host to
    enqueue `launches` calls first, so that events around a loop of short
    launches time the device, not the host's launch rate (which the caller
    measures and reports separately)."""
    import torch
    torch.cuda._sleep(int(launches * us_per_launch * 2.5e3))  # ~2.5 GHz upper bound on cycles/us


def decode_sweep(args, pk, steps, isolated_steps=200):
    """Decode-only sweep (batch 1 and 4, cache lengths 512 to 16384).  Each
    point allocates NL layer caches, NL at least the 36 attention layers of
    Qwen3-4B and large enough that together they hold at least 3x the L2
    (129 MB), every one filled with L raw N(0,1) keys/values per sequence; the `steps` timed decode steps cycle through the layers (step
    s decodes layer s mod NL, as a model's layer loop does), so each step reads
    its layer's K/V from HBM, not from L2.  The length of a layer grows by one
    per visit; bytes are counted exactly.  A GPU sleep before the loop lets the
    host enqueue the launches ahead of the device, so the events time the
    device (the host's own µs per call is reported beside it).  Per point: mean
    µs per step, K/V bytes per step and HBM GB/s (events around the whole loop:
    launch gaps included); `same_layer_us_per_step` repeats the measurement on a single
    layer (its cache can stay in L2 when small).  At B = 4, L = 2048 the point
    also times `isolated_steps` steps one by one: split plan for one launch at
    a time, a spacer kernel before each (so no launch overlaps the previous
    decode launch) and events around each launch."""
    import numpy as np
    import torch

    from gqa_attention_preallocated_qa_gb300 import binding as qa
    from gqa_attention_preallocated_qa_gb300.configs import DECODE_SWEEP

    l2_bytes = 129 * 1000 * 1000

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

    points = []
    isolated = None
    for pt in DECODE_SWEEP:
        inp = pt.inputs()
        layer_bytes = pt.B * pt.Hkv * pt.L * pt.D * 4
        NL = max(36, min(256, -(-3 * l2_bytes // layer_bytes)))
        iso = isolated_steps if (pt.B, pt.L) == (4, 2048) else 0
        visits = -(-(steps + args.warmup + iso) // NL) + args.warmup + 1
        same_steps = 200
        cap = pt.L + visits + same_steps
        h = qa.qa_cache_alloc(NL, pt.B, pt.Hq, pt.Hkv, pt.D, cap, pt.theta, pt.eps)
        ck, cv = dev(inp.cache_k), dev(inp.cache_v)
        for layer in range(NL):
            K, V, _ = qa.cache_tensors(h, layer, pt.B, pt.Hkv, cap, pt.D)
            K[:, :, :pt.L] = ck
            V[:, :, :pt.L] = cv
            qa.qa_cache_set_lengths(h, layer, [pt.L] * pt.B)
        del ck, cv
        if args.sweep_overlap:
            qa.qa_cache_set_decode_overlap(h, args.sweep_overlap)
        q, k, v, wq, wk = (dev(a) for a in (inp.dq[0], inp.dk[0], inp.dv[0], inp.wq, inp.wk))
        out = torch.empty_like(q)
        stream = torch.cuda.current_stream()
        sh = stream.cuda_stream
        lib = qa.lib
        args_c = (q.data_ptr(), k.data_ptr(), v.data_ptr(), wq.data_ptr(), wk.data_ptr(),
                  out.data_ptr())
        lens = [pt.L] * NL
        st = 0
        for i in range(args.warmup):
            st |= lib.qa_decode_step(h, i % NL, pt.B, *args_c, sh)
            lens[i % NL] += 1
        splits = qa.qa_decode_splits(h, 0, pt.B)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        byts = 0
        torch.cuda.synchronize()
        host_ahead(steps)
        e0.record(stream)
        t_host = time.perf_counter()
        for i in range(steps):
            layer = (args.warmup + i) % NL
            st |= lib.qa_decode_step(h, layer, pt.B, *args_c, sh)
            lens[layer] += 1
            byts += pt.B * pt.Hkv * lens[layer] * pt.D * 4  # keys 0..pos, K and V
        e1.record(stream)
        host_us = (time.perf_counter() - t_host) * 1e6 / steps
        torch.cuda.synchronize()
        if st or qa.qa_get_device_error(h)[0]:
            raise RuntimeError(f"decode sweep point {pt.name} failed")
        us = e0.elapsed_time(e1) * 1e3 / steps
        byts /= steps
        gbs = byts / (us * 1e-6) / 1e9
        # the same on one layer, for reference (its K/V may stay in L2)
        n1 = same_steps
        e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2.record(stream)
        for _ in range(n1):
            st |= lib.qa_decode_step(h, 0, pt.B, *args_c, sh)
        e3.record(stream)
        lens[0] += n1
        torch.cuda.synchronize()
        if st or qa.qa_get_device_error(h)[0]:
            raise RuntimeError(f"decode sweep point {pt.name} failed")
        if iso:
            qa.qa_cache_set_decode_overlap(h, 1)
            iso_splits = qa.qa_decode_splits(h, 0, pt.B)
            spacer = torch.zeros(1, device="cuda")
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(iso)]
            ib = 0
            torch.cuda.synchronize()
            host_ahead(3 * iso)
            for i in range(iso):
                layer = (args.warmup + steps + i) % NL
                spacer.add_(1.0)  # a plain kernel: this launch cannot overlap a decode launch
                evs[i][0].record(stream)
                st |= lib.qa_decode_step(h, layer, pt.B, *args_c, sh)
                evs[i][1].record(stream)
                lens[layer] += 1
                ib += pt.B * pt.Hkv * lens[layer] * pt.D * 4
            torch.cuda.synchronize()
            if st or qa.qa_get_device_error(h)[0]:
                raise RuntimeError("isolated decode steps failed")
            iso_us = statistics.mean(a.elapsed_time(b) * 1e3 for a, b in evs)
            iso_gbs = ib / iso / (iso_us * 1e-6) / 1e9
            # The floor of this measurement: the same spacer and events around
            # the library's reset kernel (one CTA zeroing a few lengths) on a
            # separate small cache.
            h0 = qa.qa_cache_alloc(1, 1, pt.Hq, pt.Hkv, pt.D, 8, pt.theta, pt.eps)
            fevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(iso)]
            torch.cuda.synchronize()
            host_ahead(3 * iso)
            for a, b in fevs:
                spacer.add_(1.0)
                a.record(stream)
                st |= lib.qa_cache_reset(h0, sh)
                b.record(stream)
            torch.cuda.synchronize()
            qa.qa_cache_free(h0)
            if st:
                raise RuntimeError("launch-floor measurement failed")
            floor_us = statistics.mean(a.elapsed_time(b) * 1e3 for a, b in fevs)
            isolated = {"B": pt.B, "L": pt.L, "steps": iso, "splits": iso_splits,
                        "us_per_step": round(iso_us, 3), "hbm_gbs": round(iso_gbs, 1),
                        "frac_of_measured_hbm": round(iso_gbs / pk["hbm_gbs"], 4),
                        "kv_bytes_per_step": round(ib / iso),
                        "launch_floor_us": round(floor_us, 3),
                        "floor_how": "the same spacer and events around a one-CTA library "
                                     "kernel (cache reset of a separate small cache): what any "
                                     "launch costs in this measurement",
                        "how": "mean of per-launch events; a spacer kernel before each launch, "
                               "layers cycled (HBM-cold), split plan for one launch, the host "
                               "ahead of the device"}
        points.append({"sweep": pt.name, "B": pt.B, "L": pt.L, "steps": steps, "layers": NL,
                       "splits": splits, "overlap": args.sweep_overlap or "per launch", "us_per_step": round(us, 3),
                       "host_us_per_call": round(host_us, 3),
                       "kv_bytes_per_step": round(byts), "hbm_gbs": round(gbs, 1),
                       "frac_of_measured_hbm": round(gbs / pk["hbm_gbs"], 4),
                       "same_layer_us_per_step": round(e2.elapsed_time(e3) * 1e3 / max(1, n1), 3)})
        qa.qa_cache_free(h)
        del inp
    return points, isolated


def run_sweep(args):
    """`--sweep`: the decode sweep alone, one JSON line per point (and one for
    the isolated step), with the clocks seen while it ran."""
    pk = peaks()
    with ClockSampler(0) as clocks:
        points, isolated = decode_sweep(args, pk, args.sweep_steps)
    for p in points:
        print(json.dumps(p), flush=True)
    print(json.dumps({"isolated_decode": isolated}), flush=True)
    print(json.dumps({"clocks": clocks.summary()}), flush=True)


def run_verify(args):
    """Multi-token query against the cache (the verify step of speculative
    decoding), served by a chunked prefill of k tokens per sequence (up to 8
    tokens: the decode kernel's multi-token form; more: the prefill kernels),
    against k decode steps of the same tokens: B = 4, cache length 2048,
    k in {2, 4, 8, 16}.
    Layers cycle as in --sweep (>= 3x L2 of caches), so K/V come from HBM.
    One JSON line per k: µs per verify call and per k decode steps."""
    import numpy as np
    import torch

    from gqa_attention_preallocated_qa_gb300 import binding as qa
    from gqa_attention_preallocated_qa_gb300.configs import SweepPoint
    from gqa_attention_preallocated_qa_gb300.inputs import layer_inputs

    pt = SweepPoint(4, 2048)
    inp = pt.inputs()
    l2_bytes = 129 * 1000 * 1000
    NL = max(1, -(-3 * l2_bytes // (pt.B * pt.Hkv * pt.L * pt.D * 4)))
    reps = 40

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

    for k in (2, 4, 8, 16):
        tok = layer_inputs(5, [k] * pt.B, pt.Hq, pt.Hkv, pt.D, k)
        cap = pt.L + 2 * k * (reps // NL + 2)
        h = qa.qa_cache_alloc(NL, pt.B, pt.Hq, pt.Hkv, pt.D, cap, pt.theta, pt.eps)
        ck, cv = dev(inp.cache_k), dev(inp.cache_v)
        for layer in range(NL):
            K, V, _ = qa.cache_tensors(h, layer, pt.B, pt.Hkv, cap, pt.D)
            K[:, :, :pt.L] = ck
            V[:, :, :pt.L] = cv
            qa.qa_cache_set_lengths(h, layer, [pt.L] * pt.B)
        q, kk, v, wq, wk = (dev(a) for a in (tok.q, tok.k, tok.v, tok.wq, tok.wk))
        out = torch.empty_like(q)
        dq, dk, dv = dev(tok.dq), dev(tok.dk), dev(tok.dv)
        dout = torch.empty((pt.B, pt.Hq, pt.D), dtype=torch.bfloat16, device="cuda")
        stream = torch.cuda.current_stream()
        sh = stream.cuda_stream
        lib = qa.lib
        lens_arr = qa._i32([k] * pt.B)
        pv = [t.data_ptr() for t in (q, kk, v, wq, wk, out)]
        pd = [(dq[s].data_ptr(), dk[s].data_ptr(), dv[s].data_ptr()) for s in range(k)]
        st = 0

        def verify(layer):
            return lib.qa_prefill(h, layer, pt.B, lens_arr, *pv, sh)

        def decode(layer):
            r = 0
            for s in range(k):
                r |= lib.qa_decode_step(h, layer, pt.B, *pd[s], pv[3], pv[4], dout.data_ptr(), sh)
            return r
        times = {}
        for name, fn in (("verify", verify), ("decode", decode)):
            for i in range(NL):  # warm-up pass over the layers
                st |= fn(i % NL)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for i in range(reps):
                st |= fn(i % NL)
            e1.record(stream)
            torch.cuda.synchronize()
            times[name] = e0.elapsed_time(e1) * 1e3 / reps
        if st or qa.qa_get_device_error(h)[0]:
            raise RuntimeError(f"verify bench k={k} failed")
        print(json.dumps({"verify": f"b{pt.B}_l{pt.L}_k{k}", "B": pt.B, "L": pt.L, "k": k,
                          "layers": NL, "verify_us": round(times["verify"], 2),
                          "decode_k_steps_us": round(times["decode"], 2),
                          "speedup_vs_decode": round(times["decode"] / times["verify"], 3)}), flush=True)
        qa.qa_cache_free(h)


def run_graph(args):
    """The multi-layer decode step: 36 attention layers, one decode step each per
    generated token, three ways: eager through qa_decode_step as a caller runs
    it (the host issues every call, so the slower of host and device sets the
    pace), the same with the host ahead of the device (device time), and one CUDA
    graph of 36 qa_decode_step_device_lengths calls replayed once per token
    (positions advance on the device; no host work per layer).  Two workloads:
    the 36-layer ragged one (B = 4, prompts 512/1024/1536/2048, capacity 2112,
    1.25 GB of caches) and B = 1 with a 1024-token prompt (capacity 1088).  The
    caches hold seeded N(0,1) keys/values (timing only; parity of this path is
    in the tests) and are far larger than L2 or cycled through 36 layers, so
    every layer reads its K/V from HBM.  One JSON line per workload."""
    import torch

    from gqa_attention_preallocated_qa_gb300 import binding as qa
    from gqa_attention_preallocated_qa_gb300.configs import RAGGED_36L, Workload

    steps = 20
    stream = torch.cuda.current_stream()
    b1 = Workload("qwen3_4b_b1_p1024_36layers", B=1, Hq=32, Hkv=8, D=128, prompt_lens=(1024,),
                  steps=64, cap=1088, layers=36, seed=6)
    for w in (RAGGED_36L, b1):
        res = {}
        for mode in ("eager_host_paced", "eager", "eager_device_lengths", "graph"):
            h = qa.qa_cache_alloc(w.layers, w.B, w.Hq, w.Hkv, w.D, w.cap, w.theta, w.eps)
            gen = torch.Generator(device="cuda").manual_seed(w.seed)
            bufs = []
            for l in range(w.layers):  # caches hold the prompts' lengths of N(0,1) keys/values
                K, V, _ = qa.cache_tensors(h, l, w.B, w.Hkv, w.cap, w.D)
                K.normal_(generator=gen)
                V.normal_(generator=gen)
                qa.qa_cache_set_lengths(h, l, list(w.prompt_lens))

                def rnd(*shape):
                    return torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
                bufs.append((rnd(w.B, w.Hq, w.D), rnd(w.B, w.Hkv, w.D), rnd(w.B, w.Hkv, w.D),
                             (1 + 0.1 * rnd(w.D).float()).to(torch.bfloat16),
                             (1 + 0.1 * rnd(w.D).float()).to(torch.bfloat16),
                             torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")))
            torch.cuda.synchronize()
            lib = qa.lib
            ptrs = [[t.data_ptr() for t in b] for b in bufs]
            fn = (lib.qa_decode_step if mode in ("eager_host_paced", "eager")
                  else lib.qa_decode_step_device_lengths)

            def step(sh):
                st = 0
                for l in range(w.layers):
                    st |= fn(h, l, w.B, *ptrs[l], sh)
                return st
            st = step(stream.cuda_stream)  # warm-up (configures the kernels outside capture)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if mode != "graph":
                if mode != "eager_host_paced":
                    host_ahead(steps * w.layers)
                e0.record(stream)
                for _ in range(steps):
                    st |= step(stream.cuda_stream)
                e1.record(stream)
            else:
                g = torch.cuda.CUDAGraph()
                side = torch.cuda.Stream()
                side.wait_stream(stream)
                with torch.cuda.stream(side):
                    with torch.cuda.graph(g):
                        st |= step(torch.cuda.current_stream().cuda_stream)
                stream.wait_stream(side)
                g.replay()  # first replay outside the timing
                e0.record(stream)
                for _ in range(steps):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            if st or qa.qa_get_device_error(h)[0]:
                raise RuntimeError(f"graph bench ({mode}) failed")
            res[mode] = e0.elapsed_time(e1) * 1e3 / steps
            qa.qa_cache_free(h)
        print(json.dumps({"graph": w.name, "layers": w.layers, "batch": w.B,
                          **{f"{m}_us_per_token": round(v, 1) for m, v in res.items()},
                          "graph_us_per_layer": round(res["graph"] / w.layers, 2),
                          "timing": "eager_host_paced: as a caller runs it; eager and "
                                    "eager_device_lengths: the host ahead of the device "
                                    "(device time); graph: replays back to back"}), flush=True)


def run_window(args):
    """Sliding-window attention against full attention: decode steps at B = 4,
    cache length 8192 (layers cycled as in --sweep, so K/V come from HBM) with
    W = 1024 and without; and the B = 4 x 2048 prefill with W = 512 and
    without.  One JSON line per case: µs and the keys each query reads."""
    import numpy as np
    import torch

    from gqa_attention_preallocated_qa_gb300 import binding as qa
    from gqa_attention_preallocated_qa_gb300.configs import QWEN3_4B_B4, SweepPoint

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    pt = SweepPoint(4, 8192)
    inp = pt.inputs()
    NL = max(1, -(-3 * 129 * 1000 * 1000 // (pt.B * pt.Hkv * pt.L * pt.D * 4)))
    reps = 200
    for window in (0, 1024):
        cap = pt.L + reps // NL + 20
        h = qa.qa_cache_alloc(NL, pt.B, pt.Hq, pt.Hkv, pt.D, cap, pt.theta, pt.eps)
        ck, cv = dev(inp.cache_k), dev(inp.cache_v)
        for layer in range(NL):
            K, V, _ = qa.cache_tensors(h, layer, pt.B, pt.Hkv, cap, pt.D)
            K[:, :, :pt.L] = ck
            V[:, :, :pt.L] = cv
            qa.qa_cache_set_lengths(h, layer, [pt.L] * pt.B)
            qa.qa_cache_set_window(h, layer, window)
        q, k, v, wq, wk = (dev(a) for a in (inp.dq[0], inp.dk[0], inp.dv[0], inp.wq, inp.wk))
        out = torch.empty_like(q)
        ptrs = [t.data_ptr() for t in (q, k, v, wq, wk, out)]
        st = 0
        for i in range(NL):
            st |= qa.lib.qa_decode_step(h, i % NL, pt.B, *ptrs, sh)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(reps):
            st |= qa.lib.qa_decode_step(h, i % NL, pt.B, *ptrs, sh)
        e1.record(stream)
        torch.cuda.synchronize()
        if st or qa.qa_get_device_error(h)[0]:
            raise RuntimeError("window bench (decode) failed")
        print(json.dumps({"window_decode": f"b4_l{pt.L}", "window": window,
                          "keys_per_query": window if window else pt.L,
                          "us_per_step": round(e0.elapsed_time(e1) * 1e3 / reps, 3)}), flush=True)
        qa.qa_cache_free(h)
    w = QWEN3_4B_B4
    pin = w.inputs()
    q, k, v, wq, wk = (dev(a) for a in (pin.q, pin.k, pin.v, pin.wq, pin.wk))
    out = torch.empty_like(q)
    lens_arr = qa._i32(w.prompt_lens)
    ptrs = [t.data_ptr() for t in (q, k, v, wq, wk, out)]
    flush = L2Flush()
    for window in (0, 512):
        h = qa.qa_cache_alloc(1, w.B, w.Hq, w.Hkv, w.D, w.cap, w.theta, w.eps)
        qa.qa_cache_set_window(h, 0, window)
        ts = []
        for it in range(13):
            flush.zero_()
            qa.lib.qa_cache_reset(h, sh)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            st = qa.lib.qa_prefill(h, 0, w.B, lens_arr, *ptrs, sh)
            e1.record(stream)
            torch.cuda.synchronize()
            if st:
                raise RuntimeError("window bench (prefill) failed")
            if it >= 3:
                ts.append(e0.elapsed_time(e1) * 1e3)
        print(json.dumps({"window_prefill": "b4_p2048", "window": window,
                          "prefill_us": round(statistics.median(ts), 2)}), flush=True)
        qa.qa_cache_free(h)


def run_profile_case(args):
    """A short program for ncu: one reset + prefill, four decode steps and one
    verify call of four tokens per sequence (the decode kernel's multi-token
    form) on the benchmark workload (B=4, prompt 2048), nothing else on the
    device; all of it twice."""
    import numpy as np
    import torch

    from gqa_attention_preallocated_qa_gb300 import binding as qa
    from gqa_attention_preallocated_qa_gb300.configs import QWEN3_4B_B4 as w
    inp = w.inputs()

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    out = torch.empty_like(q)
    h = qa.qa_cache_alloc(1, w.B, w.Hq, w.Hkv, w.D, w.cap, w.theta, w.eps)
    for rep in range(2):
        qa.qa_cache_reset(h)
        qa.qa_prefill(h, 0, list(w.prompt_lens), q, k, v, wq, wk, out)
        for s in range(4):
            dq, dk, dv = dev(inp.dq[s]), dev(inp.dk[s]), dev(inp.dv[s])
            o = torch.empty_like(dq)
            qa.qa_decode_step(h, 0, w.B, dq, dk, dv, wq, wk, o)
        # tokens 4..7 of every sequence in one call, packed sequence by sequence
        vq, vk, vv = (dev(np.ascontiguousarray(a[4:8].transpose(1, 0, 2, 3)).reshape(
            w.B * 4, *a.shape[2:])) for a in (inp.dq, inp.dk, inp.dv))
        vo = torch.empty_like(vq)
        qa.qa_prefill(h, 0, [4] * w.B, vq, vk, vv, wq, wk, vo)
    torch.cuda.synchronize()
    st, word = qa.qa_get_device_error(h)
    qa.qa_cache_free(h)
    if st:
        raise RuntimeError(f"device error {word:#x}")
    print("profile case done", flush=True)


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    """The oracle as it stands, single-threaded on the host, on a bounded sample
    of the same step per timed step; reports the extrapolated full-step time."""
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    from gqa_attention_preallocated_qa_gb300.configs import QWEN3_4B_B4 as w
    inp = w.inputs()
    model = OracleStepModel(w, inp, frac_rows=512)
    for _ in range(args.warmup):
        model.sample()
    ests, spents = [], []
    for _ in range(args.steps):
        est, sp = model.sample()
        ests.append(est)
        spents.append(sp)
    value = statistics.median(ests) * 1e6
    # Each timed step runs a bounded sample of the generate call; ms_per_step is
    # the wall time of the sample actually run, `value` the full call it stands
    # for (the sample scaled up row for row, as the description says).
    sample_ms = statistics.mean(spents) * 1e3
    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sample_ms, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": "qwen3_4b_b4_p2048_d128", "step": STEP_DEF, "batch": w.B,
                       "prompt": w.prompt_lens[0], "decode_steps": w.steps, "layers": 1},
            "extrapolated": {"value_is": "the full generate call, scaled up from each step's "
                                         "sample", "sample_ms_per_step": round(sample_ms, 3),
                             "scale": round(value / 1e3 / sample_ms, 1)},
            "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": model.desc + f"; {len(ests)} samples, "
                                                    f"{sum(spents):.1f} s"},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle timing")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="decode-only sweep over batch 1/4 and cache lengths 512..16384")
    ap.add_argument("--sweep-steps", type=int, default=1000,
                    help="timed decode steps per sweep point")
    ap.add_argument("--sweep-overlap", type=int, default=0,
                    help="decode launches the split plan fits at once in the sweep "
                         "(qa_cache_set_decode_overlap; 0: the library's default)")
    ap.add_argument("--verify", action="store_true",
                    help="k-token verify (chunked prefill) vs k decode steps, B=4, L=2048")
    ap.add_argument("--graph", action="store_true",
                    help="36-layer decode step: eager vs one CUDA graph replay")
    ap.add_argument("--window", action="store_true",
                    help="sliding-window decode (L=8192, W=1024) and prefill (W=512) vs full")
    ap.add_argument("--profile-case", action="store_true",
                    help="run one small prefill + 4 decode steps (for ncu) and exit")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    if args.profile_case:
        run_profile_case(args)
    elif args.sweep:
        run_sweep(args)
    elif args.verify or args.graph or args.window:
        # each mode's JSON lines, then the clocks seen while it ran
        with ClockSampler(0) as clocks:
            (run_verify if args.verify else run_graph if args.graph else run_window)(args)
        print(json.dumps({"clocks": clocks.summary()}), flush=True)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
