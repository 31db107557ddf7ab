"""Benchmark: one decode step (append of one token per sequence + paged decode attention)
on a synthetic in-flight batch, timed on the GPU.  Prints one JSON line.

Headline workload: the 70B-shape long-context batch (64 query / 8 KV heads, head_dim 128, bf16,
block 64, 8 sequences of 32K..128K tokens), the largest; the Llama-2-7B MHA batch, the
Llama-3-8B GQA batch and the churned 200-request FP8 pool follow as sub-records ("configs") of
the same JSON line.  `--workload` picks the headline, `--also` the sub-records.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference] [--workload c3] [--also c1,c2,c4]

For N > 1 (torchrun, one rank per GPU) every rank runs its own replica of the workload
(independent sequences, no data exchange); the value is the sum over ranks divided by the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import pkv_workloads as W  # noqa: E402

METRIC = "paged decode attention: achieved HBM GB/s (% of GB300 peak), decode tokens/s"
L2_BYTES = 126 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal, for context beside the measured peak


# ----------------------------------------------------------------------------- helpers
def algorithmic_bytes(w) -> dict:
    """Bytes the step must move at minimum.  Attention: every cached K/V element of every
    (sequence, KV head) once, fp8 scale pairs of the pages read, Q in, output out, the used
    block-table entries and the context lengths.  Append: new K/V in, stored K/V out."""
    L = w.attend_lens.astype(np.int64)
    pages = ((L + w.block_size - 1) // w.block_size).sum()
    kv = int(L.sum()) * w.Hkv * 2 * w.D * w.elem_bytes
    scales = int(pages) * w.Hkv * 8 if w.kv_dtype != "bf16" else 0
    q_out = 2 * w.B * w.Hq * w.D * 2
    meta = int(pages) * 4 + w.B * 4
    attn = kv + scales + q_out + meta
    app = (w.B * w.Hkv * w.D * 2 * 2 + w.B * w.Hkv * w.D * w.elem_bytes * 2 + w.B * 8) if w.append else 0
    return {"attention": attn, "append": app, "step": attn + app, "kv": kv}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# The sources that determine the decode attention kernel's code and launch (its own file, the
# PTX helpers, the one-byte codes its step's append writes, the pool's tensor maps and the shared
# declarations; not the ABI header's comments).
DECODE_KERNEL_SOURCES = ("paged_kv_cache_266_gb300/csrc/decode_attention.cu", "paged_kv_cache_266_gb300/csrc/ptx.cuh",
                         "paged_kv_cache_266_gb300/csrc/quant.cuh", "paged_kv_cache_266_gb300/csrc/pkv_internal.h",
                         "paged_kv_cache_266_gb300/csrc/pool.cu")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in DECODE_KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(w):
    """DRAM bytes per attention launch from the committed ncu summary, if it was taken on the
    current decode kernel sources (else None).  A workload too large to capture under the
    profiling size rule was captured on its first sequences ("c3[:2]"); its DRAM bytes are
    scaled to the full launch by the ratio of algorithmic bytes, which is how they grow (the
    DRAM/algorithmic ratio of every capture is 1.000-1.009).  Returns (bytes, note)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None, None
    src = kernel_source_hash()
    for line in open(p):
        parts = line.split()
        if len(parts) < 3 or line.startswith("#") or parts[1] != src:
            continue
        if parts[0] == w.name:
            return int(parts[2]), f"ncu capture of {parts[0]}"
        if parts[0].startswith(w.name + "[:") and parts[0].endswith("]"):
            n = int(parts[0][len(w.name) + 2:-1])
            part = algorithmic_bytes(W.truncated(w, n))["attention"]
            full = algorithmic_bytes(w)["attention"]
            return int(round(int(parts[2]) * full / part)), f"ncu capture of {parts[0]}, scaled by algorithmic bytes"
    return None, None


def append_launches(kv_dtype: str, n_tokens: int, in_step: bool = False) -> int:
    """Kernels the library launches to append n_tokens tokens: a bf16 pool takes one; a one-byte
    pool one up to 1024 tokens, three above; and none inside pkv_decode_step (in_step) on a
    one-byte pool for 1..1024 tokens, where the attention kernel appends them itself."""
    if n_tokens == 0:
        return 0
    if kv_dtype == "bf16":
        return 1
    if n_tokens <= 1024:
        return 0 if in_step else 1
    return 3


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.bus = None
        try:
            import torch
            props = torch.cuda.get_device_properties(device_index)
            self.bus = getattr(props, "pci_bus_id", None)
        except Exception:
            pass

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            rows.append(f)
        os.unlink(self.path)
        if self.bus is not None:
            mine = [r for r in rows if r[1].lower().endswith(f"{self.bus:02x}:00.0")]
            rows = mine or rows
        idx = sorted({r[0] for r in rows})
        if idx:
            rows = [r for r in rows if r[0] == idx[0]]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": float(rows[0][3]) if rows else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def dist_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle runs
def oracle_rate(w, budget_s: float, threads: int):
    """Time the oracle's decode attention over the workload's sequences, cycling through them
    until about `budget_s` seconds of CPU work are done.  Returns (GB/s of KV read, seconds,
    description of the sample)."""
    import oracle.drive as odrive
    pool, _, tables = odrive.build(w)
    q = w.query()  # drawn once: input generation stays outside the timed region
    lens = w.attend_lens.astype(np.int64)
    done_tokens, passes, spent = 0, 0, 0.0
    t0 = time.perf_counter()
    while spent < budget_s:
        for b in range(w.B):
            odrive.attention(w, pool, tables, threads=threads, seqs=[b], q=q)
            done_tokens += int(lens[b])
            spent = time.perf_counter() - t0
            if spent >= budget_s:
                break
        passes += 1
    kv = done_tokens * w.Hkv * 2 * w.D * w.elem_bytes
    return kv / spent / 1e9, spent, f"{done_tokens} context tokens of {w.name} (all heads), sequences in batch order"


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step is a bounded sample of the workload."""
    if rank != 0:
        return
    import oracle.drive as odrive
    w = W.make_workload(args.workload)
    threads = os.cpu_count() or 1
    pool, _, tables = odrive.build(w)
    q = w.query()  # drawn once: input generation stays outside the timed region
    lens = w.attend_lens.astype(np.int64)
    b_mid = int(np.argsort(lens)[len(lens) // 2])
    t0 = time.perf_counter()
    odrive.attention(w, pool, tables, threads=threads, seqs=[b_mid], q=q)
    per_seq = time.perf_counter() - t0
    budget_total = 120.0
    per_step = budget_total / max(1, args.steps + args.warmup)
    # one step = a contiguous slice of heads of one sequence (or a few sequences), sized to the budget
    n_seq = max(1, min(w.B, int(per_step / max(per_seq, 1e-9))))
    seqs = [int(b) for b in np.argsort(lens)[len(lens) // 2:][:n_seq]]
    for _ in range(args.warmup):
        odrive.attention(w, pool, tables, threads=threads, seqs=seqs, q=q)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        odrive.attention(w, pool, tables, threads=threads, seqs=seqs, q=q)
    dt = (time.perf_counter() - t0) / args.steps
    kv = int(lens[seqs].sum()) * w.Hkv * 2 * w.D * w.elem_bytes
    value = kv / dt / 1e9
    sample = f"{len(seqs)} of {w.B} sequences of {w.name} per step ({int(lens[seqs].sum())} tokens, all heads)"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- main arm
def measure_decode(w, args, world, local, stream):
    """One workload's decode step on this rank: K timed fused steps (append + attention), then
    the attention kernel alone (at least 50 launches, one event pair each), the append alone (a
    replayed graph of 50 appends) and the host-driven step through the public API.  Returns the
    workload's record (everything but the CPU baseline) and its DecodeStep."""
    import torch
    from paged_kv_cache_266_gb300 import pkv_check_device_error
    from paged_kv_cache_266_gb300.runner import DecodeStep

    step = DecodeStep(w, device=f"cuda:{local}")
    if args.seqs:
        step.limit_batch(args.seqs)
        w = W.truncated(w, args.seqs)
    nbytes = algorithmic_bytes(w)
    # append kernels per step (bf16: one; one-byte KV: one up to 1024 tokens, else three) + attention
    launches_per_step = append_launches(w.kv_dtype, w.B if w.append else 0, in_step=True) + 1

    for _ in range(args.warmup):
        step.step()
    torch.cuda.synchronize()
    if pkv_check_device_error(step.pool.handle) != 0:
        raise RuntimeError("device error flag set after warm-up")

    K = args.steps
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    # Timed region: K decode steps (append + attention, one pkv_decode_step call each).
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    ev0.record(stream)
    for _ in range(K):
        step.step()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    dist_barrier(world)
    total_ms = ev0.elapsed_time(ev1)
    # The attention kernel on its own (for the roofline): at least 50 launches whatever K is, one
    # event pair each.
    K_attn = max(50, min(K, 2000))
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(K_attn)]
    ev_c = [torch.cuda.Event(enable_timing=True) for _ in range(K_attn)]
    torch.cuda.synchronize()
    for k in range(K_attn):
        ev_b[k].record(stream)
        step.attention()
        ev_c[k].record(stream)
    torch.cuda.synchronize()
    attn_ms = [ev_b[k].elapsed_time(ev_c[k]) for k in range(K_attn)]
    # The append on its own (reported separately): the same step's K/V rewritten into their
    # slots, 50 appends captured in a CUDA graph so the device time is not bounded by how fast
    # the host issues such short launches; median over 10 replays.
    append_us = None
    if w.append:
        n_app = 50
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for _ in range(n_app):
                    step.append(side)
        stream.wait_stream(side)
        g.replay()
        torch.cuda.synchronize()
        reps = []
        for _ in range(10):
            ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ea.record(stream)
            g.replay()
            eb.record(stream)
            torch.cuda.synchronize()
            reps.append(ea.elapsed_time(eb) / n_app * 1e3)
        append_us = round(statistics.median(reps), 2)
    clocks = sampler.stop()
    ms_per_step = dist_max(total_ms / K, world)
    if pkv_check_device_error(step.pool.handle) != 0:
        raise RuntimeError("device error flag set in the timed region")

    value = world * nbytes["step"] / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    attn_mean = statistics.mean(attn_ms)
    achieved = nbytes["attention"] / (attn_mean * 1e-3) / 1e9
    traffic, traffic_note = ncu_traffic(w)

    # end to end through the public API: the caller's host arrays copied into pinned staging, the
    # allocator's tables and slots written there, one copy in, the fused step, the output back
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    for _ in range(2):
        step.step_host()
    t0 = time.perf_counter()
    h2d = d2h = 0
    for _ in range(e2e_steps):
        h2d, d2h = step.step_host()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_s = dist_max(e2e_s, world)
    e2e_value = world * nbytes["step"] / e2e_s / 1e9

    rec = {
        "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(ms_per_step, 5),
        "dtype": f"f32-accumulate on {w.kv_dtype} KV",
        "config": {"workload": w.name, "description": w.description, "batch": w.B, "q_heads": w.Hq,
                   "kv_heads": w.Hkv, "head_dim": w.D, "block_size": w.block_size, "kv_dtype": w.kv_dtype,
                   "context_tokens": int(w.attend_lens.sum()), "kv_bytes_per_step": nbytes["kv"],
                   "step_bytes": nbytes["step"], "l2": "inputs larger than L2 (KV read per step "
                   f"{nbytes['kv'] / 2**20:.0f} MiB > {L2_BYTES // 2**20} MiB)", "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(world * w.B / (ms_per_step * 1e-3), 1),
        "tokens_per_s_unit": "decode tokens per attention layer-step per second",
        "pct_of_hbm_peak": round(100 * value / (world * peak), 2),
        "kernel_us": {"attention": round(attn_mean * 1e3, 2), "attention_median": round(statistics.median(attn_ms) * 1e3, 2),
                      "step": round(ms_per_step * 1e3, 2), "attention_launches_timed": K_attn,
                      "append": append_us},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "traffic_source": traffic_note,
                     "peak_kind": peak_kind, "nominal_peak": NOMINAL_HBM_GBS,
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "kernel": "decode_kernel", "algorithmic_bytes_per_launch": nbytes["attention"]},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_s * 1e3, 4),
                "path": "caller's host q/K/V/lengths copied into pinned staging, allocator tables and slots "
                        "written there, one copy to the device, fused step, output copied back (graph-replayed)"},
        "gpu_launches": K * launches_per_step,
        "clocks": clocks,
        "wall_s_timed": round(t_wall, 3),
    }
    return rec, step, w


def run_pkv(args, world, rank, local):
    import torch
    from paged_kv_cache_266_gb300 import build as pkv_build
    pkv_build.build()

    torch.cuda.set_device(local)
    stream = torch.cuda.current_stream()

    def workload(name):
        w = W.make_workload(name)
        if args.kv and args.kv != w.kv_dtype:  # the same workload over another KV element type
            import dataclasses
            w = dataclasses.replace(w, kv_dtype=args.kv, name=f"{w.name}-{args.kv}")
        return w

    # the headline workload, then the other target workloads as sub-records of the same line
    rec, step, w = measure_decode(workload(args.workload), args, world, local, stream)
    step.close()
    del step
    cpu = None
    if rank == 0 and not args.no_cpu:
        threads = os.cpu_count() or 1
        rate, spent, sample = oracle_rate(w, args.cpu_budget, threads)
        rate1, spent1, sample1 = oracle_rate(w, max(1.0, args.cpu_budget / 3), 1)
        cpu = {"value": round(rate, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{sample}; {spent:.1f} s",
               "single_thread": {"value": round(rate1, 4), "unit": "GB/s", "cores": 1,
                                 "sample": f"{sample1}; {spent1:.1f} s"}}
    others = {}
    for name in [x for x in args.also.split(",") if x and x != args.workload]:
        sub, sstep, _ = measure_decode(workload(name), args, world, local, stream)
        sstep.close()
        del sstep
        torch.cuda.empty_cache()
        others[name] = sub

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": rec["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": rec["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": rec["dtype"], "data": "synthetic", "config": rec["config"],
    }
    for k in ("tokens_per_s", "tokens_per_s_unit", "pct_of_hbm_peak", "kernel_us", "roofline", "e2e", "gpu_launches",
              "clocks"):
        line[k] = rec[k]
    line["cpu_baseline"] = cpu
    line["wall_s_timed"] = rec["wall_s_timed"]
    if others:
        line["configs"] = others
    print(json.dumps(line), flush=True)


def run_loop(args, world, rank, local):
    """In-flight batching decode loop (one layer, Llama-3-8B shapes): sequences finish and join
    every step, blocks grow on demand, each step is a graph-replayed host-to-host decode step."""
    import torch
    from paged_kv_cache_266_gb300 import build as pkv_build
    pkv_build.build()
    import paged_kv_cache_266_gb300 as _pkv
    from paged_kv_cache_266_gb300 import pkv_check_device_error
    from paged_kv_cache_266_gb300.engine import DecodeLoop
    torch.cuda.set_device(local)
    n = args.warmup + args.steps
    sc = W.make_loop_script(index=50, n_steps=n, max_batch=args.loop_batch, Hq=32, Hkv=8, D=128, block_size=64,
                            kv_dtype="bf16", prompt_lo=128, prompt_hi=2048, p_finish=0.01)
    inputs = [sc.step_inputs(t, range(sc.max_batch)) for t in range(n)]
    # joining sequences' prompt K/V staged on the device beforehand (their prefill's output)
    dev = f"cuda:{local}"
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    prompts = {s: tuple(map(to_dev, sc.prompt_kv(s, m))) for _, joined in sc.steps for s, m in joined if m}
    loop = DecodeLoop(sc, graphs=True, device=dev, prompts=prompts)
    # each step's q / new K / new V on the device, where the layer's QKV projection would leave
    # them: the batch's input region of the loop, one device copy per step
    B = sc.max_batch  # the schedule refills the batch every step
    region, qv, kv_, vv = loop.device_input_region(B)
    staged = []
    for t in range(n):
        k, v, q = inputs[t]
        buf = torch.zeros_like(region)
        for view, arr in ((qv, q), (kv_, k), (vv, v)):
            off = view.data_ptr() - region.data_ptr()
            buf[off:off + arr.nbytes].copy_(torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1)))
        staged.append(buf)
    lib = _pkv._L()
    cs = torch.cuda.current_stream().cuda_stream
    copy_args = [(region.data_ptr(), b.data_ptr(), region.numel(), cs) for b in staged]
    for t in range(args.warmup):
        lib.pkv_stage_copy(*copy_args[t])
        loop.step(device_inputs=True)
    loop.timing = {k: 0.0 for k in loop.timing}
    kv_bytes, tokens = 0, 0
    dist_barrier(world)
    t0 = time.perf_counter()
    for t in range(args.warmup, n):
        lib.pkv_stage_copy(*copy_args[t])  # the projection's output, already on the device
        run, _ = loop.step(device_inputs=True)
        tokens += len(run)
        kv_bytes += loop.attended_tokens * sc.Hkv * 2 * sc.D * 2
    dt = dist_max(time.perf_counter() - t0, world)
    if pkv_check_device_error(loop.pool.handle) != 0:
        raise RuntimeError("device error flag set in the decode loop")
    if rank == 0:
        K = args.steps
        print(json.dumps({
            "metric": "in-flight decode loop (one layer): decode tokens/s, KV GB/s", "value": round(world * tokens / dt, 1),
            "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(dt / K * 1e3, 4), "higher_is_better": True, "scaling": "weak",
            "kv_gbs": round(world * kv_bytes / dt / 1e9, 1), "data": "synthetic",
            "config": {"workload": sc.name, "batch": sc.max_batch, "q_heads": sc.Hq, "kv_heads": sc.Hkv, "head_dim": sc.D,
                       "block_size": sc.block_size, "prompts": "U[128,2048]", "finish_prob_per_step": 0.01,
                       "joined": sum(len(j) for _, j in sc.steps[args.warmup:]), "graphs": "one per batch bucket",
                       "step_inputs": "q / new K / new V on the device (the QKV projection's output); block "
                                      "tables, slots and lengths staged on the host and copied in every step"},
            "host_ms_per_step": {k: round(v / K * 1e3, 4) for k, v in loop.timing.items()},
        }), flush=True)
    loop.close()


def run_prefix(args, world, rank, local):
    """Block reuse: 128 children of one 2048-token prompt (Llama-3-8B layer shapes, block 64), each
    with its own U[128,2048] suffix.  The same decode step is timed over the shared pool and over
    an unshared pool holding the same logical contexts; L2 is flushed before every timed step."""
    import torch
    from paged_kv_cache_266_gb300 import build as pkv_build
    pkv_build.build()
    import paged_kv_cache_266_gb300 as pkv
    from paged_kv_cache_266_gb300.runner import PrefixDecode
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    sc = W.make_prefix_script()
    row = sc.Hkv * 2 * sc.D * 2
    logical = int(sc.attend_lens.sum()) * row
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    K = max(3, min(args.steps, 500))
    res = {}
    sampler = ClockSampler(local)
    sampler.start()
    for share in (True, False):
        st = PrefixDecode(sc, share=share, device=dev)
        for _ in range(args.warmup):
            st.step()
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        dist_barrier(world)
        torch.cuda.synchronize()
        for k in range(K):
            flush.zero_()
            e0[k].record(stream)
            st.step()
            e1[k].record(stream)
        torch.cuda.synchronize()
        if pkv.pkv_check_device_error(st.pool.handle) != 0:
            raise RuntimeError("device error flag set in the timed region")
        ms = dist_max(statistics.mean(e0[k].elapsed_time(e1[k]) for k in range(K)), world)
        res[share] = {"ms_per_step": ms, "blocks": st.blocks_held, "cow_copies": st.cow_copies}
        st.close()
    clocks = sampler.stop()
    # host cost of forking: B shares of the P-token prefix on a fresh allocator
    a = pkv.pkv_allocator_create(sc.num_blocks, sc.block_size)
    pkv.pkv_seq_reserve(a, sc.parent, sc.P)
    t0 = time.perf_counter()
    for b in range(sc.B):
        pkv.pkv_seq_share_prefix(a, sc.parent, b, sc.P)
    fork_us = (time.perf_counter() - t0) / sc.B * 1e6
    pkv.pkv_allocator_destroy(a)
    if rank != 0:
        return
    sh, un = res[True], res[False]
    peak, peak_kind = measured_peaks()
    unique = sh["blocks"] * sc.block_size * row
    print(json.dumps({
        "metric": "shared-prefix decode step: logical KV bytes attended per second", "value":
        round(world * logical / (sh["ms_per_step"] * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(sh["ms_per_step"], 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32-accumulate on bf16 KV", "data": "synthetic",
        "config": {"workload": sc.name, "description": "128 children of one 2048-token prompt, suffixes U[128,2048], "
                   "Llama-3-8B layer shapes (32 q / 8 kv heads, head_dim 128), block 64", "batch": sc.B,
                   "prefix_tokens": sc.P, "context_tokens": int(sc.attend_lens.sum()), "logical_kv_bytes": logical,
                   "l2": "flushed before every timed step"},
        "shared": {"blocks_held": sh["blocks"], "pool_bytes_held": unique, "cow_copies": sh["cow_copies"],
                   "ms_per_step": round(sh["ms_per_step"], 5)},
        "unshared": {"blocks_held": un["blocks"], "pool_bytes_held": un["blocks"] * sc.block_size * row,
                     "ms_per_step": round(un["ms_per_step"], 5),
                     "logical_gbs": round(world * logical / (un["ms_per_step"] * 1e-3) / 1e9, 2)},
        "speedup_vs_unshared": round(un["ms_per_step"] / sh["ms_per_step"], 4),
        "pct_of_hbm_peak_logical": round(100 * logical / (sh["ms_per_step"] * 1e-3) / 1e9 / peak, 2),
        "peak": peak, "peak_kind": peak_kind,
        "host_fork_us_per_child": round(fork_us, 3),
        "gpu_launches": K * 2,
        "clocks": clocks,
    }), flush=True)


def run_prefill(args, world, rank, local):
    """Chunked-context prefill step: 8 sequences at seeded points of 32K prompts process one
    512-token chunk each (4096 tokens), Llama-3-8B layer shapes, block 64: append of the chunks'
    K/V then causal attention over past + chunk on the tensor cores."""
    import torch
    from paged_kv_cache_266_gb300 import build as pkv_build
    pkv_build.build()
    import paged_kv_cache_266_gb300 as pkv
    from paged_kv_cache_266_gb300.runner import PrefillStep
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    sc = W.make_prefill_script(kv_dtype=args.kv or "bf16")
    st = PrefillStep(sc, device=dev)
    flops = sc.flops()
    tokens = int(sc.cu_q[-1])
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    K = max(3, min(args.steps, 300))
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)

    def timed(fn):
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        dist_barrier(world)
        torch.cuda.synchronize()
        for k in range(K):
            flush.zero_()
            e0[k].record(stream)
            fn()
            e1[k].record(stream)
        torch.cuda.synchronize()
        return [e0[k].elapsed_time(e1[k]) for k in range(K)]

    step_ms = timed(st.step)
    attn_ms = timed(st.attention)
    clocks = sampler.stop()
    if pkv.pkv_check_device_error(st.pool.handle) != 0:
        raise RuntimeError("device error flag set in the timed region")
    ms = dist_max(statistics.mean(step_ms), world)
    attn = statistics.mean(attn_ms)
    peaks = {}
    pth = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pth):
        with open(pth) as f:
            peaks = json.load(f)
    peak = float(peaks.get("bf16_tflops", 1900.0))
    achieved = flops / (attn * 1e-3) / 1e12
    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = prefill_oracle_rate(sc, args.cpu_budget, os.cpu_count() or 1)
    if rank == 0:
        print(json.dumps({
            "metric": "chunked prefill attention over the paged pool: causal attention TFLOP/s, prompt tokens/s",
            "value": round(world * flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16 MMA, f32 accumulate" if sc.kv_dtype == "bf16" else
                     f"{sc.kv_dtype} pool widened on chip to f16, f16 MMA, f32 accumulate",
            "data": "synthetic",
            "config": {"workload": sc.name if sc.kv_dtype == "bf16" else f"{sc.name}-{sc.kv_dtype}",
                       "description": "8 sequences at seeded points of 32K prompts, one 512-token "
                       "chunk each (4096 tokens per step), Llama-3-8B layer shapes (32 q / 8 kv heads, head_dim 128), "
                       f"block 64, {sc.kv_dtype} pool", "kv_dtype": sc.kv_dtype, "batch": sc.B, "chunk_tokens": tokens, "past_tokens": [int(x) for x in sc.past],
                       "causal_flops_per_step": flops, "l2": "flushed before every timed launch"},
            "tokens_per_s": round(world * tokens / (ms * 1e-3), 1),
            "kernel_us": {"step": round(ms * 1e3, 2), "attention": round(attn * 1e3, 2),
                          "attention_median": round(statistics.median(attn_ms) * 1e3, 2)},
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4), "traffic": None,
                         "peak_kind": "measured" if peaks else "fallback", "kernel": "prefill_kernel",
                         "algorithmic_flops_per_launch": flops},
            "gpu_launches": (append_launches(sc.kv_dtype, tokens) + 1) * K,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }), flush=True)
    st.close()


def run_rope(args, world, rank, local):
    """Decode step with RoPE fused into the append (Llama-3-8B GQA batch of workload c2): the
    step's new K rows and query rows are rotated in the append kernel, then the attention runs
    as its programmatic dependent. Timed beside the same step without RoPE."""
    import torch
    from paged_kv_cache_266_gb300 import build as pkv_build
    pkv_build.build()
    import paged_kv_cache_266_gb300 as pkv
    from paged_kv_cache_266_gb300.runner import DecodeStep
    torch.cuda.set_device(local)
    w = W.make_workload("c2")
    st = DecodeStep(w, device=f"cuda:{local}")
    pos = torch.from_numpy(w.lens.astype(np.int64)).to(st.device)
    base = 500000.0
    nbytes = algorithmic_bytes(w)
    stream = torch.cuda.current_stream()
    K = max(3, min(args.steps, 2000))

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        torch.cuda.synchronize()
        for k in range(K):
            e0[k].record(stream)
            fn()
            e1[k].record(stream)
        torch.cuda.synchronize()
        return statistics.median(e0[k].elapsed_time(e1[k]) for k in range(K))

    sampler = ClockSampler(local)
    sampler.start()
    step_ms = timed(lambda: st.step())
    rope_ms = timed(lambda: pkv.pkv_decode_step_rope(st.pool.handle, st.k_new, st.v_new, st.slots_new, pos, base, st.q,
                                                     st.tables, st.lens, st.scale, st.out, st.workspace))
    append_ms = timed(lambda: st.append())
    append_rope_ms = timed(lambda: pkv.pkv_append_rope(st.pool.handle, st.k_new, st.v_new, st.slots_new, pos, base,
                                                       q=st.q))
    clocks = sampler.stop()
    if pkv.pkv_check_device_error(st.pool.handle) != 0:
        raise RuntimeError("device error flag set")
    if rank == 0:
        print(json.dumps({
            "metric": "decode step with RoPE fused into the append: KV GB/s (c2 batch)",
            "value": round(world * nbytes["step"] / (rope_ms * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(rope_ms, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32-accumulate on bf16 KV; RoPE in fp64",
            "data": "synthetic", "config": {"workload": w.name, "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv,
                                            "head_dim": w.D, "rope_base": base,
                                            "l2": "inputs larger than L2 (KV read per step > L2)"},
            "kernel_us": {"step_without_rope": round(step_ms * 1e3, 2), "step_with_rope": round(rope_ms * 1e3, 2),
                          "append": round(append_ms * 1e3, 2), "append_with_rope_and_q": round(append_rope_ms * 1e3, 2)},
            "gpu_launches": 2 * K,
            "clocks": clocks,
        }), flush=True)
    st.close()


def prefill_oracle_rate(sc, budget_s: float, threads: int):
    """The oracle's causal-attention FLOP rate on a sample of the prefill workload: the first
    rows of sequence chunks, each a one-row chunk at its own position."""
    import oracle
    threads = min(threads, sc.Hkv)  # the oracle runs one (sequence, KV head) unit per thread
    t_start = time.perf_counter()
    flops = 0
    rows = 0
    spent = 0.0  # attention calls only; the pool replica's set-up is not timed
    for b in range(sc.B):
        P, L = int(sc.past[b]), int(sc.ctx[b])
        a = oracle.Allocator(-(-L // sc.block_size) + 1, sc.block_size)
        pool = oracle.Pool(-(-L // sc.block_size) + 1, sc.block_size, sc.Hkv, sc.D, False)
        a.reserve(0, L)
        k, v = sc.kv(b, 0, L)
        pool.append(k, v, a.slot_mapping([0] * L, np.arange(L)))
        tables = a.block_tables([0], -(-L // sc.block_size))
        for i in range(0, int(sc.chunk[b]), 64):
            row = int(sc.cu_q[b]) + i
            q = sc.query(row, row + 1)
            t0 = time.perf_counter()
            pool.prefill_attention(q, np.array([0, 1], np.int32), tables,
                                   np.array([P + i + 1], np.int32), sc.Hq, 1 / math.sqrt(sc.D), threads=threads)
            spent += time.perf_counter() - t0
            flops += 4 * sc.D * sc.Hq * (P + i + 1)
            rows += 1
            if time.perf_counter() - t_start > budget_s:
                break
        if time.perf_counter() - t_start > budget_s:
            break
    return {"value": round(flops / spent / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} query rows (every 64th of each chunk), each over its full causal context; "
                      f"{spent:.1f} s of attention calls"}


def run_chunk_loop(args, world, rank, local):
    """In-flight batching with chunked context (one layer, Llama-3-8B shapes, block 64): joining
    prompts are prefilled 512 tokens per step on the tensor cores while the others decode (the
    scheduling of "TensorRT-LLM 深度实战" §7.3); every step is one prefill call plus one
    graph-replayed decode step."""
    import torch
    from paged_kv_cache_266_gb300 import build as pkv_build
    pkv_build.build()
    from paged_kv_cache_266_gb300 import pkv_check_device_error
    from paged_kv_cache_266_gb300.engine import ChunkedContextScheduler, DecodeLoop
    torch.cuda.set_device(local)
    n = args.warmup + args.steps
    sc = W.make_chunked_loop_script(index=55, n_steps=n, max_batch=args.loop_batch, Hq=32, Hkv=8, D=128,
                                    block_size=64, kv_dtype=args.kv or "bf16", prompt_lo=256, prompt_hi=4096,
                                    p_finish=0.02, chunk=args.chunk, system=args.system, reuse=not args.no_reuse)
    dev = f"cuda:{local}"
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    prompts = {}
    base = sc.system if sc.reuse else 0
    for _, joined in sc.steps:
        for s, m in joined:
            k, v, q = sc.prompt_rows(s, base, sc.system + m)
            prompts[s] = (to_dev(k), to_dev(v), to_dev(q))
    inputs = [None] * n
    loop = DecodeLoop(sc, graphs=True, device=dev, prompts=prompts, system_seq=W.SYSTEM_SEQ)
    sched = ChunkedContextScheduler(sc.chunk, sc.system, sc.reuse)  # the loop's schedule, ahead of time
    plans = []
    joined_at, first_decode = {}, {}
    for t in range(n):  # the decode inputs of each step, drawn before the timed region
        for s_ in sc.steps[t][0]:
            sched.finish(s_)
        for s_, m in sc.steps[t][1]:
            joined_at[s_] = t
            sched.admit(s_, m)
        pre, dec = sched.plan()
        sched.mark_decoded(dec)
        for s_ in dec:
            first_decode.setdefault(s_, t)
        plans.append((sum(p1 - p0 for _, p0, p1 in pre), len(dec)))
        inputs[t] = sc.step_inputs(t, dec) if dec else None
    for t in range(args.warmup):
        loop.step(inputs[t])
    torch.cuda.synchronize()
    loop.timing = {k: 0.0 for k in loop.timing}
    dist_barrier(world)
    t0 = time.perf_counter()
    for t in range(args.warmup, n):
        loop.step(inputs[t])
    torch.cuda.synchronize()
    dt = dist_max(time.perf_counter() - t0, world)
    if pkv_check_device_error(loop.pool.handle) != 0:
        raise RuntimeError("device error flag set in the chunked loop")
    pre_tok = sum(p[0] for p in plans[args.warmup:])
    dec_tok = sum(p[1] for p in plans[args.warmup:])
    ttft = [first_decode[s_] - joined_at[s_] for s_ in first_decode if joined_at[s_] >= args.warmup]
    if rank == 0:
        K = args.steps
        print(json.dumps({
            "metric": "in-flight loop with chunked context (one layer): prompt + decode tokens/s",
            "value": round(world * (pre_tok + dec_tok) / dt, 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(dt / K * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 KV; bf16 MMA / f32 accumulate" if sc.kv_dtype == "bf16" else
                     f"{sc.kv_dtype} KV; f16 MMA / f32 accumulate", "data": "synthetic",
            "config": {"workload": sc.name if sc.kv_dtype == "bf16" else f"{sc.name}-{sc.kv_dtype}",
                       "kv_dtype": sc.kv_dtype, "batch": sc.max_batch, "q_heads": sc.Hq, "kv_heads": sc.Hkv,
                       "head_dim": sc.D, "block_size": sc.block_size, "chunk": sc.chunk, "prompts": "U[256,4096]",
                       "finish_prob_per_step": 0.02, "graphs": "decode: one per batch bucket"},
            "prompt_tokens_per_s": round(world * pre_tok / dt, 1), "decode_tokens_per_s": round(world * dec_tok / dt, 1),
            "system_prompt": {"tokens": sc.system, "cached": bool(sc.system and sc.reuse)},
            "first_token_steps_mean": round(float(np.mean(ttft)), 3) if ttft else None,
            "first_token_ms_mean": round(float(np.mean(ttft)) * dt / K * 1e3, 3) if ttft else None,
            "host_ms_per_step": {k: round(v / K * 1e3, 4) for k, v in loop.timing.items()},
        }), flush=True)
    loop.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--workload", default="c3", choices=list(W.WORKLOADS))
    ap.add_argument("--also", default="c1,c2,c4",
                    help="workloads measured after the headline one, reported as sub-records ('' for none)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--seqs", type=int, default=0, help="profiling: step over the first N sequences only")
    ap.add_argument("--loop", action="store_true", help="measure the in-flight decode loop instead of one step")
    ap.add_argument("--loop-batch", type=int, default=128)
    ap.add_argument("--chunk", type=int, default=0, help="with --loop: chunked context, prompt tokens per step")
    ap.add_argument("--system", type=int, default=0, help="with --chunk: a shared system prompt of this many tokens")
    ap.add_argument("--no-reuse", action="store_true", help="with --system: every request prefills it")
    ap.add_argument("--prefix", action="store_true", help="measure decode over children of a shared prompt prefix")
    ap.add_argument("--prefill", action="store_true", help="measure the chunked-context prefill step")
    ap.add_argument("--rope", action="store_true", help="measure the decode step with RoPE fused into the append")
    ap.add_argument("--kv", default="", choices=["", "bf16", "fp8_e4m3", "int8"],
                    help="override the workload's KV element type")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.loop and args.chunk:
        run_chunk_loop(args, world, rank, local)
    elif args.loop:
        run_loop(args, world, rank, local)
    elif args.prefix:
        run_prefix(args, world, rank, local)
    elif args.prefill:
        run_prefill(args, world, rank, local)
    elif args.rope:
        run_rope(args, world, rank, local)
    else:
        run_pkv(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
