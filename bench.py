#!/usr/bin/env python
"""Aggregate greedy decode throughput of decode_step_batch on the 7B-shaped decoder.

Default workload: 32 layers, d_model 4096, 32 q / 8 kv heads (head_dim 128), SwiGLU 14336,
vocab 32000, bf16 seeded N(0, 0.02) weights; B = 8 persistent KV slabs whose context lengths
are uniform in [512, 4096] (seeded synthetic KV); greedy decode, each step feeding the
previous step's device-side next tokens.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

--impl reference times the CPU oracle on the same workload (a bounded sample of steps).
Multi-GPU runs are independent replicas (one engine and weight copy per GPU, rows never
exchange data); value = all ranks' tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "aggregate decode tok/s at B=1..32 (7B-shape) + % of HBM roofline per step"
NOMINAL_HBM_GBS = 8000.0


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


def measured_traffic(kind: str):
    """DRAM bytes (read + write) of one launch of the kernel, from the ncu capture summarised in
    profiles/traffic.json -- or None when the kernel's source changed since that capture."""
    import hashlib
    try:
        info = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))[kind]
        h = hashlib.sha256()
        for f in info.get("sources", [info.get("source")]):
            h.update(open(os.path.join(ROOT, f), "rb").read())
        if h.hexdigest() != info["sha256"]:
            return None
        return info["dram_bytes_per_launch"]
    except Exception:
        return None


def workload_by_name(name: str, layers: int | None = None):
    """A named decode workload; `layers` keeps every shape but the depth (used only to profile
    single kernels on a small device footprint; the JSON line then names the reduced model)."""
    wl = _workload_by_name(name)
    if layers:
        from dataclasses import replace
        shape = replace(wl.shape, n_layers=layers, name=f"{wl.shape.name}-{layers}-layers")
        wl = replace(wl, shape=shape, name=f"{wl.name}-{layers}-layers")
    return wl


def _workload_by_name(name: str):
    from synth.recipes import DECODE_7B_B8, LONG_7B_B32, decode_7b_fixed
    if name == "7b-bf16-b8":
        return DECODE_7B_B8
    if name == "7b-bf16-b32-long":
        return LONG_7B_B32
    if name.startswith("7b-bf16-b") and name.endswith("-ctx2048"):
        return decode_7b_fixed(int(name[len("7b-bf16-b"):-len("-ctx2048")]), 2048, "bf16")
    if name.startswith("7b-affine4-b") and name.endswith("-ctx2048"):
        return decode_7b_fixed(int(name[len("7b-affine4-b"):-len("-ctx2048")]), 2048, "affine4")
    raise SystemExit(f"unknown workload {name}")


def step_bytes(shape, ctx_lens, kv_bits: int = 16) -> float:
    """Algorithmic HBM bytes of one decode step: every linear weight once, each row's live KV
    (positions 0..t_b after the append) once, the appended K/V, the logits written.  Quantised
    KV: kv_bits / 8 bytes of code per element plus a bf16 scale and bias per 64 elements."""
    kv_tok = shape.kv_bytes_per_token() * ((kv_bits / 8 + 1 / 16) / 2 if kv_bits in (4, 8) else 1.0)
    return float(shape.weight_bytes_per_step() + sum((int(c) + 1) * kv_tok for c in ctx_lens)
                 + len(ctx_lens) * (kv_tok + 4 * shape.vocab))


def projection_bytes(shape, n: int) -> float:
    """Algorithmic bytes of one step's projections: every weight once, the operand rows in
    (fp32 activations), the outputs out (twice for a residual add)."""
    d, qd, kvd, F, V = shape.d_model, shape.q_dim, shape.kv_dim, shape.d_ff, shape.vocab
    act = shape.n_layers * (4 * n * (d + qd + 2 * kvd) + 4 * n * (qd + 2 * d) + 4 * n * (d + F)
                            + 4 * n * (F + 2 * d)) + 4 * n * (d + V)
    return float(shape.weight_bytes_per_step() + act)


def attention_bytes(shape, ctx_lens, kv_bits: int = 16) -> float:
    """Algorithmic bytes of one step's attention: each row's live KV once (positions 0..t_b),
    the new K/V appended, q in and o out, over every layer."""
    kv_tok = shape.kv_bytes_per_token() * ((kv_bits / 8 + 1 / 16) / 2 if kv_bits in (4, 8) else 1.0)
    n = len(ctx_lens)
    return float(sum((int(c) + 1) * kv_tok for c in ctx_lens) + n * kv_tok
                 + shape.n_layers * n * 4 * 2 * shape.q_dim)


def interval_union_ns(iv) -> float:
    """Total length of the union of [begin, end] intervals."""
    tot, cur_b, cur_e = 0, None, None
    for b, e in sorted(iv):
        if cur_e is None or b > cur_e:
            if cur_e is not None:
                tot += cur_e - cur_b
            cur_b, cur_e = b, e
        else:
            cur_e = max(cur_e, e)
    if cur_e is not None:
        tot += cur_e - cur_b
    return float(tot)


def stamped_class_times(eng, step, i0: int, n_steps: int):
    """Median over n_steps replayed steps of the projection and attention classes' time in the
    step (ms), from the engine's stamps; and the projection launches per step."""
    from continuous_batching_transformer_gb300 import binding as B
    B.engine_set_stamps(eng.handle, True)
    for i in range(i0, i0 + 2):  # capture the stamped step
        step(i)
    proj, attn, n_proj = [], [], 0
    for i in range(i0 + 2, i0 + 2 + n_steps):
        step(i)
        recs = B.engine_stamps(eng.handle)
        p_iv = [(b, e) for c, b, e in recs if c == B.KCLASS_PROJ and e >= b]
        a_iv = [(b, e) for c, b, e in recs if c == B.KCLASS_ATTN and e >= b]
        proj.append(interval_union_ns(p_iv) / 1e6)
        attn.append(interval_union_ns(a_iv) / 1e6)
        n_proj = len(p_iv)
    B.engine_set_stamps(eng.handle, False)
    return statistics.median(proj), statistics.median(attn), n_proj


# ---- clocks sampled during the timed region ---------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.tmp = tempfile.NamedTemporaryFile(prefix="clocks", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.close()
        rows = list(csv.reader(io.StringIO(open(self.tmp.name).read())))
        os.unlink(self.tmp.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for nm, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- the GPU arm ------------------------------------------------------------------------------
def setup_decode(wl, device, extra_positions: int, page_tokens: int = 0, kv_bits: int = 16,
                 weights=None):
    """Engine + slabs for a decode workload: synthetic KV of each row loaded into its slab,
    each row's next token ready on the device.  page_tokens > 0: a paged engine; kv_bits = 8:
    quantised KV (the arena also holds the decode rows' staging and one import's bf16 slab).
    weights: DeviceWeights of the workload's shape to reuse (else they are drawn here)."""
    import numpy as np
    import torch

    from continuous_batching_transformer_gb300 import binding as B
    from continuous_batching_transformer_gb300.model import DeviceWeights, Engine

    shape = wl.shape
    ctx = [int(c) for c in wl.context_lengths()]
    caps = [c + extra_positions for c in ctx]
    w = weights if weights is not None else DeviceWeights(shape, device)
    if page_tokens:
        arena = sum(B.slab_bytes(w.cfg, page_tokens) * (-(-c // page_tokens)) for c in caps)
    elif kv_bits in (4, 8):
        arena = (sum(B.slab_bytes_kvq(w.cfg, c, kv_bits) for c in caps) + B.slab_bytes(w.cfg, max(ctx))
                 + len(ctx) * B.slab_bytes(w.cfg, 128))
    else:
        arena = sum(B.slab_bytes(w.cfg, c) for c in caps)
    eng = Engine(w, arena_bytes=arena, max_batch=len(ctx), max_prefill_tokens=len(ctx),
                 page_tokens=page_tokens, kv_bits=kv_bits)
    slabs = []
    for r, (c, cap) in enumerate(zip(ctx, caps)):
        s = eng.kv_slab_alloc(cap)
        eng.fill_synthetic_kv(s, r, c, wl.seed)
        slabs.append(s)
    first = np.array([wl.row_tokens(r, c + 1)[c] for r, c in enumerate(ctx)], dtype=np.int32)
    tok = torch.from_numpy(first).to(device)
    return w, eng, slabs, ctx, tok


def slowest_over_ranks(seconds: float, dist=None, device=None) -> float:
    """The largest of every rank's `seconds` (each replica times its own steps; the job takes
    as long as the slowest).  Without a process group, the value itself."""
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replicas_throughput(rows_per_rank: int, steps: int, world: int, slowest_s: float) -> float:
    """Whole-job tokens per second of `world` independent replicas: every rank decodes
    `rows_per_rank` rows for `steps` steps; the job ends with the slowest rank."""
    return rows_per_rank * steps * world / slowest_s


def gpu_arm(args, rank: int, world: int):
    import torch

    import continuous_batching_transformer_gb300 as cbt
    from continuous_batching_transformer_gb300 import binding as B

    local = int(os.environ.get("LOCAL_RANK", "0"))
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    if rank == 0 or not os.path.exists(cbt._build.LIB):
        cbt.build()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        dist.barrier()
    wl = workload_by_name(args.workload, args.layers)
    K, W = args.steps, args.warmup
    w, eng, slabs, ctx, tok0 = setup_decode(wl, device, extra_positions=3 * (K + W) + 8,
                                            page_tokens=args.page_tokens, kv_bits=args.kv_bits)
    Bsz = len(slabs)
    V = wl.shape.vocab
    stream = eng.stream
    bufs = [tok0.clone(), torch.empty_like(tok0)]
    logits = torch.empty((Bsz, V), dtype=torch.float32, device=device)

    def step(i):
        eng.decode_step_batch(slabs, bufs[i % 2], logits, bufs[(i + 1) % 2])

    for i in range(W):
        step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_uuid = None
    try:
        gpu_uuid = str(torch.cuda.get_device_properties(device).uuid)
        if not gpu_uuid.startswith("GPU-"):
            gpu_uuid = "GPU-" + gpu_uuid
    except Exception:
        pass
    clocks = ClockSampler(gpu_uuid) if rank == 0 else None
    launches0 = B.kernel_launches(eng.handle)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(W, W + K):
            step(i)
        ev1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    launches = B.kernel_launches(eng.handle) - launches0
    ms = ev0.elapsed_time(ev1)
    clk = clocks.stop() if clocks else None
    # Kernel rooflines inside the replayed step: with stamps on, every projection and attention
    # launch of a step records when its CTAs could start dependent work and when the last one
    # ended (globaltimer); a class's time in the step is the union of its launches' intervals.
    KT = max(4, min(K, 16))
    proj_ms, attn_ms, proj_n = stamped_class_times(eng, step, W + K, KT)
    ms_max = slowest_over_ranks(ms, dist, device)
    code, info = eng.device_error()
    if code != 0:
        raise SystemExit(f"device error word set: code {code} info {info}")

    # end to end through the public API with host buffers: tokens in from pinned host memory,
    # next tokens back to the host, every step
    h_tok = torch.empty(Bsz, dtype=torch.int32, pin_memory=True)
    h_out = torch.empty(Bsz, dtype=torch.int32, pin_memory=True)
    h_tok.copy_(bufs[(W + K + KT + 2) % 2].cpu())
    d_tok = torch.empty_like(tok0)
    d_out = torch.empty_like(tok0)
    for i in range(3):
        d_tok.copy_(h_tok, non_blocking=True)
        eng.decode_step_batch(slabs, d_tok, None, d_out)
        h_out.copy_(d_out, non_blocking=True)
        stream.synchronize()
        h_tok.copy_(h_out)
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(K):
            d_tok.copy_(h_tok, non_blocking=True)
            eng.decode_step_batch(slabs, d_tok, None, d_out)
            h_out.copy_(d_out, non_blocking=True)
            stream.synchronize()
            h_tok.copy_(h_out)
    e2e_s = time.perf_counter() - t0
    e2e_s = slowest_over_ranks(e2e_s, dist, device)

    result = None
    ctx_mean = [c + W + K / 2.0 for c in ctx]  # mean live context over the timed steps
    if rank == 0:
        peaks = measured_peaks()
        hbm_peak = peaks["hbm_gbs"] if peaks else 6800.0
        peak_src = "of measured" if peaks else "of fallback"
        sb = step_bytes(wl.shape, ctx_mean, args.kv_bits)
        step_s = ms_max / K / 1e3
        proj_bytes = projection_bytes(wl.shape, Bsz)
        attn_bytes = attention_bytes(wl.shape, ctx_mean, args.kv_bits)
        achieved = proj_bytes / (proj_ms / 1e3) / 1e9 if proj_ms > 0 else None
        attn_gbs = attn_bytes / (attn_ms / 1e3) / 1e9 if attn_ms > 0 else None
        step_ms = ms_max / K
        if wl.shape.weight_format == "bf16":
            traffic = measured_traffic("projection")
        else:  # the 4-bit projections stream their weights once up to 16 rows, then per 16
            traffic = measured_traffic("projection_affine4")
            traffic = traffic * ((Bsz + 15) // 16) if traffic is not None else None
        result = {
            "metric": METRIC,
            "value": replicas_throughput(Bsz, K, world, ms_max / 1e3),
            "unit": "tok/s",
            "n_gpus": world,
            "steps": K,
            "warmup": W,
            "ms_per_step": ms_max / K,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": ("bf16" if wl.shape.weight_format == "bf16" else "affine4-w/bf16")
                     + (f"/kv-affine{args.kv_bits}" if args.kv_bits in (4, 8) else ""),
            "data": "synthetic (seeded N(0,0.02) weights, seeded KV slabs and tokens)",
            "config": {"workload": wl.name, "shape": wl.shape.name, "batch_per_gpu": Bsz,
                       "kv_page_tokens": args.page_tokens, "kv_bits": args.kv_bits,
                       "ctx_lengths": ctx, "parallelism": f"replicas x{world}" if world > 1 else "1 gpu",
                       "l2": "inputs larger than L2 (weights alone are %.1f GB per step)"
                             % (wl.shape.weight_bytes_per_step() / 1e9)},
            "step_roofline": {"algorithmic_bytes_per_step": sb,
                              "achieved_gbs": sb / step_s / 1e9,
                              "frac_of_8TBps": sb / step_s / 1e9 / NOMINAL_HBM_GBS,
                              "frac_of_measured_hbm": sb / step_s / 1e9 / hbm_peak},
            "roofline": {"kernel": "projection kernels (QKV, O, gate/up+SwiGLU, down, lm_head)",
                         "bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                         "peak_source": peak_src, "unit": "GB/s",
                         "frac": achieved / hbm_peak if achieved else None,
                         "share_of_step": proj_ms / step_ms if step_ms > 0 else None,
                         "launches_per_step": proj_n, "stamped_steps": KT,
                         "timing": "in the replayed step: union of the launches' globaltimer "
                                   "intervals, median over the stamped steps",
                         "traffic": traffic},
            "attention_roofline": {"kernel": "RoPE + KV append + split-K decode attention + merge",
                                   "bound": "hbm", "achieved": attn_gbs, "peak": hbm_peak,
                                   "unit": "GB/s",
                                   "frac": attn_gbs / hbm_peak if attn_gbs else None,
                                   "share_of_step": attn_ms / step_ms if step_ms > 0 else None},
            "e2e": {"value": replicas_throughput(Bsz, K, world, e2e_s), "unit": "tok/s",
                    "h2d_bytes_per_step": 4 * Bsz, "d2h_bytes_per_step": 4 * Bsz},
            "gpu_launches": int(launches),
            "clocks": clk,
        }
    eng.close()
    if result is not None and world == 1 and not args.no_sweep and not args.layers:
        result["sweep"] = sweep_arm(device, w, 10, 3, result["roofline"]["peak"])
    if dist:
        dist.destroy_process_group()
    return result


def time_steps(eng, slabs, tok0, steps: int, warmup: int) -> float:
    """Milliseconds per greedy decode step (the captured step replayed), CUDA events on the
    engine stream around `steps` steps after `warmup` untimed ones."""
    import torch
    bufs = [tok0.clone(), torch.empty_like(tok0)]
    for i in range(warmup):
        eng.decode_step_batch(slabs, bufs[i % 2], None, bufs[(i + 1) % 2])
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(eng.stream):
        ev0.record(eng.stream)
        for i in range(warmup, warmup + steps):
            eng.decode_step_batch(slabs, bufs[i % 2], None, bufs[(i + 1) % 2])
        ev1.record(eng.stream)
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1) / steps


SWEEP = ([f"7b-bf16-b{b}-ctx2048" for b in (1, 2, 4, 8, 16, 32)] + ["7b-bf16-b32-long"]
         + [f"7b-affine4-b{b}-ctx2048" for b in (1, 2, 4, 8, 16, 32)])


def sweep_arm(device, bf16_weights, steps: int, warmup: int, hbm_peak: float):
    """The batch-size sweep of the metric: bf16 and 4-bit weights at B = 1..32 (context 2048)
    and the long-context workload (32 rows of 8k-16k positions), each timed like the headline
    line, with its own step roofline."""
    import torch

    from continuous_batching_transformer_gb300.model import DeviceWeights
    from synth.recipes import MISTRAL_7B_Q4

    out = []
    q4 = None
    for name in SWEEP:
        wl = workload_by_name(name)
        if wl.shape.weight_format == "bf16":
            w = bf16_weights
        else:
            if q4 is None:
                q4 = DeviceWeights(MISTRAL_7B_Q4, device)
            w = q4
        _, eng, slabs, ctx, tok0 = setup_decode(wl, device, extra_positions=steps + warmup + 4,
                                                weights=w)
        ms = time_steps(eng, slabs, tok0, steps, warmup)
        code, info = eng.device_error()
        eng.close()
        del eng
        torch.cuda.empty_cache()
        if code != 0:
            raise SystemExit(f"{name}: device error word set: code {code} info {info}")
        ctx_mean = [c + warmup + steps / 2.0 for c in ctx]
        sb = step_bytes(wl.shape, ctx_mean)
        gbs = sb / (ms / 1e3) / 1e9
        out.append({"workload": wl.name, "batch": len(ctx), "ms_per_step": ms,
                    "tok_s": len(ctx) / (ms / 1e3), "algorithmic_bytes_per_step": sb,
                    "achieved_gbs": gbs, "frac_of_8TBps": gbs / NOMINAL_HBM_GBS,
                    "frac_of_measured_hbm": gbs / hbm_peak})
    del q4
    torch.cuda.empty_cache()
    return out


# ---- the oracle (CPU) ----------------------------------------------------------------------------
def oracle_decode_sample(wl, max_steps: int, budget_s: float, kv_bits: int = 16):
    """Time the oracle's batched decode step on the same workload (KV in the same format): all
    rows, weights streamed once per step, for up to max_steps steps or until budget_s has
    passed."""
    import numpy as np

    import oracle
    m = oracle.OracleModel(wl.shape)
    ctx = [int(c) for c in wl.context_lengths()]
    caches = []
    for r, c in enumerate(ctx):
        kc = oracle.KVCache(wl.shape, c + max_steps + 2, kv_bits=kv_bits)
        kc.fill_synthetic(r, c, wl.seed)
        caches.append(kc)
    feed = np.array([wl.row_tokens(r, c + 1)[c] for r, c in enumerate(ctx)], dtype=np.int32)
    done, t_total = 0, 0.0
    while done < max_steps and (done == 0 or t_total < budget_s):
        t0 = time.perf_counter()
        lg = oracle.decode_step_batch(m, caches, feed)
        t_total += time.perf_counter() - t0
        feed = lg.argmax(axis=1).astype(np.int32)
        done += 1
    return {"value": len(ctx) * done / t_total, "unit": "tok/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{done} decode step(s) of all {len(ctx)} rows of {wl.name} "
                      f"(full 32-layer model, {f'{kv_bits}-bit' if kv_bits in (4, 8) else 'bf16'} KV, "
                      f"{t_total:.1f} s of CPU time)"}, done, t_total


def reference_arm(args, rank: int):
    if rank != 0:
        return None
    wl = workload_by_name(args.workload, args.layers)
    cb, done, t_total = oracle_decode_sample(wl, max_steps=max(1, args.steps),
                                             budget_s=args.reference_budget, kv_bits=args.kv_bits)
    return {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "tok/s",
            "n_gpus": 0, "steps": done, "warmup": 0, "ms_per_step": 1e3 * t_total / done,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, "shape": wl.shape.name,
                                            "batch_per_gpu": len(wl.context_lengths()),
                                            "kv_bits": args.kv_bits},
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


TRACE_METRIC = "aggregate decode tok/s over a continuous-batching request trace (7B-shape)"


def trace_arm(args):
    """Continuous batching over the 64-request trace (Poisson 2 req/s, prompts U[256, 4096],
    outputs geometric with mean 256, live cap 8): every generated token over the wall-clock
    time, with time to first token, time per output token and the decode steps' roofline
    fraction.  `7b-bf16-trace` waits for the arrival times; `7b-bf16-trace-t0` lets every
    request arrive at t = 0 (a throughput replay).  `-chunked` in the name admits prompts in
    chunks of 2048 tokens with one decode step between chunks (the batching design's joiner
    prefill) instead of whole prompts at a boundary."""
    import numpy as np
    import torch

    import continuous_batching_transformer_gb300 as cbt
    from continuous_batching_transformer_gb300 import binding as B
    from continuous_batching_transformer_gb300.model import DeviceWeights, Engine
    from continuous_batching_transformer_gb300.trace import decode_gaps, percentiles, run_trace
    from synth.recipes import MISTRAL_7B, Request, agent_requests, trace_requests

    device = torch.device("cuda:0")
    torch.cuda.set_device(device)
    cbt.build()
    agents = "-agents" in args.workload
    realtime = not (args.workload.endswith("-t0") or agents)
    chunk = 2048 if "-chunked" in args.workload else None
    reuse = "share" if "-share" in args.workload else ("-reuse" in args.workload)
    if agents:  # 32 sub-agents sharing a 2048-token system prompt, all arriving at t = 0
        seed = 2
        reqs = agent_requests(32, 2048, 64, 512, 128.0, 1024, seed)
    else:
        seed = 1
        reqs = trace_requests(64, 2.0, 256, 4096, 256.0, 4096, seed)
    live_cap = 8
    w = DeviceWeights(MISTRAL_7B, device)
    cap = max(r.prompt_len + r.output_len for r in reqs) + 8
    arena = (live_cap + 1) * B.slab_bytes(w.cfg, cap)  # + a shared prefix's own slab
    # the agents' slabs differ in size and come and go: paged KV, so no extent fragments
    page = 128 if agents else 0
    if page:
        arena = (live_cap + 1) * B.slab_bytes(w.cfg, page) * (-(-cap // page))
    eng = Engine(w, arena_bytes=arena, max_batch=live_cap, page_tokens=page,
                 max_prefill_tokens=live_cap * max(r.prompt_len for r in reqs))
    # warm-up: every batch size once (captured decode steps), prefill of short prompts
    warm = [Request(0.0, 64, 4 + 2 * i, 900 + i) for i in range(live_cap)]
    run_trace(eng, warm, seed, live_cap=live_cap)
    launches0 = B.kernel_launches()
    clk = ClockSampler(None)
    res = run_trace(eng, reqs, seed, live_cap=live_cap, realtime=realtime, chunk_tokens=chunk,
                    reuse_prefix=reuse)
    clocks = clk.stop()
    launches = B.kernel_launches() - launches0
    shape = MISTRAL_7B
    kv_tok = shape.kv_bytes_per_token()
    step_frac = [(shape.weight_bytes_per_step() + kv * kv_tok) / t / 1e9 / NOMINAL_HBM_GBS
                 for kv, t in zip(res.step_kv_tokens, res.step_s)]
    out = {
        "metric": TRACE_METRIC, "value": res.generated / res.wall_s, "unit": "tok/s",
        "n_gpus": 1, "steps": res.steps, "warmup": len(warm),
        "ms_per_step": 1e3 * float(np.mean(res.step_s)) if res.step_s else None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded weights, prompts and arrival times)",
        "config": {"workload": ("agents-32req-prefix2048" if agents else
                                "trace-64req-poisson2-" + ("realtime" if realtime else "t0"))
                               + ("-chunk2048" if chunk else "") + ("-prefix-share" if reuse == "share" else
                                  "-prefix-reuse" if reuse else ""),
                   "shape": shape.name, "live_cap": live_cap, "admission_chunk": chunk,
                   "kv_page_tokens": page,
                   "parallelism": "1 gpu"},
        "trace": {"requests": len(reqs), "generated_tokens": res.generated,
                  "wall_s": res.wall_s, "decode_steps": res.steps,
                  "mean_live_rows": float(np.mean(res.step_rows)) if res.step_rows else 0.0,
                  "prefill_tokens": res.prefill_tokens, "prefill_s": res.prefill_s,
                  "kv_bytes_peak": res.kv_bytes_peak,
                  "decode_s": float(np.sum(res.step_s)),
                  "ttft_s": percentiles(res.ttft_s.values()),
                  "tpot_s": percentiles(res.tpot_s.values()),
                  "decode_gap_s": percentiles(decode_gaps(res), (50, 95, 100)),
                  "decode_step_frac_of_8TBps": percentiles(step_frac, (5, 50, 95))},
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    eng.close()
    return out


PREFILL_METRIC = "segmented prefill tok/s (7B-shape, prompts packed into one call)"


def prefill_flops(shape, seg_lens) -> float:
    """Useful FLOPs of one segmented-prefill call: every prompt token through every linear
    layer, lm_head for each segment's last token only, and causal attention inside each
    segment (Q.K^T and P.V over the keys [0, j] of query j)."""
    T = sum(seg_lens)
    layer_params = shape.linear_params() - shape.vocab * shape.d_model
    pairs = sum(n * (n + 1) // 2 for n in seg_lens)
    attn = shape.n_layers * shape.n_heads * 4.0 * shape.head_dim * pairs
    return 2.0 * layer_params * T + 2.0 * shape.vocab * shape.d_model * len(seg_lens) + attn


def prefill_arm(args):
    """Admission throughput: `7b-{bf16,affine4}-prefill` packs 4 prompts of 1024 seeded tokens
    into one prefill_segmented call on fresh slabs, K timed calls after W warm-up calls, each
    between CUDA events on the engine stream.  `roofline` is the tensor-core bound: useful
    FLOPs per call over the call's time against the measured bf16 peak (the kernels run every
    product on bf16 hi + lo operand parts, so the MMA work issued is about twice the useful
    FLOPs)."""
    import torch

    import continuous_batching_transformer_gb300 as cbt
    from continuous_batching_transformer_gb300 import binding as B
    from continuous_batching_transformer_gb300.model import DeviceWeights, Engine
    from synth.recipes import MISTRAL_7B, MISTRAL_7B_Q4

    device = torch.device("cuda:0")
    torch.cuda.set_device(device)
    cbt.build()
    shape = MISTRAL_7B_Q4 if args.workload.startswith("7b-affine4") else MISTRAL_7B
    if args.layers:
        from dataclasses import replace
        shape = replace(shape, n_layers=args.layers, name=f"{shape.name}-{args.layers}-layers")
    seg_lens = [1024] * 4
    T = sum(seg_lens)
    w = DeviceWeights(shape, device)
    arena = (len(seg_lens) + 1) * B.slab_bytes(w.cfg, max(seg_lens))
    eng = Engine(w, arena_bytes=arena, max_batch=8, max_prefill_tokens=T)
    gen = torch.Generator().manual_seed(7)
    toks = torch.randint(0, shape.vocab, (T,), generator=gen, dtype=torch.int32).to(device)
    logits = torch.empty(len(seg_lens), shape.vocab, dtype=torch.float32, device=device)
    nxt = torch.empty(len(seg_lens), dtype=torch.int32, device=device)
    st = eng.stream
    times = []
    launches0 = None
    clk = None
    for i in range(args.warmup + args.steps):
        if i == args.warmup:
            torch.cuda.synchronize()
            launches0 = B.kernel_launches()
            clk = ClockSampler(None)
        slabs = [eng.kv_slab_alloc(n) for n in seg_lens]
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        eng.prefill_segmented(slabs, seg_lens, toks, logits, nxt)
        e1.record(st)
        st.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1) / 1e3)
        for s in slabs:
            eng.kv_slab_free(s)
    clocks = clk.stop()
    launches = B.kernel_launches() - launches0
    code, info = eng.device_error()
    if code != 0:
        raise SystemExit(f"device error {code} ({info}) during prefill")
    t = statistics.median(times)
    flops = prefill_flops(shape, seg_lens)
    peaks = measured_peaks() or {}
    peak = peaks.get("bf16_tflops_sustained") or peaks.get("bf16_tflops")
    achieved = flops / t / 1e12
    out = {
        "metric": PREFILL_METRIC, "value": T / t, "unit": "tok/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 (hi+lo operand parts)" if shape.weight_format == "bf16" else "affine4 weights",
        "data": "synthetic (seeded weights and prompt tokens)",
        "config": {"workload": f"prefill-{len(seg_lens)}x{seg_lens[0]}", "shape": shape.name,
                   "tokens_per_call": T, "parallelism": "1 gpu",
                   "l2": "weights and activations stream from HBM; no flush between calls"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak if peak else None, "traffic": None,
                     "of": "measured bf16 sustained", "useful_tflop_per_call": flops / 1e12},
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    eng.close()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="7b-bf16-b8")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the B = 1..32 sweep (bf16 and 4-bit, ctx 2048) and the long-context "
                         "line that the default run appends as 'sweep'")
    ap.add_argument("--reference-budget", type=float, default=60.0)
    ap.add_argument("--kv-bits", type=int, default=16, choices=(4, 8, 16),
                    help="KV precision: 16 (bf16), 8 or 4 (affine, groups of 64)")
    ap.add_argument("--page-tokens", type=int, default=0,
                    help="paged KV with pages of this many positions (a multiple of 128)")
    ap.add_argument("--layers", type=int, default=None,
                    help="profiling aid: same shapes, fewer layers (small device footprint)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "gb300" and args.workload.startswith(("7b-bf16-trace", "7b-bf16-agents")):
        res = trace_arm(args)
    elif args.impl == "gb300" and args.workload.endswith("-prefill"):
        res = prefill_arm(args)
    elif args.impl == "reference":
        res = reference_arm(args, rank)
    else:
        res = gpu_arm(args, rank, world)
        if rank == 0 and not args.no_cpu_baseline:
            wl = workload_by_name(args.workload, args.layers)
            cb, _, _ = oracle_decode_sample(wl, max_steps=2, budget_s=15.0, kv_bits=args.kv_bits)
            res["cpu_baseline"] = cb
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
