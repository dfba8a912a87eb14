"""Decode-step benchmark: tokens/s and us/token of the captured step on GB300,
achieved HBM bandwidth against the roofline, the fp64 oracle timed beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 8b] [--impl ours|reference]

One step = one replay of the whole captured decode step (embedding, every
layer's norm/QKV/RoPE/KV-write/attention/O-proj/norm/SwiGLU MLP, final norm,
LM head, greedy argmax) over one batch of `rows` tokens.  value = tokens/s with
the slot records already in device memory (one device-to-device slot copy and
one graph launch per step); e2e = the same through dec_step with host buffers
(slot write host->device, launch, id + non-finite flag readback, bounded wait).
With --gpus N > 1 (torchrun) every rank runs an independent replica: the path
does not shard, so there is no collective on the data path.
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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s and µs/token at 1 GB300; achieved HBM GB/s vs roofline"
# committed ncu summaries: DRAM bytes per launch of the roofline kernel, valid while its source is unchanged
# (the graph strategy has no full-size capture of its gate/up GEMV committed: its traffic stays null)
PROFILES = {"persistent": (os.path.join(ROOT, "profiles", "persist_step_8b.md"), "persist.cu")}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _describe(wl, positions):
    lay = "paged KV (%d-token pages, pool %d)" % (wl.page_size, wl.num_pages) if wl.layout == "paged" \
        else "contiguous KV"
    return (f"{wl.name}: {wl.n_layers} layers, d_model {wl.d_model}, {wl.n_heads} q / {wl.n_kv_heads} kv heads "
            f"x {wl.head_dim}, SwiGLU {wl.ffn_hidden}, vocab {wl.vocab}, {wl.wdtype} weights, {lay}, "
            f"cap {wl.cap}, rows {wl.rows}, pos per step cycling {positions}")


def _positions(wl):
    import gen
    if wl.positions and len(wl.positions) == wl.rows:
        return [[int(p) for p in wl.positions]]                       # one record: fixed per-row positions
    if wl.positions:
        return [[int(p)] * wl.rows for p in wl.positions]              # cycle the listed positions
    return [[int(p) for p in gen.row_positions(wl)]]


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid
        self.proc = None
        self.out = os.path.join("/tmp", f"clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.out, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.out):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _traffic_from_profile(strategy):
    """DRAM bytes per launch of the roofline kernel from the committed ncu summary,
    or None if the summary is missing or the kernel source changed since."""
    if strategy not in PROFILES:
        return None
    path, src_name = PROFILES[strategy]
    try:
        txt = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    h = re.search(r"source_sha256:\s*([0-9a-f]+)", txt)
    if not m or not h:
        return None
    src = open(os.path.join(ROOT, "graph_replay_gb300", "csrc", src_name), "rb").read()
    if hashlib.sha256(src).hexdigest() != h.group(1):
        return None
    return float(m.group(1))


def _workload(args):
    import gen
    wl = gen.WORKLOADS[args.workload]
    over = {}
    if args.layers:
        over["n_layers"] = args.layers
    if args.vocab:
        over["vocab"] = args.vocab
    if over:   # a reduced copy of the workload, for profiler captures only
        wl = wl.replace(name=f"{wl.name}_reduced", **over)
    return wl


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """The largest value over all ranks: a replicated job takes as long as its slowest replica."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, rows: int, steps: int, seconds: float) -> float:
    """Whole-job throughput: every replica steps `rows` sequences `steps` times."""
    return world * rows * steps / seconds


PHASES = ("qkv", "attn", "o", "gu", "down")


def phase_bytes(wl) -> dict:
    """Algorithmic bytes of each phase of one step: its weight matrix, or the
    cap-swept K/V of one layer for attention."""
    es = 2 if wl.wdtype == "bf16" else 4
    kes = 2 if wl.kvdtype == "bf16" else 4
    qd, kvd = wl.n_heads * wl.head_dim, wl.n_kv_heads * wl.head_dim
    return {"qkv": (qd + 2 * kvd) * wl.d_model * es, "attn": wl.rows * 2 * wl.cap * kvd * kes,
            "o": wl.d_model * qd * es, "gu": 2 * wl.ffn_hidden * wl.d_model * es,
            "down": wl.d_model * wl.ffn_hidden * es, "head": wl.vocab * wl.d_model * es}


def summarize_timeline(stamps, wl) -> dict:
    """Per phase kind, from the in-kernel %globaltimer stamps of one step
    (ns; row p = phase p: earliest CTA start, latest CTA past its wait, earliest
    CTA end, latest CTA end): mean duration (latest end to latest end), the
    rate of the phase's algorithmic bytes over it, the spread of CTA end times,
    and the latency from the previous phase's latest end to the latest CTA
    past this phase's wait."""
    t = (np.asarray(stamps, dtype=np.float64) - float(stamps[0][0])) / 1e3
    nb = phase_bytes(wl)
    n_ph = t.shape[0]
    acc = {}
    for p in range(1, n_ph):
        k = "head" if p == n_ph - 1 else PHASES[(p - 1) % 5]
        a = acc.setdefault(k, [0, 0.0, 0.0, 0.0])
        a[0] += 1
        a[1] += t[p, 3] - t[p - 1, 3]
        a[2] += t[p, 3] - t[p, 2]
        a[3] += t[p, 1] - t[p - 1, 3]
    out = {}
    for k, (n, dur, spread, lat) in acc.items():
        out[k] = {"phases": n, "us_mean": round(dur / n, 3), "gbs": round(nb[k] / (dur / n) / 1e3, 1),
                  "end_spread_us": round(spread / n, 3), "wait_latency_us": round(lat / n, 3),
                  "us_total": round(dur, 2)}
    out["span_us"] = round(float(t[n_ph - 1, 3]), 2)
    return out


def phase_timeline(dec, dev_slots, n_rec, wl, reps=3) -> list:
    """Traced replays (outside any timed region), one summary per slot record and repeat."""
    from graph_replay_gb300 import _binding as B
    n_ph = 5 * wl.n_layers + 2
    res = []
    for i in range(n_rec):
        for _ in range(reps):
            B.dec_trace(dec.h, True)
            dec.launch(dev_slots[i])
            dec.wait()
            stamps = B.dec_trace_read(dec.h, n_ph)
            B.dec_trace(dec.h, False)
            s = summarize_timeline(stamps, wl)
            s["record"] = i
            res.append(s)
    return res


def run_ours(args, rank, world, local_rank):
    import torch

    import gen
    from gen.device import place_kv, to_tensor
    from graph_replay_gb300 import Decoder, make_config
    from graph_replay_gb300 import _binding as B

    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    wl = _workload(args)
    # weights: drawn from the seeded generator tensor by tensor, uploaded, host copy dropped
    w = {"layers": []}
    mw = gen.make_weights(wl) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    if mw is not None:
        from gen.device import upload_weights
        w = upload_weights(mw, dev)
    else:
        from gen.workloads import _draw, LAYER_ROLES
        for g in ("embed", "final_norm", "lm_head"):
            w[g] = to_tensor(_draw(wl, g, 0xFFFF), dev)
        for l in range(wl.n_layers):
            w["layers"].append({r: to_tensor(_draw(wl, r, l), dev) for r in LAYER_ROLES})
    cfg = make_config(wl.n_layers, wl.d_model, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.ffn_hidden, wl.vocab,
                      wl.wdtype, wl.kvdtype, wl.rms_eps, wl.rope_theta, device=local_rank)
    dec = Decoder(cfg, w, cap=wl.cap, rows=wl.rows, kv_layout=wl.layout, page_size=wl.page_size,
                  num_pages=wl.num_pages, strategy=args.strategy)
    slot_map = None
    if wl.layout == "paged":
        slot_map = gen.slot_map(wl)
        dec.set_slot_map(slot_map)
    plist = _positions(wl)
    maxpos = max(max(p) for p in plist)
    # KV pre-filled N(0,1) up to the largest position each row is stepped at
    for r in range(wl.rows):
        npos = max(p[r] for p in plist)
        for l in range(wl.n_layers):
            for which in (0, 1):
                place_kv(dec.kv(l, which), gen.kv_prefill(wl, l, which, r, npos), r, 0, slot_map, wl.page_size)
    toks = gen.ints(wl.seed, 0x51, 0, wl.vocab, wl.rows * len(plist)).reshape(len(plist), wl.rows)
    recs = []
    for i, p in enumerate(plist):
        wm = [int(slot_map[r][p[r] // wl.page_size]) * wl.page_size + p[r] % wl.page_size for r in range(wl.rows)] \
            if slot_map is not None else [0] * wl.rows
        recs.append(list(toks[i]) + list(p) + wm)
    dev_slots = torch.tensor(recs, dtype=torch.int32, device=dev)   # [n_records, 3*rows]
    stream = dec.stream()
    st = dec.stats()
    kernels = st["kernels_per_step"]

    def step(i):
        dec.launch(dev_slots[i % len(recs)])

    # ---- device-resident throughput ----
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    uuid = str(getattr(torch.cuda.get_device_properties(local_rank), "uuid", ""))
    clocks = Clocks(uuid if uuid.startswith("GPU-") else "GPU-" + uuid)
    clocks.start()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = e0.elapsed_time(e1)
    clk = clocks.stop()
    res = dec.wait()   # the device checks of the timed steps passed
    assert res.nonfinite.sum() == 0
    ms = max_over_ranks(ms, world, dev)
    ms_step = ms / args.steps
    tok_s = job_tokens_per_s(world, wl.rows, args.steps, ms / 1e3)

    # ---- end to end through dec_step with host buffers ----
    host_recs = [(np.array(r[:wl.rows], np.int32), np.array(r[wl.rows:2 * wl.rows], np.int32),
                  np.array(r[2 * wl.rows:], np.int32) if slot_map is not None else None) for r in recs]
    for i in range(args.warmup):
        t_, p_, w_ = host_recs[i % len(recs)]
        dec.step(t_, p_, w_, logits=False)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(args.steps):
        t_, p_, w_ = host_recs[i % len(recs)]
        dec.step(t_, p_, w_, logits=False)
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, world, dev)
    e2e_tok_s = job_tokens_per_s(world, wl.rows, args.steps, e2e_s)

    # ---- dominant kernel alone: RMSNorm + gate/up GEMV cycling the layers (graph
    # strategy), or the whole-step kernel (persistent strategy) ----
    hbm_peak, peak_kind = _peaks()
    persistent = args.strategy == "persistent"
    n_k = 16 if persistent else max(2 * wl.n_layers, 32)
    idx = [0] * n_k if persistent else [4 + 5 * (i % wl.n_layers) for i in range(n_k)]
    for i in idx[:4]:
        B.dec_launch_kernel(dec.h, i)
    k0 = torch.cuda.Event(enable_timing=True)
    k1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    k0.record(stream)
    kbytes = 0
    for i in idx:
        kbytes = B.dec_launch_kernel(dec.h, i)
    k1.record(stream)
    torch.cuda.synchronize()
    k_us = k0.elapsed_time(k1) * 1e3 / len(idx)
    k_gbs = kbytes / (k_us * 1e-6) / 1e9
    traffic = _traffic_from_profile(args.strategy) if wl.name == "8b" else None

    step_bytes = wl.step_bytes()
    step_gbs = step_bytes / (ms_step * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": round(tok_s, 3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "us_per_token": round(ms_step * 1e3 / wl.rows, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.wdtype, "data": "synthetic",
        "config": {"workload": _describe(wl, [p for p in plist]), "rows": wl.rows, "cap": wl.cap,
                   "kv_layout": wl.layout, "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2 (weights %.2f GB per step)" % (wl.weight_bytes() / 1e9),
                   "step": "1 D2D slot copy + 1 graph launch (%d kernels)" % kernels,
                   "strategy": args.strategy},
        "roofline": {"bound": "hbm",
                     "kernel": "persistent whole-step kernel" if persistent else "RMSNorm+gate/up GEMV (per layer)",
                     "achieved": round(k_gbs, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(k_gbs / hbm_peak, 4),
                     "traffic": traffic, "bytes_per_launch": kbytes, "us_per_launch": round(k_us, 3),
                     "peak_kind": peak_kind},
        "step_roofline": {"bytes_per_step": step_bytes, "achieved_gbs": round(step_gbs, 1),
                          "frac_of_measured": round(step_gbs / hbm_peak, 4),
                          "frac_of_8tbs": round(step_gbs / 8000.0, 4),
                          "weight_bytes": wl.weight_bytes(), "kv_swept_bytes": wl.kv_swept_bytes()},
        "e2e": {"value": round(e2e_tok_s, 3), "unit": "tokens/s",
                "us_per_token": round(e2e_s / args.steps * 1e6 / wl.rows, 3),
                "h2d_bytes_per_step": 3 * 4 * wl.rows, "d2h_bytes_per_step": 104,
                "readback": "greedy ids + non-finite flags + error word"},
        "gpu_launches": kernels * args.steps,
        "graph_launches_per_step": 1,
        "clocks": clk,
    }
    if args.trace:
        out["phase_timeline"] = phase_timeline(dec, dev_slots, len(recs), wl)
        for s in out["phase_timeline"]:
            print(f"record {s['record']} (pos {plist[s['record']]}): span {s['span_us']} us", file=sys.stderr)
            for k in PHASES + ("head",):
                v = s[k]
                print(f"  {k:5s} x{v['phases']:<3d} {v['us_mean']:8.2f} us  {v['gbs']:7.1f} GB/s  "
                      f"end spread {v['end_spread_us']:6.2f} us  wait latency {v['wait_latency_us']:5.2f} us",
                      file=sys.stderr)
    if world == 1 and args.prefill_tokens > 0 and wl.wdtype == "bf16":
        out["prefill"] = prefill_leg(dec, wl, args.prefill_tokens)
    dec.close()
    if persistent and world == 1 and not args.no_graph_leg:
        out["graph_strategy"] = graph_strategy_leg(args, wl, cfg, w, slot_map, dev_slots, hbm_peak)
    if mw is not None and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl, mw, plist, toks, seconds=args.cpu_seconds)
    return out


def prefill_leg(dec, wl, n_tokens, reps=3) -> dict:
    """Block prefill of one sequence (dec_prefill_block) on the same decoder,
    after the decode measurements: n_tokens prompt tokens at positions 0..n-1 of
    row 0 (or the first pages), timed with CUDA events on the handle's stream
    around the call (which waits for its own work).  Tensor-core work: every
    128-token block multiplies each weight once by 256 bf16 activation rows
    (the tokens' hi and lo parts), so the executed MMA work is twice the useful
    2 x tokens x projection-parameters."""
    import torch
    import gen
    n = min(int(n_tokens), wl.cap)
    toks = gen.ints(wl.seed, 0x77, 0, wl.vocab, n).astype(np.int32)
    pages = None
    if wl.layout == "paged":
        pages = np.arange(wl.cap // wl.page_size, dtype=np.int32)
    dec.prefill_block(toks, 0, pages=pages)   # first call: buffers, tensor maps
    stream = dec.stream()
    times = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dec.prefill_block(toks, 0, pages=pages)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = float(np.median(times))
    qd, kvd = wl.n_heads * wl.head_dim, wl.n_kv_heads * wl.head_dim
    proj_params = wl.n_layers * ((qd + 2 * kvd) * wl.d_model + wl.d_model * qd + 3 * wl.ffn_hidden * wl.d_model)
    blocks = (n + 127) // 128
    useful = 2.0 * n * proj_params
    executed = 2.0 * 256 * blocks * proj_params
    try:
        peak = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"])
    except Exception:
        peak = 1900.0
    return {"tokens": n, "ms": round(ms, 3), "tokens_per_s": round(n / (ms * 1e-3), 1),
            "useful_tflops": round(useful / (ms * 1e-3) / 1e12, 2),
            "mma_tflops": round(executed / (ms * 1e-3) / 1e12, 2),
            "mma_frac_of_bf16_peak": round(executed / (ms * 1e-3) / 1e12 / peak, 4), "bf16_peak_tflops": peak,
            "note": "whole dec_prefill_block call (projections, attention, norms, K/V writes, head); "
                    "attention runs on the tensor cores too (tcgen05, bf16 hi/lo Q and P), "
                    "its work not counted in the TFLOP/s figures"}


def graph_strategy_leg(args, wl, cfg, w, slot_map, dev_slots, hbm_peak) -> dict:
    """The pages' own strategy on the same workload, timed after the main line:
    the step's kernel sequence (embedding, 5 fused kernels per layer, head)
    recorded into one CUDA graph, one graph launch per step, same weights,
    slot records and timing method (CUDA events on the handle's stream)."""
    import torch
    from graph_replay_gb300 import Decoder
    dec = Decoder(cfg, w, cap=wl.cap, rows=wl.rows, kv_layout=wl.layout, page_size=wl.page_size,
                  num_pages=wl.num_pages, strategy="graph")
    if slot_map is not None:
        dec.set_slot_map(slot_map)
    n = len(dev_slots)
    steps = max(1, min(args.steps, 200))
    for i in range(args.warmup):
        dec.launch(dev_slots[i % n])
    torch.cuda.synchronize()
    stream = dec.stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        dec.launch(dev_slots[i % n])
    e1.record(stream)
    torch.cuda.synchronize()
    dec.wait()
    ms = e0.elapsed_time(e1) / steps
    kernels = dec.stats()["kernels_per_step"]
    dec.close()
    gbs = wl.step_bytes() / (ms * 1e-3) / 1e9
    return {"ms_per_step": round(ms, 5), "tokens_per_s": round(wl.rows / (ms * 1e-3), 3), "steps": steps,
            "kernels_per_step": kernels, "achieved_gbs": round(gbs, 1), "frac": round(gbs / hbm_peak, 4),
            "frac_of_8tbs": round(gbs / 8000.0, 4)}


def cpu_baseline(wl, mw, plist, toks, seconds=20.0, steps_cap=None):
    """The fp64 oracle as it stands, on this host's cores, over a bounded sample
    of the same workload (same weights, pre-filled KV, positions, tokens)."""
    import gen
    import oracle
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    orcs = []
    for r in range(wl.rows):
        o = oracle.Oracle(mw, cap=wl.cap, rows=1)
        npos = max(p[r] for p in plist)
        for l in range(wl.n_layers):
            o.K[0][l][:npos] = gen.kv_prefill(wl, l, 0, r, npos)
            o.V[0][l][:npos] = gen.kv_prefill(wl, l, 1, r, npos)
        orcs.append(o)
    n = 0
    t0 = time.perf_counter()
    while True:
        p = plist[n % len(plist)]
        for r in range(wl.rows):
            orcs[r].step(0, int(toks[n % len(plist)][r]), int(p[r]))
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or (steps_cap and n >= steps_cap):
            break
    return {"value": round(wl.rows * n / el, 5), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} fp64 oracle decode steps of the {wl.name} workload ({wl.rows} rows, same positions and "
                      f"pre-filled KV), {el:.1f} s"}


def run_reference(args):
    import gen
    wl = _workload(args)
    mw = gen.make_weights(wl)
    plist = _positions(wl)
    toks = gen.ints(wl.seed, 0x51, 0, wl.vocab, wl.rows * len(plist)).reshape(len(plist), wl.rows)
    # warm-up steps are part of the bounded sample budget: W short steps, then K timed
    budget = max(5.0, min(120.0, args.cpu_seconds))
    cpu_baseline(wl, mw, plist, toks, seconds=0.0, steps_cap=max(1, min(args.warmup, 2)))
    cb = cpu_baseline(wl, mw, plist, toks, seconds=budget, steps_cap=args.steps)
    # the same oracle on one thread: one decode step (one per row), reported beside the line
    import oracle
    try:
        if oracle.set_threads(1) != 1:
            raise RuntimeError("the oracle did not switch to one thread")
        one = cpu_baseline(wl, mw, plist, toks, seconds=0.0, steps_cap=1)
        cb["single_thread"] = {"value": one["value"], "unit": one["unit"], "cores": 1, "sample": one["sample"]}
    except Exception as e:   # reported, never fatal: the line's value is the multi-core sample
        cb["single_thread"] = {"unavailable": str(e)[:200]}
    finally:
        oracle.set_threads(cb["cores"])
    return {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": _describe(wl, plist), "rows": wl.rows, "cap": wl.cap, "kv_layout": wl.layout},
            "cpu_baseline": cb, "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="8b")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-tokens", type=int, default=1024,
                    help="tokens of the block-prefill leg timed after the decode line (0: skip)")
    ap.add_argument("--no-graph-leg", action="store_true",
                    help="skip timing the multi-kernel graph strategy beside the persistent line")
    ap.add_argument("--strategy", default="persistent", choices=["graph", "persistent"],
                    help="graph: the step's kernel sequence in one CUDA graph; persistent: one whole-step kernel")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (reduced case for profilers)")
    ap.add_argument("--vocab", type=int, default=0, help="override the vocabulary (reduced case for profilers)")
    ap.add_argument("--trace", action="store_true",
                    help="after the timed region, replay each slot record with the in-kernel phase trace on and "
                         "report per-phase durations (stderr, and phase_timeline in the JSON line)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
