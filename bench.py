#!/usr/bin/env python3
"""Benchmark of the paged-KV decode hot path on GB300.

One step = the whole hot path for one batch: pa_reshape_and_cache of every
sequence's new token, then pa_decode (partition kernel + split-K merge) over
the paged cache. Default workload: the Llama-3-8B-shaped GQA decode batch
(64 sequences, context U{128..4096} seeded, 32 q / 8 KV heads, head_dim 128,
bf16, block 16, random block placement in a pool 1.25x the blocks needed).

value = KV bytes read per step (K and V of every attended token) / device
time per step, whole job (all ranks). The KV pool and the step's inputs are
resident in HBM when the timed region starts; the 586 MB KV stream is 4.5x
the 129 MB L2, so no flush is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
       python bench.py --impl reference ...   (the fp64 CPU oracle arm)
Under torchrun (N > 1) each rank runs an independent replica of the workload
(decode shards by sequence with no exchange), timing is bracketed by a
barrier and synchronize, and the max time over ranks is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV-read HBM GB/s (fraction of peak), tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
DEFAULT_WORKLOAD = "gqa_8b"
WORKLOAD_LAYERS = {"tiny_mha": 1, "mha_7b": 32, "gqa_8b": 32, "gqa_70b_cow": 80, "mixed": 32,
                   "gqa_8b_fp8": 32, "swa_mistral": 32}
# ncu DRAM bytes per launch of the decode partition kernel, per workload,
# each tagged with the hash of the kernel sources it was taken on (written
# from an ncu CSV by `bench.py --record-traffic CSV --workload W`)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
TRAFFIC_KERNELS = ("pa_decode_partition_kernel", "pa_decode_mma_kernel")
TRAFFIC_COMMAND = ("ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none "
                   "-k regex:'pa_decode_(partition|mma)' -s 5 -c 2 --csv --log-file dram_{w}.csv "
                   "python bench.py --workload {w} --steps 20 --warmup 3 --skip-baselines --no-prefill-leg")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=["tiny_mha", "mha_7b", "gqa_8b", "gqa_70b_cow", "mixed", "gqa_8b_fp8",
                             "swa_mistral", "swap_8b", "prefix_cache"])
    ap.add_argument("--partition-tokens", type=int, default=int(os.environ.get("PA_PARTITION_TOKENS", "0")),
                    help="decode context partition size (0 = library default; env PA_PARTITION_TOKENS)")
    ap.add_argument("--nvtx", action="store_true",
                    help="mark the warm-up and timed regions and every step with NVTX ranges")
    ap.add_argument("--skip-baselines", action="store_true",
                    help="skip the CPU oracle and end-to-end legs (profiling runs)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="host time the reference arm (the oracle) aims to spend on warmup + steps")
    ap.add_argument("--record-traffic", metavar="CSV",
                    help="store the decode kernel's ncu DRAM bytes per launch from CSV for --workload "
                         "in profiles/traffic.json, then exit")
    ap.add_argument("--no-plan", action="store_true",
                    help="decode without the host-built work plan (pa_decode / _fp8 / _window in grid order)")
    ap.add_argument("--no-prefill-leg", action="store_true",
                    help="skip the tensor-core prefill leg of the default run")
    return ap.parse_args()


# ----------------------------------------------------------------- helpers --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max_ms(local_ms: float, dist_mod=None, device=None) -> float:
    """Slowest rank's elapsed time (the whole job ends when the last rank
    does). A host-side timing reduction only: no data of the hot path crosses
    ranks."""
    if dist_mod is None or not dist_mod.is_initialized() or dist_mod.get_world_size() == 1:
        return float(local_ms)
    import torch
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device or "cpu")
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(bytes_per_step_per_rank: int, steps: int, world: int, t_max_ms: float) -> float:
    """Weak scaling: every rank processes its own replica of the batch."""
    return world * bytes_per_step_per_rank * steps / (t_max_ms / 1e3) / 1e9


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", FALLBACK_HBM_GBS)), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense bf16 TFLOP/s measured as a burst: the prefill is timed over tens
    of milliseconds, not a seconds-long loop under the power cap (fp16, which
    its P.V product uses, has the same dense rate)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured bf16 dense TFLOP/s, burst (MEASURED_PEAKS.json bf16_tflops)"
    return 1900.0, "fallback bf16 dense TFLOP/s, burst"


def unique_kv_tokens(tables, ctx, window=None) -> int:
    """Distinct (physical block, offset) slots attended by the batch: positions
    0..ctx-1, or the last window+1 of them with a sliding window."""
    import numpy as np
    ids = []
    for b, c in enumerate(ctx):
        c = int(c)
        first = max(0, c - 1 - window) if window is not None else 0
        if c <= first:
            continue
        pos = np.arange(first, c)
        ids.append(tables[b, pos // 16].astype(np.int64) * 16 + pos % 16)
    return int(np.unique(np.concatenate(ids)).size) if ids else 0


TRAFFIC_SOURCES = ("decode.cu", "pa_common.cuh", "tc_sm100.cuh")


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_59_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str = None):
    """DRAM bytes (read + write) per launch of the decode partition kernel
    for this workload from the committed ncu figures, if they were taken on
    the current kernel sources (else None)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        entry = json.load(f).get("entries", {}).get(workload or DEFAULT_WORKLOAD)
    if not entry or entry.get("source_sha") != kernel_source_sha():
        return None
    return float(entry["dram_bytes_per_launch"])


def record_traffic(csv_path: str, workload: str) -> dict:
    """Reads an ncu CSV (dram__bytes_read.sum and dram__bytes_write.sum of
    the decode partition kernel's launches) and stores the mean bytes per
    launch for `workload` in the traffic file, tagged with the current kernel
    source hash."""
    import csv
    per_launch = {}
    names = {}
    with open(csv_path) as f:
        rows = [ln for ln in f if ln.startswith('"')]
    for row in csv.DictReader(rows):
        name = row.get("Kernel Name", "")
        if not any(k in name for k in TRAFFIC_KERNELS):
            continue
        if row.get("Metric Name") not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}[row.get("Metric Unit", "byte")]
        val = float(row["Metric Value"].replace(",", "")) * scale
        per_launch[row["ID"]] = per_launch.get(row["ID"], 0.0) + val
        names[row["ID"]] = name
    if not per_launch:
        raise SystemExit(f"{csv_path}: no DRAM figures of {TRAFFIC_KERNELS}")
    data = {"entries": {}}
    if os.path.exists(TRAFFIC_FILE):
        with open(TRAFFIC_FILE) as f:
            data = json.load(f)
    data["source_files"] = ["paged_kv_cache_59_gb300/csrc/" + f for f in TRAFFIC_SOURCES]
    entry = {"kernel": sorted(set(n.split("(")[0] for n in names.values())),
             "launches": len(per_launch),
             "dram_bytes_per_launch": round(sum(per_launch.values()) / len(per_launch)),
             "source_sha": kernel_source_sha(),
             "command": TRAFFIC_COMMAND.format(w=workload)}
    data.setdefault("entries", {})[workload] = entry
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")
    return entry


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        deadline = time.time() + 5
        while not self.rows and time.time() < deadline:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "begin":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.06)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        inside = [r for t, r in self.rows if self.t0 is not None and self.t0 <= t <= (self.t1 or t)]
        used = inside
        if not used and self.rows:                    # region shorter than one sample period
            ref = self.t1 or self.t0 or 0
            used = [min(self.rows, key=lambda tr: abs(tr[0] - ref))[1]]
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in used:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples_in_region": len(inside)}


# ------------------------------------------------------------- our arm ------

def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import paged_kv_cache_59_gb300 as pk
    from paged_kv_cache_59_gb300 import build as pk_build
    from workloads import make_workload

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    if rank == 0 or world == 1:
        pk_build.build()
    if world > 1:
        dist.barrier()
    pk.load()
    dev = torch.device("cuda", local)

    wl = make_workload(args.workload, fill="zero", keep_logical=False)
    H, Hk, D = wl.n_heads, wl.n_kv_heads, wl.head_dim
    B = len(wl.dec_ctx)
    max_ctx = int(wl.dec_ctx.max())
    window = wl.meta.get("window")
    # algorithmic KV bytes: the distinct cached tokens the batch attends to (a
    # block shared by several tables, like a common prompt prefix, counts once)
    uniq_tok = unique_kv_tokens(wl.dec_tables, wl.dec_ctx, window)
    # pa_decode's kernel choice: tensor cores at head_dim 128 for groups of 8 and E4M3 caches
    tc_path = D == 128 and (H // Hk == 8 or wl.meta.get("kv_dtype") == "fp8_e4m3")
    if window is not None:   # tokens each query attends to: ctx-1-W .. ctx-1
        sum_ctx = int(sum(min(int(c), window + 1) for c in wl.dec_ctx))
    else:
        sum_ctx = int(wl.dec_ctx.sum())
    fp8 = wl.meta.get("kv_dtype") == "fp8_e4m3"
    eb = 1 if fp8 else 2                       # bytes per cached element
    kv_bytes = uniq_tok * Hk * D * 2 * eb
    alg_bytes = (kv_bytes + 2 * wl.q.nbytes + wl.dec_tables.nbytes + wl.dec_ctx.nbytes)

    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(dev)

    # this step's new tokens: one per decode sequence, plus every chunk token
    # of the prefill sequences (mixed workload)
    has_pf = wl.q_pf is not None
    n_dec_new = len(wl.slot_mapping) if wl.slot_mapping is not None else 0
    new_k, new_v = wl.new_k[:n_dec_new], wl.new_v[:n_dec_new]
    slots = wl.slot_mapping[:n_dec_new]
    pf_flops = pf_kv_bytes = 0
    if has_pf:
        for si in range(len(wl.pf_ctx)):
            L = int(wl.q_start_loc[si + 1] - wl.q_start_loc[si]); c = int(wl.pf_ctx[si])
            pf_flops += 4 * D * H * sum(c - L + i + 1 for i in range(L))
            pf_kv_bytes += c * Hk * D * 2 * 2
        kv_bytes += pf_kv_bytes
    kp, vp = to_dev(wl.k_pool), to_dev(wl.v_pool)
    del wl.k_pool, wl.v_pool
    q = to_dev(wl.q)
    out = torch.empty_like(q)
    nk, nv, sl = to_dev(new_k), to_dev(new_v), to_dev(slots)
    tabs, ctx = to_dev(wl.dec_tables), to_dev(wl.dec_ctx)
    if has_pf:
        q_pf, pf_tabs, pf_ctx, qsl = to_dev(wl.q_pf), to_dev(wl.pf_tables), to_dev(wl.pf_ctx), to_dev(wl.q_start_loc)
        out_pf = torch.empty_like(q_pf)
        max_chunk = int(np.max(np.diff(wl.q_start_loc)))
        # key ranges split into pieces so the grid fills whole waves of SMs
        ws_pf = pk.prefill_workspace(q_pf, len(wl.pf_ctx), Hk, max_chunk, 0)
    pt = args.partition_tokens
    ws = pk.decode_workspace(q, max_ctx, pt)
    stream = torch.cuda.current_stream()
    if fp8:
        ks, vs = to_dev(wl.meta["k_scale"]), to_dev(wl.meta["v_scale"])
        alg_bytes += ks.numel() * 4 * 2

    def write_cache():
        if fp8:
            pk.pa_reshape_and_cache_fp8(nk, nv, kp, vp, sl, ks, vs)
        else:
            pk.pa_reshape_and_cache(nk, nv, kp, vp, sl)

    # the decode call's work plan, built on the host from the batch's lengths
    # (which do not change between the steps) and kept on the device like the tables
    plan_host = None if args.no_plan else pk.pa_decode_plan(
        wl.dec_ctx, H, Hk, D, wl.dec_tables.shape[1], max_ctx, wl.num_blocks,
        window=-1 if window is None else window, elem_bytes=eb, partition_tokens=pt)
    plan = to_dev(plan_host) if plan_host is not None else None

    def decode():
        if plan is not None:
            pk.pa_decode_planned(out, q, kp, vp, tabs, ctx, wl.scale, max_ctx, plan,
                                 k_scale=ks if fp8 else None, v_scale=vs if fp8 else None,
                                 window=-1 if window is None else window, workspace=ws, partition_tokens=pt)
        elif fp8:
            pk.pa_decode_fp8(out, q, kp, vp, ks, vs, tabs, ctx, wl.scale, max_ctx, workspace=ws,
                             partition_tokens=pt)
        elif window is not None:
            pk.pa_decode_window(out, q, kp, vp, tabs, ctx, wl.scale, max_ctx, window, workspace=ws,
                                partition_tokens=pt)
        else:
            pk.pa_decode(out, q, kp, vp, tabs, ctx, wl.scale, max_ctx, workspace=ws, partition_tokens=pt)
    # cache write, prefill (plan + main + merge of the cut pairs in balanced mode), decode
    # (partition kernel, plus the split-K merge kernel when some context spans partitions)
    launches_per_step = ((1 if n_dec_new else 0) + ((3 if ws_pf is not None else 1) if has_pf else 0)
                         + 1 + (1 if pk.pa_decode_workspace_bytes(B, H, D, max_ctx, pt) else 0))

    def step_body(ev_pair=None, pf_pair=None):
        if n_dec_new:
            write_cache()
        if has_pf:
            if pf_pair is not None:
                pf_pair[0].record(stream)
            pk.pa_prefill_paged_ex(out_pf, q_pf, kp, vp, pf_tabs, pf_ctx, qsl, wl.scale, max_chunk,
                                   splits=0, workspace=ws_pf)
            if pf_pair is not None:
                pf_pair[1].record(stream)
        if ev_pair is not None:
            ev_pair[0].record(stream)
        decode()
        if ev_pair is not None:
            ev_pair[1].record(stream)

    nvtx = torch.cuda.nvtx if args.nvtx else None

    def step(ev_pair=None, pf_pair=None):
        if nvtx is not None:
            nvtx.range_push("step")
        step_body(ev_pair, pf_pair)
        if nvtx is not None:
            nvtx.range_pop()

    if nvtx is not None:
        nvtx.range_push("warmup")
    for _ in range(max(args.warmup, 3)):
        step()
    if nvtx is not None:
        nvtx.range_pop()
    torch.cuda.synchronize()
    assert pk.pa_get_device_error() == 0

    # An event between two kernels stops the next one's programmatic dependent
    # launch from overlapping the previous one's tail, so the per-call events of
    # the roofline are recorded on every `every`-th timed step only (at least
    # every 4th; at most 16 samples), the other steps run back to back.
    every = max(4, -(-args.steps // 16))
    sampled = [i % every == 0 for i in range(args.steps)]

    def timed_region():
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) if sampled[i] else None
               for i in range(args.steps)]
        pfe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               if has_pf and sampled[i] else None for i in range(args.steps)]
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        sampler.mark("begin")
        if nvtx is not None:
            nvtx.range_push("timed")
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i], pfe[i])
        t_end.record(stream)
        if nvtx is not None:
            nvtx.range_pop()
        torch.cuda.synchronize()
        sampler.mark("end")
        if world > 1:
            dist.barrier()
        total_ms = t_start.elapsed_time(t_end)
        dec_ms = [e[0].elapsed_time(e[1]) for e in evs if e is not None]
        timed_region.pf_ms = [e[0].elapsed_time(e[1]) for e in pfe if e is not None] if has_pf else []
        return total_ms, dec_ms

    vis = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    sampler = ClockSampler(vis[local] if local < len(vis) else str(local))
    sampler.start()
    total_ms, dec_ms = timed_region()
    clocks = sampler.stop()
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(clocks.get("reasons", [])):
        sampler = ClockSampler(sampler.gpu)
        sampler.start()
        total_ms, dec_ms = timed_region()
        clocks = sampler.stop()
        clocks["remeasured"] = True

    t_max = reduce_max_ms(total_ms, dist if world > 1 else None, dev)
    ms_per_step = t_max / args.steps
    graph = graph_replay(torch, step, args.steps, kv_bytes)
    clocks = merge_clocks(clocks, clock_leg(torch, graph_replay.replay or step, sampler.gpu))
    value = whole_job_gbps(kv_bytes, args.steps, world, t_max)

    # roofline of the decode call (partition kernel + merge kernel)
    dec_ms_sorted = sorted(dec_ms)
    dec_avg = sum(dec_ms) / len(dec_ms)
    peak, peak_kind = measured_peaks()
    achieved = alg_bytes / (dec_avg / 1e3) / 1e9
    traffic = profiled_traffic(args.workload) if pt == 0 else None

    step_tokens = B + (int(wl.q_start_loc[-1]) if has_pf else 0)
    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8_e4m3" if fp8 else "bf16",
        "data": ("synthetic: cached K/V as seeded E4M3 codes (uniform over finite codes) with "
                 "per-KV-head fp32 scales, N(0,1) q and new tokens rounded to bf16, seeded context "
                 "lengths, random physical block placement" if fp8 else
                 "synthetic: seeded N(0,1) q/K/V rounded to bf16, seeded context lengths, "
                 "random physical block placement"),
        "config": {
            "workload": wl.name,
            "n_seqs": B, "n_heads": H, "n_kv_heads": Hk, "head_dim": D, "block_size": 16,
            "sum_context_tokens": sum_ctx, "distinct_cached_tokens_read": uniq_tok,
            "max_context": max_ctx, "num_blocks": wl.num_blocks,
            "kv_bytes_per_step": kv_bytes,
            "step": (("pa_reshape_and_cache_fp8 (1 new token/seq, encoded) + pa_decode_fp8 (partition "
                      "kernel + split-K merge)" if fp8 else
                      f"pa_reshape_and_cache (1 new token/seq) + pa_decode_window (window {window})"
                      if window is not None else
                      "pa_reshape_and_cache (1 new token/seq) + pa_decode (partition kernel + split-K merge)")
                     + ("; the decode as pa_decode_planned" if plan_host is not None else "")),
            "l2": f"no flush: the KV stream ({kv_bytes / 1e6:.0f} MB/step) exceeds the 129 MB L2",
            "partition_tokens": pt or pk.pa_decode_partition_tokens(
                B, H, Hk, D, max_ctx, window if window is not None else -1, eb),
            "decode_plan": ("none: the decode call's CTAs in grid order" if plan_host is None else
                            f"pa_decode_planned over a host-built plan (pa_decode_plan) of {len(plan_host)} "
                            "work items, longest partitions first, built once (the lengths do not change "
                            "between steps) and resident like the block tables"),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        # tokens the step produces: one per decode sequence, plus every prefill
        # chunk token on the mixed workload
        "tokens_per_s": round(world * step_tokens / (ms_per_step / 1e3), 1),
        "kv_tokens_per_s": round(world * sum_ctx / (ms_per_step / 1e3), 1),
        "attention_only_model_tokens_per_s": round(
            world * step_tokens / (ms_per_step / 1e3) / WORKLOAD_LAYERS[args.workload], 1),
        "hbm_frac_of_measured": round(value / world / peak, 4),
        "hbm_frac_of_nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "roofline": {
            "bound": "hbm",
            "kernel": (("pa_decode_mma_kernel (warp-level tensor-core MMAs)" if tc_path else
                        "pa_decode_partition_kernel") + " + pa_decode_merge_kernel (one decode call"
                       + (", CTAs from the host-built plan)" if plan_host is not None else ")")),
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_source": f"{peak_kind} HBM copy GB/s",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": alg_bytes,
            "launch_ms_avg": round(dec_avg, 5),
            "launch_ms_median": round(dec_ms_sorted[len(dec_ms) // 2], 5),
            "launch_ms_p10_p90": [round(dec_ms_sorted[len(dec_ms) // 10], 5),
                                  round(dec_ms_sorted[(9 * len(dec_ms)) // 10], 5)],
            "launches_timed": len(dec_ms),
            "timing": (f"CUDA events around the decode call on every {every}th timed step "
                       f"({len(dec_ms)} of {args.steps}); the other steps carry no events, which would "
                       "stop the next kernel's programmatic launch from overlapping the previous one"),
        },
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "graph_replay": graph,
    }
    if has_pf:
        result["config"]["step"] = ("pa_reshape_and_cache (decode tokens + chunk tokens) + "
                                    "pa_prefill_paged_ex (tcgen05, balanced) + pa_decode")
        result["config"]["prefill_flop_per_step"] = pf_flops
        result["config"]["prefill_splits"] = ("balanced (0): %d bytes of workspace" % ws_pf.numel()
                                              if ws_pf is not None else 1)
        result["prefill_roofline"] = prefill_roofline(pf_flops, timed_region.pf_ms, ws_pf)

    if not args.skip_baselines:
        result["e2e"] = run_e2e(args, pk, wl, new_k, new_v, slots, kp, vp, dev, kv_bytes, world,
                                dist if world > 1 else None,
                                (ks, vs) if fp8 else None, plan_host)
        if rank == 0:
            # an oracle process holds its own host copy of the pools plus numpy's working arrays
            child_bytes = int(1.2 * 2 * kp.numel() * kp.element_size()) + (256 << 20)
            result["cpu_baseline"] = run_cpu_baseline(args.workload, args.cpu_seconds, child_bytes)
            if has_pf:
                result["prefill_roofline"]["cpu_baseline"] = run_cpu_prefill_baseline(args.cpu_seconds,
                                                                                      child_bytes)
    if not has_pf and args.workload == DEFAULT_WORKLOAD and not args.no_prefill_leg:
        # the tensor-core row of the path, after the decode legs; the decode
        # batch's pools are freed first (the prefill leg brings its own)
        del kp, vp
        torch.cuda.empty_cache()
        result["prefill_roofline"] = prefill_leg(args, pk, torch, dev, sampler.gpu)
        result["gpu_launches_prefill_leg"] = result["prefill_roofline"]["calls_timed"] * \
            result["prefill_roofline"]["launches_per_call"]
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def graph_replay(torch, step, n, kv_bytes):
    """The same step captured once as a CUDA graph and replayed n times back
    to back, inputs resident (launch overhead removed; reported beside the
    eager timing, which is the bench value)."""
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # warm the launch path off the capture
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / n
        graph_replay.replay = g.replay
        return {"ms_per_step": round(ms, 5), "value": round(kv_bytes / (ms / 1e3) / 1e9, 1), "unit": "GB/s",
                "how": f"the step captured once as a CUDA graph, {n} replays back to back"}
    except Exception as e:  # report, do not hide
        graph_replay.replay = None
        return {"error": str(e)[-200:]}


def clock_leg(torch, fn, gpu, seconds=1.2):
    """SM clock under load: fn (one step, or one graph replay) run back to back
    for at least `seconds` while nvidia-smi samples the clocks. Not part of
    the timed region; it only shows the clock the kernels run at."""
    sampler = ClockSampler(gpu)
    sampler.start()
    torch.cuda.synchronize()
    sampler.mark("begin")
    t0 = time.perf_counter()
    calls = 0
    while True:
        for _ in range(64):
            fn()
        calls += 64
        torch.cuda.synchronize()
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    sampler.mark("end")
    c = sampler.stop()
    return {"sm_mhz": c["sm_mhz"], "sm_max_mhz": c["sm_max_mhz"], "reasons": c["reasons"],
            "samples": c.get("samples_in_region", 0), "seconds": round(dt, 3), "calls": calls}


def merge_clocks(region, leg):
    """The timed region's clock record, with the load leg's median SM clock
    standing in when the region was too short for the 50 ms sampler."""
    out = dict(region)
    out["load_leg"] = leg
    if leg and leg.get("sm_mhz") is not None and region.get("samples_in_region", 0) < 3:
        out["sm_mhz"] = leg["sm_mhz"]
        out["sm_mhz_source"] = (f"load leg: {leg['samples']} samples over {leg['seconds']} s of back-to-back "
                                "steps (the timed region is shorter than a few sample periods)")
        out["reasons"] = sorted(set(region.get("reasons", [])) | set(leg.get("reasons", [])))
    else:
        out["sm_mhz_source"] = "timed region"
    return out


def prefill_leg(args, pk, torch, dev, gpu):
    """The tensor-core contraction of the path, timed in the default run
    beside the decode step: the mixed workload's chunked prefill (4 sequences
    x a 512-token causal chunk at 32,768 context, 32 q / 8 KV heads, head_dim
    128, bf16 cache), one pa_prefill_paged_ex call (balanced: plan, tcgen05
    main kernel, merge of the cut pairs) per iteration, CUDA events around
    every call, then a clock leg of >= 1 s of calls."""
    import numpy as np
    from workloads import make_workload

    wl = make_workload("mixed", fill="zero", keep_logical=False)
    H, Hk, D = wl.n_heads, wl.n_kv_heads, wl.head_dim

    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(dev)

    kp, vp = to_dev(wl.k_pool), to_dev(wl.v_pool)
    del wl.k_pool, wl.v_pool
    pk.pa_reshape_and_cache(to_dev(wl.new_k), to_dev(wl.new_v), kp, vp, to_dev(wl.slot_mapping))
    q_pf, tabs, ctx, qsl = to_dev(wl.q_pf), to_dev(wl.pf_tables), to_dev(wl.pf_ctx), to_dev(wl.q_start_loc)
    out = torch.empty_like(q_pf)
    max_chunk = int(np.max(np.diff(wl.q_start_loc)))
    ws = pk.prefill_workspace(q_pf, len(wl.pf_ctx), Hk, max_chunk, 0)
    flops = 0
    for si in range(len(wl.pf_ctx)):
        L = int(wl.q_start_loc[si + 1] - wl.q_start_loc[si]); c = int(wl.pf_ctx[si])
        flops += 4 * D * H * sum(c - L + i + 1 for i in range(L))
    stream = torch.cuda.current_stream()

    def call():
        pk.pa_prefill_paged_ex(out, q_pf, kp, vp, tabs, ctx, qsl, wl.scale, max_chunk, splits=0, workspace=ws)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    assert pk.pa_get_device_error() == 0
    n = max(20, min(args.steps, 100))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    sampler = ClockSampler(gpu)
    sampler.start()
    torch.cuda.synchronize()
    sampler.mark("begin")
    for a, b in evs:
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    sampler.mark("end")
    clocks = merge_clocks(sampler.stop(), clock_leg(torch, call, gpu))
    assert pk.pa_get_device_error() == 0
    ms = sorted(a.elapsed_time(b) for a, b in evs)
    res = prefill_roofline(flops, ms, ws)
    res.update({"workload": "mixed: 4 x 512-token causal chunk at 32,768 context, 32 q / 8 KV heads, d 128",
                "calls_timed": n, "launches_per_call": 3 if ws is not None else 1, "clocks": clocks})
    del kp, vp, q_pf, out, ws
    torch.cuda.empty_cache()
    return res


def prefill_roofline(flops, ms, ws):
    avg = sum(ms) / len(ms)
    tpk, tpk_kind = measured_tensor_peak()
    ms = sorted(ms)
    return {
        "bound": "tensor",
        "kernel": ("pa_prefill_plan_kernel + pa_prefill_tc_kernel (one CTA per SM) + pa_prefill_merge_cut_kernel"
                   if ws is not None else "pa_prefill_tc_kernel"),
        "achieved": round(flops / (avg / 1e3) / 1e12, 1), "peak": tpk,
        "peak_source": tpk_kind, "unit": "TFLOP/s",
        "frac": round(flops / (avg / 1e3) / 1e12 / tpk, 4),
        "flop_per_call": flops,
        "launch_ms_avg": round(avg, 4),
        "launch_ms_median": round(ms[len(ms) // 2], 4),
        "launch_ms_p10_p90": [round(ms[len(ms) // 10], 4), round(ms[(9 * len(ms)) // 10], 4)],
        "note": "algorithmic FLOPs 4*D*H*sum(positions attended); the kernel also runs the "
                "masked halves of the diagonal tiles; CUDA events around each call"}


def run_e2e(args, pk, wl, new_k, new_v, slots, kp, vp, dev, kv_bytes, world, dist, fp8_scales=None,
            plan_host=None):
    """Same metric through the public API with host buffers. Each step copies
    its inputs (q, new K/V, slots, tables, context lengths) from page-locked
    host memory, runs the hot path and copies the output back, then the host
    waits for it. The inputs sit in one pinned buffer (one host-to-device
    copy; the API calls take views into its device twin) and the output comes
    back in one copy; the whole step - copies and kernels - is captured once
    as a CUDA graph and replayed."""
    import numpy as np
    import torch

    has_pf = wl.q_pf is not None
    srcs = [wl.q, new_k, new_v, slots, wl.dec_tables, wl.dec_ctx]
    if has_pf:
        srcs += [wl.q_pf, wl.pf_tables, wl.pf_ctx, wl.q_start_loc]
    i_plan = len(srcs)
    if plan_host is not None:  # the decode plan travels with the other inputs
        srcs.append(plan_host)
    srcs = [np.ascontiguousarray(x) for x in srcs]
    offs, off = [], 0
    for x in srcs:                                  # 256-byte aligned slots in one buffer
        offs.append(off)
        off += (x.nbytes + 255) // 256 * 256
    h_buf = torch.empty(off, dtype=torch.uint8).pin_memory()
    d_buf = torch.empty(off, dtype=torch.uint8, device=dev)
    tdt = {np.uint16: torch.int16, np.int16: torch.int16, np.int32: torch.int32, np.int64: torch.int64}
    d_in = []
    for x, o in zip(srcs, offs):
        h_buf[o:o + x.nbytes].copy_(torch.from_numpy(x.view(np.uint8).reshape(-1)))
        d_in.append(d_buf[o:o + x.nbytes].view(tdt[x.dtype.type]).view(x.shape))
    out_shapes = [wl.q.shape] + ([wl.q_pf.shape] if has_pf else [])
    out_bytes = [int(np.prod(sh)) * 2 for sh in out_shapes]
    oo = [0, (out_bytes[0] + 255) // 256 * 256][:len(out_shapes)]
    h_out = torch.empty(sum((b + 255) // 256 * 256 for b in out_bytes), dtype=torch.uint8).pin_memory()
    d_outb = torch.empty_like(h_out, device=dev)
    d_out = [d_outb[o:o + nb].view(torch.int16).view(sh) for o, nb, sh in zip(oo, out_bytes, out_shapes)]
    max_ctx = int(wl.dec_ctx.max())
    max_chunk = int(np.max(np.diff(wl.q_start_loc))) if has_pf else 0
    ws = pk.decode_workspace(d_in[0], max_ctx, args.partition_tokens)
    ws_pf = pk.prefill_workspace(d_in[6], len(wl.pf_ctx), wl.n_kv_heads, max_chunk, 0) if has_pf else None
    h2d = int(h_buf.numel())
    d2h = int(h_out.numel())

    def body():
        d_buf.copy_(h_buf, non_blocking=True)
        q, nk, nv, sl, tabs, ctx = d_in[:6]
        if len(slots):
            if fp8_scales is not None:
                pk.pa_reshape_and_cache_fp8(nk, nv, kp, vp, sl, *fp8_scales)
            else:
                pk.pa_reshape_and_cache(nk, nv, kp, vp, sl)
        if has_pf:
            q_pf, pf_tabs, pf_ctx, qsl = d_in[6:10]
            pk.pa_prefill_paged_ex(d_out[1], q_pf, kp, vp, pf_tabs, pf_ctx, qsl, wl.scale, max_chunk,
                                   splits=0, workspace=ws_pf)
        if plan_host is not None:
            pk.pa_decode_planned(d_out[0], q, kp, vp, tabs, ctx, wl.scale, max_ctx, d_in[i_plan],
                                 k_scale=fp8_scales[0] if fp8_scales else None,
                                 v_scale=fp8_scales[1] if fp8_scales else None,
                                 window=-1 if wl.meta.get("window") is None else wl.meta["window"],
                                 workspace=ws, partition_tokens=args.partition_tokens)
        elif fp8_scales is not None:
            pk.pa_decode_fp8(d_out[0], q, kp, vp, *fp8_scales, tabs, ctx, wl.scale, max_ctx, workspace=ws,
                             partition_tokens=args.partition_tokens)
        elif wl.meta.get("window") is not None:
            pk.pa_decode_window(d_out[0], q, kp, vp, tabs, ctx, wl.scale, max_ctx, wl.meta["window"],
                                workspace=ws, partition_tokens=args.partition_tokens)
        else:
            pk.pa_decode(d_out[0], q, kp, vp, tabs, ctx, wl.scale, max_ctx, workspace=ws,
                         partition_tokens=args.partition_tokens)
        h_out.copy_(d_outb, non_blocking=True)

    for _ in range(max(args.warmup, 3)):             # first calls set kernel attributes (not capturable)
        body()
    torch.cuda.synchronize()
    graph = None
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            body()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            body()
        torch.cuda.synchronize()
    except Exception as e:  # report and run the same step eagerly
        graph = None
        graph_error = str(e)[-200:]
    stream = torch.cuda.current_stream()

    def step():
        if graph is not None:
            graph.replay()
        else:
            body()
        stream.synchronize()                       # the host reads this step's result

    for _ in range(max(args.warmup, 3)):
        step()
    n = args.steps
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n):
        step()
    torch.cuda.synchronize()
    dt = reduce_max_ms((time.perf_counter() - t0) * 1e3, dist, dev) / 1e3
    res = {"value": round(world * kv_bytes * n / dt / 1e9, 1), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": round(dt * 1e3 / n, 5),
           "how": "wall clock over K steps; each step: one pinned host-to-device copy of all inputs (with the "
                  "decode plan, when used), the "
                  "step's kernels, one device-to-host copy of the output, host waits; the step is "
                  + ("replayed as a captured CUDA graph" if graph is not None else "run eagerly")}
    if graph is None:
        res["graph_error"] = graph_error
    return res


# ------------------------------------------------------ CPU oracle timing ---

_CPU_CHILD = r"""
import json, sys, time
import numpy as np
sys.path.insert(0, {root!r})
from workloads import make_workload
from oracle.attention import paged_decode, paged_decode_window
from oracle.cache_ops import reshape_and_cache
from oracle import fp8 as ofp8
wl = make_workload({workload!r}, fill="zero", keep_logical=False)
fp8 = wl.meta.get("kv_dtype") == "fp8_e4m3"
B, H, Hk = len(wl.dec_ctx), wl.n_heads, wl.n_kv_heads
G = H // Hk
n_new = min(B, len(wl.slot_mapping)) if wl.slot_mapping is not None else 0
budget, per_step = {seconds}, {per_step}
# The unit of work is one (sequence, KV head): its G query heads attend over
# the sequence's blocks. Each unit runs through the unchanged oracle on a
# compact copy of just that sequence's blocks of that KV head (built here,
# outside the timed region), so a unit costs what its arithmetic costs.
units = [(b, h) for b in range(B) for h in range(Hk)]
W = wl.meta.get("window")
def prepare(b, h):
    nblk = (int(wl.dec_ctx[b]) + 15) // 16
    blk0 = max(0, int(wl.dec_ctx[b]) - 1 - W) // 16 if W is not None else 0
    ids = wl.dec_tables[b, blk0:nblk]                  # blocks the unit reads (held blocks only)
    kp = np.ascontiguousarray(wl.k_pool[ids, h:h + 1])
    vp = np.ascontiguousarray(wl.v_pool[ids, h:h + 1])
    table = np.concatenate([np.full(blk0, -1, np.int32), np.arange(nblk - blk0, dtype=np.int32)])[None, :]
    slot = None
    if b < n_new:
        s = int(wl.slot_mapping[b]); blk, off = s // 16, s % 16
        idx = int(np.nonzero(ids == blk)[0][0])        # the block's place in the compact pool
        slot = np.array([idx * 16 + off], dtype=np.int64)
    return kp, vp, table, slot
kv_tok = 2 * wl.head_dim * (1 if fp8 else 2)   # K + V bytes of one token of one KV head
def run_unit(b, h, kp, vp, table, slot):
    if fp8:
        ks, vs = wl.meta["k_scale"][h:h + 1], wl.meta["v_scale"][h:h + 1]
        if slot is not None:
            kp, vp = ofp8.reshape_and_cache_fp8(wl.new_k[b:b + 1, h:h + 1], wl.new_v[b:b + 1, h:h + 1],
                                                kp, vp, slot, ks, vs)
        ofp8.paged_decode_fp8(wl.q[b:b + 1, h * G:(h + 1) * G], kp, vp, table, wl.dec_ctx[b:b + 1],
                              wl.scale, ks, vs)
    else:
        if slot is not None:
            kp, vp = reshape_and_cache(wl.new_k[b:b + 1, h:h + 1], wl.new_v[b:b + 1, h:h + 1], kp, vp,
                                       slot)
        if W is not None:
            paged_decode_window(wl.q[b:b + 1, h * G:(h + 1) * G], kp, vp, table, wl.dec_ctx[b:b + 1],
                                wl.scale, W)
        else:
            paged_decode(wl.q[b:b + 1, h * G:(h + 1) * G], kp, vp, table, wl.dec_ctx[b:b + 1], wl.scale)
done_tok = 0
n_units = 0
u = {start} % len(units)
dt = 0.0
while True:
    sel = [units[(u + i) % len(units)] for i in range(per_step)]
    u = (u + per_step) % len(units)
    prep = [prepare(b, h) for b, h in sel]
    t0 = time.perf_counter()
    for (b, h), args in zip(sel, prep):
        run_unit(b, h, *args)
    dt += time.perf_counter() - t0
    for b, h in sel:
        done_tok += int(wl.dec_ctx[b]) if W is None else min(int(wl.dec_ctx[b]), W + 1)
    n_units += len(sel)
    if {fixed_steps} and n_units >= {fixed_steps} * per_step:
        break
    if not {fixed_steps} and dt >= budget:
        break
print(json.dumps({{"seconds": dt, "tokens": done_tok, "units": n_units, "kv_bytes": done_tok * kv_tok}}))
"""


_CPU_PREFILL_CHILD = r"""
import json, sys, time
import numpy as np
sys.path.insert(0, {root!r})
from workloads import make_workload
from oracle.attention import paged_prefill
from oracle.cache_ops import reshape_and_cache
wl = make_workload("mixed", fill="zero", keep_logical=False)
H, Hk, D = wl.n_heads, wl.n_kv_heads, wl.head_dim
G = H // Hk
budget = {seconds}
# The unit of work is one chunk row of one KV head's group: its G query heads
# attend causally over positions 0..p of the sequence through the unchanged
# oracle, given that KV head's pools (so its gather reads one head). Units
# cycle over (sequence, KV head, row), rows spread over the chunk. The cache
# write of the chunk tokens runs once, outside the timed region.
n_seq = len(wl.pf_ctx)
n_dec = len(wl.dec_ctx)
kp, vp = reshape_and_cache(wl.new_k[n_dec:], wl.new_v[n_dec:], wl.k_pool, wl.v_pool,
                           wl.slot_mapping[n_dec:])
units = []
for i in range(0, 512, 37):
    for s in range(n_seq):
        for kh in range(Hk):
            units.append((s, kh, i))
u = {start} % len(units)
dt, flops, n_units = 0.0, 0, 0
while dt < budget:
    s, kh, i = units[u]
    u = (u + 1) % len(units)
    r = int(wl.q_start_loc[s]) + i
    L = int(wl.q_start_loc[s + 1] - wl.q_start_loc[s])
    p = int(wl.pf_ctx[s]) - L + i
    rows = [(r, g) for g in range(G)]
    t0 = time.perf_counter()
    paged_prefill(wl.q_pf[:, kh * G:(kh + 1) * G], kp[:, kh:kh + 1], vp[:, kh:kh + 1], wl.pf_tables,
                  wl.pf_ctx, wl.q_start_loc, wl.scale, rows=rows)
    dt += time.perf_counter() - t0
    flops += 4 * D * G * (p + 1)
    n_units += 1
print(json.dumps({{"seconds": dt, "flops": flops, "units": n_units}}))
"""


def _oracle_cmd(workload, seconds, per_step, fixed_steps=0, start=0, mode="decode"):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    if mode == "prefill":
        code = _CPU_PREFILL_CHILD.format(root=ROOT, seconds=seconds, start=start)
    else:
        code = _CPU_CHILD.format(root=ROOT, workload=workload, seconds=seconds, per_step=per_step,
                                 fixed_steps=fixed_steps, start=start)
    return [sys.executable, "-c", code], env


def run_cpu_prefill_baseline(seconds, bytes_per_child):
    """The fp64 oracle on sampled chunk rows of the mixed workload's prefill
    (1 thread, then one single-threaded process per host core), in TFLOP/s of
    the same algorithmic FLOPs as the GPU figure."""
    def one(start):
        return _oracle_cmd("mixed", seconds, 1, start=start, mode="prefill")
    try:
        cmd, env = one(0)
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=3600)
        if r.returncode != 0:
            raise RuntimeError(r.stderr[-2000:])
        res = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # report, do not hide
        return {"value": None, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "error": str(e)[-300:]}
    out = {"value": round(res["flops"] / res["seconds"] / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
           "kind": "oracle",
           "sample": f"{res['units']} chunk rows x {4} query heads of one KV head (cycled over the 4 "
                     f"sequences, 8 KV heads and every 37th chunk row) through the fp64 numpy oracle's "
                     f"causal prefill in {res['seconds']:.1f} s on 1 host thread (BLAS pinned to 1)",
           "host_logical_cores": os.cpu_count()}
    cores = os.cpu_count() or 1
    try:
        free = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError):
        free = 0
    n = max(1, min(cores, int(free // 2 // max(bytes_per_child, 1)))) if free else 1
    procs = []
    try:
        for i in range(n):
            cmd, env = one(i * 31)
            procs.append(subprocess.Popen(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
        outs = [p.communicate(timeout=3600) for p in procs]
        if any(p.returncode != 0 for p in procs):
            raise RuntimeError(next(e for p, (_, e) in zip(procs, outs) if p.returncode != 0)[-2000:])
        rs = [json.loads(o.strip().splitlines()[-1]) for o, _ in outs]
        out["all_cores"] = {"value": round(sum(x["flops"] / x["seconds"] for x in rs) / 1e12, 6),
                            "unit": "TFLOP/s", "cores": n,
                            "sample": f"{n} single-threaded oracle processes at once, each timing about "
                                      f"{seconds:.0f} s of chunk rows; the rate is the sum of theirs"}
    except Exception as e:  # report, do not hide
        for p in procs:
            if p.poll() is None:
                p.kill()
        out["all_cores"] = {"value": None, "cores": n, "error": str(e)[-300:]}
    return out


def _oracle_child(workload, seconds, per_step, fixed_steps=0):
    cmd, env = _oracle_cmd(workload, seconds, per_step, fixed_steps)
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=3600)
    if r.returncode != 0:
        raise RuntimeError(f"oracle child failed:\n{r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_cpu_baseline(workload, seconds, bytes_per_child):
    try:
        res = _oracle_child(workload, seconds, per_step=1)
    except Exception as e:  # report, do not hide
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle", "error": str(e)[-300:]}
    return {"value": round(res["kv_bytes"] / res["seconds"] / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{res['units']} (sequence, KV head) units of the {workload} batch (cycled in "
                      f"order; {res['tokens']} context tokens, each unit's cache write and decode) "
                      f"through the fp64 numpy oracle in {res['seconds']:.1f} s on 1 host thread "
                      f"(BLAS pinned to 1 thread)",
            "host_logical_cores": os.cpu_count(),
            "all_cores": run_cpu_all_cores(workload, seconds, bytes_per_child)}


def run_cpu_all_cores(workload, seconds, bytes_per_child):
    """The same oracle in one single-threaded process per host core, run at
    the same time, each starting at its own place in the unit list; the
    reported rate is the sum of the processes' rates. The process count is
    capped so that their copies of the workload take at most half of the
    host's free memory."""
    cores = os.cpu_count() or 1
    try:
        free = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError):
        free = 0
    n = max(1, min(cores, int(free // 2 // max(bytes_per_child, 1)))) if free else 1
    procs = []
    try:
        for i in range(n):
            cmd, env = _oracle_cmd(workload, seconds, per_step=1, start=i * 997)
            procs.append(subprocess.Popen(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                          text=True))
        outs = [p.communicate(timeout=3600) for p in procs]
        if any(p.returncode != 0 for p in procs):
            err = next(e for p, (_, e) in zip(procs, outs) if p.returncode != 0)
            raise RuntimeError(f"oracle child failed:\n{err[-2000:]}")
        res = [json.loads(o.strip().splitlines()[-1]) for o, _ in outs]
    except Exception as e:  # report, do not hide
        for p in procs:
            if p.poll() is None:
                p.kill()
        return {"value": None, "cores": n, "error": str(e)[-300:]}
    rate = sum(r["kv_bytes"] / r["seconds"] for r in res) / 1e9
    return {"value": round(rate, 4), "unit": "GB/s", "cores": n,
            "sample": f"{n} single-threaded oracle processes at once, each timing about {seconds:.0f} s "
                      f"of units ({sum(r['units'] for r in res)} units, {sum(r['tokens'] for r in res)} "
                      f"context tokens in all); the rate is the sum of theirs"}


# --------------------------------------------------------- reference arm ----

def run_reference(args):
    """The oracle as the reference arm: the same metric and unit on the host
    cores, each step a bounded sample (whole sequences) of the workload."""
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return
    # size the per-step sample so that warmup + steps stay within ~2 minutes
    calib = _oracle_child(args.workload, 2.0, per_step=1)
    sec_per_unit = calib["seconds"] / max(calib["units"], 1)
    budget = args.ref_seconds
    total_steps = args.steps + args.warmup
    per_step = max(1, int(budget / total_steps / sec_per_unit))
    per_step = min(per_step, 512)
    if args.warmup:
        _oracle_child(args.workload, 0, per_step=per_step, fixed_steps=args.warmup)
    res = _oracle_child(args.workload, 0, per_step=per_step, fixed_steps=args.steps)
    value = res["kv_bytes"] / res["seconds"] / 1e9
    sample = (f"each step: {per_step} (sequence, KV head) unit(s) of the {args.workload} batch, "
              f"cycled in order, through the fp64 numpy oracle (reshape_and_cache + decode) on 1 "
              f"host thread")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(res["seconds"] * 1e3 / max(args.steps, 1), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic: the same seeded workload as the GPU arm",
        "config": {"workload": args.workload, "sample_units_per_step": per_step,
                   "unit": "one (sequence, KV head): its query heads over its context"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


SWAP_METRIC = "KV block swap between HBM and page-locked host memory, GB/s (out + in)"


def run_swap(args):
    """Preemption by swapping on the 8B-GQA block shape: each step swaps 4,096
    blocks (16 sequences x 4,096 tokens; 32 KiB of K and 32 KiB of V each) out
    to page-locked host memory and back into other blocks. The roofline
    denominator is a contiguous cudaMemcpyAsync of the same bytes each way,
    measured in the same run."""
    import numpy as np
    import torch

    import paged_kv_cache_59_gb300 as pk
    from paged_kv_cache_59_gb300 import build as pk_build

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    pk_build.build()
    pk.load()
    dev = torch.device("cuda", local)
    Hk, D, BS = 8, 128, 16
    n_move, n_pool = 4096, 8192
    rng = np.random.default_rng(8)
    kp = torch.zeros((n_pool, Hk, BS, D), dtype=torch.int16, device=dev)
    vp = torch.zeros_like(kp)
    ids_out = torch.from_numpy(rng.permutation(n_pool)[:n_move].astype(np.int32)).to(dev)
    ids_in = torch.from_numpy(rng.permutation(n_pool)[:n_move].astype(np.int32)).to(dev)
    hk = torch.empty((n_move, Hk, BS, D), dtype=torch.int16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    block_bytes = Hk * BS * D * 2 * 2          # K + V
    bytes_each_way = n_move * block_bytes
    stream = torch.cuda.current_stream()

    def step(evs=None):
        if evs: evs[0].record(stream)
        pk.pa_swap_out_blocks(kp, vp, ids_out, hk, hv)
        if evs: evs[1].record(stream)
        pk.pa_swap_in_blocks(hk, hv, kp, vp, ids_in)
        if evs: evs[2].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert pk.pa_get_device_error() == 0
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    vis = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    sampler = ClockSampler(vis[local] if local < len(vis) else str(local))
    sampler.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    sampler.mark("begin")
    t0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    sampler.mark("end")
    clocks = sampler.stop()
    total_ms = t0.elapsed_time(t1)
    out_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    in_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    # the link's contiguous copy rate, same bytes, both directions
    dk = torch.empty((n_move, Hk, BS, D), dtype=torch.int16, device=dev)
    dv = torch.empty_like(dk)
    def memcpy_ms(to_host):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(3):
            (hk.copy_(dk, non_blocking=True), hv.copy_(dv, non_blocking=True)) if to_host else \
                (dk.copy_(hk, non_blocking=True), dv.copy_(hv, non_blocking=True))
        a.record(stream)
        for _ in range(10):
            (hk.copy_(dk, non_blocking=True), hv.copy_(dv, non_blocking=True)) if to_host else \
                (dk.copy_(hk, non_blocking=True), dv.copy_(hv, non_blocking=True))
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 10
    m_out, m_in = memcpy_ms(True), memcpy_ms(False)
    gbs = lambda ms: bytes_each_way / (ms / 1e3) / 1e9
    value = 2 * bytes_each_way / (total_ms / args.steps / 1e3) / 1e9
    peak = 2 * bytes_each_way / ((m_out + m_in) / 1e3) / 1e9
    result = {
        "metric": SWAP_METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: 4,096 of 8,192 pool blocks (random ids) out to host memory and back into "
                "4,096 other random blocks",
        "config": {"workload": "swap_8b_4096blocks", "n_kv_heads": Hk, "head_dim": D, "block_size": BS,
                   "bytes_each_way_per_step": bytes_each_way, "blocks_per_step": n_move,
                   "step": "pa_swap_out_blocks + pa_swap_in_blocks (one kernel each)"},
        "swap_out_gbs": round(gbs(out_ms), 1), "swap_in_gbs": round(gbs(in_ms), 1),
        "roofline": {"bound": "host link", "kernel": "swap_blocks_kernel (out and in)",
                     "achieved": round(value, 1), "peak": round(peak, 1),
                     "peak_source": "contiguous cudaMemcpyAsync of the same bytes, pinned host <-> HBM, "
                                    "measured in this run (out %.1f, in %.1f GB/s)" % (gbs(m_out), gbs(m_in)),
                     "unit": "GB/s", "frac": round(value / peak, 4), "traffic": None},
        "gpu_launches": 2 * args.steps, "clocks": clocks,
    }
    print(json.dumps(result), flush=True)


PREFIX_METRIC = "prefix-cached admissions per second (host block manager)"


def run_prefix_cache(args):
    """Host-side measurement of the block manager's prefix cache: requests
    that share a 2,048-token system prompt plus a distinct 37-token query
    (the shared-prompt case the pages describe) are admitted (longest cached
    prefix adopted, remaining tokens appended, full blocks registered) and
    freed, in a pool small enough that the cache keeps evicting old queries'
    blocks. Each step admits and frees 1,000 requests; the C++ manager is
    called through the C ABI (token arrays prepared outside the timed loop)."""
    import ctypes as C
    import numpy as np

    from paged_kv_cache_59_gb300 import _capi
    from paged_kv_cache_59_gb300 import build as pk_build

    pk_build.build()
    lib = _capi.load()
    rng = np.random.default_rng(12)
    prompt = rng.integers(0, 32000, 2048).astype(np.int32)
    reqs = [np.ascontiguousarray(np.concatenate([prompt, rng.integers(0, 32000, 37).astype(np.int32)]))
            for _ in range(1000)]
    ptrs = [r.ctypes.data_as(C.POINTER(C.c_int32)) for r in reqs]
    bm = lib.pa_bm_create(128 + 64 * 3 + 256, 16)
    n_cached, n_added, ncow = C.c_int64(0), C.c_int(0), C.c_int(0)
    slots = (C.c_int64 * 4096)()
    cow = (C.c_int64 * 2)()
    hits = tok_total = 0
    sid = 0

    def step():
        nonlocal sid, hits, tok_total
        live = []
        for r, p in zip(reqs, ptrs):
            assert lib.pa_bm_add_seq_cached(bm, sid, p, len(r), C.byref(n_cached)) == 0
            rest = len(r) - n_cached.value
            assert lib.pa_bm_append_tokens(bm, sid, rest, slots, cow, 1, C.byref(ncow)) == 0
            assert lib.pa_bm_cache_blocks(bm, sid, p, len(r), C.byref(n_added)) == 0
            hits += n_cached.value
            tok_total += len(r)
            live.append(sid)
            sid += 1
            if len(live) == 64:                  # keep 64 resident
                assert lib.pa_bm_free_seq(bm, live.pop(0)) == 0
        for s_ in live:
            assert lib.pa_bm_free_seq(bm, s_) == 0

    for _ in range(max(args.warmup, 3)):
        step()
    hits = tok_total = 0
    steps = min(args.steps, 20)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    dt = time.perf_counter() - t0
    lib.pa_bm_destroy(bm)
    per_s = steps * len(reqs) / dt
    print(json.dumps({
        "metric": PREFIX_METRIC, "value": round(per_s, 1), "unit": "admissions/s", "n_gpus": 0,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / steps, 3),
        "higher_is_better": True, "scaling": "none", "vs_baseline": None, "dtype": "int32 tokens",
        "data": "synthetic: 1,000 requests = one 2,048-token prompt + distinct 37-token queries",
        "config": {"workload": "prefix_cache_2048_shared_prompt", "block_size": 16, "pool_blocks": 576,
                   "resident": 64, "step": "admit (add_seq_cached + append + cache_blocks) and free 1,000 "
                   "requests through the C ABI"},
        "cached_token_fraction": round(hits / max(tok_total, 1), 4),
        "us_per_admission": round(dt * 1e6 / (steps * len(reqs)), 2),
        "host_cores_used": 1,
    }), flush=True)


def main():
    args = parse_args()
    if args.record_traffic:
        print(json.dumps(record_traffic(args.record_traffic, args.workload)))
    elif args.impl == "reference":
        run_reference(args)
    elif args.workload == "swap_8b":
        run_swap(args)
    elif args.workload == "prefix_cache":
        run_prefix_cache(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
