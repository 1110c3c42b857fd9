"""Benchmark: one decode step of load-balanced split-KV GQA attention.

A step is the whole path over one synthetic batch: Task Assign (hpa_plan),
split-KV attention (hpa_decode_attn) and the combine (hpa_combine), on one
stream.  Default workload: the mixed-length batch (40 requests log-uniform
in [1K, 128K] + one each of 1K/4K/16K/64K/128K; 64/8 heads, d=128; bf16 KV
in 64-token pages with shuffled page ids; tile 512; one partition per
resident attention CTA).  Its KV (about 7 GB) is far larger than L2, so no
flush is needed between steps.

  python bench.py [--gpus N --steps K --warmup W] [--config 1..5] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own batch
(seeded by rank) on its own GPU -- data-parallel replicas with no collective
on the data path -- and the timing is the max over ranks.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "mixed-length decode attention: µs/batch, KV-read HBM GB/s and % of peak"
UNIT = "us/batch"

# DRAM traffic of one decode_attn_kernel launch from an ncu capture, valid only
# for the kernel source it was taken on (sha256 of decode_attn.cu) and for the
# workload it was taken on; else null.  Expressed per algorithmic KV byte and
# scaled to the full batch, since traffic grows with the KV read.
TRAFFIC_PROFILE = {
    "config": 3,
    "source_sha256": "67e86ff851789597537dc8fc07e83fbc9e8a369d6e98cd1044fef4e76cc1ff91",
    "bytes_per_kv_byte": (2574309376 + 3269120) / 2572926976,
    "workload": "mixed_45req_1k_128k_paged, first 12 requests (2.57 GB KV)",
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_sha():
    src = os.path.join(ROOT, "load_balanced_split_gb300", "csrc", "decode_attn.cu")
    return hashlib.sha256(open(src, "rb").read()).hexdigest()


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.f = None

    def __enter__(self):
        try:
            self.f = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.dev)], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.f is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.f.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- ranks
def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def per_batch_us(ms_per_step: float, world: int) -> float:
    """Whole-job µs per batch: every rank processes one batch per step."""
    return ms_per_step * 1e3 / world


# ----------------------------------------------------------------------------- our arm
def traced_groups(rows: int, attn: str):
    """Row groups of the CTA trace the bench can take for the kernel it times, or None.

    hpa_decode_attn_traced runs the kernel hpa_decode_attn picks: the tcgen05 kernel
    above 16 query rows per KV head (no row-group axis), else mma.sync (one CTA per
    group of 16 rows); the all-heads variant traces itself.  A forced kernel that
    differs from that choice has no trace."""
    groups = (rows + 15) // 16
    if attn == "allheads":
        return groups
    traced_tc = rows > 16
    timed_tc = attn == "tc" or (attn == "auto" and rows > 16)
    if timed_tc != traced_tc:
        return None
    return 1 if traced_tc else groups


def step_distribution(step_ms):
    """Median and p10 / p90 of single-step times (µs), from the breakdown pass: events
    around every kernel of every step, so each step pays its own event overhead."""
    if not step_ms:
        return None
    x = np.sort(np.asarray(step_ms, dtype=np.float64) * 1e3)
    pick = lambda f: round(float(np.quantile(x, f)), 2)
    return {"median": pick(0.5), "p10": pick(0.1), "p90": pick(0.9), "steps": int(x.size),
            "source": "per-step CUDA events (breakdown pass, rank 0)"}


def run_ours(args, rank, world, local_rank):
    import torch
    import load_balanced_split_gb300 as hpa

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    b = W.make_config(args.config, seed=args.seed + rank, max_requests=args.requests,
                      q_len=args.q_len)
    if args.tile:
        b.tile = args.tile
    kv = hpa.KV_BF16 if b.kv_dtype == "bf16" else hpa.KV_E4M3
    tc = args.attn == "tc"
    allh = args.attn == "allheads"
    mma = args.attn == "mma"
    default_c = (hpa.hpa_default_num_ctas_tc if tc else
                 hpa.hpa_default_num_ctas_allheads if allh else
                 hpa.hpa_default_num_ctas_mma if mma else hpa.hpa_default_num_ctas)
    if args.num_ctas == 0:        # the device default, even where the workload fixes a count
        C = default_c(b.Hkv, b.q_len, kv, b.Hq)
    else:
        C = args.num_ctas or b.num_ctas or default_c(b.Hkv, b.q_len, kv, b.Hq)
    groups = (b.Hq // b.Hkv * b.q_len + 15) // 16  # query-row groups per (partition, head)
    q = b.q.to(dev)
    k, v = b.k_pool.to(dev), b.v_pool.to(dev)
    ks = vs = None
    if kv == hpa.KV_E4M3:
        ks = torch.from_numpy(b.k_scale).to(dev)
        vs = torch.from_numpy(b.v_scale).to(dev)
    lens = torch.from_numpy(b.seq_lens).to(dev)
    indptr = torch.from_numpy(b.page_indptr).to(dev)
    indices = torch.from_numpy(b.page_indices).to(dev)
    ws = hpa.Workspace(b.B, b.q_len, b.Hq, b.d, num_ctas=C, device=dev,
                       weighted=args.plan == "weighted")
    out = torch.empty((b.B, b.q_len, b.Hq, b.d), dtype=torch.bfloat16, device=dev)
    out_lse = torch.empty((b.B, b.q_len, b.Hq), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(w=ws, ev=None):
        if ev is not None:
            ev[0].record(stream)
        w.plan(lens, b.tile, stream)
        if ev is not None:
            ev[1].record(stream)
        if allh:
            hpa.hpa_decode_attn_allheads(q, k, v, indptr, indices, w.taskmap, w.num_ctas,
                                         w.partial_o, w.partial_lse, ks, vs, stream=stream)
        else:
            hpa.hpa_decode_attn(q, k, v, indptr, indices, w.taskmap, w.num_ctas, w.partial_o,
                                w.partial_lse, ks, vs, stream=stream, tc=tc, mma=mma)
        if ev is not None:
            ev[2].record(stream)
        hpa.hpa_combine(w.partial_o, w.partial_lse, w.taskmap, w.num_ctas, out, out_lse, stream)
        if ev is not None:
            ev[3].record(stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def timed(fn, steps, warmup, breakdown=True, join=None):
        """ms per step over `steps` back-to-back steps (events only at the two ends, so
        consecutive kernels keep their programmatic-dependent-launch overlap), then,
        if asked, a second pass with events around each kernel for the breakdown.
        join(), if given, makes `stream` wait for work the steps left on other streams
        before the end event."""
        for _ in range(warmup):
            fn()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        t0.record(stream)
        for _ in range(steps):
            fn()
        if join is not None:
            join()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        total = t0.elapsed_time(t1)
        if not breakdown:
            return total / steps, [], [], [], []
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        for i in range(steps):
            fn(ev=evs[i])
        torch.cuda.synchronize(dev)
        attn = [e[1].elapsed_time(e[2]) for e in evs]
        plan = [e[0].elapsed_time(e[1]) for e in evs]
        comb = [e[2].elapsed_time(e[3]) for e in evs]
        whole = [e[0].elapsed_time(e[3]) for e in evs]
        return total / steps, attn, plan, comb, whole

    with ClockSampler(local_rank) as clk:
        ms, attn, plan_ms, comb_ms, step_ms = timed(step, args.steps, args.warmup)
    clocks = clk.summary()
    torch.cuda.synchronize(dev)
    status = ws.status()
    if status != 0:
        raise RuntimeError("task map status %d after the timed steps" % status)

    ms = max_over_ranks(ms, world, dev)       # the slowest rank sets the step time

    def traced_tail(w, reps=3):
        """Per-CTA timestamps of the attention kernel (outside the timed region)."""
        groups_t = traced_groups(b.Hq // b.Hkv * b.q_len, args.attn)
        if groups_t is None:
            return None
        heads_axis = 1 if allh else b.Hkv  # CTAs per partition and row group
        tr = torch.zeros(4 * w.num_ctas * heads_axis * groups, dtype=torch.int64, device=dev)
        out_t = None
        for _ in range(reps):
            w.plan(lens, b.tile, stream)
            if allh:
                hpa.hpa_decode_attn_allheads(q, k, v, indptr, indices, w.taskmap, w.num_ctas,
                                             w.partial_o, w.partial_lse, ks, vs, trace=tr,
                                             stream=stream)
            else:
                hpa.hpa_decode_attn_traced(q, k, v, indptr, indices, w.taskmap, w.num_ctas,
                                           w.partial_o, w.partial_lse, tr, ks, vs, stream=stream)
            torch.cuda.synchronize(dev)
            out_t = hpa.trace_summary(tr, w.num_ctas, heads_axis, groups_t)
        return {k2: round(v2, 3) if isinstance(v2, float) else v2 for k2, v2 in out_t.items()}

    tail = traced_tail(ws)

    def event_floor_us(reps=200):
        """The same event bracket around a one-element fill (a launch that does almost
        nothing): what any small kernel in the breakdown pays for its launch and events."""
        dummy = torch.zeros(1, dtype=torch.int32, device=dev)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                e0.record(stream)
                dummy.fill_(0)
                e1.record(stream)
        torch.cuda.synchronize(dev)
        return round(statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs) * 1e3, 2)

    floor_us = event_floor_us()

    # the same step with the combine folded into the attention launch (one kernel fewer)
    def fused_step(ev=None):
        hpa.decode_step(ws, q, k, v, lens, indptr, indices, out, out_lse, ks, vs, tile=b.tile,
                        stream=stream, fused=True)

    fused_ms = None if (tc or allh) else max_over_ranks(
        timed(fused_step, args.steps, args.warmup, breakdown=False)[0], world, dev)

    # static split-KV comparators through the same kernels (heuristic and best of a sweep)
    comparator = None
    if not args.no_static and rank == 0:
        max_tiles = int((b.seq_lens.max() + b.tile - 1) // b.tile)
        heur = max(1, min(max_tiles, math.ceil(C / b.B)))
        sweep = sorted(set([heur] + [s for s in (1, 2, 4, 8, 16, 32, 64, 128) if s <= max_tiles]))
        res = {}
        for s in sweep:
            wss = hpa.Workspace(b.B, b.q_len, b.Hq, b.d, splits=s, device=dev)
            res[s] = timed(lambda ev=None, w=wss: step(w, ev), max(3, args.steps // 2), 3,
                           breakdown=False)[0]
        best = min(res, key=res.get)
        wsb = hpa.Workspace(b.B, b.q_len, b.Hq, b.d, splits=best, device=dev)
        _, attn_b, _, _, _ = timed(lambda ev=None, w=wsb: step(w, ev), max(3, args.steps // 2), 3)
        comparator = {
            "static_heuristic": {"splits": heur, "us_per_batch": round(res[heur] * 1e3, 2)},
            "static_best": {"splits": best, "us_per_batch": round(res[best] * 1e3, 2),
                            "attention_us": round(statistics.mean(attn_b) * 1e3, 2),
                            "tail": traced_tail(wsb)},
            "sweep_us": {str(s): round(t * 1e3, 2) for s, t in res.items()},
            "speedup_vs_static_heuristic": round(res[heur] / ms, 3),
            "speedup_vs_static_best": round(res[best] / ms, 3),
        }

    # End to end through the public API with host buffers.  A step's inputs (q,
    # lengths, page table) sit back to back in one pinned host buffer and one device
    # buffer, and its outputs (out, lse) likewise, so a step moves them with one copy
    # each way; the device tensors the calls take are views into those buffers.
    # Every step copies its inputs in and its result out inside the timed region, on
    # two copy streams and two sets of device buffers, so that step i + 1's input copy
    # and step i's result copy run while the neighbouring step computes (as a serving
    # loop would pipeline them).
    def packed(tensors, device):
        offs, total = [], 0
        for t in tensors:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = (torch.empty(total, dtype=torch.uint8, device=device) if device is not None
               else torch.empty(total, dtype=torch.uint8).pin_memory())
        views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                 for o, t in zip(offs, tensors)]
        return buf, views

    inputs = [b.q, torch.from_numpy(b.seq_lens), torch.from_numpy(b.page_indptr),
              torch.from_numpy(b.page_indices)]
    in_h, in_h_views = packed(inputs, None)
    for dst, src in zip(in_h_views, inputs):
        dst.copy_(src)
    in_ds = [packed(inputs, dev) for _ in range(2)]            # (buffer, views) per set
    out_ds = [packed([out, out_lse], dev) for _ in range(2)]
    out_hs = [packed([out, out_lse], None)[0] for _ in range(2)]
    h2d = in_h.numel()
    d2h = out_hs[0].numel()
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    h2d_ev = [torch.cuda.Event() for _ in range(2)]
    comp_ev = [torch.cuda.Event() for _ in range(2)]
    d2h_ev = [torch.cuda.Event() for _ in range(2)]
    e2e_count = [0]

    def e2e_step(ev=None):
        cur = e2e_count[0] % 2
        e2e_count[0] += 1
        in_d, (q_e, lens_e, indptr_e, indices_e) = in_ds[cur]
        out_d, (out_e, lse_e) = out_ds[cur]
        # inputs: after the step two back (which read this buffer set) has computed
        h2d_stream.wait_event(comp_ev[cur])
        with torch.cuda.stream(h2d_stream):
            in_d.copy_(in_h, non_blocking=True)
        h2d_ev[cur].record(h2d_stream)
        stream.wait_event(h2d_ev[cur])
        stream.wait_event(d2h_ev[cur])  # the result buffer's previous copy-out is done
        hpa.decode_step(ws, q_e, k, v, lens_e, indptr_e, indices_e, out_e, lse_e, ks, vs,
                        tile=b.tile, stream=stream, tc=tc, allheads=allh, mma=mma)
        comp_ev[cur].record(stream)
        d2h_stream.wait_event(comp_ev[cur])
        with torch.cuda.stream(d2h_stream):
            out_hs[cur].copy_(out_d, non_blocking=True)
        d2h_ev[cur].record(d2h_stream)

    def e2e_join():
        stream.wait_stream(h2d_stream)
        stream.wait_stream(d2h_stream)

    e2e_ms = max_over_ranks(timed(e2e_step, args.steps, args.warmup, breakdown=False,
                                  join=e2e_join)[0], world, dev)

    def e2e_serial_step(ev=None):
        """The same step with both copies on the compute stream (nothing overlaps)."""
        in_d, (q_e, lens_e, indptr_e, indices_e) = in_ds[0]
        out_d, (out_e, lse_e) = out_ds[0]
        with torch.cuda.stream(stream):
            in_d.copy_(in_h, non_blocking=True)
        hpa.decode_step(ws, q_e, k, v, lens_e, indptr_e, indices_e, out_e, lse_e, ks, vs,
                        tile=b.tile, stream=stream, tc=tc, allheads=allh, mma=mma)
        with torch.cuda.stream(stream):
            out_hs[0].copy_(out_d, non_blocking=True)

    e2e_serial_ms = max_over_ranks(
        timed(e2e_serial_step, args.steps, args.warmup, breakdown=False)[0], world, dev)

    feeder = None if args.no_feeder else feeder_measure(hpa, dev, stream, args, timed)
    return dict(b=b, C=C, ms=ms, attn=attn, plan=plan_ms, comb=comb_ms, step_ms=step_ms,
                clocks=clocks, tail=tail, floor_us=floor_us,
                feeder=feeder,
                fused_ms=fused_ms, comparator=comparator, e2e_ms=e2e_ms,
                e2e_serial_ms=e2e_serial_ms, h2d=h2d, d2h=d2h)


def feeder_measure(hpa, dev, stream, args, timed, n_tokens=65536):
    """hpa_store_kv on a 64K-token chunk (RoPE + RMSNorm + Hadamard + E4M3 + paged store).

    Algorithmic bytes per token: K and V in (8 heads x 128 x bf16 x 2 = 4096 B), the
    token's cos/sin row (512 B) and the E4M3 K and V written (2048 B)."""
    import torch
    b = W.make_batch([n_tokens], q_len=1, kv_dtype="e4m3", seed=args.seed + 99)
    fi = W.make_feeder_inputs(args.seed + 99, 1, n_tokens, max_pos=n_tokens)
    k, v = b.k_pool.to(dev), b.v_pool.to(dev)
    ks, vs = torch.from_numpy(b.k_scale).to(dev), torch.from_numpy(b.v_scale).to(dev)
    lens = torch.from_numpy(b.seq_lens).to(dev)
    ip, ix = torch.from_numpy(b.page_indptr).to(dev), torch.from_numpy(b.page_indices).to(dev)
    kn, vn = fi.k_new.to(dev), fi.v_new.to(dev)
    cs, w = torch.from_numpy(fi.cos_sin).to(dev), torch.from_numpy(fi.norm_w).to(dev)

    def f(ev=None):
        hpa.hpa_store_kv(kn, vn, lens, ip, ix, cs, w, k, v, eps=fi.eps, use_hadamard=True,
                         k_scale=ks, v_scale=vs, stream=stream)

    ms = timed(f, max(10, args.steps // 10), args.warmup, breakdown=False)[0]
    nbytes = n_tokens * (4096 + 512 + 2048)
    return {"workload": "store %d new tokens, 8 KV heads, E4M3 cache, Hadamard on" % n_tokens,
            "us_per_call": round(ms * 1e3, 2), "algorithmic_bytes": nbytes,
            "achieved_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(b, target_s):
    """Time the oracle on a prefix of the batch's requests (about target_s seconds).

    Returns (seconds per batch extrapolated by token count, threads, description)."""
    import oracle
    threads = os.cpu_count() or 1
    order = list(range(b.B))
    # calibrate on the first request, then take a prefix worth ~target_s
    t0 = time.perf_counter()
    oracle.attention(b, items=[(0, 0, int(b.seq_lens[0]))], n_threads=threads)
    t1 = time.perf_counter() - t0
    rate = int(b.seq_lens[0]) / max(t1, 1e-6)                # tokens per second
    want = max(int(rate * target_s), 1)
    items, tok = [], 0
    for r in order:
        if tok >= want:
            break
        items.append((r, 0, int(b.seq_lens[r])))
        tok += int(b.seq_lens[r])
    # when the whole batch is quicker than target_s, repeat it to fill the time
    reps, dt = 0, 0.0
    while reps == 0 or (dt < target_s and reps < 50):
        t0 = time.perf_counter()
        oracle.attention(b, items=items, n_threads=threads)
        dt += time.perf_counter() - t0
        reps += 1
    total = int(b.seq_lens.astype(np.int64).sum())
    per_batch = dt / reps * total / tok
    desc = ("fp64 C oracle, unsplit attention of the first %d of %d requests (%d of %d tokens, "
            "all %d heads), %d run(s), %.1f s of CPU time, scaled to the batch by token count"
            % (len(items), b.B, tok, total, b.Hq, reps, dt))
    return per_batch, threads, desc


def run_reference(args, rank, world):
    if rank != 0:
        return None
    b = W.make_config(args.config, seed=args.seed, max_requests=args.requests)
    # the whole run (warm-up + timed steps) is budgeted at about two minutes of CPU time
    per_step_s = max(0.05, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(b, per_step_s)
    secs, threads, desc = [], 0, ""
    t_begin = time.perf_counter()
    for _ in range(args.steps):
        s, threads, desc = oracle_sample(b, per_step_s)
        secs.append(s)
    wall = time.perf_counter() - t_begin
    us = statistics.mean(secs) * 1e6
    return {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(us / 1e3, 3), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": W.CONFIGS[args.config], "batch": int(b.B),
                       "kv_tokens": int(b.seq_lens.sum()), "q_len": b.q_len,
                       "heads": "64q/8kv", "head_dim": 128, "kv_dtype": b.kv_dtype,
                       "seed": args.seed},
            "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": threads,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": round(wall, 1)}


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--requests", type=int, default=None,
                    help="keep only the first N requests of the workload (smaller case)")
    ap.add_argument("--tile", type=int, default=None, help="tile size in tokens (default 512)")
    ap.add_argument("--q-len", type=int, default=None,
                    help="query tokens per request (default: the workload's, 1 or 2)")
    ap.add_argument("--plan", default="tiles", choices=["tiles", "weighted"],
                    help="tile budgets (the pages' method) or the token-weighted variant")
    ap.add_argument("--num-ctas", type=int, default=None,
                    help="partitions per KV head (default: the workload's own count, else the "
                         "device default; 0: the device default)")
    ap.add_argument("--attn", default="auto", choices=["auto", "mma", "tc", "allheads"],
                    help="attention kernel: hpa_decode_attn's own choice by query rows per KV "
                         "head (auto), mma.sync (hpa_decode_attn_mma), tcgen05 "
                         "(hpa_decode_attn_tc), or mma.sync with every KV head inside the CTA "
                         "(hpa_decode_attn_allheads)")
    ap.add_argument("--no-static", action="store_true", help="skip the static comparators")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-feeder", action="store_true", help="skip the KV-store feeder timing")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.init_process_group("nccl")

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    r = run_ours(args, rank, world, local_rank)
    if rank != 0:
        return
    b = r["b"]
    kv_bytes = b.kv_bytes
    peak, peak_kind = peaks()
    attn_ms = statistics.mean(r["attn"])
    achieved = kv_bytes / (attn_ms * 1e-3) / 1e9
    us_batch = per_batch_us(r["ms"], world)
    traffic = None
    rows = b.Hq // b.Hkv * b.q_len
    on_tc = args.attn == "tc" or (args.attn == "auto" and rows > 16)
    kernel_name = "decode_attn_tc_kernel" if on_tc else "decode_attn_kernel"
    if (args.attn in ("auto", "mma") and not on_tc and args.config == TRAFFIC_PROFILE["config"]
            and TRAFFIC_PROFILE["source_sha256"] == kernel_sha()
            and TRAFFIC_PROFILE["bytes_per_kv_byte"]):
        traffic = int(TRAFFIC_PROFILE["bytes_per_kv_byte"] * kv_bytes)
    cpu = None
    if not args.no_cpu_baseline:
        s, threads, desc = oracle_sample(b, 15.0)
        cpu = {"value": round(s * 1e6, 1), "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": desc}
    line = {
        "metric": METRIC, "value": round(us_batch, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["ms"], 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": b.kv_dtype, "data": "synthetic",
        "config": {"workload": W.CONFIGS[args.config] + (
                       "" if args.requests is None else " (first %d requests)" % b.B),
                   "batch": int(b.B),
                   "kv_tokens": int(b.seq_lens.sum()), "q_len": b.q_len, "heads": "64q/8kv",
                   "head_dim": 128, "page": 64, "tile": b.tile, "num_ctas": int(r["C"]),
                   "kv_dtype": b.kv_dtype, "kv_bytes": int(kv_bytes), "plan": args.plan,
                   "attention_kernel": ("mma.sync, all KV heads per CTA" if args.attn == "allheads"
                                        else "tcgen05" if on_tc else "mma.sync"),
                   "l2": "inputs larger than L2 (%.2f GB KV), no flush" % (kv_bytes / 1e9),
                   "parallelism": "dp%d replicas" % world, "seed": args.seed},
        "kv_gbs": round(kv_bytes / (r["ms"] * 1e-3) / 1e9, 1),
        "pct_of_hbm_peak": round(100.0 * kv_bytes / (r["ms"] * 1e-3) / 1e9 / peak, 1),
        "breakdown_us": {"plan": round(statistics.mean(r["plan"]) * 1e3, 2),
                         "attention": round(attn_ms * 1e3, 2),
                         "combine": round(statistics.mean(r["comb"]) * 1e3, 2),
                         "event_floor": r["floor_us"]},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": kernel_name,
                     "peak_kind": peak_kind + " (hbm_gbs)"},
        "step_us_distribution": step_distribution(r["step_ms"]),
        "tail": r["tail"],
        "kv_store_feeder": r["feeder"],
        "fused_combine": None if r["fused_ms"] is None else {
            "us_per_batch": round(per_batch_us(r["fused_ms"], world), 2),
            "speedup_vs_three_calls": round(r["ms"] / r["fused_ms"], 3)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(per_batch_us(r["e2e_ms"], world), 2), "unit": UNIT,
                "h2d_bytes_per_step": int(r["h2d"]), "d2h_bytes_per_step": int(r["d2h"]),
                "copies": "every step's input and result copies inside the timed region, on "
                          "two copy streams with double-buffered device buffers, overlapping "
                          "the neighbouring steps",
                "serial_value": round(per_batch_us(r["e2e_serial_ms"], world), 2)},
        "gpu_launches": 3 * args.steps,
        "clocks": r["clocks"],
        "comparator": r["comparator"],
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
