#!/usr/bin/env python
"""Benchmark of the per-decode-step KV-cache eviction engine.

One step = one decode step of every layer of the 70B-shaped H2O workload
(80 layers, 16 sequences x 8 KV heads, group 8, d=128, bf16, 16384-token
prompts = 86 GB of K/V, budget 3276 = 1638 heavy + 1638 recent): split-K
attention + score epilogue, bottom-k selection, eviction, admission and
gated relocation, through the C ABI.  The prompt is prefilled and the first
(mass-eviction) decode step runs inside the warm-up; the timed steps are the
steady state.  Every layer call streams ~215 MB of K/V, more than the 129 MB
L2, so no L2 flush is needed between steps.

Metric: KV bytes scored + evicted per step (K/V rows read by the attention,
the H2O score read-modify-write, 1 KB per relocated token) / step time, in
GB/s, as in the task's metric; tokens scored per second alongside.
"""
import argparse
import contextlib
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

METRIC = "KV GB/s scored+evicted per decode step (frac. of HBM peak); tokens scored/s"
UNIT = "GB/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=48)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--workload", default="h2o_70b")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--cpu-lanes", type=int, default=96)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-layers", type=int, default=0,
                    help="profiling only: run the workload with this many layers (not a bench number)")
    ap.add_argument("--kernel-table", action="store_true",
                    help="time the engine's other kernels on their own workloads (DropKV window scoring at "
                         "32K and 128K, selection, forced compaction, the SnapKV and toy decode steps), one "
                         "JSON line each, instead of the decode-step bench line")
    ap.add_argument("--only", default="",
                    help="with --kernel-table: comma-separated subset of d3_32k, d3_128k, snapkv_pf_32k, "
                         "snapkv_pf_128k, snapkv, dropkv_decode, toy, reloc")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        time.sleep(0.3)

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.p.terminate()
        self.p.wait()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[2]))
                smax.append(float(r[3]))
                for nm, v in zip(names, r[6:10]):
                    if v.strip().lower() == "active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# oracle baseline (CPU) on a bounded sample of lanes
# ---------------------------------------------------------------------------
def _oracle_lane_job(job):
    import types
    import numpy as np
    from oracle.engine import Engine as Oracle
    K, V, steps, f = job
    cfg = types.SimpleNamespace(policy=f["policy"], num_layers=1, batch=1, num_q_heads=f["g"], num_kv_heads=1,
                                head_dim=f["d"], blocks_per_pool=f["blocks"], budget=f["budget"],
                                recent_window=f["R"], obs_window=f["W"], pool_kernel=f["pk"],
                                theta_f=f["theta"])
    o = Oracle(cfg)
    o.prefill(0, K[None, None].astype(np.float64), V[None, None].astype(np.float64))
    q, kn, vn, pos = steps[0]
    o.decode_step(0, q[None].astype(np.float64), kn[None, None].astype(np.float64),
                  vn[None, None].astype(np.float64), pos)         # mass eviction: warm-up
    t0 = time.perf_counter()
    nbytes = tokens = 0
    for q, kn, vn, pos in steps[1:]:
        n = o.layers[0].lanes[0].pos.size
        r = o.decode_step(0, q[None].astype(np.float64), kn[None, None].astype(np.float64),
                          vn[None, None].astype(np.float64), pos)
        tokens += n + 1
        nbytes += (n + 1) * 2 * f["d"] * 2 + n * 8 + len(r["moves"]) * 4 * f["d"] * 2
    return time.perf_counter() - t0, nbytes, tokens


def oracle_baseline(lane_inputs, f, workers):
    """Times the oracle's steady-state decode steps on the sampled lanes in a
    spawn pool of single-threaded workers; returns (GB/s, tokens/s, seconds)."""
    import multiprocessing as mp
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    jobs = [(K, V, steps, f) for K, V, steps in lane_inputs]
    t0 = time.perf_counter()
    with mp.get_context("spawn").Pool(workers) as pool:
        res = pool.map(_oracle_lane_job, jobs)
    wall = time.perf_counter() - t0
    busy = sum(r[0] for r in res)
    nbytes = sum(r[1] for r in res)
    tokens = sum(r[2] for r in res)
    # per-core throughput x cores used (the workers run concurrently)
    gbs = nbytes / busy * workers / 1e9
    return gbs, tokens / busy * workers, busy, wall


def lane_sample_inputs(wl, shp, n_lanes, n_steps, device):
    """Context and step inputs of the first n_lanes lanes of layer 0, as
    float32 numpy arrays (bf16 values are exact in float32)."""
    import torch
    K, V = wl.context(0, device=device)
    g = shp.group
    out = []
    steps_all = [wl.step(0, t, device=device) for t in range(n_steps)]
    for lane in range(n_lanes):
        b, h = divmod(lane, shp.num_kv_heads)
        steps = [(q[b, h * g:(h + 1) * g].float().cpu().numpy(), kn[b, h].float().cpu().numpy(),
                  vn[b, h].float().cpu().numpy(), pos) for q, kn, vn, pos in steps_all]
        out.append((K[b, h].float().cpu().numpy(), V[b, h].float().cpu().numpy(), steps))
    del K, V
    if device != "cpu":
        torch.cuda.empty_cache()
    return out


def oracle_fields(shp):
    per_lane = -(-shp.max_tokens // 16) + -(-shp.budget // 16) + 2
    return dict(policy=shp.policy, g=shp.group, d=shp.head_dim, blocks=per_lane, budget=shp.budget,
                R=shp.recent_window, W=shp.obs_window, pk=shp.pool_kernel, theta=float(shp.theta_f))


# ---------------------------------------------------------------------------
# measured peaks and committed counters
# ---------------------------------------------------------------------------
def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return float(json.load(open(p))["hbm_gbs"]), "measured"
        except (KeyError, ValueError):
            pass
    return 6800.0, "fallback"


def committed_traffic():
    """DRAM bytes per launch of the decode attention kernel from the
    committed ncu summary, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "d1_attend_h2o70b.json")
    src = os.path.join(ROOT, "kv_cache_token_gb300", "csrc", "attend.cu")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if d.get("attend_cu_sha256_16") != h:
            return None
        return d.get("dram_bytes_per_launch_full_size")
    except (ValueError, OSError):
        return None


# ---------------------------------------------------------------------------
# ranks: one replica per GPU, no collective on the data path
# ---------------------------------------------------------------------------
def rank_shape(shp, rank):
    """The workload of one rank: the same shapes with the rank's own seed
    (lanes are independent, so each GPU serves its own sequences: weak
    scaling); rank 0 keeps the single-GPU seed."""
    import dataclasses
    return shp if rank == 0 else dataclasses.replace(shp, seed=shp.seed + 7919 * rank)


def aggregate_over_ranks(ms_per_step, step_bytes, attended_per_step, device="cpu"):
    """Whole-job figures: the slowest rank's step time, and the bytes and
    tokens every rank processed (timing only; nothing of the data moves)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms_per_step, step_bytes, attended_per_step
    t = torch.tensor([ms_per_step, step_bytes, attended_per_step], dtype=torch.float64, device=device)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    sm = t.clone()
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(sm[1]), float(sm[2])


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist
    import __graft_entry__
    __graft_entry__.build()
    from kv_cache_token_gb300 import Engine, config_from
    from workloads import Workload, shape

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    shp = rank_shape(shape(args.workload), rank)
    if args.profile_layers:
        import dataclasses
        shp = dataclasses.replace(shp, num_layers=args.profile_layers)
    assert shp.kind == "decode"
    assert args.warmup >= 1 and args.warmup + args.steps + args.e2e_steps <= shp.steps, "the workload has %d decode steps" % shp.steps
    wl = Workload(shp)
    eng = Engine(config_from(shp))
    eng.reset()
    cpu_lanes = None
    t_setup = time.time()
    for layer in range(shp.num_layers):
        if layer == 0 and rank == 0 and not args.no_cpu_baseline:
            cpu_lanes = lane_sample_inputs(wl, shp, args.cpu_lanes, args.warmup + args.steps, "cuda")
        K, V = wl.context(layer, device="cuda")
        eng.prefill(layer, K, V)
        del K, V
    torch.cuda.synchronize()
    code, msg = eng.last_error()
    assert code == 0, msg
    total_steps = args.warmup + args.steps + args.e2e_steps
    inputs = [[wl.step(layer, t, device="cuda")[:3] for layer in range(shp.num_layers)]
              for t in range(args.warmup + args.steps)]
    L, B, Hq, d = shp.num_layers, shp.batch, shp.num_q_heads, shp.head_dim
    outs = [torch.empty((B, Hq, d), dtype=torch.float32, device="cuda") for _ in range(L)]
    lses = [torch.empty((B, Hq), dtype=torch.float32, device="cuda") for _ in range(L)]
    vics = [torch.empty((eng.lanes, shp.max_tokens), dtype=torch.int32, device="cuda") for _ in range(L)]
    nvs = [torch.empty((eng.lanes,), dtype=torch.int32, device="cuda") for _ in range(L)]
    stream = torch.cuda.current_stream()

    def step(t):
        pos = shp.ctx + t
        for layer in range(L):
            q, kn, vn = inputs[t][layer]
            eng.decode_step(layer, q, kn, vn, pos, outs[layer], lses[layer], vics[layer], nvs[layer])

    for t in range(args.warmup):
        step(t)
    torch.cuda.synchronize()
    code, msg = eng.last_error()
    assert code == 0, msg
    counts_before = eng.counts.sum(dim=1).cpu().numpy().astype(np.int64)          # per layer
    stats_before = eng.stats_buf.sum(dim=0).cpu().numpy()
    setup_s = time.time() - t_setup

    sampler = ClockSampler(local)
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    elapsed_ms = e0.elapsed_time(e1)
    # dominant kernel: the split-K attention of every layer, replayed on the
    # steady-state tables (it changes no engine state).  Average launch
    # duration: events around each replay of the L launches issued back to
    # back as in a step (consecutive launches overlap only their launch
    # latency); the per-launch figure with events around every launch (no
    # overlap at all) is reported beside it.
    reps = 3
    tlast = args.warmup + args.steps - 1
    b2b = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    iso = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps * L)]
    torch.cuda.synchronize()
    for rep in range(reps):
        b2b[rep][0].record(stream)
        for layer in range(L):
            q, kn, vn = inputs[tlast][layer]
            eng.attend(layer, q, kn, vn)
        b2b[rep][1].record(stream)
    for rep in range(reps):
        for layer in range(L):
            q, kn, vn = inputs[tlast][layer]
            ev = iso[rep * L + layer]
            ev[0].record(stream)
            eng.attend(layer, q, kn, vn)
            ev[1].record(stream)
    torch.cuda.synchronize()
    code, msg = eng.last_error()
    assert code == 0, msg
    counts_after = eng.counts.sum(dim=1).cpu().numpy().astype(np.int64)
    stats_after = eng.stats_buf.sum(dim=0).cpu().numpy()
    assert np.array_equal(counts_before, counts_after), "timed steps are not in steady state"
    lanes = eng.lanes
    attended = int((counts_before + lanes).sum()) * args.steps             # kept + new, every layer
    kv_bytes = attended * 2 * d * 2
    score_bytes = int(counts_before.sum()) * 8 * args.steps
    moved = int(stats_after[5] - stats_before[5])
    move_bytes = moved * 4 * d * 2
    step_bytes = (kv_bytes + score_bytes + move_bytes) / args.steps
    ms_per_step = elapsed_ms / args.steps
    d1_ms = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in b2b) / L
    d1_iso_ms = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in iso)
    fin_ms = ms_per_step / L - d1_ms
    d1_bytes = int((counts_before + lanes).mean()) * 2 * d * 2   # K/V rows per launch (one layer)
    peak, peak_kind = hbm_peak()
    d1_gbs = d1_bytes / (d1_ms * 1e-3) / 1e9

    # end to end through the public call, host buffers, copies in the timed
    # region: each step's inputs of all layers go up in one pinned buffer per
    # tensor kind on a copy stream (double-buffered on the device, so step
    # t+1's upload overlaps step t's compute) and its outputs come back the
    # same way once the step's last layer is done.
    e2e = None
    if args.e2e_steps > 0:
        base = args.warmup + args.steps
        kread = 16
        host_in = []
        for t in range(args.e2e_steps):
            per = [wl.step(layer, base + t)[:3] for layer in range(L)]
            host_in.append(tuple(torch.stack([p[i] for p in per]).pin_memory() for i in range(3)))
        dev_in = [tuple(torch.empty_like(x, device="cuda") for x in host_in[0]) for _ in range(2)]
        out_all = torch.empty((L, B, Hq, d), dtype=torch.float32, device="cuda")
        lse_all = torch.empty((L, B, Hq), dtype=torch.float32, device="cuda")
        nv_all = torch.empty((L, lanes), dtype=torch.int32, device="cuda")
        vic_all = torch.empty((L, lanes, shp.max_tokens), dtype=torch.int32, device="cuda")
        host_out = (torch.empty(out_all.shape, dtype=torch.float32).pin_memory(),
                    torch.empty(lse_all.shape, dtype=torch.float32).pin_memory(),
                    torch.empty(nv_all.shape, dtype=torch.int32).pin_memory(),
                    torch.empty((L, lanes, kread), dtype=torch.int32).pin_memory())
        h2d = sum(x.numel() * x.element_size() for x in host_in[0])
        d2h = sum(x.numel() * x.element_size() for x in host_out)
        cs = torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(args.e2e_steps)]
        ev_done = [torch.cuda.Event() for _ in range(args.e2e_steps)]
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        ea.record(stream)
        cs.wait_stream(stream)

        def upload(t):
            with torch.cuda.stream(cs):
                if t >= 2:
                    cs.wait_event(ev_done[t - 2])          # its device buffer is free again
                for dst, src in zip(dev_in[t % 2], host_in[t]):
                    dst.copy_(src, non_blocking=True)
                ev_in[t].record(cs)

        upload(0)
        for t in range(args.e2e_steps):
            if t + 1 < args.e2e_steps:
                upload(t + 1)
            stream.wait_event(ev_in[t])
            pos = shp.ctx + base + t
            qa, ka, va = dev_in[t % 2]
            for layer in range(L):
                eng.decode_step(layer, qa[layer], ka[layer], va[layer], pos, out_all[layer], lse_all[layer],
                                vic_all[layer], nv_all[layer])
            ev_done[t].record(stream)
            with torch.cuda.stream(cs):
                cs.wait_event(ev_done[t])
                host_out[0].copy_(out_all, non_blocking=True)
                host_out[1].copy_(lse_all, non_blocking=True)
                host_out[2].copy_(nv_all, non_blocking=True)
                host_out[3].copy_(vic_all[:, :, :kread], non_blocking=True)
        stream.wait_stream(cs)
        eb.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = ea.elapsed_time(eb) / args.e2e_steps
        counts_e2e = eng.counts.sum(dim=1).cpu().numpy().astype(np.int64)
        e2e_bytes = (int((counts_e2e + lanes).sum()) * 2 * d * 2 + int(counts_e2e.sum()) * 8)
        e2e = {"value": round(e2e_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 4)}
        code, msg = eng.last_error()
        assert code == 0, msg

    # aggregate over ranks: units processed by all / max time
    ms_per_step, all_bytes, all_attended = aggregate_over_ranks(ms_per_step, step_bytes, attended / args.steps,
                                                                device="cuda")
    value = all_bytes / (ms_per_step * 1e-3) / 1e9
    tokens_s = all_attended / (ms_per_step * 1e-3)

    cpu = None
    if rank == 0 and cpu_lanes is not None:
        workers = max(1, min(len(cpu_lanes), os.cpu_count() or 1, 16))
        gbs, tps, busy, wall = oracle_baseline(cpu_lanes, oracle_fields(shp), workers)
        cpu = {"value": round(gbs, 4), "unit": UNIT, "cores": workers, "kind": "oracle",
               "tokens_scored_per_s": round(tps, 1),
               "sample": "%d lanes of layer 0 x %d steady-state decode steps (after the mass-eviction step), "
                         "numpy float64 oracle, %d single-threaded processes, %.1f s of CPU work"
                         % (len(cpu_lanes), args.warmup + args.steps - 1, workers, busy)}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "tokens_scored_per_s": round(tokens_s, 1),
        "config": {"workload": "h2o_70b: 80 layers, batch 16, 64 q / 8 KV heads, d 128, bf16, context 16384 "
                               "(86 GB K/V), H2O budget 3276 (1638 recent), steady-state decode steps",
                   "global_batch": B * world, "seq_len": shp.ctx, "parallelism": "replica per GPU" if world > 1 else "1 GPU",
                   "l2": "no flush: every layer call streams ~215 MB of K/V, above the 129 MB L2",
                   "bytes_per_step": int(step_bytes), "moved_tokens_timed": moved,
                   "attend_ms_per_layer": round(d1_ms, 5), "rest_of_step_ms_per_layer": round(fin_ms, 5),
                   "setup_s": round(setup_s, 1)},
        "roofline": {"bound": "hbm", "kernel": "attend_bf16_kernel (split-K decode attention)",
                     "achieved": round(d1_gbs, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(d1_gbs / peak, 4), "traffic": committed_traffic(),
                     "algorithmic_bytes_per_launch": d1_bytes, "avg_launch_ms": round(d1_ms, 5),
                     "launches_timed": reps * L, "isolated_launch_ms": round(d1_iso_ms, 5),
                     "isolated_frac": round(d1_bytes / (d1_iso_ms * 1e-3) / 1e9 / peak, 4)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": eng.kernels_per_decode_step() * L * args.steps,
    }
    if args.profile_layers:
        line["profile_only"] = "%d layers: for profiling, not a bench number" % L
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# reference arm: the oracle on host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from workloads import Workload, shape
    shp = shape(args.workload)
    wl = Workload(shp)
    lanes = max(1, args.cpu_lanes)
    steps = min(args.warmup + args.steps, shp.steps)
    t0 = time.time()
    inputs = lane_sample_inputs(wl, shp, lanes, steps, "cpu")
    workers = max(1, min(lanes, os.cpu_count() or 1, 16))
    gbs, tps, busy, wall = oracle_baseline(inputs, oracle_fields(shp), workers)
    bytes_per_step = None
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "tokens_scored_per_s": round(tps, 1),
        "config": {"workload": "h2o_70b: 80 layers, batch 16, 64 q / 8 KV heads, d 128, bf16, context 16384 "
                               "(86 GB K/V), H2O budget 3276 (1638 recent), steady-state decode steps",
                   "seq_len": shp.ctx, "bytes_per_step": bytes_per_step},
        "cpu_baseline": {"value": round(gbs, 4), "unit": UNIT, "cores": workers, "kind": "oracle",
                         "sample": "%d lanes of layer 0 x %d steady-state decode steps, numpy float64 oracle, "
                                   "%d single-threaded processes (%.1f s CPU, %.1f s total)"
                                   % (lanes, steps - 1, workers, busy, time.time() - t0)},
        "e2e": {"value": round(gbs, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# kernel table: the other kernels, each on its own workload
# ---------------------------------------------------------------------------
def tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return float(json.load(open(p))["bf16_tflops"]), "measured"
        except (KeyError, ValueError):
            pass
    return 1900.0, "fallback"


def run_kernel_table(args):
    import numpy as np
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from kv_cache_token_gb300 import Engine, config_from
    from workloads import Workload, shape

    hbm, hbm_kind = hbm_peak()
    tc, tc_kind = tensor_peak()
    only = set(x for x in args.only.split(",") if x)
    stream = torch.cuda.current_stream()

    def timed(fn, reps, warm=2):
        for _ in range(warm):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for a, b in evs:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        ms = sorted(a.elapsed_time(b) for a, b in evs)
        return ms[len(ms) // 2], ms[max(0, len(ms) // 10)], ms[min(len(ms) - 1, (9 * len(ms)) // 10)]

    def emit(row, workload, ms, p10, p90, nbytes=None, flops=None, extra=None):
        line = {"kernel_table": row, "workload": workload, "ms_median": round(ms, 4), "ms_p10": round(p10, 4),
                "ms_p90": round(p90, 4)}
        fr = {}
        if nbytes is not None:
            gbs = nbytes / (ms * 1e-3) / 1e9
            line["hbm"] = {"algorithmic_bytes": int(nbytes), "achieved_gbs": round(gbs, 1), "peak_gbs": hbm,
                           "peak_kind": hbm_kind, "frac": round(gbs / hbm, 4)}
            fr["hbm"] = gbs / hbm
        if flops is not None:
            tf = flops / (ms * 1e-3) / 1e12
            line["tensor"] = {"flops": int(flops), "achieved_tflops": round(tf, 1), "peak_tflops": tc,
                              "peak_kind": tc_kind, "frac": round(tf / tc, 4)}
            fr["tensor"] = tf / tc
        if fr:
            line["bound"] = max(fr, key=fr.get)
        if extra:
            line.update(extra)
        print(json.dumps(line), flush=True)

    # D3 window scoring, selection and (128K) forced compaction
    for tag, name in (("d3_32k", "dropkv_prefill"), ("d3_128k", "paged_128k")):
        if only and tag not in only:
            continue
        shp = shape(name)
        wl = Workload(shp)
        eng = Engine(config_from(shp))
        eng.reset()
        K, V = wl.context(0, device="cuda")
        eng.prefill(0, K, V)
        del K, V
        q, qp = wl.window(0, device="cuda")
        lanes, w, g, d, n = eng.lanes, shp.window, shp.group, shp.head_dim, shp.ctx
        lse = torch.empty((shp.batch, shp.num_q_heads, w), dtype=torch.float32, device="cuda")
        a_out = torch.empty((shp.batch, shp.num_q_heads, w, d), dtype=torch.float32, device="cuda")
        scores = torch.zeros((lanes, shp.max_tokens), dtype=torch.float32, device="cuda")
        ms, p10, p90 = timed(lambda: eng.score(0, q, qp, lse, a_out, scores), reps=10)
        # K and V read once per pass; QK^T and PV (pass 1), QK^T and a V^T (pass 2), full key range per row
        rows = g * w
        emit("D3 DropKV window scoring (pass 1, combine, pass 2, finalize)", name, ms, p10, p90,
             nbytes=2 * lanes * n * 2 * d * 2, flops=4 * 2 * lanes * rows * n * d)
        pos, cnt = eng.positions[0], eng.counts[0]
        victims = torch.full((lanes, shp.max_tokens), -1, dtype=torch.int32, device="cuda")
        nvic = torch.zeros((lanes,), dtype=torch.int32, device="cuda")
        ms, p10, p90 = timed(lambda: eng.select(scores, pos, cnt, shp.budget, shp.recent_window, victims, nvic),
                             reps=10)
        emit("D4 bottom-k selection (radix descent on (key, position))", name, ms, p10, p90,
             nbytes=lanes * n * (4 + 4))
        if tag == "d3_128k":
            samples = []
            for rep in range(3):
                if rep:
                    eng.reset()
                    K, V = wl.context(0, device="cuda")
                    eng.prefill(0, K, V)
                    del K, V
                    eng.score(0, q, qp, lse, a_out, scores)
                    eng.select(scores, pos, cnt, shp.budget, shp.recent_window, victims, nvic)
                if rep == 0:
                    # the block-granular counterfactual of the same eviction
                    # (vToken review, Sec. 2 and Eq. (1)): only blocks whose 16
                    # tokens all died are freed, nothing moves
                    torch.cuda.synchronize()
                    slots_h = eng.slots[0].cpu().numpy()
                    cnt_h = eng.counts[0].cpu().numpy()
                    pos_h = eng.positions[0].cpu().numpy()
                    vic_h, nv_h = victims.cpu().numpy(), nvic.cpu().numpy()
                    bg = {"freed_blocks": 0, "blocks": 0, "live": 0, "half_empty": 0}
                    blocks_before = 0
                    for l in range(lanes):
                        n_l = int(cnt_h[l])
                        dead = np.isin(pos_h[l, :n_l], vic_h[l, :int(nv_h[l])])
                        blk = slots_h[l, :n_l] // 16
                        live = np.bincount(blk[~dead], minlength=int(blk.max()) + 1)
                        held = np.bincount(blk, minlength=live.size) > 0
                        blocks_before += int(held.sum())
                        bg["freed_blocks"] += int((held & (live == 0)).sum())
                        bg["blocks"] += int((held & (live > 0)).sum())
                        bg["live"] += int(live.sum())
                        bg["half_empty"] += int((held & (live > 0) & (live <= 8)).sum())
                    bg["waste_F"] = round(1.0 - bg["live"] / (16.0 * bg["blocks"]), 4) if bg["blocks"] else 0.0
                # outputs allocated outside the timed call
                freed = torch.empty((shp.blocks_per_pool,), dtype=torch.int32, device="cuda")
                moves = torch.empty((lanes * shp.max_tokens, 6), dtype=torch.int32, device="cuda")
                n_freed = torch.empty((1,), dtype=torch.int32, device="cuda")
                n_moves = torch.empty((1,), dtype=torch.int32, device="cuda")
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                eng.compact(0, victims, nvic, freed, n_freed, moves, n_moves)
                e1.record(stream)
                torch.cuda.synchronize()
                samples.append(e0.elapsed_time(e1))
            moved, nf = int(n_moves.item()), int(n_freed.item())
            st = eng.stats(0).cpu().tolist()
            samples.sort()
            emit("D5 token-level compaction (plan, allocate, gather, release)", name, samples[1], samples[0],
                 samples[-1], nbytes=moved * 2 * d * 2 * 2 + int(nvic.sum().item()) * 3 * 4,
                 extra={"moved_tokens": moved, "freed_blocks": nf, "blocks_after": st[9], "live_after": st[10],
                        "blocks_before": blocks_before,
                        "token_level": {"freed_blocks": blocks_before - st[9], "blocks": st[9], "live": st[10],
                                        "half_empty": st[11],
                                        "waste_F": round(1.0 - st[10] / (16.0 * st[9]), 4) if st[9] else 0.0},
                        "block_granular": bg})
        code, msg = eng.last_error()
        assert code == 0, msg
        del eng
        torch.cuda.empty_cache()

    # SnapKV's one-shot prefill selection: window attention mass (K read in
    # both passes, no V), pooled keys, bottom-k at 1/16 of the prompt
    for tag, name in (("snapkv_pf_32k", "snapkv_prefill"), ("snapkv_pf_128k", "snapkv_prefill_128k")):
        if only and tag not in only:
            continue
        shp = shape(name)
        wl = Workload(shp)
        eng = Engine(config_from(shp))
        eng.reset()
        K, V = wl.context(0, device="cuda")
        eng.prefill(0, K, V)
        del K, V
        q, qp = wl.window(0, device="cuda")
        lanes, w, g, d, n = eng.lanes, shp.window, shp.group, shp.head_dim, shp.ctx
        lse = torch.empty((shp.batch, shp.num_q_heads, w), dtype=torch.float32, device="cuda")
        scores = torch.zeros((lanes, shp.max_tokens), dtype=torch.float32, device="cuda")
        ms, p10, p90 = timed(lambda: eng.score_mass(0, q, qp, 0, lse, scores), reps=10)
        rows = g * w
        emit("SnapKV prefill keys (LSE pass, attention-mass pass, pooling)", name, ms, p10, p90,
             nbytes=2 * lanes * n * d * 2 + lanes * n * 4, flops=2 * 2 * lanes * rows * n * d)
        pos, cnt = eng.positions[0], eng.counts[0]
        victims = torch.full((lanes, shp.max_tokens), -1, dtype=torch.int32, device="cuda")
        nvic = torch.zeros((lanes,), dtype=torch.int32, device="cuda")
        ms, p10, p90 = timed(lambda: eng.select(scores, pos, cnt, shp.budget, shp.recent_window, victims, nvic),
                             reps=10)
        emit("D4 bottom-k selection (radix descent on (key, position))", name, ms, p10, p90,
             nbytes=lanes * n * (4 + 4))
        code, msg = eng.last_error()
        assert code == 0, msg
        del eng
        torch.cuda.empty_cache()

    # decode steps of the SnapKV workload and of the H2O toy (latency-bound)
    # the DropKV decode variant runs on the SnapKV workload's data (same
    # prompts, queries and new tokens), with its residual-output scores in a
    # 32-step ring and no pooling
    import dataclasses
    variants = {"dropkv_decode": lambda: dataclasses.replace(shape("snapkv_decode"), policy=2, pool_kernel=1)}
    for tag, name, first in (("snapkv", "snapkv_decode", 1), ("dropkv_decode", "dropkv_decode", 1),
                             ("toy", "h2o_toy", 1)):
        if only and tag not in only:
            continue
        shp = variants[name]() if name in variants else shape(name)
        wl = Workload(shp)
        eng = Engine(config_from(shp))
        eng.reset()
        K, V = wl.context(0, device="cuda")
        eng.prefill(0, K, V)
        del K, V
        steps = [wl.step(0, t, device="cuda") for t in range(shp.steps)]
        B, Hq, d = shp.batch, shp.num_q_heads, shp.head_dim
        out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
        lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
        for t in range(first):
            q, kn, vn, p = steps[t]
            eng.decode_step(0, q, kn, vn, p, out, lse)
        torch.cuda.synchronize()
        n_before = int(eng.counts[0].sum().item())
        timed_steps = list(range(first, shp.steps))
        # the timed steps are captured into one CUDA graph and replayed once,
        # so the per-call host work of the binding is not on the timeline
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.graph(graph, stream=cap):
            for t in timed_steps:
                q, kn, vn, p = steps[t]
                eng.decode_step(0, q, kn, vn, p, out, lse)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / len(timed_steps)
        lanes = eng.lanes
        es = 2 if shp.kv_dtype == "bf16" else 4
        # K and V rows; the ring policies add the ring write, the window
        # sum's reads and the key, and the DropKV variant a second V read
        per_tok = 2 * d * es + (8 if shp.policy == 0 else 4 + 4 * shp.obs_window + 8)
        if shp.policy == 2:
            per_tok += d * es
        emit("decode step (attention, score epilogue, selection, eviction, admission)", name, ms, ms, ms,
             nbytes=(n_before + lanes) * per_tok,
             extra={"steps_timed": len(timed_steps), "us_per_step": round(ms * 1e3, 2),
                    "note": "the timed steps captured into one CUDA graph through the C ABI and replayed once"})
        code, msg = eng.last_error()
        assert code == 0, msg
        del eng
        torch.cuda.empty_cache()

    # the mass-eviction step of the 70B-shaped workload (8 of its 80 layers,
    # full lane count and context): relocation inside each layer's step
    # versus deferred to a second stream behind events (vToken review,
    # Sec. 3.3 Stage 4), where layer l's relocation overlaps layer l+1's step
    if not only or "reloc" in only:
        shp = dataclasses.replace(shape("h2o_70b"), num_layers=8)
        wl = Workload(shp)
        eng = Engine(config_from(shp))
        L, B, Hq, d = shp.num_layers, shp.batch, shp.num_q_heads, shp.head_dim
        first = [wl.step(l, 0, device="cuda") for l in range(L)]
        out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
        lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
        freed = torch.empty((shp.blocks_per_pool,), dtype=torch.int32, device="cuda")
        moves = torch.empty((eng.lanes * shp.max_tokens, 6), dtype=torch.int32, device="cuda")
        n_freed = torch.empty((1,), dtype=torch.int32, device="cuda")
        n_moves = torch.empty((1,), dtype=torch.int32, device="cuda")
        side = torch.cuda.Stream()
        for mode in ("in_step", "side_stream"):
            samples, moved = [], 0
            for rep in range(3):
                eng.reset()
                for l in range(L):
                    K, V = wl.context(l, device="cuda")
                    eng.prefill(l, K, V)
                    del K, V
                eng.defer_relocation(mode != "in_step")
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for l in range(L):
                    q, kn, vn, p = first[l]
                    eng.decode_step(l, q, kn, vn, p, out, lse)
                    if mode != "in_step":
                        ev = torch.cuda.Event()
                        ev.record(stream)
                        side.wait_event(ev)
                        eng.relocate(l, freed, n_freed, moves, n_moves, stream=side)
                if mode != "in_step":
                    ev = torch.cuda.Event()
                    ev.record(side)
                    stream.wait_event(ev)
                e1.record(stream)
                torch.cuda.synchronize()
                samples.append(e0.elapsed_time(e1))
                moved = sum(int(eng.stats(l)[5].item()) for l in range(L))
            eng.defer_relocation(False)
            samples.sort()
            attended = L * eng.lanes * (shp.ctx + 1)
            emit("mass-eviction decode step, relocation " + ("in the step" if mode == "in_step"
                                                            else "on a second stream (vToken Stage 4)"),
                 "h2o_70b, 8 of 80 layers", samples[1], samples[0], samples[-1],
                 nbytes=attended * 2 * d * 2 + moved * 2 * d * 2 * 2,
                 extra={"moved_tokens": moved, "layers": L})
        code, msg = eng.last_error()
        assert code == 0, msg
        del eng
        torch.cuda.empty_cache()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.kernel_table:
        run_kernel_table(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
