#!/usr/bin/env python
"""Benchmark of the per-decode-step KV-cache eviction engine.

Default (`python bench.py`): one step = one decode step of every layer of the
70B-shaped H2O workload (80 layers, 16 sequences x 8 KV heads, group 8,
d=128, bf16, 16384-token prompts = 86 GB of K/V, budget 3276 = 1638 heavy +
1638 recent): split-K attention + score epilogue, bottom-k selection,
eviction, admission and gated relocation, through the C ABI.  The prompt is
prefilled and the first (mass-eviction) decode step runs inside the warm-up;
the timed steps are the steady state.  Every layer call streams ~215 MB of
K/V, more than the 129 MB L2, so no L2 flush is needed between steps.

`--workload` picks another configuration, each printed as the same kind of
line (clocks, roofline, CPU oracle baseline, end-to-end figure):
  h2o_70b_mass   the first decode step of the 70B-shaped workload over all
                 80 layers (16,385 -> 3,276 tokens per lane, relocation)
  h2o_toy        1 lane, d=64, fp32, context 512, 32 steps
  snapkv_decode  32 lanes x 4096, obsWindow 32, poolKernel 7, 256 steps
  dropkv_decode  the DropKV decode variant on the SnapKV workload's data
  dropkv_prefill DropKV window-64 scoring at 32K, selection to 5%, compaction
  paged_128k     the same at 128K (8192 blocks per lane), compaction into
                 dense blocks, token-level vs block-granular metrics
`--all-workloads` prints one line per workload; `--kernel-table` times the
engine's other kernels on their own.

Metric: KV bytes scored + evicted per step (K/V rows read by the attention or
the scoring passes, the score state read and written, 1 KB per relocated
token) / step time, in GB/s, as in the task's metric; tokens scored per
second alongside.
"""
import argparse
import contextlib
import dataclasses
import hashlib
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV GB/s scored+evicted per decode step (frac. of HBM peak); tokens scored/s"
UNIT = "GB/s"
L2_BYTES = 129 * 2 ** 20
WORKLOADS = ("h2o_70b", "h2o_70b_mass", "h2o_toy", "snapkv_decode", "dropkv_decode", "dropkv_prefill",
             "paged_128k")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=48)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--workload", default="h2o_70b", choices=WORKLOADS)
    ap.add_argument("--all-workloads", action="store_true",
                    help="one line per workload (the default one first)")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--cpu-lanes", type=int, default=96)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-layers", type=int, default=0,
                    help="profiling only: run the workload with this many layers (not a bench number)")
    ap.add_argument("--kernel-table", action="store_true",
                    help="time the engine's other kernels on their own workloads (DropKV window scoring at "
                         "32K and 128K, selection, forced compaction, SnapKV prefill selection, relocation), "
                         "one JSON line each, instead of the decode-step bench line")
    ap.add_argument("--only", default="",
                    help="with --kernel-table: comma-separated subset of d3_32k, d3_128k, snapkv_pf_32k, "
                         "snapkv_pf_128k, reloc")
    ap.add_argument("--selftest-cpu", action="store_true",
                    help="the rank launcher and the cross-rank aggregation on CPU ranks (gloo) with a tiny "
                         "stand-in numpy step per rank; prints the aggregated line, no GPU")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# ranks: `--gpus N` without a launcher starts N ranks itself
# ---------------------------------------------------------------------------
def _free_port():
    with contextlib.closing(socket.socket(socket.AF_INET, socket.SOCK_STREAM)) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def maybe_spawn_ranks(args):
    """With --gpus N > 1 and no WORLD_SIZE in the environment, re-run this
    script under torch.distributed.run with N processes on this node
    (127.0.0.1 rendezvous) and return its exit code; None when this process
    is a rank (or N = 1)."""
    if args.gpus <= 1 or "WORLD_SIZE" in os.environ:
        return None
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", str(args.gpus),
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.abspath(__file__)]
    cmd += sys.argv[1:]
    env = dict(os.environ)
    env.setdefault("NCCL_DEBUG", "INFO")   # each rank's NCCL log shows the job's rank count
    return subprocess.call(cmd, env=env)


def rank_shape(shp, rank):
    """The workload of one rank: the same shapes with the rank's own seed
    (lanes are independent, so each GPU serves its own sequences: weak
    scaling); rank 0 keeps the single-GPU seed."""
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


def selftest_cpu(args):
    """Launcher and aggregation on CPU ranks: each rank times a few steps of
    stand-in work on its own seeded copy of a small workload's context
    (numpy softmax-weighted sums of its rows; gloo barrier before and after,
    slowest rank's time, all ranks' work) and rank 0 prints the aggregated
    line.  No GPU is touched."""
    import numpy as np
    import torch.distributed as dist
    from workloads import Workload, scaled
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        dist.init_process_group("gloo")
    shp = rank_shape(scaled("h2o_70b", num_layers=1, batch=1, num_kv_heads=2, num_q_heads=16, ctx=256,
                            steps=6, budget=64, recent_window=32), rank)
    wl = Workload(shp)
    K, V = (x.float().numpy() for x in wl.context(0))
    steps = [wl.step(0, t) for t in range(shp.steps)]
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    attended = 0
    for q, _, _, _ in steps:
        qn = q.float().numpy()
        for lane in range(shp.lanes):
            b, h = divmod(lane, shp.num_kv_heads)
            s = qn[b, h * shp.group:(h + 1) * shp.group] @ K[b, h].T
            p = np.exp(s - s.max(axis=1, keepdims=True))
            _ = (p / p.sum(axis=1, keepdims=True)) @ V[b, h]
            attended += K.shape[2]
    if world > 1:
        dist.barrier()
    ms = (time.perf_counter() - t0) * 1e3 / shp.steps
    per = attended / shp.steps
    ms, total_bytes, total_tok = aggregate_over_ranks(ms, per * 2 * shp.head_dim * 2, per)
    if rank == 0:
        print(json.dumps({"metric": METRIC, "value": round(total_bytes / (ms * 1e-3) / 1e9, 6), "unit": UNIT,
                          "n_gpus": world, "steps": shp.steps - 1, "warmup": 1, "ms_per_step": round(ms, 4),
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                          "data": "synthetic; CPU self-test of the rank launcher (stand-in numpy work, gloo), "
                                  "not a bench number",
                          "tokens_scored_per_s": round(total_tok / (ms * 1e-3), 1),
                          "config": {"workload": shp.name, "ranks": world}}))
    if world > 1:
        dist.destroy_process_group()


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
# oracle baseline (CPU) on bounded samples of lanes, in a spawn pool
# ---------------------------------------------------------------------------
def _oracle_cfg(f):
    import types
    return types.SimpleNamespace(policy=f["policy"], num_layers=1, batch=1, num_q_heads=f["g"], num_kv_heads=1,
                                 head_dim=f["d"], blocks_per_pool=f["blocks"], budget=f["budget"],
                                 recent_window=f["R"], obs_window=f["W"], pool_kernel=f["pk"],
                                 theta_f=f["theta"])


def _oracle_decode_job(job):
    """One lane through the oracle: prefill, `untimed` decode steps, then the
    timed steps; returns (seconds, bytes, tokens) of the timed steps."""
    import numpy as np
    from oracle.engine import Engine as Oracle
    K, V, steps, f, untimed = job
    o = Oracle(_oracle_cfg(f))
    o.prefill(0, K[None, None].astype(np.float64), V[None, None].astype(np.float64))

    def run(st):
        q, kn, vn, pos = st
        n = o.layers[0].lanes[0].pos.size
        r = o.decode_step(0, q[None].astype(np.float64), kn[None, None].astype(np.float64),
                          vn[None, None].astype(np.float64), pos)
        return n, r

    for st in steps[:untimed]:
        run(st)
    t0 = time.perf_counter()
    nbytes = tokens = 0
    for st in steps[untimed:]:
        n, r = run(st)
        tokens += n + 1
        nbytes += (n + 1) * f["tok_bytes"] + n * f["score_bytes"] + len(r["moves"]) * 4 * f["d"] * f["es"]
    return time.perf_counter() - t0, nbytes, tokens


def _oracle_score_job(job):
    """One lane of a prefill-scoring configuration through the oracle:
    window scores, selection to the budget, forced compaction; returns
    (seconds, bytes, tokens)."""
    import numpy as np
    from oracle.engine import Engine as Oracle
    from oracle.engine import select as oselect
    K, V, qw, qp, f = job
    o = Oracle(_oracle_cfg(f))
    o.prefill(0, K[None, None].astype(np.float64), V[None, None].astype(np.float64))
    n = K.shape[0]
    t0 = time.perf_counter()
    r = o.score(0, qw[None].astype(np.float64), qp)
    L = o.layers[0].lanes[0]
    vict = oselect([r["scores"][0]], [L.pos], [n], f["budget"], f["R"])
    c = o.compact(0, vict)
    dt = time.perf_counter() - t0
    return dt, n * f["tok_bytes"] + len(c["moves"]) * 4 * f["d"] * 2, n


def oracle_pool(fn, jobs, workers):
    """Runs the jobs in a spawn pool of single-threaded workers; returns
    (GB/s, tokens/s, busy seconds, wall seconds) as per-core throughput x
    cores used (the workers run concurrently)."""
    import multiprocessing as mp
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    t0 = time.perf_counter()
    with mp.get_context("spawn").Pool(workers) as pool:
        res = pool.map(fn, jobs)
    wall = time.perf_counter() - t0
    busy = sum(r[0] for r in res)
    nbytes = sum(r[1] for r in res)
    tokens = sum(r[2] for r in res)
    return nbytes / busy * workers / 1e9, tokens / busy * workers, busy, wall


def oracle_fields(shp, score_bytes=8, tok_bytes=None):
    per_lane = -(-shp.max_tokens // 16) + -(-shp.budget // 16) + 2
    es = 2 if shp.kv_dtype == "bf16" else 4
    return dict(policy=shp.policy, g=shp.group, d=shp.head_dim, blocks=per_lane, budget=shp.budget,
                R=shp.recent_window, W=shp.obs_window, pk=shp.pool_kernel, theta=float(shp.theta_f), es=es,
                score_bytes=score_bytes, tok_bytes=tok_bytes if tok_bytes is not None else 2 * shp.head_dim * es)


def decode_lane_jobs(wl, shp, lanes, n_steps, f, untimed, device):
    """Per sampled lane of layer 0: (K, V, steps, fields, untimed) as
    float32 numpy (bf16 values are exact in float32)."""
    import torch
    K, V = wl.context(0, device=device)
    g = shp.group
    steps_all = [wl.step(0, t, device=device) for t in range(n_steps)]
    jobs = []
    for lane in lanes:
        b, h = divmod(lane, shp.num_kv_heads)
        steps = [(q[b, h * g:(h + 1) * g].float().cpu().numpy(), kn[b, h].float().cpu().numpy(),
                  vn[b, h].float().cpu().numpy(), pos) for q, kn, vn, pos in steps_all]
        jobs.append((K[b, h].float().cpu().numpy(), V[b, h].float().cpu().numpy(), steps, f, untimed))
    del K, V
    if device != "cpu":
        torch.cuda.empty_cache()
    return jobs


def score_lane_jobs(wl, shp, lanes, f, device):
    import torch
    K, V = wl.context(0, device=device)
    qw, qp = wl.window(0, device=device)
    g = shp.group
    jobs = []
    for lane in lanes:
        b, h = divmod(lane, shp.num_kv_heads)
        jobs.append((K[b, h].float().cpu().numpy(), V[b, h].float().cpu().numpy(),
                     qw[b, h * g:(h + 1) * g].float().cpu().numpy(), qp.cpu().numpy(), f))
    del K, V
    if device != "cpu":
        torch.cuda.empty_cache()
    return jobs


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


def tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return float(json.load(open(p))["bf16_tflops"]), "measured"
        except (KeyError, ValueError):
            pass
    return 1900.0, "fallback"


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
# GPU arm: shared pieces
# ---------------------------------------------------------------------------
class Gpu:
    """Process-level setup of the GPU arm: device, ranks, barrier."""

    def __init__(self):
        import torch
        import torch.distributed as dist
        import __graft_entry__
        __graft_entry__.build()
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(self.local)
        if self.world > 1 and not dist.is_initialized():
            dist.init_process_group("nccl", device_id=torch.device("cuda", self.local))
        self.stream = torch.cuda.current_stream()
        self._flush = None

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()

    def flush_l2(self):
        """Writes a buffer twice the size of L2 (outside any timed region)."""
        import torch
        if self._flush is None:
            self._flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
        self._flush.fill_(1.0)

    def hold(self):
        """Keeps the stream busy for ~0.2 ms (a spinning kernel) so that the
        host has enqueued the timed region before the GPU reaches it: the
        events then bracket device time, not launch latency."""
        import torch
        torch.cuda._sleep(400000)

    def finish(self, line):
        import torch.distributed as dist
        if self.rank == 0:
            print(json.dumps(line), flush=True)
        if self.world > 1 and dist.is_initialized():
            dist.destroy_process_group()


def line_base(g, args, value, ms_per_step, tokens_s, dtype, workload, extra_config, steps, warmup):
    return {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": g.world, "steps": steps,
            "warmup": warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "tokens_scored_per_s": round(tokens_s, 1),
            "config": dict({"workload": workload, "parallelism": "replica per GPU" if g.world > 1 else "1 GPU"},
                           **extra_config)}


def hbm_roofline(kernel, nbytes, ms, extra=None):
    peak, kind = hbm_peak()
    gbs = nbytes / (ms * 1e-3) / 1e9
    r = {"bound": "hbm", "kernel": kernel, "achieved": round(gbs, 1), "peak": peak, "peak_kind": kind,
         "unit": "GB/s", "frac": round(gbs / peak, 4), "traffic": None, "algorithmic_bytes_per_launch": int(nbytes),
         "avg_launch_ms": round(ms, 5)}
    if extra:
        r.update(extra)
    return r


# ---------------------------------------------------------------------------
# GPU arm: the 70B-shaped steady state (the default line)
# ---------------------------------------------------------------------------
def run_h2o70b(args, g):
    import numpy as np
    import torch
    from kv_cache_token_gb300 import Engine, config_from
    from workloads import Workload, shape

    shp = rank_shape(shape("h2o_70b"), g.rank)
    if args.profile_layers:
        shp = dataclasses.replace(shp, num_layers=args.profile_layers)
    assert args.warmup >= 1 and args.warmup + args.steps + args.e2e_steps <= shp.steps, \
        "the workload has %d decode steps" % shp.steps
    ser_steps = min(4, shp.steps - (args.warmup + args.steps + args.e2e_steps))
    wl = Workload(shp)
    eng = Engine(config_from(shp))
    eng.reset()
    cpu_jobs = None
    t_setup = time.time()
    for layer in range(shp.num_layers):
        if layer == 0 and g.rank == 0 and not args.no_cpu_baseline:
            f = oracle_fields(shp)
            cpu_jobs = decode_lane_jobs(wl, shp, range(args.cpu_lanes), args.warmup + args.steps, f, 1, "cuda")
        K, V = wl.context(layer, device="cuda")
        eng.prefill(layer, K, V)
        del K, V
    torch.cuda.synchronize()
    code, msg = eng.last_error()
    assert code == 0, msg
    inputs = [[wl.step(layer, t, device="cuda")[:3] for layer in range(shp.num_layers)]
              for t in range(args.warmup + args.steps)]
    ser_base = args.warmup + args.steps + args.e2e_steps
    ser_inputs = [[wl.step(layer, ser_base + t, device="cuda")[:3] for layer in range(shp.num_layers)]
                  for t in range(ser_steps)]
    L, B, Hq, d = shp.num_layers, shp.batch, shp.num_q_heads, shp.head_dim
    outs = [torch.empty((B, Hq, d), dtype=torch.float32, device="cuda") for _ in range(L)]
    lses = [torch.empty((B, Hq), dtype=torch.float32, device="cuda") for _ in range(L)]
    vics = [torch.empty((eng.lanes, shp.max_tokens), dtype=torch.int32, device="cuda") for _ in range(L)]
    nvs = [torch.empty((eng.lanes,), dtype=torch.int32, device="cuda") for _ in range(L)]
    stream = g.stream
    one = torch.zeros((1,), dtype=torch.float32, device="cuda")

    def step(t, serialize=False):
        pos = shp.ctx + t
        for layer in range(L):
            q, kn, vn = ser_inputs[t - ser_base][layer] if serialize else inputs[t][layer]
            eng.decode_step(layer, q, kn, vn, pos, outs[layer], lses[layer], vics[layer], nvs[layer])
            if serialize:
                one.add_(1.0)   # an ordinary kernel: the next layer starts only once this one is complete

    for t in range(args.warmup):
        step(t)
    torch.cuda.synchronize()
    code, msg = eng.last_error()
    assert code == 0, msg
    counts_before = eng.counts.sum(dim=1).cpu().numpy().astype(np.int64)          # per layer
    stats_before = eng.stats_buf.sum(dim=0).cpu().numpy()
    setup_s = time.time() - t_setup

    sampler = ClockSampler(g.local)
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    e1.record(stream)
    torch.cuda.synchronize()
    g.barrier()
    clocks = sampler.stop()
    elapsed_ms = e0.elapsed_time(e1)
    # the split-K attention of every layer, replayed on the steady-state
    # tables (it changes no engine state): average launch duration from
    # events around each replay of the L launches issued back to back; the
    # per-launch figure with events around every launch beside it
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
    d1_bytes = int((counts_before + lanes).mean()) * 2 * d * 2   # K/V rows per launch (one layer)
    peak, peak_kind = hbm_peak()

    e2e = None
    if args.e2e_steps > 0:
        e2e = h2o70b_e2e(args, g, eng, wl, shp, L, B, Hq, d)
    # The layers of one timed step overlap: each layer's epilogue runs beside
    # the next layer's attention, which may start while this layer's
    # attention drains (the queries of all layers are given).  For reference,
    # the workload's last steps with the layers one after another: a
    # one-element torch kernel between layers (no early start across it).
    ser_ms = None
    if ser_steps > 0:
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s0.record(stream)
        for i in range(ser_steps):
            step(ser_base + i, serialize=True)
        s1.record(stream)
        torch.cuda.synchronize()
        ser_ms = s0.elapsed_time(s1) / ser_steps
        code, msg = eng.last_error()
        assert code == 0, msg

    ms_per_step, all_bytes, all_attended = aggregate_over_ranks(ms_per_step, step_bytes, attended / args.steps,
                                                                device="cuda")
    value = all_bytes / (ms_per_step * 1e-3) / 1e9
    tokens_s = all_attended / (ms_per_step * 1e-3)

    cpu = None
    if g.rank == 0 and cpu_jobs is not None:
        workers = max(1, min(len(cpu_jobs), os.cpu_count() or 1, 16))
        gbs, tps, busy, wall = oracle_pool(_oracle_decode_job, cpu_jobs, workers)
        cpu = {"value": round(gbs, 4), "unit": UNIT, "cores": workers, "kind": "oracle",
               "tokens_scored_per_s": round(tps, 1),
               "sample": "%d lanes of layer 0 x %d steady-state decode steps (after the mass-eviction step), "
                         "numpy float64 oracle, %d single-threaded processes, %.1f s of CPU work"
                         % (len(cpu_jobs), args.warmup + args.steps - 1, workers, busy)}

    line = line_base(g, args, value, ms_per_step, tokens_s, "bf16",
                     "h2o_70b: 80 layers, batch 16, 64 q / 8 KV heads, d 128, bf16, context 16384 (86 GB K/V), "
                     "H2O budget 3276 (1638 recent), steady-state decode steps",
                     {"global_batch": B * g.world, "seq_len": shp.ctx,
                      "l2": "no flush: every layer call streams ~215 MB of K/V, above the 129 MB L2",
                      "bytes_per_step": int(step_bytes), "moved_tokens_timed": moved,
                      "layers_overlap": "layer l's epilogue runs beside layer l+1's attention, which may start "
                                        "while layer l's attention drains (all layers' queries are given)",
                      "serialized_layers": None if ser_ms is None else {
                          "ms_per_step": round(ser_ms, 4), "value": round(step_bytes / (ser_ms * 1e-3) / 1e9, 2),
                          "how": "the workload's last steps with a one-element torch kernel between layers, so "
                                 "each layer starts after the previous one is complete",
                          "steps": ser_steps},
                      "setup_s": round(setup_s, 1)},
                     args.steps, args.warmup)
    line["roofline"] = hbm_roofline(
        "decode step (split-K attention + lean score epilogue, layers streamed): step bytes / step time",
        step_bytes / L, ms_per_step / L,
        {"per": "layer (step / 80)",
         "attention_only": {"kernel": "attend_bf16_kernel (split-K decode attention)",
                            "achieved": round(d1_bytes / (d1_ms * 1e-3) / 1e9, 1),
                            "frac": round(d1_bytes / (d1_ms * 1e-3) / 1e9 / peak, 4),
                            "traffic": committed_traffic(), "algorithmic_bytes_per_launch": d1_bytes,
                            "avg_launch_ms": round(d1_ms, 5), "launches_timed": reps * L,
                            "isolated_launch_ms": round(d1_iso_ms, 5),
                            "isolated_frac": round(d1_bytes / (d1_iso_ms * 1e-3) / 1e9 / peak, 4),
                            "how": "the 80 attention launches replayed back to back on the steady-state "
                                   "tables, CUDA events around each replay"}})
    line["cpu_baseline"] = cpu
    line["e2e"] = e2e
    line["clocks"] = clocks
    line["gpu_launches"] = eng.kernels_per_decode_step() * L * args.steps
    if args.profile_layers:
        line["profile_only"] = "%d layers: for profiling, not a bench number" % L
    g.finish(line)


def h2o70b_e2e(args, g, eng, wl, shp, L, B, Hq, d):
    """The same metric through kvevict_decode_step with host buffers: each
    step's q / k / v for all layers go up from pinned memory in one copy per
    tensor kind on a copy stream (double-buffered on the device, so the next
    step's upload overlaps this step's compute), and out / LSE / victim
    counts / first victims come back the same way, all inside the timed
    region."""
    import torch
    stream = g.stream
    lanes = eng.lanes
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
    g.barrier()
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
    g.barrier()
    e2e_ms = ea.elapsed_time(eb) / args.e2e_steps
    counts_e2e = eng.counts.sum(dim=1).cpu().numpy()
    e2e_bytes = (int((counts_e2e + lanes).sum()) * 2 * d * 2 + int(counts_e2e.sum()) * 8)
    code, msg = eng.last_error()
    assert code == 0, msg
    return {"value": round(e2e_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 4)}


# ---------------------------------------------------------------------------
# GPU arm: the 70B-shaped mass-eviction step over all 80 layers
# ---------------------------------------------------------------------------
def run_h2o70b_mass(args, g):
    import numpy as np
    import torch
    from kv_cache_token_gb300 import Engine, config_from
    from workloads import Workload, shape

    shp = rank_shape(shape("h2o_70b"), g.rank)
    wl = Workload(shp)
    eng = Engine(config_from(shp))
    L, B, Hq, d = shp.num_layers, shp.batch, shp.num_q_heads, shp.head_dim
    lanes = eng.lanes
    first = [wl.step(l, 0, device="cuda") for l in range(L)]
    out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    stream = g.stream
    cpu_jobs = None
    if g.rank == 0 and not args.no_cpu_baseline:
        f = oracle_fields(shp)
        cpu_jobs = decode_lane_jobs(wl, shp, range(16), 1, f, 0, "cuda")

    def prefill_all():
        eng.reset()
        for l in range(L):
            K, V = wl.context(l, device="cuda")
            eng.prefill(l, K, V)
            del K, V
        torch.cuda.synchronize()

    reps = max(1, min(args.steps, 3))
    samples, moved = [], 0
    sampler = ClockSampler(g.local)
    for rep in range(reps + args.warmup):
        prefill_all()
        if rep == args.warmup:
            sampler.start()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for l in range(L):
            q, kn, vn, p = first[l]
            eng.decode_step(l, q, kn, vn, p, out, lse)
        e1.record(stream)
        torch.cuda.synchronize()
        g.barrier()
        if rep >= args.warmup:
            samples.append(e0.elapsed_time(e1))
        moved = int(eng.stats_buf[:, 5].sum().item())
    clocks = sampler.stop()
    code, msg = eng.last_error()
    assert code == 0, msg
    kept_after = int(eng.counts.sum().item())
    ms = statistics.median(samples)
    attended = L * lanes * (shp.ctx + 1)
    step_bytes = attended * 2 * d * 2 + L * lanes * shp.ctx * 8 + moved * 4 * d * 2
    # end to end: one more mass-eviction step with its inputs uploaded from
    # pinned host memory and its outputs read back, inside the timed region
    prefill_all()
    host_in = tuple(torch.stack([first[l][i] for l in range(L)]).cpu().pin_memory() for i in range(3))
    dev_in = tuple(torch.empty_like(x, device="cuda") for x in host_in)
    out_all = torch.empty((L, B, Hq, d), dtype=torch.float32, device="cuda")
    lse_all = torch.empty((L, B, Hq), dtype=torch.float32, device="cuda")
    nv_all = torch.empty((L, lanes), dtype=torch.int32, device="cuda")
    vic_all = torch.empty((L, lanes, shp.max_tokens), dtype=torch.int32, device="cuda")
    kread = shp.ctx + 1 - shp.budget
    host_out = (torch.empty(out_all.shape, dtype=torch.float32).pin_memory(),
                torch.empty(lse_all.shape, dtype=torch.float32).pin_memory(),
                torch.empty(nv_all.shape, dtype=torch.int32).pin_memory(),
                torch.empty((L, lanes, kread), dtype=torch.int32).pin_memory())
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ea.record(stream)
    for dst, src in zip(dev_in, host_in):
        dst.copy_(src, non_blocking=True)
    for l in range(L):
        eng.decode_step(l, dev_in[0][l], dev_in[1][l], dev_in[2][l], first[l][3], out_all[l], lse_all[l],
                        vic_all[l], nv_all[l])
    for dst, src in zip(host_out, (out_all, lse_all, nv_all, vic_all[:, :, :kread])):
        dst.copy_(src, non_blocking=True)
    eb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = ea.elapsed_time(eb)
    code, msg = eng.last_error()
    assert code == 0, msg
    e2e = {"value": round(step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
           "h2d_bytes_per_step": int(sum(x.numel() * x.element_size() for x in host_in)),
           "d2h_bytes_per_step": int(sum(x.numel() * x.element_size() for x in host_out)),
           "ms_per_step": round(e2e_ms, 4)}

    ms, all_bytes, all_attended = aggregate_over_ranks(ms, step_bytes, attended, device="cuda")
    value = all_bytes / (ms * 1e-3) / 1e9
    cpu = None
    if cpu_jobs is not None:
        workers = max(1, min(len(cpu_jobs), os.cpu_count() or 1, 16))
        gbs, tps, busy, wall = oracle_pool(_oracle_decode_job, cpu_jobs, workers)
        cpu = {"value": round(gbs, 4), "unit": UNIT, "cores": workers, "kind": "oracle",
               "tokens_scored_per_s": round(tps, 1),
               "sample": "the mass-eviction step of 16 lanes of layer 0 (16,385 -> 3,276 tokens each), numpy "
                         "float64 oracle, %d single-threaded processes, %.1f s of CPU work" % (workers, busy)}
    line = line_base(g, args, value, ms, all_attended / (ms * 1e-3), "bf16",
                     "h2o_70b_mass: the first decode step of the 70B-shaped workload over all 80 layers "
                     "(16,385 -> 3,276 tokens per lane, admission, relocation in the step)",
                     {"global_batch": B * g.world, "seq_len": shp.ctx, "bytes_per_step": int(step_bytes),
                      "moved_tokens": moved, "kept_after": kept_after, "samples_ms": [round(x, 3) for x in samples],
                      "l2": "no flush: the step reads 86 GB of K/V",
                      "timing": "each sample: prefill every layer (untimed), then the 80 layers' first decode step"},
                     reps, args.warmup)
    line["roofline"] = hbm_roofline("decode step over 80 layers (attention over the full prompt, the large "
                                    "epilogue's selection and relocation): step bytes / step time",
                                    step_bytes / L, ms / L, {"per": "layer (step / 80)"})
    line["cpu_baseline"] = cpu
    line["e2e"] = e2e
    line["clocks"] = clocks
    line["gpu_launches"] = eng.kernels_per_decode_step() * L * reps
    g.finish(line)


# ---------------------------------------------------------------------------
# GPU arm: single-layer decode workloads (toy, SnapKV, DropKV decode variant)
# ---------------------------------------------------------------------------
def small_decode_shape(name):
    from workloads import shape
    if name == "dropkv_decode":
        # the SnapKV workload's data, residual-output scores in a 32-step
        # ring, no pooling
        return dataclasses.replace(shape("snapkv_decode"), policy=2, pool_kernel=1)
    return shape(name)


def per_token_bytes(shp):
    d = shp.head_dim
    es = 2 if shp.kv_dtype == "bf16" else 4
    if shp.policy == 0:
        return 2 * d * es, 8
    extra = d * es if shp.policy == 2 else 0      # the DropKV variant's second V read
    return 2 * d * es + extra, 4 + 4 * shp.obs_window + 8


def run_small_decode(args, g, name):
    import numpy as np
    import torch
    from kv_cache_token_gb300 import Engine, config_from
    from workloads import Workload

    shp = rank_shape(small_decode_shape(name), g.rank)
    wl = Workload(shp)
    eng = Engine(config_from(shp))
    eng.reset()
    K, V = wl.context(0, device="cuda")
    eng.prefill(0, K, V)
    del K, V
    steps = [wl.step(0, t, device="cuda") for t in range(shp.steps)]
    B, Hq, d = shp.batch, shp.num_q_heads, shp.head_dim
    lanes = eng.lanes
    out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    stream = g.stream
    first = max(1, args.warmup)        # the first step evicts down to the budget
    # e2e steps are the last few; the timed device steps the ones before
    n_e2e = min(max(args.e2e_steps, 0), max(0, shp.steps - first - 4))
    timed = list(range(first, shp.steps - n_e2e))
    for t in range(first):
        q, kn, vn, p = steps[t]
        eng.decode_step(0, q, kn, vn, p, out, lse)
    torch.cuda.synchronize()
    # each timed step is captured into its own CUDA graph (the binding's
    # per-call host work is then off the timeline), replayed once with L2
    # flushed before it (the lane state fits in L2)
    graphs = []
    cap = torch.cuda.Stream()
    for t in timed:
        gr = torch.cuda.CUDAGraph()
        cap.wait_stream(stream)
        q, kn, vn, p = steps[t]
        with torch.cuda.graph(gr, stream=cap):
            eng.decode_step(0, q, kn, vn, p, out, lse)
        graphs.append(gr)
        stream.wait_stream(cap)
    torch.cuda.synchronize()
    # capturing records the launches without running them: the state is
    # still the one after the warm-up steps
    counts = []
    ms_steps = []
    sampler = ClockSampler(g.local)
    sampler.start()
    g.barrier()
    stats_before = eng.stats_buf.sum(dim=0).cpu().numpy()
    # first half: L2 flushed before each step (the line's value); second
    # half: the steps back to back with warm caches, for reference
    half = max(1, len(graphs) // 2)
    for gr in graphs[:half]:
        counts.append(int(eng.counts[0].sum().item()))
        g.flush_l2()
        g.hold()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gr.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms_steps.append(e0.elapsed_time(e1))
    warm_us = None
    if len(graphs) > half:
        g.hold()
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        for gr in graphs[half:]:
            gr.replay()
        w1.record(stream)
        torch.cuda.synchronize()
        warm_us = w0.elapsed_time(w1) * 1e3 / (len(graphs) - half)
    g.barrier()
    clocks = sampler.stop()
    stats_after = eng.stats_buf.sum(dim=0).cpu().numpy()
    code, msg = eng.last_error()
    assert code == 0, msg
    tokb, scoreb = per_token_bytes(shp)
    # the moved-token count covers both halves; the byte count takes the
    # flushed half's share of it
    stats_after = stats_before + (stats_after - stats_before) * half / len(graphs)
    attended = sum(c + lanes for c in counts)
    moved = int(stats_after[5] - stats_before[5])
    es = 2 if shp.kv_dtype == "bf16" else 4
    total_bytes = attended * tokb + sum(counts) * scoreb + moved * 4 * d * es
    ms = sum(ms_steps) / len(ms_steps)
    step_bytes = total_bytes / len(ms_steps)
    # end to end: the last steps through kvevict_decode_step with host
    # buffers, each step's inputs uploaded from pinned memory and its
    # outputs read back inside its timed region (L2 flushed before each)
    e2e = None
    if n_e2e:
        e2e_ms, e2e_bytes = [], 0
        h_in = [tuple(x.cpu().pin_memory() for x in steps[t][:3]) for t in range(shp.steps - n_e2e, shp.steps)]
        d_in = tuple(torch.empty_like(x, device="cuda") for x in h_in[0])
        h_out = (torch.empty(out.shape, dtype=torch.float32).pin_memory(),
                 torch.empty(lse.shape, dtype=torch.float32).pin_memory(),
                 torch.empty((lanes,), dtype=torch.int32).pin_memory(),
                 torch.empty((lanes, 8), dtype=torch.int32).pin_memory())
        for j, t in enumerate(range(shp.steps - n_e2e, shp.steps)):
            c = int(eng.counts[0].sum().item())
            g.flush_l2()
            torch.cuda.synchronize()
            g.hold()
            ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ea.record(stream)
            for dst, src in zip(d_in, h_in[j]):
                dst.copy_(src, non_blocking=True)
            _, _, vic, nv = eng.decode_step(0, d_in[0], d_in[1], d_in[2], steps[t][3], out, lse)
            for dst, src in zip(h_out, (out, lse, nv, vic[:, :8])):
                dst.copy_(src, non_blocking=True)
            eb.record(stream)
            torch.cuda.synchronize()
            e2e_ms.append(ea.elapsed_time(eb))
            e2e_bytes += (c + lanes) * tokb + c * scoreb
        code, msg = eng.last_error()
        assert code == 0, msg
        em = sum(e2e_ms) / len(e2e_ms)
        e2e = {"value": round(e2e_bytes / len(e2e_ms) / (em * 1e-3) / 1e9, 2), "unit": UNIT,
               "h2d_bytes_per_step": int(sum(x.numel() * x.element_size() for x in h_in[0])),
               "d2h_bytes_per_step": int(sum(x.numel() * x.element_size() for x in h_out)),
               "ms_per_step": round(em, 4), "steps": n_e2e}
    ms, all_bytes, all_attended = aggregate_over_ranks(ms, step_bytes, attended / len(ms_steps), device="cuda")
    value = all_bytes / (ms * 1e-3) / 1e9
    cpu = None
    if g.rank == 0 and not args.no_cpu_baseline:
        f = oracle_fields(shp, score_bytes=scoreb, tok_bytes=tokb)
        n_lanes = min(lanes, 32)
        n_steps = shp.steps if lanes <= 8 else min(shp.steps, 1 + 96)
        jobs = decode_lane_jobs(wl, shp, range(n_lanes), n_steps, f, 1, "cpu")
        workers = max(1, min(len(jobs), os.cpu_count() or 1, 16))
        gbs, tps, busy, wall = oracle_pool(_oracle_decode_job, jobs, workers)
        cpu = {"value": round(gbs, 6), "unit": UNIT, "cores": workers, "kind": "oracle",
               "tokens_scored_per_s": round(tps, 1),
               "sample": "%d lanes x %d decode steps after the first, numpy float64 oracle, %d single-threaded "
                         "processes, %.1f s of CPU work" % (n_lanes, n_steps - 1, workers, busy)}
    desc = {"h2o_toy": "h2o_toy: 1 lane, d 64, fp32, context 512, budget 128 (64 recent), 32 steps",
            "snapkv_decode": "snapkv_decode: batch 4, 32 q / 8 KV heads, d 128, bf16, context 4096, obsWindow 32, "
                             "poolKernel 7, recent 256, budget 1024, 256 steps",
            "dropkv_decode": "dropkv_decode: the SnapKV workload's data, DropKV residual-output scores in a "
                             "32-step ring, no pooling, budget 1024, 256 steps"}[name]
    line = line_base(g, args, value, ms, all_attended / (ms * 1e-3), shp.kv_dtype if shp.kv_dtype != "fp32" else "f32",
                     desc, {"l2": "flushed before every timed step (a %d MB buffer written)" % (2 * L2_BYTES >> 20),
                            "timing": "each step captured into its own CUDA graph through the C ABI, replayed once "
                                      "between CUDA events, the stream held busy by a short spin before them",
                            "us_per_step": round(ms * 1e3, 2), "bytes_per_step": int(step_bytes),
                            "moved_tokens": moved,
                            "warm_l2_us_per_step": None if warm_us is None else round(warm_us, 2),
                            "warm_l2": "the other half of the steps replayed back to back, no flush"},
                     len(ms_steps), first)
    line["roofline"] = hbm_roofline("decode step (attention, score epilogue, keys, selection, eviction, "
                                    "admission): latency-bound at this size", step_bytes, ms)
    line["cpu_baseline"] = cpu
    line["e2e"] = e2e
    line["clocks"] = clocks
    line["gpu_launches"] = eng.kernels_per_decode_step() * len(ms_steps)
    g.finish(line)


# ---------------------------------------------------------------------------
# GPU arm: prefill-window scoring + selection + compaction (configs 3 and 5)
# ---------------------------------------------------------------------------
def run_prefill(args, g, name):
    import numpy as np
    import torch
    from kv_cache_token_gb300 import Engine, config_from
    from workloads import Workload, shape

    shp = rank_shape(shape(name), g.rank)
    wl = Workload(shp)
    eng = Engine(config_from(shp))
    lanes, w, grp, d, n = eng.lanes, shp.window, shp.group, shp.head_dim, shp.ctx
    q, qp = wl.window(0, device="cuda")
    lse = torch.empty((shp.batch, shp.num_q_heads, w), dtype=torch.float32, device="cuda")
    a_out = torch.empty((shp.batch, shp.num_q_heads, w, d), dtype=torch.float32, device="cuda")
    scores = torch.zeros((lanes, shp.max_tokens), dtype=torch.float32, device="cuda")
    victims = torch.full((lanes, shp.max_tokens), -1, dtype=torch.int32, device="cuda")
    nvic = torch.zeros((lanes,), dtype=torch.int32, device="cuda")
    freed = torch.empty((shp.blocks_per_pool,), dtype=torch.int32, device="cuda")
    moves = torch.empty((lanes * shp.max_tokens, 6), dtype=torch.int32, device="cuda")
    n_freed = torch.empty((1,), dtype=torch.int32, device="cuda")
    n_moves = torch.empty((1,), dtype=torch.int32, device="cuda")
    K, V = wl.context(0, device="cuda")
    stream = g.stream

    def prefill():
        eng.reset()
        eng.prefill(0, K, V)
        torch.cuda.synchronize()

    def step():
        eng.score(0, q, qp, lse, a_out, scores)
        eng.select(scores, eng.positions[0], eng.counts[0], shp.budget, shp.recent_window, victims, nvic)
        eng.compact(0, victims, nvic, freed, n_freed, moves, n_moves)

    reps = max(3, min(args.steps, 10))
    samples = []
    sampler = ClockSampler(g.local)
    for rep in range(args.warmup + reps):
        prefill()
        if rep == args.warmup:
            sampler.start()
            g.barrier()
        g.hold()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        if rep >= args.warmup:
            samples.append(e0.elapsed_time(e1))
    g.barrier()
    clocks = sampler.stop()
    code, msg = eng.last_error()
    assert code == 0, msg
    moved, nf = int(n_moves.item()), int(n_freed.item())
    st = eng.stats(0).cpu().tolist()
    ms = statistics.median(samples)
    # K and V read in both scoring passes, the scores written and read by the
    # selection with the positions, 1 KB per relocated token
    step_bytes = lanes * n * (2 * 2 * d * 2 + 4 + 8) + moved * 4 * d * 2
    flops = 4 * 2 * lanes * grp * w * n * d
    # end to end: the window queries uploaded from pinned memory, the scores,
    # victims and freed list read back
    prefill()
    hq, hqp = q.cpu().pin_memory(), qp.cpu().pin_memory()
    dq, dqp = torch.empty_like(q), torch.empty_like(qp)
    h_out = (torch.empty(scores.shape, dtype=torch.float32).pin_memory(),
             torch.empty(victims.shape, dtype=torch.int32).pin_memory(),
             torch.empty(nvic.shape, dtype=torch.int32).pin_memory(),
             torch.empty(freed.shape, dtype=torch.int32).pin_memory(),
             torch.empty((1,), dtype=torch.int32).pin_memory())
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g.hold()
    ea.record(stream)
    dq.copy_(hq, non_blocking=True)
    dqp.copy_(hqp, non_blocking=True)
    eng.score(0, dq, dqp, lse, a_out, scores)
    eng.select(scores, eng.positions[0], eng.counts[0], shp.budget, shp.recent_window, victims, nvic)
    eng.compact(0, victims, nvic, freed, n_freed, moves, n_moves)
    for dst, src in zip(h_out, (scores, victims, nvic, freed, n_freed)):
        dst.copy_(src, non_blocking=True)
    eb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = ea.elapsed_time(eb)
    e2e = {"value": round(step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
           "h2d_bytes_per_step": int(hq.numel() * hq.element_size() + hqp.numel() * hqp.element_size()),
           "d2h_bytes_per_step": int(sum(x.numel() * x.element_size() for x in h_out)),
           "ms_per_step": round(e2e_ms, 4)}
    code, msg = eng.last_error()
    assert code == 0, msg
    del K, V
    ms_all, all_bytes, all_tok = aggregate_over_ranks(ms, step_bytes, lanes * n, device="cuda")
    value = all_bytes / (ms_all * 1e-3) / 1e9
    cpu = None
    if g.rank == 0 and not args.no_cpu_baseline:
        f = oracle_fields(shp, tok_bytes=2 * 2 * d * 2 + 4 + 8)
        n_lanes = 8 if n <= 32768 else 4
        jobs = score_lane_jobs(wl, shp, range(n_lanes), f, "cpu")
        workers = max(1, min(len(jobs), os.cpu_count() or 1, 16))
        gbs, tps, busy, wall = oracle_pool(_oracle_score_job, jobs, workers)
        cpu = {"value": round(gbs, 6), "unit": UNIT, "cores": workers, "kind": "oracle",
               "tokens_scored_per_s": round(tps, 1),
               "sample": "%d lanes: window scores, selection to the budget and forced compaction, numpy float64 "
                         "oracle, %d single-threaded processes, %.1f s of CPU work" % (n_lanes, workers, busy)}
    tc, tc_kind = tensor_peak()
    tflops = flops / (ms * 1e-3) / 1e12
    desc = {"dropkv_prefill": "dropkv_prefill: batch 1, 32 q / 8 KV heads, d 128, bf16, context 32768, window 64, "
                              "keep 1638 per KV head: window scoring, selection, compaction",
            "paged_128k": "paged_128k: batch 1, 32 q / 8 KV heads, d 128, bf16, context 131072 in 16-token "
                          "blocks, window 64, keep 6553 per KV head: window scoring, selection, token-level "
                          "compaction into dense blocks"}[name]
    line = line_base(g, args, value, ms_all, all_tok / (ms_all * 1e-3), "bf16", desc,
                     {"l2": "no flush: each pass reads %d MB of K/V, above the 129 MB L2" % (lanes * n * 512 >> 20),
                      "timing": "each sample: reset and prefill (untimed), a short spin to hold the stream, then "
                                "scoring + selection + compaction between CUDA events",
                      "samples_ms": [round(x, 4) for x in samples], "bytes_per_step": int(step_bytes),
                      "moved_tokens": moved, "freed_blocks": nf, "blocks_after": st[9], "live_after": st[10],
                      "half_empty_after": st[11]},
                     reps, args.warmup)
    line["roofline"] = hbm_roofline("window scoring (two tcgen05 passes) + selection + compaction",
                                    step_bytes, ms, {"tensor": {"flops": int(flops),
                                                                "achieved_tflops": round(tflops, 1),
                                                                "peak_tflops": tc, "peak_kind": tc_kind,
                                                                "frac": round(tflops / tc, 4)}})
    line["cpu_baseline"] = cpu
    line["e2e"] = e2e
    line["clocks"] = clocks
    line["gpu_launches"] = None
    g.finish(line)


def run_gpu(args):
    g = Gpu()
    name = args.workload
    if name == "h2o_70b":
        run_h2o70b(args, g)
    elif name == "h2o_70b_mass":
        run_h2o70b_mass(args, g)
    elif name in ("h2o_toy", "snapkv_decode", "dropkv_decode"):
        run_small_decode(args, g, name)
    else:
        run_prefill(args, g, name)


# ---------------------------------------------------------------------------
# reference arm: the oracle on host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from workloads import Workload, shape
    name = args.workload
    t0 = time.time()
    if name in ("h2o_70b", "h2o_70b_mass"):
        shp = shape("h2o_70b")
        wl = Workload(shp)
        f = oracle_fields(shp)
        if name == "h2o_70b":
            lanes, steps, untimed = max(1, args.cpu_lanes), min(args.warmup + args.steps, shp.steps), 1
            sample = "%d lanes of layer 0 x %d steady-state decode steps" % (lanes, steps - 1)
        else:
            lanes, steps, untimed = 16, 1, 0
            sample = "the mass-eviction step of 16 lanes of layer 0"
        jobs = decode_lane_jobs(wl, shp, range(lanes), steps, f, untimed, "cpu")
        fn = _oracle_decode_job
    elif name in ("h2o_toy", "snapkv_decode", "dropkv_decode"):
        shp = small_decode_shape(name)
        wl = Workload(shp)
        tokb, scoreb = per_token_bytes(shp)
        f = oracle_fields(shp, score_bytes=scoreb, tok_bytes=tokb)
        lanes = min(shp.lanes, 32)
        steps = shp.steps if shp.lanes <= 8 else min(shp.steps, 1 + 96)
        jobs = decode_lane_jobs(wl, shp, range(lanes), steps, f, 1, "cpu")
        fn = _oracle_decode_job
        sample = "%d lanes x %d decode steps after the first" % (lanes, steps - 1)
    else:
        shp = shape(name)
        wl = Workload(shp)
        f = oracle_fields(shp, tok_bytes=2 * 2 * shp.head_dim * 2 + 4 + 8)
        lanes = 8 if shp.ctx <= 32768 else 4
        jobs = score_lane_jobs(wl, shp, range(lanes), f, "cpu")
        fn = _oracle_score_job
        sample = "%d lanes: window scores, selection and forced compaction" % lanes
    workers = max(1, min(len(jobs), os.cpu_count() or 1, 16))
    gbs, tps, busy, wall = oracle_pool(fn, jobs, workers)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 6), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "tokens_scored_per_s": round(tps, 1),
        "config": {"workload": name, "seq_len": shp.ctx},
        "cpu_baseline": {"value": round(gbs, 6), "unit": UNIT, "cores": workers, "kind": "oracle",
                         "sample": "%s, numpy float64 oracle, %d single-threaded processes (%.1f s CPU, %.1f s total)"
                                   % (sample, workers, busy, time.time() - t0)},
        "e2e": {"value": round(gbs, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# kernel table: the other kernels, each on its own workload
# ---------------------------------------------------------------------------
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

    sampler = ClockSampler(0)
    sampler.start()

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

    # D3 window scoring and selection alone
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
    print(json.dumps({"kernel_table": "clocks over the table", "clocks": sampler.stop()}), flush=True)


def main():
    args = parse()
    rc = maybe_spawn_ranks(args)
    if rc is not None:
        sys.exit(rc)
    if args.selftest_cpu:
        selftest_cpu(args)
    elif args.impl == "reference":
        if args.all_workloads:
            for name in WORKLOADS:
                args.workload = name
                run_reference(args)
        else:
            run_reference(args)
    elif args.kernel_table:
        run_kernel_table(args)
    elif args.all_workloads:
        # each workload in its own process (each frees its device memory)
        rc = 0
        for name in WORKLOADS:
            cmd = [sys.executable, os.path.abspath(__file__), "--workload", name]
            for a in ("--steps", "--warmup", "--e2e-steps", "--cpu-lanes"):
                cmd += [a, str(getattr(args, a[2:].replace("-", "_")))]
            if args.no_cpu_baseline:
                cmd.append("--no-cpu-baseline")
            rc |= subprocess.call(cmd)
        sys.exit(rc)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
