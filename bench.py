"""Benchmark of the DynaSpec draft head + verification step on GB300.

One step = one chain speculation step of the Llama-3-8B-shaped drafter head on one sequence:
for each of the 6 draft positions the router MLP + position-aware top-k + shortlist build
(side stream) and the gathered head with the Gumbel-max draw (main stream), then rejection-
sampling verification over the full 128,256-token vocabulary.  The metric is draft tokens/s
(B * gamma tokens per step).  Inputs are seeded synthetic tensors of the stated shapes.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]

`--impl reference` times the CPU oracle (plain C, fp64) on the same workload: the only
reference implementation of this path is the one written from the DynaSpec pages.
Under torchrun every rank runs its own replica (independent sequences, no collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np   # noqa: E402

METRIC = "draft-head tokens/s (router+gather-GEMM+sample+verify)"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 512 << 20        # > 129 MB L2: written between timed steps ...
L2_CLEAN_BYTES = 256 << 20        # ... then this much is read, so the written lines leave L2 too
TIMED_HEAD_STEPS = 256                 # instrumented replays for the per-head times (the event clock
                                      # ticks in ~2 us steps: many samples average the ticks out)
FALLBACK_HBM_GBS = 6800.0
HEAD_KERNEL_SOURCES = ["dynamic_vocab_draft_gb300/csrc/head.cu", "dynamic_vocab_draft_gb300/csrc/common.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="llama_b1")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure only the --config workload (by default the llama_b1 run also "
                         "measures the batched, tree and large workloads, key per_config)")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), \
        int(os.environ.get("WORLD_SIZE", "1"))


def max_over_ranks(ms, device=None):
    """The slowest rank's time: every replica ran the same number of steps on its own
    sequences, so the job's time is the maximum (all_reduce MAX; identity for one process)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_step, steps, job_ms):
    """Units per second over all ranks: each of `world` replicas did units_per_step * steps."""
    return world * units_per_step * steps / (job_ms * 1e-3)


def workload_config(cfg):
    kind = (f"chain drafting, B={cfg.B}, gamma={cfg.gamma}" if cfg.mode == "chain" else
            f"tree drafting, B={cfg.B}, depth {cfg.gamma} x {cfg.width} nodes")
    if cfg.static:
        kind += f", one fixed {cfg.static}-token shortlist (no router)"
    return {"workload": f"{cfg.name}: {kind}, V={cfg.V}, d={cfg.d}, T={cfg.T}",
            "V": cfg.V, "d": cfg.d, "clusters": cfg.M, "router": f"{cfg.d}->{cfg.Hr}->{cfg.M} {cfg.act}",
            "B": cfg.B, "gamma": cfg.gamma, "budget": list(cfg.budget), "T": cfg.T,
            "sigma_p": cfg.sigma_p, "seed": None,
            "l2": (f"flushed before every timed step ({L2_FLUSH_BYTES >> 20} MB write, then "
                   f"{L2_CLEAN_BYTES >> 20} MB read: no input of the step and no dirty line in L2)"),
            "parallelism": "replicas (independent sequences per GPU, no collective)"}


# ---------------------------------------------------------------------------------------
# Reference arm: the CPU oracle
# ---------------------------------------------------------------------------------------
def oracle_sample(inp, budget_s, max_steps, warmup):
    """Time whole oracle steps on the host (one position + verify per step, positions cycled)
    until max_steps are done or budget_s is spent.  Returns (tokens/s, steps, seconds)."""
    import oracle
    cfg = inp["cfg"]
    gamma = cfg.gamma
    ref = oracle.chain_step(inp, seqs=[0])       # warm (and needed for the verify sample)
    pos = ref[0]["positions"]
    for i in range(max(0, warmup)):
        oracle.chain_step(inp, seqs=[0], positions=[i % gamma], verify=False)
    t0 = time.perf_counter()
    n = 0
    while n < max_steps and (time.perf_counter() - t0) < budget_s:
        t = n % gamma
        oracle.chain_step(inp, seqs=[0], positions=[t], verify=False)
        if t == gamma - 1:
            oracle.verify_chain(inp["z"][:1], [[p["logits"] for p in pos]], [[p["S"] for p in pos]],
                                np.array([[p["idx"] for p in pos]]), inp["u"][:1], cfg.T)
        n += 1
    dt = time.perf_counter() - t0
    return n / dt, n, dt


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    import oracle
    import workloads as wl
    cfg = wl.config(args.config)
    if cfg.mode == "chain":
        inp = wl.chain_inputs(cfg, args.seed)
        warm = args.warmup
        value, n, dt = oracle_sample(inp, budget_s=90.0, max_steps=args.steps, warmup=warm)
        sample = (f"{n} oracle draft positions of sequence 0 (router + top-k + shortlist + head + sample; "
                  f"verification of the whole chain after every {cfg.gamma}th), {dt:.1f} s")
        ms_per_step = 1e3 * dt / max(n, 1) * cfg.gamma * cfg.B
    else:
        inp = wl.tree_inputs(cfg, args.seed)
        warm = min(args.warmup, 2)                 # a whole tree step of the oracle takes seconds
        for _ in range(warm):
            oracle.tree_step(inp, seqs=[0])
        t0 = time.perf_counter()
        n = 0
        while n < max(1, min(args.steps, 3)) and time.perf_counter() - t0 < 90.0:
            oracle.tree_step(inp, seqs=[0])
            n += 1
        dt = time.perf_counter() - t0
        value = n * cfg.gamma * cfg.width / dt
        sample = f"{n} whole tree steps of sequence 0 ({cfg.gamma * cfg.width} nodes each + verification), {dt:.1f} s"
        ms_per_step = 1e3 * dt / n * cfg.B
    cores = oracle.get_threads()
    # the same workload description as the GPU arm's line (the L2 flush it names is the GPU
    # arm's timing rule; the oracle runs on the host cores)
    cfgd = workload_config(cfg)
    cfgd["seed"] = args.seed
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": n, "warmup": warm, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": cfgd,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def head_source_hash():
    h = hashlib.sha256()
    for rel in HEAD_KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_head_profile():
    """The committed ncu summary's per-launch figures for the batch-1 head (DRAM bytes, mean
    duration in µs), if it was taken on the current kernel source (else {})."""
    path = os.path.join(ROOT, "profiles", "head_gemv_llama_b1.md")
    try:
        text = open(path).read()
    except OSError:
        return {}
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha") != head_source_hash():
        return {}
    out = {}
    for key, name in (("traffic", "dram_bytes_per_launch"), ("launch_us", "ncu_launch_us_mean")):
        try:
            out[key] = float(vals[name])
        except (KeyError, ValueError):
            pass
    return out


def committed_traffic():
    """DRAM bytes per head launch from the committed ncu summary, if it was taken on the
    current kernel source (else None)."""
    return committed_head_profile().get("traffic")


_HEAD_CACHE = {}


def device_head(cfg, seed, dev, torch, host=False):
    """The LM head W [V, d] on the device (host=True: its host bits too, for the oracle);
    workloads with the same (V, d, seed) share one copy."""
    import workloads as wl
    key = (cfg.V, cfg.d, seed)
    if key not in _HEAD_CACHE:
        _HEAD_CACHE.clear()                      # keep one head resident at a time
        W = wl.lm_head(cfg, seed)
        _HEAD_CACHE[key] = (W, torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16))
    return _HEAD_CACHE[key] if host else _HEAD_CACHE[key][1]


def build_drafter(cfg, inp, dev, pkg, torch, W):
    """Drafter + pinned host copies of the per-step inputs (name -> (host, device buffer))."""
    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def pinned_bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()

    common = (W, bf(inp["W1"]), bf(inp["b1"]), bf(inp["W2"]), bf(inp["b2"]),
              torch.as_tensor(inp["csr_off"]), torch.as_tensor(inp["csr_tok"]))
    if cfg.mode == "chain":
        if cfg.static:
            d = pkg.pipeline.StaticChainDrafter(W, inp["static_ids"], B=cfg.B, gamma=cfg.gamma, T=cfg.T,
                                                seed=inp["gumbel_seed"])
        else:
            d = pkg.pipeline.ChainDrafter(*common, B=cfg.B, gamma=cfg.gamma, budget=cfg.budget, act=cfg.act,
                                          T=cfg.T, seed=inp["gumbel_seed"])
        host = {"H": (pinned_bf(inp["H"].transpose(1, 0, 2)), d.H),
                "z": (torch.from_numpy(inp["z"]).pin_memory(), d.z),
                "u": (torch.from_numpy(inp["u"]).pin_memory(), d.u)}
        tokens = cfg.B * cfg.gamma
    else:
        d = pkg.pipeline.TreeDrafter(*common, inp["parent"], B=cfg.B, D=cfg.gamma, Wd=cfg.width,
                                     budget=cfg.budget, act=cfg.act, T=cfg.T, seed=inp["gumbel_seed"])
        host = {"Hr_h": (pinned_bf(inp["Hr_h"].transpose(1, 0, 2)), d.Hr_h),
                "Hn": (pinned_bf(inp["Hn"]), d.Hn),
                "z": (torch.from_numpy(inp["z"]).pin_memory(), d.z),
                "u_node": (torch.from_numpy(inp["u_node"]).pin_memory(), d.u_node),
                "u_res": (torch.from_numpy(inp["u_res"]).pin_memory(), d.u_res)}
        tokens = cfg.B * cfg.gamma * cfg.width
    for h, dv in host.values():
        dv.copy_(h)
    return d, host, tokens


def algorithmic_bytes(cfg, d):
    """Per head launch (list) and per step, counted once per byte the path must move: every W row of
    the (per-position) union once, the router weights once per position, each target row once, the
    ids, logits and hidden states once."""
    V, dd, M, Hr = cfg.V, cfg.d, cfg.M, cfg.Hr
    G = 1 if cfg.mode == "chain" else cfg.width
    n_pos = cfg.gamma
    offs = d.vs_offsets.cpu().numpy()
    sizes = np.diff(offs, axis=1)                                       # [pos, B]
    if not getattr(d, "union", True):
        union = None
    elif cfg.static:
        union = np.full(n_pos, cfg.static)                              # the one list is the union
    else:
        union = d.union_count.cpu().numpy()[:, 0]
    heads = []
    for t in range(n_pos):
        S = float(sizes[t].sum())
        rows = S if union is None else float(union[t])                   # W rows streamed
        ids_bytes = 4 * rows if union is None else 8 * rows              # list ids / union ids + clusters
        heads.append(rows * 2 * dd + ids_bytes + 4 * S * G + cfg.B * G * 2 * dd)
    router = 0 if cfg.static else 2 * (Hr * dd + Hr + M * Hr + M) + cfg.B * (2 * dd + 4 * Hr * 2 + 4 * M)
    rows_target = cfg.gamma + 1 if cfg.mode == "chain" else 1 + cfg.gamma * cfg.width
    verify = 4 * cfg.B * rows_target * V
    return heads, float(sum(heads) + n_pos * router + verify), (union.tolist() if union is not None else None), sizes


class Flusher:
    """Evicts the previous step's inputs from the 129 MB L2 before every timed step: a 512 MB
    write, then a 256 MB read so the written lines leave L2 too (no dirty line left for the
    step to write back)."""

    def __init__(self, dev, torch):
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.clean = torch.zeros(L2_CLEAN_BYTES // 4, dtype=torch.int32, device=dev)
        self.sink = torch.zeros((), dtype=torch.int64, device=dev)

    def __call__(self, i):
        self.flush.fill_(i & 0xFF)
        self.sink.copy_(self.clean.sum())


def measure(cfg, seed, dev, pkg, torch, world, local_rank, steps, warmup, e2e_steps, head_steps, flush):
    """Time `steps` whole steps of workload cfg (device-resident inputs), then the per-head times
    from the instrumented graph, then `e2e_steps` steps with their host transfers.  Returns the
    measured figures and the inputs (for the oracle baseline)."""
    import workloads as wl
    inp = (wl.chain_inputs(cfg, seed, with_head=False) if cfg.mode == "chain"
           else wl.tree_inputs(cfg, seed, with_head=False))
    W = device_head(cfg, seed, dev, torch)
    d, host, tokens_per_step = build_drafter(cfg, inp, dev, pkg, torch, W)
    d.enable_head_timing()
    d.capture()
    main = torch.cuda.current_stream(dev)
    for _ in range(max(3, warmup)):
        flush(1)
        d.replay()
    torch.cuda.synchronize()
    d.check_status()

    K = steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    t_wall = time.perf_counter()
    for i in range(K):
        flush(i)
        starts[i].record(main)
        d.replay()
        ends[i].record(main)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = max_over_ranks(sum(step_ms), dev)
    d.check_status()
    value = whole_job_rate(world, tokens_per_step, K, total_ms)
    # per-head launch times and the step's breakdown, from the instrumented graph (same step
    # plus event records around every head), replayed after the timed region
    head_ms, breakdown = [], []
    for i in range(max(1, min(K, head_steps))):
        flush(i)
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(main)
        d.replay(timed=True)
        s1.record(main)
        torch.cuda.synchronize()
        head_ms.append(d.head_times_ms())
        h0, hl = d.head_events[0][0], d.head_events[-1][1]
        breakdown.append((s0.elapsed_time(h0), h0.elapsed_time(hl), hl.elapsed_time(s1)))

    # e2e through the public API: every step copies its inputs from pinned host memory (the
    # ones only verification reads on a copy stream beside the drafting stages) and its
    # results (accepted lengths, corrections, draft tokens) back to pinned host memory
    Ke = max(1, min(K, e2e_steps))
    out_h = torch.empty(d.out.shape, dtype=d.out.dtype).pin_memory()
    late_names = ("z", "u", "u_node", "u_res")
    d.capture_io([v for k, v in host.items() if k not in late_names],
                 [v for k, v in host.items() if k in late_names], out_h)
    for _ in range(max(3, warmup)):             # untimed, like the device leg's warm-up
        flush(1)
        d.replay_io()
    torch.cuda.synchronize()
    e2e_ms = 0.0
    for i in range(Ke):
        flush(i)
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(main)
        d.replay_io()
        e.record(main)
        e.synchronize()
        e2e_ms += s.elapsed_time(e)
    d.check_status()
    h2d = sum(h.numel() * h.element_size() for h, _ in host.values())
    d2h = out_h.numel() * out_h.element_size()
    e2e_ms = max_over_ranks(e2e_ms, dev)
    e2e_value = whole_job_rate(world, tokens_per_step, Ke, e2e_ms)

    peak, peak_src = load_peak()
    hm = np.array(head_ms)                               # [samples, positions] ms
    head_bytes, step_bytes, union, sizes = algorithmic_bytes(cfg, d)
    per_row = cfg.mode == "chain" and cfg.B == 1
    achieved = float(sum(head_bytes) / (hm.mean(axis=0).sum() * 1e-3) / 1e9)
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": committed_traffic() if per_row and cfg.name == "llama_b1" else None,
            "kernel": ("head_gemv_kernel (gathered head, per-row path: one warp per W row, 8 KB in flight)"
                       if per_row else "tc::gemm_kernel<MT, UnionEp> + head_rowstats_kernel (gathered head "
                       "over the union of the lists on tcgen05, then the row statistics and draws)"),
            "algorithmic_bytes_per_launch": float(np.mean(head_bytes)),
            "avg_launch_us": float(hm.mean() * 1e3), "peak_source": peak_src,
            "shortlist_sizes": sizes.sum(axis=1).tolist(), "union_rows": union}
    if per_row and cfg.name == "llama_b1":
        # the same launches' mean duration in the committed ncu launch list (cold, serialised;
        # without the latency of the events that bracket each head inside the graph)
        prof = committed_head_profile()
        if "launch_us" in prof:
            roof["ncu_avg_launch_us"] = prof["launch_us"]
            roof["ncu_frac"] = float(np.mean(head_bytes)) / (prof["launch_us"] * 1e-6) / 1e9 / peak
    step_us = total_ms / K * 1e3
    res = dict(
        cfg=cfg, inp=inp, value=value, total_ms=total_ms, K=K, tokens_per_step=tokens_per_step, roofline=roof,
        step_roofline={"algorithmic_bytes": step_bytes, "achieved_gbs": step_bytes / (step_us * 1e-6) / 1e9,
                       "frac": step_bytes / (step_us * 1e-6) / 1e9 / peak},
        e2e={"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
             "steps": Ke, "ms_per_step": e2e_ms / Ke},
        breakdown_us={
            "before_first_head": 1e3 * float(np.median([x[0] for x in breakdown])),
            "heads_span": 1e3 * float(np.median([x[1] for x in breakdown])),
            "heads_busy": 1e3 * float(np.median(hm.sum(axis=1))),
            "after_last_head (verify)": 1e3 * float(np.median([x[2] for x in breakdown])),
            "per_position_head": [1e3 * float(x) for x in np.median(hm, axis=0)]},
        gpu_launches=d.launches_per_step() * K, clocks=clk, wall_s=t_wall,
        step_ms_p50=float(np.median(step_ms)), step_ms_min=float(np.min(step_ms)))
    del d, host
    return res


STANDIN_F = 14336                 # drafter stand-in MLP width (Llama-3-8B's)


def measure_overlap(cfg, seed, dev, pkg, torch, steps, warmup, flush):
    """The router's overlap with the drafter at batch 1 (DynaSpec summary, Pipeline Flow: the
    router runs on its own stream beside the drafter).  A drafter stand-in with the weight bytes
    of an EAGLE step runs before every head (ds_drafter_standin, scale 0 so the hidden states stay
    the workload's); router t+1 waits for the drafter step that computes its input.  The same
    step with the routers serialised on the main stream gives the router's full cost, so
    serial - overlapped = the router time the overlap hides."""
    import workloads as wl
    inp = wl.chain_inputs(cfg, seed, with_head=False)
    W = device_head(cfg, seed, dev, torch)
    d, host, tokens_per_step = build_drafter(cfg, inp, dev, pkg, torch, W)
    g = torch.Generator(device=dev).manual_seed(seed + 101)
    mk = lambda *shape: (torch.randn(*shape, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    d.attach_drafter(mk(cfg.d, 2 * cfg.d), mk(cfg.d, cfg.d), mk(2 * STANDIN_F, cfg.d), mk(cfg.d, STANDIN_F),
                     scale=0.0)
    d.H_base.copy_(d.H)
    d.x0.fill_(int(inp["csr_tok"][0]))
    standin_bytes = 2 * (2 * cfg.d * cfg.d + cfg.d * cfg.d + 3 * STANDIN_F * cfg.d)
    main = torch.cuda.current_stream(dev)
    out = {"standin_weight_bytes_per_step": standin_bytes * cfg.gamma, "standin_F": STANDIN_F}
    for serial in (False, True):
        d.serial_router = serial
        d.head_events = None
        d.route_events = None
        if not serial:
            d.enable_head_timing()
            d.enable_overlap_timing()
        d.capture()
        for _ in range(max(3, warmup)):
            flush(1)
            d.replay()
        torch.cuda.synchronize()
        d.check_status()
        ms = []
        for i in range(steps):
            flush(i)
            a = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            a.record(main)
            d.replay()
            e.record(main)
            e.synchronize()
            ms.append(a.elapsed_time(e))
        out["serial_us" if serial else "overlapped_us"] = 1e3 * float(np.median(ms))
        if not serial:
            ov = []
            for i in range(max(1, min(steps, 16))):
                flush(i)
                d.replay(timed=True)
                torch.cuda.synchronize()
                ov.append(d.overlap_times_ms())
            ov = np.median(np.array(ov), axis=0)           # [gamma, 6] ms
            out["router_us_per_position"] = [1e3 * float(x) for x in ov[:, 1] - ov[:, 0]]
            out["drafter_us_per_position"] = [1e3 * float(x) for x in ov[:, 3] - ov[:, 2]]
            out["head_us_per_position"] = [1e3 * float(x) for x in ov[:, 5] - ov[:, 4]]
            # router t (t >= 1) starts after drafter step t-1; what the head of t waits for beyond
            # its own drafter step is the exposed part
            out["router_exposed_us_per_position"] = [1e3 * float(max(0.0, ov[t, 1] - ov[t, 3]))
                                                     for t in range(cfg.gamma)]
    d.check_status()
    out["hidden_router_us_per_step"] = out["serial_us"] - out["overlapped_us"]
    out["router_total_us_per_step"] = float(sum(out["router_us_per_position"]))
    out["tokens_per_s_overlapped"] = tokens_per_step / (out["overlapped_us"] * 1e-6)
    del d, host
    return out


# Workloads measured after the headline, in the same process (same flush and timing).
PER_CONFIG = ["llama_b1_static32k", "batched", "tree", "large_b1_f5", "large_b64_f100"]


def run_ours(args):
    import torch
    import workloads as wl
    import dynamic_vocab_draft_gb300 as pkg

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pkg.load_library()
    cfg = wl.config(args.config)
    seed = args.seed + rank                      # each replica drafts its own sequences
    flush = Flusher(dev, torch)
    r = measure(cfg, seed, dev, pkg, torch, world, local_rank, args.steps, args.warmup, args.e2e_steps,
                TIMED_HEAD_STEPS, flush)
    inp = r.pop("inp")
    inp["W"] = device_head(cfg, seed, dev, torch, host=True)[0]      # the oracle baseline reads it

    per_config = None
    if args.config == "llama_b1" and not args.no_per_config:
        per_config = {}
        for name in PER_CONFIG:
            torch.cuda.empty_cache()
            c = wl.config(name)
            q = measure(c, seed, dev, pkg, torch, world, local_rank, args.steps, args.warmup,
                        args.e2e_steps, min(args.steps, 64), flush)
            q.pop("inp")
            unit = "nodes/s" if c.mode == "tree" else "tokens/s"
            per_config[name] = {
                "workload": workload_config(c)["workload"], "value": q["value"], "unit": unit,
                "us_per_step": q["total_ms"] / q["K"] * 1e3, "steps": q["K"],
                "head_frac": q["roofline"]["frac"], "head_us": q["roofline"]["avg_launch_us"],
                "head_kernel": q["roofline"]["kernel"],
                "step_frac": q["step_roofline"]["frac"], "step_algorithmic_bytes": q["step_roofline"]["algorithmic_bytes"],
                "e2e": {"value": q["e2e"]["value"], "unit": unit, "ms_per_step": q["e2e"]["ms_per_step"],
                        "h2d_bytes_per_step": q["e2e"]["h2d_bytes_per_step"],
                        "d2h_bytes_per_step": q["e2e"]["d2h_bytes_per_step"]},
                "breakdown_us": q["breakdown_us"], "clocks": q["clocks"], "gpu_launches": q["gpu_launches"]}
        torch.cuda.empty_cache()
        per_config["llama_b1_drafter_overlap"] = measure_overlap(
            wl.config("llama_b1"), seed, dev, pkg, torch, max(args.steps, 20), args.warmup, flush)
        _HEAD_CACHE.clear()

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, inp)
    cfgd = workload_config(cfg)
    cfgd["seed"] = args.seed
    line = {"metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": world, "steps": r["K"],
            "warmup": max(3, args.warmup), "ms_per_step": r["total_ms"] / r["K"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": cfgd, "roofline": r["roofline"], "step_roofline": r["step_roofline"],
            "cpu_baseline": cpu, "e2e": r["e2e"], "breakdown_us": r["breakdown_us"],
            "gpu_launches": r["gpu_launches"], "clocks": r["clocks"], "wall_s_timed_region": r["wall_s"],
            "step_ms_p50": r["step_ms_p50"], "step_ms_min": r["step_ms_min"]}
    if per_config is not None:
        line["per_config"] = per_config
    print(json.dumps(line), flush=True)


def cpu_baseline(cfg, inp):
    """The oracle on the host cores, on a bounded sample of the same workload: all cores (the
    line's value) and one thread."""
    import oracle
    all_cores = oracle.get_threads()
    out = {}
    for threads, budget_s in ((all_cores, 12.0), (1, 8.0)):
        oracle.set_threads(threads)
        if cfg.mode == "chain":
            v, n, dt = oracle_sample(inp, budget_s=budget_s, max_steps=10 ** 9, warmup=1)
            sample = (f"{n} oracle draft positions of sequence 0 of this workload "
                      f"(+ chain verification every {cfg.gamma}th), {dt:.1f} s")
        else:
            t0 = time.perf_counter()
            oracle.tree_step(inp, seqs=[0])
            dt = time.perf_counter() - t0
            v = cfg.gamma * cfg.width / dt
            sample = f"one whole tree step of sequence 0 ({cfg.gamma * cfg.width} nodes + tree verification), {dt:.1f} s"
        out[threads] = (v, sample)
    oracle.set_threads(all_cores)
    v, sample = out[all_cores]
    return {"value": v, "unit": UNIT, "cores": all_cores, "kind": "oracle", "sample": sample,
            "single_thread": {"value": out[1][0], "unit": UNIT, "cores": 1, "sample": out[1][1]}}


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
