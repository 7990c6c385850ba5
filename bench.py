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
L2_FLUSH_BYTES = 512 << 20        # > 129 MB L2: written between timed steps
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
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), \
        int(os.environ.get("WORLD_SIZE", "1"))


def workload_config(cfg):
    return {"workload": f"{cfg.name}: chain drafting, Llama-3-8B-shaped LM head, "
                        f"B={cfg.B}, gamma={cfg.gamma}, T={cfg.T}",
            "V": cfg.V, "d": cfg.d, "clusters": cfg.M, "router": f"{cfg.d}->{cfg.Hr}->{cfg.M} {cfg.act}",
            "B": cfg.B, "gamma": cfg.gamma, "budget": list(cfg.budget), "T": cfg.T,
            "sigma_p": cfg.sigma_p, "seed": None,
            "l2": f"flushed before every timed step ({L2_FLUSH_BYTES >> 20} MB write)",
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
    for _ in range(max(0, min(warmup, 1))):
        oracle.chain_step(inp, seqs=[0], positions=[0], verify=False)
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
    inp = wl.chain_inputs(cfg, args.seed)
    value, n, dt = oracle_sample(inp, budget_s=90.0, max_steps=args.steps, warmup=args.warmup)
    cores = oracle.get_threads()
    sample = (f"{n} oracle draft positions of sequence 0 (router + top-k + shortlist + head + sample; "
              f"verification of the whole chain after every {cfg.gamma}th), {dt:.1f} s")
    cfgd = workload_config(cfg)
    cfgd["seed"] = args.seed
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": n, "warmup": min(args.warmup, 1), "ms_per_step": 1e3 * dt / max(n, 1) * cfg.gamma,
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


def committed_traffic():
    """DRAM bytes per head launch from the committed ncu summary, if it was taken on the
    current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "head_gemv_llama_b1.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha") != head_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


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
    assert cfg.mode == "chain"
    seed = args.seed + rank                      # each replica drafts its own sequences
    inp = wl.chain_inputs(cfg, seed)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    d = pkg.pipeline.ChainDrafter(bf(inp["W"]), bf(inp["W1"]), bf(inp["b1"]), bf(inp["W2"]), bf(inp["b2"]),
                                  torch.as_tensor(inp["csr_off"]), torch.as_tensor(inp["csr_tok"]),
                                  B=cfg.B, gamma=cfg.gamma, budget=cfg.budget, act=cfg.act, T=cfg.T,
                                  seed=inp["gumbel_seed"])
    # step inputs in pinned host memory (the e2e leg copies them every step)
    H_host = torch.from_numpy(np.ascontiguousarray(inp["H"].transpose(1, 0, 2)).view(np.int16)) \
        .view(torch.bfloat16).pin_memory()
    z_host = torch.from_numpy(inp["z"]).pin_memory()
    u_host = torch.from_numpy(inp["u"]).pin_memory()
    d.H.copy_(H_host)
    d.z.copy_(z_host)
    d.u.copy_(u_host)
    d.enable_head_timing()
    d.capture()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    main = torch.cuda.current_stream(dev)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        d.replay()
    torch.cuda.synchronize()
    d.check_status()
    sizes = np.diff(d.vs_offsets.cpu().numpy(), axis=1)[:, 0] if cfg.B == 1 else None

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    head_ms = []
    breakdown = []                           # (router before the first head, heads span, verify) ms
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    t_wall = time.perf_counter()
    for i in range(K):
        flush.fill_(i & 0xFF)
        starts[i].record(main)
        d.replay()
        ends[i].record(main)
        if i % 16 == 15 or i == K - 1:      # head timings are overwritten by the next replay
            torch.cuda.synchronize()
            head_ms.append(d.head_times_ms())
            h0, hl = d.head_events[0][0], d.head_events[-1][1]
            breakdown.append((starts[i].elapsed_time(h0), h0.elapsed_time(hl), hl.elapsed_time(ends[i])))
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = sum(step_ms)
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    d.check_status()
    tokens_per_step = cfg.B * cfg.gamma
    value = world * tokens_per_step * K / (total_ms * 1e-3)

    # e2e through the public API: pinned host inputs -> device, step, results -> host
    Ke = min(K, args.e2e_steps)
    acc_h = torch.empty(cfg.B, dtype=torch.int32).pin_memory()
    cor_h = torch.empty(cfg.B, dtype=torch.int32).pin_memory()
    tok_h = torch.empty(cfg.gamma, cfg.B, dtype=torch.int32).pin_memory()
    e2e_ms = 0.0
    for i in range(Ke):
        flush.fill_(i & 0xFF)
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(main)
        d.H.copy_(H_host, non_blocking=True)
        d.z.copy_(z_host, non_blocking=True)
        d.u.copy_(u_host, non_blocking=True)
        d.replay()
        acc_h.copy_(d.accepted, non_blocking=True)
        cor_h.copy_(d.correction, non_blocking=True)
        tok_h.copy_(d.tokens, non_blocking=True)
        e.record(main)
        e.synchronize()
        e2e_ms += s.elapsed_time(e)
    h2d = H_host.numel() * 2 + z_host.numel() * 4 + u_host.numel() * 4
    d2h = (acc_h.numel() + cor_h.numel() + tok_h.numel()) * 4
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(t.item())
    e2e_value = world * tokens_per_step * Ke / (e2e_ms * 1e-3)

    # roofline of the dominant kernel: the gathered head (algorithmic bytes per launch)
    peak, peak_src = load_peak()
    hm = np.array(head_ms)                               # [samples, gamma] ms
    if sizes is not None:
        head_bytes = sizes.astype(np.float64) * (2 * cfg.d + 8) + 2 * cfg.d   # W rows + id + logit, h
    else:
        head_bytes = None
    roof = None
    if head_bytes is not None:
        achieved = float(head_bytes.sum() / (hm.mean(axis=0).sum() * 1e-3) / 1e9)
        traffic = committed_traffic()
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic, "kernel": "head_gemv_kernel (gathered head, per-row path, software-pipelined 16-byte loads)",
                "algorithmic_bytes_per_launch": float(head_bytes.mean()),
                "avg_launch_us": float(hm.mean() * 1e3), "peak_source": peak_src,
                "shortlist_sizes": sizes.tolist()}
    step_bytes = None
    if sizes is not None:
        router_bytes = 2 * (cfg.Hr * cfg.d + cfg.Hr + cfg.M * cfg.Hr + cfg.M) + 4 * cfg.Hr * 2 + 4 * cfg.M * 2
        verify_bytes = 4 * cfg.B * (cfg.gamma + 1) * cfg.V
        step_bytes = float(head_bytes.sum() + cfg.gamma * router_bytes + verify_bytes)

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        v, n, dt = oracle_sample(inp, budget_s=20.0, max_steps=10 ** 9, warmup=1)
        cpu = {"value": v, "unit": UNIT, "cores": oracle.get_threads(), "kind": "oracle",
               "sample": f"{n} oracle draft positions of sequence 0 of this workload "
                         f"(+ chain verification every {cfg.gamma}th), {dt:.1f} s"}
    cfgd = workload_config(cfg)
    cfgd["seed"] = args.seed
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": total_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": cfgd, "roofline": roof,
            "step_roofline": None if step_bytes is None else {
                "algorithmic_bytes": step_bytes, "achieved_gbs": step_bytes / (total_ms / K * 1e-3) / 1e9,
                "frac": step_bytes / (total_ms / K * 1e-3) / 1e9 / peak},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": Ke, "ms_per_step": e2e_ms / Ke},
            "breakdown_us": {
                "before_first_head": 1e3 * float(np.median([x[0] for x in breakdown])),
                "heads_span": 1e3 * float(np.median([x[1] for x in breakdown])),
                "heads_busy": 1e3 * float(np.median(hm.sum(axis=1))),
                "after_last_head (verify)": 1e3 * float(np.median([x[2] for x in breakdown])),
                "per_position_head": [1e3 * float(x) for x in np.median(hm, axis=0)]},
            "gpu_launches": d.launches_per_step() * K,
            "clocks": clk,
            "wall_s_timed_region": t_wall,
            "step_ms_p50": float(np.median(step_ms)), "step_ms_min": float(np.min(step_ms))}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
