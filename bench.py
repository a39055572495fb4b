"""Benchmark of one paged q_len=1 decode step (RoPE + append, attention, combine).

Default workload: the c=64 Talker decode batch (64 rows, 16 q / 8 kv heads,
head_dim 128, pages of 16 tokens, lengths uniform in [200, 1200]).  A "step"
is the whole path for one layer over the batch: vh_rope_kv_append,
vh_paged_decode_attn and vh_decode_combine.  Metric: decode tokens/s (active
rows per second per layer call) and achieved HBM GB/s.

Timing: inputs resident in HBM; K steps captured in CUDA graphs that cycle
over enough KV-pool replicas to exceed 4x the L2 size, so every step reads
its K/V from HBM; CUDA events on the launching stream, synchronize and a
barrier on both sides, max over ranks.  The attention kernel alone is timed
the same way for the roofline figure.  `e2e` goes through the public Python
call with pinned host buffers: per step the new q/k/v, lengths, flags and
page table are copied in and the output is copied out.

--impl reference times the float64 CPU oracle on the host cores instead (each
step one row of the same workload).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "decode-attn tokens/s and achieved HBM GB/s (% of GB300 peak) at c=64"
WORKLOAD = "c64"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=list(workloads.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    return ap.parse_args()


def dist_setup(n_gpus):
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def step_bytes(inp) -> dict:
    """Algorithmic bytes of one step and of one attention launch."""
    lens = inp.seq_lens.cpu().long()
    act = inp.active.cpu().long()
    Lact = lens[act.bool()]
    Bact = int(act.sum())
    kv = int(Lact.sum()) * inp.Hkv * inp.D * 2 * 2
    pt = int(((Lact + inp.P - 1) // inp.P).sum()) * 4
    q_bf16 = Bact * inp.Hq * inp.D * 2
    kv_new = Bact * 2 * inp.Hkv * inp.D * 2
    out = Bact * inp.Hq * inp.D * 2
    q_rot = Bact * inp.Hq * inp.D * 4
    lens_b = 8 * inp.B
    step = kv + q_bf16 + kv_new + kv_new + out + pt + lens_b
    attn = kv + q_rot + out + pt + lens_b
    return {"step": step, "attn": attn, "kv": kv, "active": Bact}


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def run_ours(args, rank, world):
    import paged_len_decode_gb300 as vh

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = workloads.WORKLOADS[args.workload]
    inp = workloads.make_inputs(args.workload, layer=rank, device=dev)
    B, Hq, Hkv, D, P = inp.B, inp.Hq, inp.Hkv, inp.D, inp.P
    by = step_bytes(inp)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    pool_bytes = inp.pool.numel() * 2
    R = max(2, math.ceil(4 * l2 / pool_bytes))
    pools = [inp.pool] + [inp.pool.clone() for _ in range(R - 1)]

    max_pos = inp.max_pages_per_seq * P
    cos_sin = torch.empty((max_pos, D), dtype=torch.float32, device=dev)
    vh.vh_rope_table(cos_sin, inp.theta)
    q_rot = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    ws = vh.alloc_workspace(B, Hq, Hkv, D, P, device=dev)
    n_ctas = vh.vh_decode_num_ctas(B, Hq, Hkv, D, P)

    def step(r):
        vh.decode_step(inp.q, inp.k_new, inp.v_new, cos_sin, pools[r][:, 0], pools[r][:, 1], inp.page_table,
                       inp.seq_lens, inp.active, q_rot, out, ws)

    def attn_only(r):
        vh.vh_paged_decode_attn(q_rot, pools[r][:, 0], pools[r][:, 1], inp.page_table, inp.seq_lens,
                                inp.active, out, ws)

    for r in range(R):  # first calls outside capture; also fills every replica's new slot
        step(r)
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=dev)

    def capture(fn, n):
        g = torch.cuda.CUDAGraph()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    fn(i % R)
        torch.cuda.current_stream().wait_stream(stream)
        return g

    chunk = R * max(1, 240 // R)  # steps per graph replay (a multiple of the replica count)

    def timed(fn, K, clocks=None):
        full = capture(fn, chunk)
        rem = K % chunk
        tail = capture(fn, rem) if rem else None
        with torch.cuda.stream(stream):
            full.replay()  # warm the graph itself
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        if clocks:
            clocks.start()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(K // chunk):
                full.replay()
            if tail is not None:
                tail.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ck = clocks.stop() if clocks else None
        barrier(world)
        ms = e0.elapsed_time(e1)
        return max_over_ranks(ms, world), ck

    # warm-up steps (untimed)
    for i in range(args.warmup):
        step(i % R)
    torch.cuda.synchronize()

    clocks = Clocks(dev.index)
    ms_total, ck = timed(step, args.steps, clocks)
    ms_step = ms_total / args.steps
    ms_attn_total, _ = timed(attn_only, args.steps)
    ms_attn = ms_attn_total / args.steps

    tokens_per_s = by["active"] * world / (ms_step * 1e-3)
    step_gbs = by["step"] / (ms_step * 1e-3) / 1e9
    attn_gbs = by["attn"] / (ms_attn * 1e-3) / 1e9
    peak, peak_kind = peaks()

    # ---- e2e through the public call with host buffers ----
    pin = lambda t: t.cpu().pin_memory()
    h_in = {k: pin(getattr(inp, k)) for k in ("q", "k_new", "v_new", "page_table", "seq_lens", "active")}
    d_in = {k: torch.empty_like(getattr(inp, k)) for k in h_in}
    h_out = torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = h_out.numel() * h_out.element_size()
    K_e2e = min(args.steps, 2000)

    def e2e_step(r):
        for k in h_in:
            d_in[k].copy_(h_in[k], non_blocking=True)
        vh.decode_step(d_in["q"], d_in["k_new"], d_in["v_new"], cos_sin, pools[r][:, 0], pools[r][:, 1],
                       d_in["page_table"], d_in["seq_lens"], d_in["active"], q_rot, out, ws)
        h_out.copy_(out, non_blocking=True)

    for i in range(10):
        e2e_step(i % R)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(K_e2e):
        e2e_step(i % R)
    e1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    e2e_ms = max_over_ranks(max(e0.elapsed_time(e1), wall * 1e3), world) / K_e2e
    e2e_tps = by["active"] * world / (e2e_ms * 1e-3)

    res = {
        "metric": METRIC, "value": round(tokens_per_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "accum_dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{args.workload}: B={B} (active {by['active']}), Hq={Hq}, Hkv={Hkv}, "
                               f"D={D}, P={P}, lengths {w.dist} [{w.len_lo},{w.len_hi}]",
                   "global_batch": B * world, "kv_bytes_per_step": by["kv"],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"{R} KV-pool replicas cycled ({R * pool_bytes / 1e6:.0f} MB >= 4x L2 "
                         f"{l2 / 1e6:.0f} MB): inputs larger than L2",
                   "ctas": n_ctas},
        "hbm_gbs": round(step_gbs, 1), "hbm_frac_of_peak": round(step_gbs / peak, 4),
        "roofline": {"bound": "hbm", "kernel": "decode_attn_kernel", "achieved": round(attn_gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(attn_gbs / peak, 4), "traffic": None,
                     "peak_kind": peak_kind, "ms_per_launch": round(ms_attn, 6),
                     "algorithmic_bytes_per_launch": by["attn"]},
        "clocks": ck,
        "e2e": {"value": round(e2e_tps, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 6), "steps": K_e2e},
        "gpu_launches": 3 * args.steps,
    }
    return res, inp


def cpu_oracle_rate(inp_cpu, seconds: float, max_steps: int | None = None):
    """Oracle steps on single rows of the workload (round robin): rows/s."""
    import oracle

    pool = inp_cpu.pool.clone()
    B = inp_cpu.B
    rows = [b for b in range(B) if int(inp_cpu.active[b])]
    n, t0 = 0, time.perf_counter()
    while True:
        b = rows[n % len(rows)]
        act = torch.zeros(B, dtype=torch.int32)
        act[b] = 1
        q_rot, pool_after, _ = oracle.rope_kv_append(inp_cpu.q, inp_cpu.k_new, inp_cpu.v_new, pool,
                                                     inp_cpu.page_table, inp_cpu.seq_lens, act,
                                                     P=inp_cpu.P, theta=inp_cpu.theta, in_place=True)
        oracle.decode_attn(q_rot, pool_after, inp_cpu.page_table, inp_cpu.seq_lens, act, P=inp_cpu.P,
                           rows=[b])
        n += 1
        el = time.perf_counter() - t0
        if (max_steps is not None and n >= max_steps) or (max_steps is None and el >= seconds):
            return n / el, n, el, oracle.num_threads()


def main():
    args = parse()
    rank, world = dist_setup(args.gpus)
    if args.impl == "reference":
        if rank != 0:
            return
        inp = workloads.make_inputs(args.workload, device="cpu")
        cpu_oracle_rate(inp, 0, max_steps=max(3, args.warmup) if args.warmup else 3)
        rate, n, el, cores = cpu_oracle_rate(inp, 0, max_steps=args.steps)
        res = {"impl": "reference", "metric": METRIC, "value": round(rate, 3), "unit": "tokens/s",
               "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
               "ms_per_step": round(el / n * 1e3, 4), "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "f64", "data": "synthetic",
               "config": {"workload": f"{args.workload} (one row per step, round robin)"},
               "cpu_baseline": {"value": round(rate, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"{n} single-row oracle steps of the {args.workload} workload"},
               "e2e": {"value": round(rate, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                       "d2h_bytes_per_step": 0}}
        print(json.dumps(res))
        return
    res, inp = run_ours(args, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, n, el, cores = cpu_oracle_rate(inp.to("cpu"), args.cpu_seconds)
        res["cpu_baseline"] = {"value": round(rate, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                               "sample": f"{n} single-row oracle steps (RoPE+append+attention) of the "
                                         f"{args.workload} workload in {el:.1f} s"}
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
