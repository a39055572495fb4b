"""Benchmark of the paged q_len=1 decode step (RoPE + append, attention, merge).

Default workload: the c=64 Talker decode batch (64 rows, 16 q / 8 kv heads,
head_dim 128, pages of 16 tokens, lengths uniform in [200, 1200]).  A "step"
is the whole path for one layer over the batch.  The headline runs it as one
launch (vh_decode_fused), each step a programmatic dependent of the previous
one; the three-call form (vh_rope_kv_append, vh_paged_decode_attn,
vh_decode_combine) is timed beside it.  Metric: decode tokens/s (active rows
per layer call per second) and the achieved HBM GB/s of the step.

Timing: inputs resident in HBM; K steps captured in CUDA graphs that cycle
over enough KV-pool replicas to exceed 4x the L2 size, so every step reads
its K/V from HBM; CUDA events on the launching stream, synchronize and a
barrier on both sides, max over ranks.  `e2e` goes through the public Python
call with pinned host buffers: per step the new q/k/v, lengths, flags and page
table (one input arena) are copied in and the output is copied out.  The
headline e2e replays a CUDA graph of many steps with two input arenas and two
outputs, the copies on their own streams overlapping the neighbouring steps'
kernels, as a serving runtime pipelines its decode steps; `e2e.serial` is one
graph per step (copy in, call, copy out, in order) and `e2e.eager` issues the
same copies and call from Python each step.

--impl reference times the float64 CPU oracle on the host cores instead (each
step one row of the same workload).  --ncu-case runs a few eager launches on
one pool only (for profiler captures).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
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
KERNEL_SOURCES = ["paged_len_decode_gb300/csrc/decode_attn.cu", "paged_len_decode_gb300/csrc/vh_common.cuh",
                  "paged_len_decode_gb300/csrc/vh_kernels.h", "paged_len_decode_gb300/csrc/vh_plan.cu",
                  "paged_len_decode_gb300/csrc/vh_plan.h"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=list(workloads.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "fp16"],
                    help="16-bit element type of q, k, v, the cache and the output")
    ap.add_argument("--layout", default=None, choices=["NHD", "HND", "CONTIG"],
                    help="cache layout: token-major pages [NP,2,P,Hkv,D], head-major pages "
                         "[NP,2,Hkv,P,D] or one contiguous cache per row [2,B,Hkv,P,D] "
                         "(default: the workload's)")
    ap.add_argument("--interleaved", action="store_true",
                    help="interleaved (2i, 2i+1) RoPE pairing instead of rotate-half")
    ap.add_argument("--pdl-kv", type=int, default=1,
                    help="fused steps request their first cached K/V tiles before the wait on the "
                         "previous step (VH_FLAG_PDL_KV; each step reads another pool)")
    ap.add_argument("--pdl", type=int, default=1,
                    help="programmatic dependent launch between the timed fused steps (1/0; 0 also turns "
                         "off the early K/V requests)")
    ap.add_argument("--e2e-pdl", type=int, default=0,
                    help="programmatic dependent launch between the pipelined e2e steps (1/0)")
    ap.add_argument("--qk-norm", action="store_true",
                    help="per-head RMSNorm of q and the new key before RoPE (unit weights, eps 1e-6)")
    ap.add_argument("--layers", type=int, default=None,
                    help="layer calls per step (default: the workload's own count, 28 for 'high')")
    ap.add_argument("--ncu-case", action="store_true",
                    help="eager launches of the fused and the three-call step on one pool (profiling)")
    return ap.parse_args()


def dist_setup():
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
    try:
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, path: str | None = None):
    """DRAM bytes per launch of the fused kernel from the committed ncu summary,
    if that capture was taken of the current kernel sources; else None."""
    path = path or os.path.join(ROOT, "profiles", f"decode_fused_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    sha = re.search(r"kernel source sha256\[:16\]:\s*([0-9a-f]{16})", text)
    val = re.search(r"dram bytes per launch \(read \+ write\):\s*([0-9]+)", text)
    if not sha or not val or sha.group(1) != kernel_source_sha():
        return None
    return int(val.group(1))


def step_bytes(inp) -> dict:
    """Algorithmic bytes of one decode step: K/V of every active row (L_b keys), the
    new q/k/v, the appended k/v, the output, the page-table entries and the
    lengths/flags; plus the attention-only variant (fp32 q_rot instead of q/k/v)."""
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


class Setup:
    """Device buffers of one workload: KV pools and the step's outputs.

    One layer: R replicas of the pool, cycled so that their total exceeds 4x L2.
    Several layers (the high-concurrency workload has 28): one pool and one set
    of inputs per layer, each drawn with its own layer seed; a step runs all
    layers in order."""

    def __init__(self, name: str, rank: int, dev, replicas: int | None = None, layers: int | None = None,
                 qk_norm: bool = False, dtype: str = "bf16", interleaved: bool = False, layout: str = "NHD"):
        import paged_len_decode_gb300 as vh
        self.vh = vh
        self.L = layers or workloads.WORKLOADS[name].layers
        et = torch.float16 if dtype == "fp16" else torch.bfloat16
        if self.L > 1:
            self.layer_inputs = [workloads.make_inputs(name, layer=rank * self.L + l, device=dev, dtype=et,
                                                       layout=layout) for l in range(self.L)]
            inp = self.layer_inputs[0]
        else:
            self.layer_inputs = None
            inp = workloads.make_inputs(name, layer=rank, device=dev, dtype=et, layout=layout)
        self.inp = inp
        self.B, self.Hq, self.Hkv, self.D, self.P = inp.B, inp.Hq, inp.Hkv, inp.D, inp.P
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.pool_bytes = inp.pool.numel() * 2
        if self.layer_inputs:
            # one pool per layer; small layer sets are repeated (fresh copies)
            # until they exceed 4x L2, and a step cycles through them
            reps = replicas or max(1, math.ceil(4 * self.l2 / (self.L * self.pool_bytes)))
            self.pools = [li.pool for li in self.layer_inputs]
            self.pools += [li.pool.clone() for _ in range(reps - 1) for li in self.layer_inputs]
            self.R = self.L * reps
        else:
            self.R = replicas or max(2, math.ceil(4 * self.l2 / self.pool_bytes))
            self.pools = [inp.pool] + [inp.pool.clone() for _ in range(self.R - 1)]
        self.cos_sin = torch.empty((inp.max_pages_per_seq * self.P, self.D), dtype=torch.float32, device=dev)
        vh.vh_rope_table(self.cos_sin, inp.theta)
        self.q_rot = torch.empty((self.B, self.Hq, self.D), dtype=torch.float32, device=dev)
        self.out = torch.empty((self.B, self.Hq, self.D), dtype=et, device=dev)
        self.ws3 = vh.alloc_workspace(self.B, self.Hq, self.Hkv, self.D, self.P, device=dev)
        self.wsf = vh.alloc_workspace(self.B, self.Hq, self.Hkv, self.D, self.P, device=dev)
        self.n_ctas = vh.vh_decode_num_ctas(self.B, self.Hq, self.Hkv, self.D, self.P)
        self.pdl_kv = False
        self.norm = {"interleaved": interleaved}
        if qk_norm:
            w = torch.ones(self.D, dtype=torch.float32, device=dev)
            self.norm.update({"q_norm_w": w, "k_norm_w": w, "norm_eps": 1e-6})

    def inputs(self, r):
        return self.layer_inputs[r % self.L] if self.layer_inputs else self.inp

    def step_bytes(self) -> dict:
        if not self.layer_inputs:
            return step_bytes(self.inp)
        per = [step_bytes(li) for li in self.layer_inputs]
        return {k: (sum(x[k] for x in per) if k != "active" else per[0][k]) for k in per[0]}

    def kv(self, r):
        """[NP, P, Hkv, D] K and V views of pool r (strided unless token-major)."""
        pool = self.pools[r]
        if self.inp.layout == "CONTIG":
            return pool[0].transpose(1, 2), pool[1].transpose(1, 2)
        if self.inp.layout == "HND":
            return pool[:, 0].transpose(1, 2), pool[:, 1].transpose(1, 2)
        return pool[:, 0], pool[:, 1]

    def fused(self, r, pdl=True, src=None, out=None):
        s = src or self.inputs(r)
        k, v = self.kv(r)
        self.vh.vh_decode_fused(s.q, s.k_new, s.v_new, self.cos_sin, k, v, s.api_page_table, s.seq_lens,
                                s.active, self.out if out is None else out, self.wsf, pdl=pdl,
                                pdl_kv=pdl and self.pdl_kv, **self.norm)

    def three(self, r):
        i = self.inputs(r)
        k, v = self.kv(r)
        self.vh.decode_step(i.q, i.k_new, i.v_new, self.cos_sin, k, v,
                            i.api_page_table, i.seq_lens, i.active, self.q_rot, self.out, self.ws3, **self.norm)


def run_ncu_case(args):
    """A few eager launches on one pool: 3 fused, 3 three-call steps."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = Setup(args.workload, 0, dev, replicas=1, layers=1, dtype=args.dtype, interleaved=args.interleaved,
              layout=args.layout)
    for _ in range(3):
        s.fused(0, pdl=False)
    for _ in range(3):
        s.three(0)
    torch.cuda.synchronize()
    print(json.dumps({"ncu_case": args.workload, "ok": True}))


def e2e_measure(s, inp, R, by, args, world, dev, stream):
    """e2e through the public call with host buffers (one fused launch per step)."""
    # The step's inputs live in one pinned host arena and one device arena (the
    # way a serving runtime stages a step), so each step is one host->device
    # copy, the call, and one device->host copy of the output.
    names = ("q", "k_new", "v_new", "page_table", "seq_lens", "active")
    offs, total = {}, 0
    for k in names:
        t = getattr(inp, k)
        offs[k] = total
        total += -(-t.numel() * t.element_size() // 256) * 256
    h_arena = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for k in names:
        t = getattr(inp, k)
        n = t.numel() * t.element_size()
        h_arena[offs[k]:offs[k] + n].copy_(t.contiguous().view(torch.uint8).view(-1).cpu())

    def device_arena():
        d_arena = torch.zeros(total, dtype=torch.uint8, device=dev)
        views = {}
        for k in names:
            t = getattr(inp, k)
            n = t.numel() * t.element_size()
            views[k] = d_arena[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
        d_in = workloads.DecodeInputs(**{**{k: getattr(inp, k) for k in (
            "B", "Hq", "Hkv", "D", "P", "max_pages_per_seq", "num_pages", "theta", "pool", "layout")}, **views})
        return d_arena, d_in

    d_arenas, d_ins = zip(*[device_arena() for _ in range(2)])
    outs = [s.out, torch.empty_like(s.out)]
    h_outs = [torch.empty((s.B, s.Hq, s.D), dtype=s.out.dtype).pin_memory() for _ in range(2)]
    h2d = total
    d2h = h_outs[0].numel() * h_outs[0].element_size()
    K_e2e = min(args.steps, 2000)

    def e2e_step(r):
        d_arenas[0].copy_(h_arena, non_blocking=True)
        s.fused(r, pdl=False, src=d_ins[0])
        h_outs[0].copy_(s.out, non_blocking=True)

    def e2e_time(run, n, per):
        for i in range(3):
            run(i)
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(n):
            run(i)
        e1.record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        return max_over_ranks(max(e0.elapsed_time(e1), wall * 1e3), world) / (n * per)

    # eager: the Python call issued per step
    e2e_eager_ms = e2e_time(lambda i: e2e_step(i % R), K_e2e, 1)
    # one CUDA graph per step (host->device copy of the step's inputs, the
    # fused call, device->host copy of the output), replayed each step
    graphs = []
    for r in range(R):
        g = torch.cuda.CUDAGraph()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                e2e_step(r)
        torch.cuda.current_stream().wait_stream(stream)
        graphs.append(g)
    e2e_serial_ms = e2e_time(lambda i: graphs[i % R].replay(), K_e2e, 1)

    # pipelined serving pattern: two device input arenas and two outputs; the
    # host->device copy of step i+1 runs on its own stream while step i
    # computes, the device->host copy of step i on a third stream.  Every
    # step still copies its whole input arena in and its output out.
    M = R * max(1, 64 // R)  # steps per graph
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event() for _ in range(M)]
    k_done = [torch.cuda.Event() for _ in range(M)]
    d2h_done = [torch.cuda.Event() for _ in range(M)]
    gp = torch.cuda.CUDAGraph()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(gp, stream=stream):
            s_h2d.wait_stream(stream)
            s_d2h.wait_stream(stream)
            for i in range(M):
                b = i % 2
                with torch.cuda.stream(s_h2d):
                    if i >= 2:
                        s_h2d.wait_event(k_done[i - 2])  # step i-2 has read this arena
                    d_arenas[b].copy_(h_arena, non_blocking=True)
                    h2d_done[i].record(s_h2d)
                stream.wait_event(h2d_done[i])
                if i >= 2:
                    stream.wait_event(d2h_done[i - 2])  # this output has been copied out
                # programmatic dependent launch on the previous step's kernel: the
                # inputs this launch reads before its wait come from its own
                # copy, a full dependency
                s.fused(i % R, pdl=args.e2e_pdl, src=d_ins[b], out=outs[b])
                k_done[i].record(stream)
                with torch.cuda.stream(s_d2h):
                    s_d2h.wait_event(k_done[i])
                    h_outs[b].copy_(outs[b], non_blocking=True)
                    d2h_done[i].record(s_d2h)
            stream.wait_stream(s_h2d)
            stream.wait_stream(s_d2h)
    torch.cuda.current_stream().wait_stream(stream)
    e2e_ms = e2e_time(lambda i: gp.replay(), max(1, K_e2e // M), M)
    e2e_tps = by["active"] * world / (e2e_ms * 1e-3)

    return {"value": round(e2e_tps, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 6), "steps": max(1, K_e2e // M) * M,
            "call": "paged_len_decode_gb300.vh_decode_fused, one pinned-host->device copy of the step's "
                    "input arena and one device->host copy of its output per step; CUDA graph of "
                    f"{M} steps with two input arenas and two outputs, the copies on their own streams "
                    "overlapping the neighbouring steps' kernels"
                    + (", PDL between the kernels" if args.e2e_pdl else ""),
            "serial": {"value": round(by["active"] * world / (e2e_serial_ms * 1e-3), 1),
                       "ms_per_step": round(e2e_serial_ms, 6),
                       "call": "one CUDA graph per step: copy in, call, copy out, in order"},
            "eager": {"value": round(by["active"] * world / (e2e_eager_ms * 1e-3), 1),
                      "ms_per_step": round(e2e_eager_ms, 6)}}


def run_ours(args, rank, world):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = workloads.WORKLOADS[args.workload]
    s = Setup(args.workload, rank, dev, layers=args.layers, qk_norm=args.qk_norm, dtype=args.dtype,
              interleaved=args.interleaved, layout=args.layout)
    inp, R, L = s.inp, s.R, s.L
    s.pdl_kv = bool(args.pdl_kv) and bool(args.pdl) and R > 1  # consecutive steps read different pools
    by = s.step_bytes()

    for r in range(R):  # first calls outside capture (launch attributes, every replica's new slot)
        s.three(r)
        s.fused(r, pdl=False)
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
        return max_over_ranks(e0.elapsed_time(e1), world), ck

    for i in range(args.warmup):  # untimed warm-up steps
        s.fused(i % R)
        s.three(i % R)
    torch.cuda.synchronize()

    clocks = Clocks(dev.index)
    ms_fused_total, ck = timed(lambda r: s.fused(r, pdl=bool(args.pdl)), args.steps * L, clocks)  # L calls per step
    ms_step = ms_fused_total / args.steps
    ms_three_total, _ = timed(s.three, args.steps * L)
    ms_three = ms_three_total / args.steps

    tokens_per_s = by["active"] * world / (ms_step * 1e-3)
    step_gbs = by["step"] / (ms_step * 1e-3) / 1e9
    peak, peak_kind = peaks()

    e2e = None
    if L == 1:
        e2e = e2e_measure(s, inp, R, by, args, world, dev, stream)

    res = {
        "metric": METRIC, "value": round(tokens_per_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if args.dtype == "fp16" else "bf16",
        "accum_dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{args.workload}: B={s.B} (active {by['active']}), Hq={s.Hq}, Hkv={s.Hkv}, "
                               f"D={s.D}, P={s.P}, lengths {w.dist} [{w.len_lo},{w.len_hi}]",
                   "global_batch": s.B * world, "kv_bytes_per_step": by["kv"],
                   "step": (f"{L} layer calls, " if L > 1 else "") +
                           "one vh_decode_fused launch (RoPE+append+attention+merge) per layer call, " +
                           ("PDL between launches" if args.pdl else "no PDL between launches") +
                           (", first cached K/V tiles requested before the wait "
                                                     "(VH_FLAG_PDL_KV)" if s.pdl_kv else ""),
                   "layers": L, "qk_norm": bool(args.qk_norm), "rope": "interleaved" if args.interleaved
                   else "rotate-half", "elements": args.dtype, "pages": s.inp.layout,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": (f"{R} KV pools, one per layer call ({R // L} sets of {L} layers, "
                          f"{R * s.pool_bytes / 1e6:.0f} MB" if L > 1 else
                          f"{R} KV-pool replicas cycled ({R * s.pool_bytes / 1e6:.0f} MB")
                         + f" >= 4x L2 {s.l2 / 1e6:.0f} MB): inputs larger than L2",
                   "ctas": s.n_ctas},
        "hbm_gbs": round(step_gbs, 1), "hbm_frac_of_peak": round(step_gbs / peak, 4),
        "roofline": {"bound": "hbm", "kernel": f"decode_attn_kernel<{s.D},{s.Hq // s.Hkv},1,"
                               f"{'ElemF16' if args.dtype == 'fp16' else 'ElemBf16'}> (fused step)",
                     "achieved": round(step_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(step_gbs / peak, 4), "traffic": (recorded_traffic(args.workload)
                                                    if args.dtype == "bf16" and not args.interleaved
                                                    and s.inp.layout == "NHD" else None),
                     "peak_kind": peak_kind, "ms_per_launch": round(ms_step / L, 6),
                     "algorithmic_bytes_per_launch": by["step"] // L},
        "three_call": {"ms_per_step": round(ms_three, 6),
                       "value": round(by["active"] * world / (ms_three * 1e-3), 1), "unit": "tokens/s",
                       "launches_per_step": 3 * L},
        "clocks": ck,
        "e2e": e2e if e2e is not None else {"value": None, "unit": "tokens/s",
                                            "note": "measured for single-layer steps only"},
        "gpu_launches": args.steps * L,
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
    if args.ncu_case:
        run_ncu_case(args)
        return
    rank, world = dist_setup()
    if args.impl == "reference":
        if rank != 0:
            return
        inp = workloads.make_inputs(args.workload, device="cpu")
        cpu_oracle_rate(inp, 0, max_steps=max(3, args.warmup))
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
