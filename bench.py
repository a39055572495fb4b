"""Benchmark of the paged q_len=1 decode step (RoPE + append, attention, merge).

Headline workload: the c=64 Talker decode batch (64 rows, 16 q / 8 kv heads,
head_dim 128, pages of 16 tokens, lengths uniform in [200, 1200]).  A "step"
is the whole path for one layer over the batch (for the 28-layer workload,
all 28 layer calls).  The headline runs it as one launch (vh_decode_fused),
each step a programmatic dependent of the previous one; the same steps
without programmatic dependent launch (`no_pdl`) and the three-call form
(vh_rope_kv_append, vh_paged_decode_attn, vh_decode_combine) are timed
beside it.  Metric: decode tokens/s (active rows per layer call per second)
and the achieved HBM GB/s of the step, as a fraction of the measured copy
bandwidth and of the 8 TB/s HBM3e specification.  The default run also
measures the long-context, padded-batch and 28-layer high-concurrency
workloads (`workloads` in the JSON line).

Timing: inputs resident in HBM; the K steps of one replay are captured in a
CUDA graph that cycles over enough KV-pool replicas to exceed 4x the L2
size, so every step reads its K/V from HBM.  The graph is warmed by 3
replays, then replayed at least 20 times (and for about a second), each
replay bracketed by CUDA events on the launching stream; ms_per_step is the
median replay time / K.  A synchronize and a barrier bracket the whole timed
region, and the max over ranks is taken.  nvidia-smi samples the clocks
across all replays.  `e2e` goes through the public Python call with pinned
host buffers: per step the new q/k/v, lengths, flags and page table (one
input arena) move from host to device and the output back.  The headline
e2e lets each step's kernel read its inputs from the pinned host arena and
write its output to pinned host memory in place (VH_FLAG_HOST_IO, over the
NVLink-C2C link), in a CUDA graph of many steps linked by programmatic
dependent launch; `e2e.copies` copies the arena in and the output out with
copy operations on their own streams overlapping the neighbouring steps'
kernels, as a runtime without host I/O in the kernel pipelines its steps;
`e2e.serial` is one graph per step (copy in, call, copy out, in order) and
`e2e.eager` issues the same copies and call from Python each step.

`cpu_baseline` and --impl reference time the float64 CPU oracle as it
stands on whole steps of the same workload (every active row per call),
on all host cores and on one core, in the same tokens/s and GB/s columns;
`cpu_baseline.accuracy` compares the output of one timed fused step with
the oracle's.  Also in the line: the attention's flops (reported, not the
bound), the host-side warm-up times (first calls, graph capture, first
replay), an L2-hot side note (every launch on one pool) and the pages'
whole-pipeline serving figures as context.
--ncu-case runs a few eager launches on one pool only (for profiler
captures).
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
    ap.add_argument("--steps", type=int, default=240,
                    help="steps per timed graph replay (each replay is timed; the median is reported)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--replays", type=int, default=20, help="minimum number of timed replays")
    ap.add_argument("--seconds", type=float, default=1.0,
                    help="the timed replays of each measurement last at least about this long")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=list(workloads.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="oracle time on all host cores (the one-core sample gets the same budget)")
    ap.add_argument("--extra-workloads", default=None,
                    help="comma-separated workloads measured beside the headline (default with the c64 "
                         "headline and default options: long,padded,high; '' for none)")
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
    ap.add_argument("--e2e-pdl", type=int, default=1,
                    help="programmatic dependent launch between the pipelined e2e steps' kernels (1/0; each "
                         "kernel still waits for its own input copy)")
    ap.add_argument("--qk-norm", action="store_true",
                    help="per-head RMSNorm of q and the new key before RoPE (unit weights, eps 1e-6)")
    ap.add_argument("--layers", type=int, default=None,
                    help="layer calls per step (default: the workload's own count, 28 for 'high')")
    ap.add_argument("--ncu-case", action="store_true",
                    help="eager launches of the fused and the three-call step on one pool (profiling)")
    ap.add_argument("--planned", action="store_true",
                    help="with --ncu-case: the launches read a per-step plan (vh_decode_plan, written once)")
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
    lengths/flags; plus the attention-only variant (fp32 q_rot instead of q/k/v)
    and the attention's flops (reported beside the bytes, not the bound)."""
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
    flops = 4 * inp.Hq * inp.D * int(Lact.sum())  # q.K and p.V over every key of every q head
    return {"step": step, "attn": attn, "kv": kv, "active": Bact, "flops": flops}


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

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

    @classmethod
    def summarise(cls, lines) -> dict:
        """Median SM clock over the samples taken under load (GPU utilisation
        >= 50 %, or all samples if none is), and every throttle reason seen."""
        rows = []
        for line in lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                sm, smax = float(f[1]), float(f[2])
            except ValueError:
                continue
            try:
                util = float(f[9])
            except ValueError:
                util = -1.0
            try:
                pw = float(f[3])
            except ValueError:
                pw = None
            rows.append((sm, smax, util, pw, [n for n, v in zip(cls.NAMES, f[5:9]) if v.lower() == "active"]))
        loaded = [r for r in rows if r[2] >= 50.0]
        use = loaded or rows
        reasons = sorted({n for r in use for n in r[4]})
        pws = [r[3] for r in use if r[3] is not None]
        return {"sm_mhz": statistics.median(r[0] for r in use) if use else None,
                "sm_max_mhz": use[-1][1] if use else None, "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_median": round(statistics.median(pws), 1) if pws else None}

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        return self.summarise(out.strip().splitlines())


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

    def fused(self, r, pdl=True, src=None, out=None, planned=False, host_io=False):
        s = src or self.inputs(r)
        k, v = self.kv(r)
        self.vh.vh_decode_fused(s.q, s.k_new, s.v_new, self.cos_sin, k, v, s.api_page_table, s.seq_lens,
                                s.active, self.out if out is None else out, self.wsf, pdl=pdl,
                                pdl_kv=pdl and self.pdl_kv, planned=planned, host_io=host_io, **self.norm)

    def plan(self, r):
        """The step's work list for the fused launches (vh_decode_plan)."""
        s = self.inputs(r)
        k, _ = self.kv(r)
        self.vh.vh_decode_plan(s.seq_lens, s.active, s.api_page_table, self.wsf, Hq=self.Hq, Hkv=self.Hkv,
                               D=self.D, page_size=self.P, num_pages=k.shape[0],
                               max_pages_per_seq=s.max_pages_per_seq, max_pos=self.cos_sin.shape[0],
                               fp16=s.pool.dtype == torch.float16)

    def three(self, r):
        i = self.inputs(r)
        k, v = self.kv(r)
        self.vh.decode_step(i.q, i.k_new, i.v_new, self.cos_sin, k, v,
                            i.api_page_table, i.seq_lens, i.active, self.q_rot, self.out, self.ws3, **self.norm)


def run_ncu_case(args):
    """A few eager launches on one pool: 3 fused, 3 three-call steps (with
    --planned the fused launches read a plan written once before them)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = Setup(args.workload, 0, dev, replicas=1, layers=1, dtype=args.dtype, interleaved=args.interleaved,
              layout=args.layout)
    if args.planned:
        s.plan(0)
    for _ in range(3):
        s.fused(0, pdl=False, planned=args.planned)
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
    K_e2e = min(max(args.steps, 640), 2000)

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
                # programmatic dependent launch on the previous step's kernel
                # (which writes another pool and the other output): the inputs
                # this launch reads before its wait come from its own copy, a
                # full dependency of the launch
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

    # in place over the host link (VH_FLAG_HOST_IO): every step's kernel reads
    # the step's inputs from the pinned host arena and writes its output into
    # pinned host memory; no copy nodes, so no copy-to-kernel joins in the
    # graph, and each kernel is a programmatic dependent of the previous one
    h_views = {}
    for k in names:
        t = getattr(inp, k)
        n = t.numel() * t.element_size()
        h_views[k] = h_arena[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
    h_in = workloads.DecodeInputs(**{**{k: getattr(inp, k) for k in (
        "B", "Hq", "Hkv", "D", "P", "max_pages_per_seq", "num_pages", "theta", "pool", "layout")}, **h_views})
    io_bytes_in = sum(getattr(inp, k).numel() * getattr(inp, k).element_size() for k in names)
    s.fused(0, pdl=False, src=h_in, out=h_outs[0], host_io=True)
    torch.cuda.synchronize()
    gz = torch.cuda.CUDAGraph()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(gz, stream=stream):
            for i in range(M):
                s.fused(i % R, pdl=True, src=h_in, out=h_outs[i % 2], host_io=True)
    torch.cuda.current_stream().wait_stream(stream)
    io_ms = e2e_time(lambda i: gz.replay(), max(1, K_e2e // M), M)

    rate = lambda ms: round(by["active"] * world / (ms * 1e-3), 1)
    copies = {"value": rate(e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
              "ms_per_step": round(e2e_ms, 6), "steps": max(1, K_e2e // M) * M,
              "call": "paged_len_decode_gb300.vh_decode_fused, one pinned-host->device copy of the step's "
                      "input arena and one device->host copy of its output per step; CUDA graph of "
                      f"{M} steps with two input arenas and two outputs, the copies on their own streams "
                      "overlapping the neighbouring steps' kernels"
                      + (", PDL between the kernels" if args.e2e_pdl else "")}
    host_io = {"value": rate(io_ms), "unit": "tokens/s", "h2d_bytes_per_step": io_bytes_in,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(io_ms, 6), "steps": max(1, K_e2e // M) * M,
               "call": "paged_len_decode_gb300.vh_decode_fused with VH_FLAG_HOST_IO: each step's kernel reads "
                       "the step's inputs (q, k_new, v_new, page table, lengths, flags) from pinned host memory "
                       "and writes its output to pinned host memory, over the NVLink-C2C link; CUDA graph of "
                       f"{M} steps, PDL between the kernels"}
    return {**host_io, "copies": copies,
            "serial": {"value": rate(e2e_serial_ms), "ms_per_step": round(e2e_serial_ms, 6),
                       "call": "one CUDA graph per step: copy in, call, copy out, in order"},
            "eager": {"value": rate(e2e_eager_ms), "ms_per_step": round(e2e_eager_ms, 6)}}


SPEC_HBM_GBS = 8000.0  # HBM3e specification of a GB300 (about 8 TB/s)
EXTRA_WORKLOADS = ("long", "padded", "high")
# layer calls that share one per-step plan in a one-layer workload: the
# 28-layer Talker of the pages' c=64 serving figures (VoxCPM2's MiniCPM4 Talker)
PLAN_LAYERS = 28


def step_graphs(s, fn, K, stream, plan_every: int = 0):
    """CUDA graphs of K steps (K*L launches) that continue one cycle over the
    R pools: graph j starts at pool (j*K*L) mod R, so replaying the graphs in
    turn never reads the same pool in two consecutive launches.  plan_every >
    0: a vh_decode_plan launch before the first launch of each replay and then
    before every plan_every-th launch."""
    n_launch = K * s.L
    n_graphs = s.R // math.gcd(s.R, n_launch)
    graphs = []
    for j in range(n_graphs):
        start = (j * n_launch) % s.R
        g = torch.cuda.CUDAGraph()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(n_launch):
                    if plan_every and i % plan_every == 0:
                        s.plan((start + i) % s.R)
                    fn((start + i) % s.R)
        torch.cuda.current_stream().wait_stream(stream)
        graphs.append(g)
    return graphs


def time_replays(graphs, K, stream, world, min_replays, seconds):
    """Warm the graphs with 3 replays, then time at least `min_replays` replays
    (and about `seconds` of them), each bracketed by its own CUDA events on the
    launching stream.  Returns (median ms per step, mean ms per step, replays),
    the median taken as the max over ranks."""
    n_g = len(graphs)
    with torch.cuda.stream(stream):
        for i in range(max(3, n_g)):
            graphs[i % n_g].replay()
    torch.cuda.synchronize()
    # replay time estimate from 3 more replays
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(3):
            graphs[i % n_g].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    est = max(e0.elapsed_time(e1) / 3, 1e-3)
    n = int(min(200000, max(min_replays, math.ceil(seconds * 1e3 / est))))
    n = -(-n // n_g) * n_g
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(n):
            ev[i][0].record(stream)
            graphs[i % n_g].replay()
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    per_step = [a.elapsed_time(b) / K for a, b in ev]
    med = max_over_ranks(statistics.median(per_step), world)
    return med, statistics.fmean(per_step), n


def rates(by, ms_step, world, peak, L):
    """tokens/s, GB/s and fractions of one step time."""
    gbs = by["step"] / (ms_step * 1e-3) / 1e9
    return {"ms_per_step": round(ms_step, 6), "tokens_per_s": round(by["active"] * world / (ms_step * 1e-3), 1),
            "hbm_gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
            "frac_of_spec": round(gbs / SPEC_HBM_GBS, 4), "ms_per_launch": round(ms_step / L, 6),
            **({"tflops": round(by["flops"] / (ms_step * 1e-3) / 1e12, 3)} if "flops" in by else {})}


def workload_desc(name, s, by):
    w = workloads.WORKLOADS[name]
    return (f"{name}: B={s.B} (active {by['active']}), Hq={s.Hq}, Hkv={s.Hkv}, D={s.D}, P={s.P}, "
            f"lengths {w.dist} [{w.len_lo},{w.len_hi}]" + (f", {s.L} layer calls per step" if s.L > 1 else ""))


def l2_desc(s):
    return ((f"{s.R} KV pools, one per layer call ({s.R // s.L} sets of {s.L} layers, "
             f"{s.R * s.pool_bytes / 1e6:.0f} MB" if s.L > 1 else
             f"{s.R} KV-pool replicas cycled ({s.R * s.pool_bytes / 1e6:.0f} MB")
            + f" >= 4x L2 {s.l2 / 1e6:.0f} MB): inputs larger than L2")


def measure_workload(name, args, rank, world, dev, stream, *, headline: bool):
    """Build one workload's pools and time its fused step with programmatic
    dependent launch (and early K/V requests), the same steps without it,
    and (headline only) the three-call step and the end-to-end figures."""
    s = Setup(name, rank, dev, layers=args.layers if headline else None,
              qk_norm=args.qk_norm if headline else False, dtype=args.dtype if headline else "bf16",
              interleaved=args.interleaved if headline else False, layout=args.layout if headline else None)
    by = s.step_bytes()
    pdl = bool(args.pdl) if headline else True
    s.pdl_kv = (bool(args.pdl_kv) if headline else True) and pdl and s.R > 1  # consecutive launches read other pools
    # first calls outside capture (launch plan, tensor maps, module load,
    # every pool's new slot); the first of each form is timed on the host
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    s.fused(0, pdl=False)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    s.three(0)
    torch.cuda.synchronize()
    warm = {"first_fused_call_ms": round((t1 - t0) * 1e3, 3),
            "first_three_call_ms": round((time.perf_counter() - t1) * 1e3, 3)}
    for r in range(1, s.R):
        s.three(r)
        s.fused(r, pdl=False)
    t0 = time.perf_counter()
    for i in range(args.warmup * s.L):  # untimed warm-up steps
        s.fused(i % s.R)
        s.three(i % s.R)
    torch.cuda.synchronize()
    warm["warmup_steps_ms"] = round((time.perf_counter() - t0) * 1e3, 3)
    peak, _ = peaks()
    K = args.steps
    res = {"workload": workload_desc(name, s, by), "steps_per_replay": K, "layers": s.L,
           "algorithmic_bytes_per_step": by["step"], "kv_bytes_per_step": by["kv"], "l2": l2_desc(s),
           "ctas": s.n_ctas}
    t0 = time.perf_counter()
    g = step_graphs(s, lambda r: s.fused(r, pdl=pdl), K, stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    with torch.cuda.stream(stream):
        g[0].replay()
    torch.cuda.synchronize()
    warm.update({"graph_capture_ms": round((t1 - t0) * 1e3, 3), "graphs": len(g),
                 "first_replay_ms": round((time.perf_counter() - t1) * 1e3, 3)})
    med, mean, n = time_replays(g, K, stream, world, args.replays, args.seconds)
    del g
    if headline:
        # the output of the last timed launch (every pool holds the same
        # cache and every launch the same inputs), for the accuracy check
        # against the float64 oracle in the CPU-baseline leg
        torch.cuda.synchronize()
        res["_out"] = s.out.cpu()
    res.update(rates(by, med, world, peak, s.L))
    res["warmup_host_ms"] = warm
    res.update({"ms_per_step_mean": round(mean, 6), "replays": n, "pdl": pdl, "pdl_kv": s.pdl_kv,
                "traffic": (recorded_traffic(name) if (not headline or (args.dtype == "bf16" and not args.interleaved
                            and not args.qk_norm and s.inp.layout == "NHD")) else None)})
    if pdl:
        g = step_graphs(s, lambda r: s.fused(r, pdl=False), K, stream)
        med_np, mean_np, n_np = time_replays(g, K, stream, world, args.replays, args.seconds)
        del g
        res["no_pdl"] = {**rates(by, med_np, world, peak, s.L), "replays": n_np,
                         "step": "the same fused launches, each waiting for the previous one to complete"}
    # the same steps with the work list planned once per model step
    every = s.L if s.L > 1 else PLAN_LAYERS
    for key, pl in (("planned", pdl), ("planned_no_pdl", False)) if pdl else (("planned", False),):
        s.plan(0)
        s.fused(0, pdl=False, planned=True)
        torch.cuda.synchronize()
        g = step_graphs(s, lambda r, pl=pl: s.fused(r, pdl=pl, planned=True), K, stream, plan_every=every)
        med_p, _, n_p = time_replays(g, K, stream, world, args.replays, args.seconds)
        del g
        res[key] = {**rates(by, med_p, world, peak, s.L), "replays": n_p,
                    "step": (f"one vh_decode_plan launch per {every} layer calls (and at the start of each "
                             f"replay of {K * s.L}), the fused launches reading it (VH_FLAG_PLANNED)"
                             + (", PDL between the fused launches" if pl else ", no PDL"))}
    if headline:
        g = step_graphs(s, s.three, K, stream)
        med3, _, n3 = time_replays(g, K, stream, world, args.replays, args.seconds)
        del g
        res["three_call"] = {**rates(by, med3, world, peak, s.L), "replays": n3, "launches_per_step": 3 * s.L}
        res["e2e"] = (e2e_measure(s, s.inp, s.R, by, args, world, dev, stream) if s.L == 1 else
                      {"value": None, "unit": "tokens/s", "note": "measured for single-layer steps only"})
        if s.L == 1:
            res["l2_hot"] = l2_hot_measure(s, by, K, args, world, stream, pdl)
            res["stack"] = stack_measure(s, by, K, args, world, stream, peak)
        res["_setup"] = s
        res["_by"] = by
    else:
        del s
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return res


def stack_measure(s, by, K, args, world, stream, peak):
    """The fused step inside a layer stack: each step first runs a stand-in
    QKV projection (three cuBLAS GEMMs from a hidden state of Hq*D to q, k_new
    and v_new, weight replicas cycled beyond 4x L2 as a stack's per-layer
    weights would be), then the fused step reads the projections' outputs.
    The attention's cost in the stack is the step time minus that of the
    same GEMMs alone, with programmatic dependent launch on the GEMMs (the
    cached K/V requested before the wait), without it, and with PDL and the
    per-step plan (one vh_decode_plan per PLAN_LAYERS layer calls)."""
    dev, et = s.out.device, s.out.dtype
    hidden = s.Hq * s.D
    wbytes = hidden * (s.Hq + 2 * s.Hkv) * s.D * 2
    n_w = max(2, math.ceil(4 * s.l2 / wbytes))
    g = torch.Generator(device="cpu").manual_seed(20260777)
    x = (torch.randn(s.B, hidden, generator=g) * 0.5).to(dev, et)
    ws = [[(torch.randn(hidden, n * s.D, generator=g) * hidden ** -0.5).to(dev, et)
           for n in (s.Hq, s.Hkv, s.Hkv)] for _ in range(n_w)]
    q = torch.empty(s.B, s.Hq, s.D, dtype=et, device=dev)
    k_new = torch.empty(s.B, s.Hkv, s.D, dtype=et, device=dev)
    v_new = torch.empty_like(k_new)
    src = workloads.DecodeInputs(**{**{k: getattr(s.inp, k) for k in (
        "B", "Hq", "Hkv", "D", "P", "max_pages_per_seq", "num_pages", "theta", "pool", "layout", "page_table",
        "seq_lens", "active")}, "q": q, "k_new": k_new, "v_new": v_new})

    def proj(i):
        wq, wk, wv = ws[i % n_w]
        torch.matmul(x, wq, out=q.view(s.B, -1))
        torch.matmul(x, wk, out=k_new.view(s.B, -1))
        torch.matmul(x, wv, out=v_new.view(s.B, -1))

    def graph(with_attn, pdl, planned=False):
        proj(0)
        if planned:
            s.plan(0)
        if with_attn:
            s.fused(0, pdl=False, src=src, planned=planned)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            with torch.cuda.graph(gr, stream=stream):
                for i in range(K):
                    if planned and i % PLAN_LAYERS == 0:
                        s.plan(i % s.R)  # the step's work list, once per PLAN_LAYERS layer calls
                    proj(i)
                    if with_attn:
                        s.fused(i % s.R, pdl=pdl, src=src, planned=planned)
        torch.cuda.current_stream().wait_stream(stream)
        return [gr]

    out = {}
    pdl_kv, s.pdl_kv = s.pdl_kv, s.R > 1
    for key, fn in (("gemm_only", lambda: graph(False, False)), ("with_attn_pdl", lambda: graph(True, True)),
                    ("with_attn_no_pdl", lambda: graph(True, False)),
                    ("with_attn_planned_pdl", lambda: graph(True, True, planned=True))):
        gr = fn()
        out[key], _, _ = time_replays(gr, K, stream, world, args.replays, min(args.seconds, 0.5))
        del gr
    s.pdl_kv = pdl_kv
    res = {"gemm_ms_per_step": round(out["gemm_only"], 6), "weight_replicas": n_w,
           "note": "stand-in QKV projection (cuBLAS bf16 GEMMs, [B, Hq*D] x [Hq*D, (Hq+2*Hkv)*D], weights cycled "
                   "beyond 4x L2) before every fused step; attention cost = step minus the GEMMs alone"}
    for key, pl in (("pdl", "with_attn_pdl"), ("no_pdl", "with_attn_no_pdl"),
                    ("planned_pdl", "with_attn_planned_pdl")):
        attn = out[pl] - out["gemm_only"]
        r = rates(by, attn, world, peak, s.L)
        res[key] = {"step_ms": round(out[pl], 6), "attn_ms_per_step": r["ms_per_step"],
                    "hbm_gbs": r["hbm_gbs"], "frac_of_peak": r["frac_of_peak"], "frac_of_spec": r["frac_of_spec"]}
    return res


def l2_hot_measure(s, by, K, args, world, stream, pdl):
    """Side note: the same fused steps, every launch on the first pool, so the
    cache is read from L2 as far as it fits (no early K/V requests: each launch
    reads the slots the previous one appended)."""
    pdl_kv, s.pdl_kv = s.pdl_kv, False
    g = torch.cuda.CUDAGraph()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for _ in range(K * s.L):
                s.fused(0, pdl=pdl)
    torch.cuda.current_stream().wait_stream(stream)
    med, _, n = time_replays([g], K, stream, world, args.replays, min(args.seconds, 0.5))
    del g
    s.pdl_kv = pdl_kv
    r = rates(by, med, world, peaks()[0], s.L)
    return {"ms_per_step": r["ms_per_step"], "tokens_per_s": r["tokens_per_s"], "step_bytes_per_s_gbs": r["hbm_gbs"],
            "replays": n, "pool_mb": round(s.pool_bytes / 1e6, 1), "l2_mb": round(s.l2 / 1e6, 1),
            "note": "one pool re-read by every launch (L2-resident as far as it fits), without the early K/V "
                    "requests (each launch reads the slot the previous one appended), hence slower than the "
                    "steps cycling over pools in HBM that request their first tiles before the wait; a side "
                    "note, not the metric"}


# The pages' own figures are whole-pipeline TTS serving throughputs on other
# hardware ("Engineering TTS inference in vLLM-Omni", performance data
# section): printed beside the kernel numbers as context only.
PAGES_CONTEXT = {
    "note": "end-to-end TTS serving throughput (LM, sampler, codec, scheduler) on NVIDIA H20; context only, "
            "not kernel results and not comparable with tokens/s",
    "figures": [
        {"system": "VoxCPM2 (28-layer Talker, paged attention), with CFM batching", "value": 33.07,
         "unit": "audio-s/s", "hardware": "H20 x1", "concurrency": 64},
        {"system": "Fish Speech S2 Pro (q_len=1 decode-attention kernel)", "value": 23.72, "unit": "audio-s/s",
         "hardware": "H20 x1", "concurrency": 64},
        {"system": "Higgs Audio V3", "value": 35.26, "unit": "audio-s/s", "hardware": "H20 x1",
         "concurrency": 16},
    ],
}


def run_ours(args, rank, world):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    peak, peak_kind = peaks()
    default_variant = (args.dtype == "bf16" and not args.interleaved and not args.qk_norm and args.layout is None
                       and args.layers is None and args.pdl and args.pdl_kv)
    if args.extra_workloads is None:
        extras = list(EXTRA_WORKLOADS) if (args.workload == WORKLOAD and default_variant) else []
    else:
        extras = [x for x in args.extra_workloads.split(",") if x]

    clocks = Clocks(dev.index)
    clocks.start()
    h = measure_workload(args.workload, args, rank, world, dev, stream, headline=True)
    s, by = h.pop("_setup"), h.pop("_by")
    e2e = h.pop("e2e")
    gpu_out = h.pop("_out")
    inp_cpu = s.inp.to("cpu") if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    # the last timed launch is a call of the last layer (graphs start at a
    # multiple of the layer count and hold whole steps)
    check = {"inp": inp_cpu, "out": gpu_out, "out_inp": s.inputs(s.L - 1).to("cpu"),
             "opts": {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in s.norm.items()}} \
        if inp_cpu is not None else None
    del s
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    extra = {}
    for name in extras:
        if name == args.workload:
            continue
        extra[name] = measure_workload(name, args, rank, world, dev, stream, headline=False)
    ck = clocks.stop()

    w = workloads.WORKLOADS[args.workload]
    L = h["layers"]
    ms_step = h["ms_per_step"]
    kname = (f"decode_attn_kernel<{w.D},{w.Hq // w.Hkv},1,{'ElemF16' if args.dtype == 'fp16' else 'ElemBf16'}> "
             "(fused step)")
    n_replays = h["replays"]
    res = {
        "metric": METRIC, "value": h["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if args.dtype == "fp16" else "bf16",
        "accum_dtype": "f32", "data": "synthetic",
        "config": {"workload": h["workload"], "global_batch": w.B * world, "kv_bytes_per_step": by["kv"],
                   "step": (f"{L} layer calls, " if L > 1 else "") +
                           "one vh_decode_fused launch (RoPE+append+attention+merge) per layer call, " +
                           ("PDL between launches" if h["pdl"] else "no PDL between launches") +
                           (", first cached K/V tiles requested before the wait (VH_FLAG_PDL_KV)"
                            if h["pdl_kv"] else ""),
                   "timing": (f"CUDA graph of {args.steps} steps, warmed by 3 replays, then {n_replays} timed "
                              "replays, each bracketed by CUDA events on the launching stream; ms_per_step = "
                              "median replay time / steps"),
                   "layers": L, "qk_norm": bool(args.qk_norm), "rope": "interleaved" if args.interleaved
                   else "rotate-half", "elements": args.dtype, "pages": args.layout or w.layout,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": h["l2"], "ctas": h["ctas"]},
        "hbm_gbs": h["hbm_gbs"], "hbm_frac_of_peak": h["frac_of_peak"], "hbm_frac_of_spec": h["frac_of_spec"],
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": h["hbm_gbs"], "peak": peak, "unit": "GB/s",
                     "frac": h["frac_of_peak"], "traffic": h["traffic"], "peak_kind": peak_kind,
                     "spec_peak": SPEC_HBM_GBS, "frac_of_spec": h["frac_of_spec"],
                     "ms_per_launch": h["ms_per_launch"], "algorithmic_bytes_per_launch": by["step"] // L},
        "ms_per_step_mean": h["ms_per_step_mean"],
        "algorithmic_flops_per_step": by["flops"], "tflops": h.get("tflops"),
        "warmup_host_ms": h["warmup_host_ms"],
        "no_pdl": h.get("no_pdl"),
        "planned": h.get("planned"),
        "planned_no_pdl": h.get("planned_no_pdl"),
        "three_call": h["three_call"],
        "l2_hot": h.get("l2_hot"),
        "stack": h.get("stack"),
        "workloads": extra,
        "clocks": ck,
        "e2e": e2e,
        "gpu_launches": n_replays * args.steps * L,
        "pages_context": PAGES_CONTEXT,
    }
    return res, check


def cpu_oracle_steps(inp_cpu, *, seconds: float | None = None, max_steps: int | None = None,
                     threads: int | None = None):
    """Whole oracle steps on the workload: RoPE + append of every active row,
    then the attention of every row (OpenMP over rows and q heads).  Returns
    (steps/s, steps, seconds, threads used)."""
    import oracle

    if inp_cpu.layout != "NHD":
        inp_cpu = inp_cpu.as_nhd()
    before = oracle.num_threads()
    if threads is not None:
        oracle.set_num_threads(threads)
    try:
        used = oracle.num_threads()
        pool = inp_cpu.pool.contiguous().clone()
        n, t0 = 0, time.perf_counter()
        while True:
            q_rot, pool_after, _ = oracle.rope_kv_append(inp_cpu.q, inp_cpu.k_new, inp_cpu.v_new, pool,
                                                         inp_cpu.page_table, inp_cpu.seq_lens, inp_cpu.active,
                                                         P=inp_cpu.P, theta=inp_cpu.theta, in_place=True)
            oracle.decode_attn(q_rot, pool_after, inp_cpu.page_table, inp_cpu.seq_lens, inp_cpu.active, P=inp_cpu.P)
            n += 1
            el = time.perf_counter() - t0
            if (max_steps is not None and n >= max_steps) or (seconds is not None and el >= seconds):
                return n / el, n, el, used
    finally:
        oracle.set_num_threads(before)


def oracle_accuracy(inp_cpu, gpu_out, opts) -> dict:
    """The output of the last timed launch against the float64 oracle on the
    same inputs (its pool holds the same cache as the first), active rows,
    with the parity tolerance |gpu - ref| <= 2e-3 + 1e-2 |ref|."""
    import oracle

    ref = oracle.reference_step(inp_cpu.as_nhd(), q_norm_w=opts.get("q_norm_w"), k_norm_w=opts.get("k_norm_w"),
                                norm_eps=opts.get("norm_eps", 1e-6), interleaved=opts.get("interleaved", False))
    act = inp_cpu.active.bool()
    r, g = ref["out"].double()[act], gpu_out.double()[act]
    err = (g - r).abs()
    excess = err - (2e-3 + 1e-2 * r.abs())
    return {"vs": "float64 oracle, every active row of the last timed step", "max_abs_err": float(err.max()),
            "mean_abs_err": float(err.mean()), "worst_margin": float(excess.max()),
            "within_tolerance": bool((excess <= 0).all() and torch.isfinite(g).all()),
            "tolerance": "|gpu - ref| <= 2e-3 + 1e-2 |ref|"}


def cpu_baseline(inp_cpu, name, seconds: float, max_steps: int | None = None, all_cores=None, check=None):
    """The oracle on all host cores and on one core, in tokens/s and GB/s.
    all_cores: an (steps/s, steps, seconds, threads) result already taken;
    check: the GPU output of the timed step and its options, compared with
    the oracle's output (`accuracy`)."""
    by = step_bytes(inp_cpu)
    rate, n, el, cores = all_cores or cpu_oracle_steps(inp_cpu, seconds=seconds, max_steps=max_steps)
    rate1, n1, el1, _ = cpu_oracle_steps(inp_cpu, seconds=seconds, max_steps=max_steps, threads=1)
    extra = {"accuracy": oracle_accuracy(check["out_inp"], check["out"], check["opts"])} if check else {}
    return {**extra, "value": round(rate * by["active"], 3), "unit": "tokens/s", "cores": cores, "nproc": os.cpu_count(),
            "kind": "oracle", "hbm_gbs": round(rate * by["step"] / 1e9, 4), "ms_per_step": round(el / n * 1e3, 3),
            "sample": f"{n} whole oracle steps (RoPE+append+attention of all {by['active']} active rows) of the "
                      f"{name} workload in {el:.1f} s on {cores} threads; {n1} steps in {el1:.1f} s on 1 thread",
            "single_core": {"value": round(rate1 * by["active"], 3), "unit": "tokens/s", "cores": 1,
                            "hbm_gbs": round(rate1 * by["step"] / 1e9, 4), "ms_per_step": round(el1 / n1 * 1e3, 3)}}


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
        by = step_bytes(inp)
        cpu_oracle_steps(inp, max_steps=max(1, args.warmup))  # untimed warm-up steps
        rate, n, el, cores = cpu_oracle_steps(inp, max_steps=args.steps)
        cb = cpu_baseline(inp, args.workload, seconds=min(args.cpu_seconds, 5.0), max_steps=args.steps,
                          all_cores=(rate, n, el, cores))
        tps = rate * by["active"]
        res = {"impl": "reference", "metric": METRIC, "value": round(tps, 3), "unit": "tokens/s",
               "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
               "ms_per_step": round(el / n * 1e3, 4), "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "f64", "data": "synthetic",
               "hbm_gbs": round(rate * by["step"] / 1e9, 4),
               "config": {"workload": f"{args.workload} (whole steps: RoPE+append+attention of every active row)",
                          "global_batch": inp.B},
               "cpu_baseline": cb,
               "e2e": {"value": round(tps, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                       "d2h_bytes_per_step": 0}}
        print(json.dumps(res))
        return
    res, check = run_ours(args, rank, world)
    if check is not None:
        res["cpu_baseline"] = cpu_baseline(check["inp"], args.workload, args.cpu_seconds, check=check)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
