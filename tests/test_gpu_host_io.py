"""The fused step with its per-step inputs and output in pinned host memory
(VH_FLAG_HOST_IO), against the float64 oracle.

The kernel reads q, k_new, v_new, the lengths, flags, positions and page
table from host memory and writes its output there; the caches, the RoPE
table and the workspace stay on the device.  Checked on the serving
workloads, with a per-step plan, with fp16 and the RoPE / RMSNorm options,
and as a chain of launches linked by programmatic dependent launch inside a
CUDA graph (how the benchmark's end-to-end form runs it).
"""
import pytest
import torch

import gpu_harness as H
import oracle
import workloads

pytestmark = pytest.mark.gpu


def _pinned(t):
    return None if t is None else t.detach().cpu().contiguous().pin_memory()


def run_host_io(inp, *, planned=False, interleaved=False, norm=None, positions=None, pdl_chain=0):
    """One fused step (or pdl_chain + 1 launches on copies of the pool, in a
    CUDA graph) with host-memory inputs and output; returns (out, pool_after, err)."""
    v = H.vh()
    g = inp.to("cuda").clone()
    B, Hq, Hkv, D, P = g.B, g.Hq, g.Hkv, g.D, g.P
    cos_sin = torch.empty((g.max_pages_per_seq * P, D), dtype=torch.float32, device="cuda")
    v.vh_rope_table(cos_sin, g.theta)
    ws = v.alloc_workspace(B, Hq, Hkv, D, P, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hq, hk, hv = _pinned(g.q), _pinned(g.k_new), _pinned(g.v_new)
    hl, ha, hpos = _pinned(g.seq_lens), _pinned(g.active), _pinned(positions)
    hpt = None if g.api_page_table is None else _pinned(g.api_page_table)
    out = torch.full((B, Hq, D), float("nan"), dtype=g.pool.dtype).pin_memory()
    nq = nk = None
    eps = 1e-6
    if norm is not None:
        nq, nk, eps = norm["q"].to("cuda"), norm["k"].to("cuda"), norm["eps"]
    pools = [g.pool] + [g.pool.clone() for _ in range(pdl_chain)]

    def views(pool):
        if g.layout == "CONTIG":
            return pool[0].transpose(1, 2), pool[1].transpose(1, 2)
        if g.layout == "HND":
            return pool[:, 0].transpose(1, 2), pool[:, 1].transpose(1, 2)
        return pool[:, 0], pool[:, 1]

    def call(pool, pdl):
        k, vv = views(pool)
        v.vh_decode_fused(hq, hk, hv, cos_sin, k, vv, hpt, hl, ha, out, ws, positions=hpos, err_flag=err,
                          pdl=pdl, pdl_kv=pdl, q_norm_w=nq, k_norm_w=nk, norm_eps=eps, interleaved=interleaved,
                          planned=planned, host_io=True)

    if planned:
        v.vh_decode_plan(g.seq_lens, g.active, g.api_page_table, ws, Hq=Hq, Hkv=Hkv, D=D, page_size=P,
                         num_pages=views(g.pool)[0].shape[0], max_pages_per_seq=g.max_pages_per_seq,
                         positions=None if positions is None else positions.to("cuda", torch.int32),
                         max_pos=cos_sin.shape[0], fp16=g.pool.dtype == torch.float16)
    if pdl_chain:
        saved = [p.clone() for p in pools]
        for i, p in enumerate(pools):     # first calls outside the capture
            call(p, pdl=False)
        torch.cuda.synchronize()
        for p, s0 in zip(pools, saved):
            p.copy_(s0)
        out.fill_(float("nan"))
        cg = torch.cuda.CUDAGraph()
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            with torch.cuda.graph(cg, stream=st):
                for i, p in enumerate(pools):
                    call(p, pdl=i > 0)
        torch.cuda.current_stream().wait_stream(st)
        cg.replay()
    else:
        call(g.pool, pdl=False)
    torch.cuda.synchronize()
    g.pool = pools[-1]
    return out.clone(), g.nhd_pool().contiguous().cpu(), int(err.item())


@pytest.mark.parametrize("planned", [False, True])
@pytest.mark.parametrize("name", ["tiny", "c64", "padded", "long", "fastar"])
def test_host_io_workloads(name, planned):
    inp = workloads.make_inputs(name, device="cuda")
    cpu = inp.to("cpu").as_nhd()
    ref = oracle.reference_step(cpu)
    out, pool, err = run_host_io(inp, planned=planned)
    assert err == 0
    H.check_out(cpu, ref["out"], out)
    H.check_append(cpu, ref, pool)


def test_host_io_options():
    g = torch.Generator().manual_seed(71)
    norm = {"q": (1.0 + 0.2 * torch.randn(128, generator=g)).float(),
            "k": (1.0 + 0.2 * torch.randn(128, generator=g)).float(), "eps": 1e-6}
    inp = workloads.make_case(B=6, Hq=32, Hkv=8, D=128, P=16, seq_lens=[900, 1, 17, 300, 64, 2000],
                              active=[1, 1, 1, 0, 1, 1], seed=72, device="cuda", dtype=torch.float16, layout="HND")
    cpu = inp.to("cpu").as_nhd()
    ref = oracle.reference_step(cpu, q_norm_w=norm["q"], k_norm_w=norm["k"], norm_eps=norm["eps"], interleaved=True)
    out, pool, err = run_host_io(inp, interleaved=True, norm=norm)
    assert err == 0
    H.check_out(cpu, ref["out"], out)
    H.check_append(cpu, ref, pool, rel=H.MIDPOINT_REL_NORM, interleaved=True)


@pytest.mark.parametrize("name", ["c64", "long"])
def test_host_io_pdl_chain_in_a_graph(name):
    # three launches on three copies of the pool, each a programmatic
    # dependent of the previous one, inputs read from host memory: the last
    # launch's output and cache must match the oracle
    inp = workloads.make_inputs(name, device="cuda")
    cpu = inp.to("cpu").as_nhd()
    ref = oracle.reference_step(cpu)
    out, pool, err = run_host_io(inp, pdl_chain=2)
    assert err == 0
    H.check_out(cpu, ref["out"], out)
    H.check_append(cpu, ref, pool)
