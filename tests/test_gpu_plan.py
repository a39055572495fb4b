"""The per-step plan (vh_decode_plan) and 8-token pages, against the float64 oracle.

A plan is written once per decode step and read by every attention launch of
that step (each layer's call on its own KV pool).  Checked here: both paths
on every workload with a plan, one plan reused by the 28 layer calls of a
high-concurrency step (programmatic dependent launches between them, as a
model runs them), plans that do not match the launch (another CTA count,
the other path, none written) being ignored, and the data-error flags the
plan raises, and the benchmark's chain (one plan, then layer launches
linked by programmatic dependent launch) captured in a CUDA graph, and
plans that change from step to step read by the programmatic dependent
launched right after each plan.  Pages of
8 tokens (every 16-token tile spans two pages) are checked on both paths,
both page layouts, with and without a plan.
"""
import pytest
import torch

import gpu_harness as H
import oracle
import workloads

pytestmark = pytest.mark.gpu


def case(lens, *, active=None, Hq=8, Hkv=2, D=128, P=16, seed=1, mps=None, **kw):
    return workloads.make_case(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, P=P, seq_lens=lens, active=active,
                               max_pages_per_seq=mps, seed=seed, device="cuda", **kw)


# ---------------------------------------------------------------- planned launches

@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("name", ["tiny", "c64", "padded", "long", "high", "fastar"])
def test_planned_workload_parity(name, path):
    inp = workloads.make_inputs(name, device="cuda")
    H.full_check(inp, path=path, planned=True, rows=list(range(0, inp.B, 4)) if name == "high" else None)


@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("name", ["c64", "padded", "long"])
def test_planned_fused_with_early_kv_and_repeats(name, graph):
    inp = workloads.make_inputs(name, device="cuda")
    H.full_check(inp, path="fused", planned=True, pdl=True, pdl_kv=True, graph=graph, repeat=3)


@pytest.mark.parametrize("path", H.PATHS)
def test_planned_edge_cases(path):
    for inp in (case([1, 1, 1], seed=40), case([16, 32, 4096, 1, 17], seed=41),
                case([200, 1, 500], active=[1, 0, 1], seed=42), case([1], active=[0], seed=43)):
        H.full_check(inp, path=path, planned=True)
    for n in (1, 3, 1000):
        H.full_check(case([300, 17, 1200, 5], Hq=16, Hkv=8, seed=44), path=path, planned=True, num_ctas=n)


def _layer_step(path, L, rows_every):
    """One plan, then L layer calls of the high-concurrency step (each layer
    its own pool, q, k and v; one batch).  Returns the per-layer outputs and
    pools after the step."""
    v = H.vh()
    layers = [workloads.make_inputs("high", layer=l, device="cuda") for l in range(L)]
    g0 = layers[0]
    B, Hq, Hkv, D, P = g0.B, g0.Hq, g0.Hkv, g0.D, g0.P
    cos_sin = torch.empty((g0.max_pages_per_seq * P, D), dtype=torch.float32, device="cuda")
    v.vh_rope_table(cos_sin, g0.theta)
    ws = v.alloc_workspace(B, Hq, Hkv, D, P, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_rot = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    outs = [torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    v.vh_decode_plan(g0.seq_lens, g0.active, g0.page_table, ws, Hq=Hq, Hkv=Hkv, D=D, page_size=P,
                     num_pages=g0.num_pages, max_pos=cos_sin.shape[0], err_flag=err, three_call=path == "three")
    for l, li in enumerate(layers):
        if path == "fused":
            # each launch a programmatic dependent of the previous layer's, its
            # first cached tiles requested before the wait (another pool)
            v.vh_decode_fused(li.q, li.k_new, li.v_new, cos_sin, li.pool[:, 0], li.pool[:, 1], g0.page_table,
                              g0.seq_lens, g0.active, outs[l], ws, err_flag=err, pdl=l > 0, pdl_kv=l > 0,
                              planned=True)
        else:
            v.decode_step(li.q, li.k_new, li.v_new, cos_sin, li.pool[:, 0], li.pool[:, 1], g0.page_table,
                          g0.seq_lens, g0.active, q_rot, outs[l], ws, err_flag=err, planned=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = list(range(0, B, rows_every))
    for l, li in enumerate(layers):
        fresh = workloads.make_inputs("high", layer=l, device="cuda").to("cpu")
        ref = oracle.reference_step(fresh, rows=rows)
        H.check_out(fresh, ref["out"], outs[l].cpu(), rows=rows)
        if l in (0, L - 1):
            H.check_append(fresh, ref, li.pool.cpu())
        del fresh, ref
        layers[l] = None


@pytest.mark.parametrize("path", H.PATHS)
def test_one_plan_reused_by_the_28_layer_calls_of_a_step(path):
    _layer_step(path, 28, rows_every=16)


def test_plan_that_does_not_match_the_launch_is_ignored():
    v = H.vh()
    inp = case([300, 17, 1200, 5, 64], Hq=16, Hkv=8, seed=45)
    cpu = inp.to("cpu")
    ref = oracle.reference_step(cpu)
    for plan_kw, call in [({"num_ctas": 7}, {"num_ctas": 0}),          # another CTA count
                          ({"three_call": True}, {}),                  # planned for the other path
                          (None, {})]:                                 # never planned
        g = inp.clone()
        B, Hq, Hkv, D, P = g.B, g.Hq, g.Hkv, g.D, g.P
        cos_sin = torch.empty((g.max_pages_per_seq * P, D), dtype=torch.float32, device="cuda")
        v.vh_rope_table(cos_sin, g.theta)
        ws = v.alloc_workspace(B, Hq, Hkv, D, P, 7, device="cuda")
        ws_auto = v.vh_decode_workspace_bytes(B, Hq, Hkv, D, P)
        if ws.numel() < ws_auto:
            ws = torch.zeros(ws_auto, dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        if plan_kw is not None:
            v.vh_decode_plan(g.seq_lens, g.active, g.page_table, ws, Hq=Hq, Hkv=Hkv, D=D, page_size=P,
                             num_pages=g.num_pages, max_pos=cos_sin.shape[0], err_flag=err, **plan_kw)
        v.vh_decode_fused(g.q, g.k_new, g.v_new, cos_sin, g.pool[:, 0], g.pool[:, 1], g.page_table, g.seq_lens,
                          g.active, out, ws, err_flag=err, planned=True, **call)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        H.check_out(cpu, ref["out"], out.cpu())
        H.check_append(cpu, ref, g.pool.cpu())


@pytest.mark.parametrize("path", H.PATHS)
def test_plan_flags_bad_lengths_and_positions(path):
    inp = case([50, 60, 70], seed=46)
    inp.seq_lens[1] = inp.max_pages_per_seq * inp.P + 5
    got = H.run_step(inp, path=path, planned=True)
    assert got["err"] & 1
    assert not got["out"][1].any()
    inp = case([20, 30], seed=47)
    got = H.run_step(inp, positions=torch.tensor([3, 10_000], dtype=torch.int32), max_pos=64, path=path,
                     planned=True)
    assert got["err"] & 4
    if path == "fused":
        assert not got["out"][1].any(), "a row with an invalid position is treated as padding"


# ---------------------------------------------------------------- 8-token pages

@pytest.mark.parametrize("planned", [False, True])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("path", H.PATHS)
def test_eight_token_pages(path, layout, planned):
    # lengths on and around page and tile boundaries: a tile's second page
    # missing (<= 8 live tokens), present, and the new token in either page
    for lens, seed in ([1, 7, 8, 9, 15, 16, 17, 24, 25, 300], 50), ([1023, 512, 33, 2], 51):
        inp = case(lens, P=8, Hq=16, Hkv=8, seed=seed, layout=layout)
        H.full_check(inp, path=path, planned=planned)
    inp = case([100, 9, 64], P=8, Hq=8, Hkv=8, D=64, seed=52, layout=layout, dtype=torch.float16)
    H.full_check(inp, path=path, planned=planned, interleaved=True)


@pytest.mark.parametrize("path", H.PATHS)
def test_eight_token_pages_split_rows_and_early_kv(path):
    inp = case([4000, 3, 2500], P=8, Hq=32, Hkv=8, seed=53)
    H.full_check(inp, path=path, num_ctas=200)
    if path == "fused":
        H.full_check(inp, path=path, pdl=True, pdl_kv=True, graph=True, repeat=2, planned=True)


def test_plan_and_layer_chain_captured_in_a_graph():
    # the chain the benchmark times: one plan, then four layers' fused launches
    # (each its own pool, one batch), each a programmatic dependent of the
    # previous with its first K/V tiles requested before the wait, captured
    # in a CUDA graph and replayed twice
    v = H.vh()
    base = workloads.make_inputs("c64", device="cuda")
    layers = []
    for l in range(4):
        li = base.clone()
        g = torch.Generator(device="cuda").manual_seed(900 + l)
        live = ~torch.isnan(li.pool.float())
        li.pool[live] = torch.randn(int(live.sum()), generator=g, device="cuda").to(li.pool.dtype)
        li.q.copy_(torch.randn(li.q.shape, generator=g, device="cuda").to(li.q.dtype))
        li.k_new.copy_(torch.randn(li.k_new.shape, generator=g, device="cuda").to(li.k_new.dtype))
        li.v_new.copy_(torch.randn(li.v_new.shape, generator=g, device="cuda").to(li.v_new.dtype))
        layers.append(li)
    refs = [oracle.reference_step(li.to("cpu")) for li in layers]
    B, Hq, Hkv, D, P = base.B, base.Hq, base.Hkv, base.D, base.P
    cos_sin = torch.empty((base.max_pages_per_seq * P, D), dtype=torch.float32, device="cuda")
    v.vh_rope_table(cos_sin, base.theta)
    ws = v.alloc_workspace(B, Hq, Hkv, D, P, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in layers]
    pools0 = [li.pool.clone() for li in layers]

    def step():
        v.vh_decode_plan(base.seq_lens, base.active, base.page_table, ws, Hq=Hq, Hkv=Hkv, D=D, page_size=P,
                         num_pages=base.num_pages, max_pos=cos_sin.shape[0], err_flag=err)
        for l, li in enumerate(layers):
            v.vh_decode_fused(li.q, li.k_new, li.v_new, cos_sin, li.pool[:, 0], li.pool[:, 1], base.page_table,
                              base.seq_lens, base.active, outs[l], ws, err_flag=err, pdl=l > 0, pdl_kv=l > 0,
                              planned=True)

    step()  # first calls outside the capture
    torch.cuda.synchronize()
    cg = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(cg, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        for l, li in enumerate(layers):
            li.pool.copy_(pools0[l])
            outs[l].fill_(float("nan"))
        cg.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for l, li in enumerate(layers):
            cpu = li.to("cpu")
            H.check_out(cpu, refs[l]["out"], outs[l].cpu())
            H.check_append(cpu, refs[l], li.pool.cpu())  # (uses the lengths, flags and page table only)


@pytest.mark.parametrize("graph", [False, True])
def test_alternating_plans_read_by_programmatic_dependents(graph):
    # every step writes a new plan (other lengths, flags and page table, same
    # shape) and the fused launch right after it is its programmatic
    # dependent, which reads the plan before its own wait (with its first K/V
    # tiles requested there too): a plan not yet visible would put the other
    # step's tile ranges and page ids on this step's cache
    v = H.vh()
    steps = [case([700, 1, 300, 1200, 64, 900, 17, 450], active=[1, 1, 1, 1, 0, 1, 1, 1], Hq=16, Hkv=8,
                  seed=71, mps=80),
             case([33, 1100, 1, 512, 980, 5, 640, 256], active=[1, 1, 0, 1, 1, 1, 1, 1], Hq=16, Hkv=8,
                  seed=72, mps=80)]
    refs = [oracle.reference_step(st.to("cpu")) for st in steps]
    B, Hq, Hkv, D, P = 8, 16, 8, 128, 16
    cos_sin = torch.empty((80 * P, D), dtype=torch.float32, device="cuda")
    v.vh_rope_table(cos_sin, steps[0].theta)
    ws = v.alloc_workspace(B, Hq, Hkv, D, P, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in steps]
    pools0 = [st.pool.clone() for st in steps]

    def run(order):
        for i in order:
            st = steps[i]
            v.vh_decode_plan(st.seq_lens, st.active, st.page_table, ws, Hq=Hq, Hkv=Hkv, D=D, page_size=P,
                             num_pages=st.num_pages, max_pos=cos_sin.shape[0], err_flag=err)
            v.vh_decode_fused(st.q, st.k_new, st.v_new, cos_sin, st.pool[:, 0], st.pool[:, 1], st.page_table,
                              st.seq_lens, st.active, outs[i], ws, err_flag=err, pdl=True, pdl_kv=True,
                              planned=True)

    def check():
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for i, st in enumerate(steps):
            cpu = st.to("cpu")
            H.check_out(cpu, refs[i]["out"], outs[i].cpu())
            H.check_append(cpu, refs[i], st.pool.cpu())

    if not graph:
        run([0, 1, 0, 1, 1, 0])  # appends rewrite the same slots with the same values
        check()
        return
    run([0, 1])  # first calls outside the capture
    torch.cuda.synchronize()
    cg = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(cg, stream=s):
            run([0, 1, 1, 0, 1])
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        for i, st in enumerate(steps):
            st.pool.copy_(pools0[i])
            outs[i].fill_(float("nan"))
        cg.replay()
        check()


@pytest.mark.parametrize("path", H.PATHS)
def test_many_pieces_fp16_interleaved_rmsnorm(path):
    # the staged merge of many pieces with fp16 outputs, next to the other options
    g = torch.Generator().manual_seed(61)
    norm = {"q": (1.0 + 0.2 * torch.randn(128, generator=g)).float(),
            "k": (1.0 + 0.2 * torch.randn(128, generator=g)).float(), "eps": 1e-6}
    inp = case([2500, 900, 3], Hq=16, Hkv=4, D=128, seed=62, dtype=torch.float16, layout="HND")
    H.full_check(inp, path=path, num_ctas=80, interleaved=True, norm=norm)
