"""Helpers for the GPU tests: run the CUDA path through the C interface and
compare it with the float64 oracle on the same seeded inputs.

Tolerance for float outputs (the attention output, bf16 or fp16): elementwise
|gpu - ref| <= 2e-3 + 1e-2 * |ref|.  The rotated q (fp32) must agree to
1e-5 + 1e-5 * |ref| (fp32 RoPE with fp32 cos/sin against float64).  The KV
append must be bit-exact, except rotated-key elements whose float64 value
lies within the fp32 rotation's error bound of a rounding midpoint of the
element type (bf16 or fp16),
where fp32 and float64 rotation may round to different neighbours.  For
x' = x_i cos - x_{i+D/2} sin computed in fp32 (cos/sin rounded to fp32, two
products, one subtraction) the error is below 3 * 2^-24 * (|x_i| + |x_{i+D/2}|);
the exemption window is 2^-21 * (|x_i| + |x_{i+D/2}|), a margin of about 2.7.
"""
from __future__ import annotations

import torch

import oracle

ATOL, RTOL = 2e-3, 1e-2
QROT_ATOL, QROT_RTOL = 1e-5, 1e-5
MIDPOINT_REL = 2.0 ** -21
MIDPOINT_REL_NORM = 2.0 ** -20  # with the RMSNorm before RoPE (a few more fp32 roundings)


def vh():
    import paged_len_decode_gb300 as v
    return v


PATHS = ("three", "fused")


def run_step(inp, *, path="three", num_ctas=0, positions=None, sm_scale=0.0, max_pos=None, graph=False,
             repeat=1, pdl=False, norm=None, interleaved=False, pdl_kv=False, planned=False, host_io=False):
    """Run one decode step on `inp` (CPU or CUDA DecodeInputs) through the C interface.

    path "three": vh_rope_kv_append + vh_paged_decode_attn + vh_decode_combine;
    path "fused": vh_decode_fused (one launch; q_rot is not produced).
    planned: vh_decode_plan once, then the attention launches take their
    work list from it (all `repeat` calls share the one plan).
    host_io (fused path): q, k_new, v_new, the lengths, flags, positions,
    page table and the output are pinned host memory the kernel reads and
    writes in place (VH_FLAG_HOST_IO).
    Returns dict(q_rot, out, pool_after, err) on the CPU (pool_after token-major);
    `inp` is not modified.
    """
    v = vh()
    dev = torch.device("cuda")
    g = inp.to(dev).clone()
    B, Hq, Hkv, D, P = g.B, g.Hq, g.Hkv, g.D, g.P
    max_pos = max_pos or g.max_pages_per_seq * P
    cos_sin = torch.empty((max_pos, D), dtype=torch.float32, device=dev)
    v.vh_rope_table(cos_sin, g.theta)
    q_rot = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=dev)
    out = torch.full((B, Hq, D), float("nan"), dtype=g.pool.dtype, device=dev)
    ws = v.alloc_workspace(B, Hq, Hkv, D, P, num_ctas, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pos = positions.to(dev, torch.int32) if positions is not None else None
    k_cache, v_cache = g.k_cache(), g.v_cache()   # [NP, P, Hkv, D] views of either page layout
    nq = nk = None
    eps = 1e-6
    if norm is not None:
        nq = None if norm["q"] is None else norm["q"].to(dev)
        nk = None if norm["k"] is None else norm["k"].to(dev)
        eps = norm["eps"]

    def plan():
        v.vh_decode_plan(g.seq_lens, g.active, g.api_page_table, ws, Hq=Hq, Hkv=Hkv, D=D, page_size=P,
                         num_pages=k_cache.shape[0], max_pages_per_seq=g.max_pages_per_seq, positions=pos,
                         max_pos=max_pos, num_ctas=num_ctas, err_flag=err, fp16=g.pool.dtype == torch.float16,
                         three_call=path != "fused")

    fin = {"q": g.q, "k_new": g.k_new, "v_new": g.v_new, "pt": g.api_page_table, "lens": g.seq_lens,
           "act": g.active, "pos": pos}
    if host_io:
        assert path == "fused"
        fin = {k: None if t is None else t.cpu().contiguous().pin_memory() for k, t in fin.items()}
        out = out.cpu().pin_memory()

    def step():
        if planned:
            plan()
        for _ in range(repeat):
            if path == "fused":
                v.vh_decode_fused(fin["q"], fin["k_new"], fin["v_new"], cos_sin, k_cache, v_cache, fin["pt"],
                                  fin["lens"], fin["act"], out, ws, positions=fin["pos"], sm_scale=sm_scale,
                                  num_ctas=num_ctas, err_flag=err, pdl=pdl, q_norm_w=nq, k_norm_w=nk, norm_eps=eps,
                                  interleaved=interleaved, pdl_kv=pdl_kv, planned=planned, host_io=host_io)
            else:
                v.decode_step(g.q, g.k_new, g.v_new, cos_sin, k_cache, v_cache, g.api_page_table, g.seq_lens,
                              g.active, q_rot, out, ws, positions=pos, sm_scale=sm_scale, num_ctas=num_ctas,
                              err_flag=err, q_norm_w=nq, k_norm_w=nk, norm_eps=eps, interleaved=interleaved,
                              planned=planned)

    if graph:
        # first call outside capture (sets per-device launch attributes)
        step()
        torch.cuda.synchronize()
        out.fill_(float("nan"))
        cg = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(cg, stream=s):
                step()
        torch.cuda.current_stream().wait_stream(s)
        cg.replay()
    else:
        step()
    torch.cuda.synchronize()
    # pool_after in token-major order whatever the layout, for comparison with the oracle
    return {"q_rot": q_rot.cpu(), "out": out.cpu(), "pool_after": g.nhd_pool().contiguous().cpu(),
            "err": int(err.item())}


def bits16(t):
    return t.contiguous().view(torch.int16).to(torch.int32) & 0xFFFF


# significand bits and smallest quantum (subnormal step) of the 16-bit types
_GRID = {torch.bfloat16: (8, -133), torch.float16: (11, -24)}


def midpoint_mask(x: torch.Tensor, k_in: torch.Tensor, rel: float = MIDPOINT_REL,
                  dtype=torch.bfloat16, interleaved: bool = False) -> torch.Tensor:
    """Elements of the rotated keys x (float64 [..., D]) that lie within the fp32
    rotation error bound of a rounding midpoint of `dtype`; k_in are the keys
    fed to the rotation, whose pair magnitudes set the bound (pairs (i, i+D/2),
    or (2i, 2i+1) when interleaved)."""
    bits, qmin = _GRID[dtype]
    ax = x.abs()
    nz = ax > 0
    e = torch.frexp(torch.where(nz, ax, torch.ones_like(ax))).exponent
    ulp = torch.ldexp(torch.ones_like(ax), (e - bits).clamp(min=qmin))
    frac = torch.remainder(ax / ulp, 1.0)
    k = k_in.double().abs()
    if interleaved:
        pair = k[..., 0::2] + k[..., 1::2]
        scale = torch.stack([pair, pair], dim=-1).flatten(-2)
    else:
        h = k.shape[-1] // 2
        pair = k[..., :h] + k[..., h:]
        scale = torch.cat([pair, pair], dim=-1)
    return nz & ((frac - 0.5).abs() * ulp <= rel * scale)


def check_append(inp, ref, gpu_pool, rel=MIDPOINT_REL, interleaved=False):
    """Bit-exact placement: pool after the GPU append == pool after the oracle append,
    except midpoint-exempt rotated-key elements.  Returns (number of exempt
    elements, number that actually differ)."""
    a, b = bits16(gpu_pool), bits16(ref["pool_after"])
    diff = a != b
    if not diff.any():
        return 0, 0
    # allowed differences: K elements of appended slots whose float64 value is a near-midpoint
    allowed = torch.zeros_like(diff)
    act = inp.active.cpu().bool()
    lens = inp.seq_lens.cpu()
    pt = inp.page_table.cpu()
    mid = midpoint_mask(ref["k_rot"], ref["k_pre"], rel, dtype=gpu_pool.dtype, interleaved=interleaved)
    n = 0
    for bb in torch.nonzero(act).flatten().tolist():
        L = int(lens[bb])
        page, off = int(pt[bb, (L - 1) // inp.P]), (L - 1) % inp.P
        allowed[page, 0, off] |= mid[bb]
        n += int(mid[bb].sum())
    bad = diff & ~allowed
    assert not bad.any(), f"{int(bad.sum())} pool elements differ outside the midpoint exemption, " \
                          f"first at {torch.nonzero(bad)[0].tolist()}"
    # and every differing element is the rounding of a value within the fp32
    # error window of the exact rotated key: |gpu - exact| <= window + one step
    # of the element type (near zero, after cancellation, that may be several
    # bit patterns away, or the other sign)
    bits_, qmin = _GRID[gpu_pool.dtype]
    k = ref["k_pre"].double().abs()
    if interleaved:
        pair = k[..., 0::2] + k[..., 1::2]
        scale = torch.stack([pair, pair], dim=-1).flatten(-2)
    else:
        h = k.shape[-1] // 2
        pair = k[..., :h] + k[..., h:]
        scale = torch.cat([pair, pair], dim=-1)
    for bb in torch.nonzero(act).flatten().tolist():
        L = int(lens[bb])
        page, off = int(pt[bb, (L - 1) // inp.P]), (L - 1) % inp.P
        dd = diff[page, 0, off]
        if not dd.any():
            continue
        got = gpu_pool[page, 0, off].double()[dd]
        exact = ref["k_rot"][bb][dd]
        mag = torch.maximum(got.abs(), exact.abs())
        e = torch.frexp(torch.where(mag > 0, mag, torch.ones_like(mag))).exponent
        step = torch.ldexp(torch.ones_like(mag), (e - bits_).clamp(min=qmin))
        assert ((got - exact).abs() <= rel * scale[bb][dd] + step).all(), \
            f"row {bb}: an exempt element is further than the window from the exact key"
    return n, int(diff.sum())


def check_out(inp, ref_out, gpu_out, rows=None):
    act = inp.active.cpu().bool()
    rows = list(range(inp.B)) if rows is None else rows
    got = gpu_out.double()
    for_rows = torch.tensor(rows, dtype=torch.long)
    a = act[for_rows]
    live = for_rows[a]
    dead = for_rows[~a]
    if len(dead):
        assert torch.equal(gpu_out[dead], torch.zeros_like(gpu_out[dead])), "padding rows must be zero"
    if len(live):
        g_, r_ = got[live], ref_out[live]
        assert torch.isfinite(g_).all(), "non-finite output in a live row"
        err = (g_ - r_).abs()
        tol = ATOL + RTOL * r_.abs()
        worst = (err - tol).max().item()
        assert worst <= 0, f"max |d| {err.max().item():.3e} exceeds tolerance by {worst:.3e}"
        return err.max().item()
    return 0.0


def check_q_rot(inp, ref_q_rot, gpu_q_rot):
    act = inp.active.cpu().bool()
    g_, r_ = gpu_q_rot[act].double(), ref_q_rot[act]
    if g_.numel() == 0:
        return 0.0
    err = (g_ - r_).abs()
    assert (err <= QROT_ATOL + QROT_RTOL * r_.abs()).all(), f"q_rot max |d| {err.max().item():.3e}"
    return err.max().item()


def full_check(inp, *, path="three", num_ctas=0, rows=None, positions=None, sm_scale=0.0, graph=False,
               max_pos=None, repeat=1, pdl=False, norm=None, interleaved=False, pdl_kv=False, planned=False,
               host_io=False):
    """Run the GPU path and the oracle on `inp`; check q_rot (three-call path),
    the append bits and the output.  norm: dict(q, k, eps) of RMSNorm weights.
    The element type (bf16 / fp16) and page layout are those of inp; the oracle
    always sees the token-major copy of the same pool."""
    cpu = inp.to("cpu").as_nhd()
    nk = {} if norm is None else {"q_norm_w": norm["q"], "k_norm_w": norm["k"], "norm_eps": norm["eps"]}
    ref = oracle.reference_step(cpu, positions=positions, rows=rows, sm_scale=sm_scale, interleaved=interleaved,
                                **nk)
    got = run_step(inp, path=path, num_ctas=num_ctas, positions=positions, sm_scale=sm_scale, graph=graph,
                   max_pos=max_pos, repeat=repeat, pdl=pdl, norm=norm, interleaved=interleaved, pdl_kv=pdl_kv,
                   planned=planned, host_io=host_io)
    assert got["err"] == 0, f"device error flag {got['err']}"
    exempt, n_diff = check_append(cpu, ref, got["pool_after"], MIDPOINT_REL if norm is None else MIDPOINT_REL_NORM,
                                  interleaved=interleaved)
    qerr = check_q_rot(cpu, ref["q_rot"], got["q_rot"]) if path == "three" else 0.0
    oerr = check_out(cpu, ref["out"], got["out"], rows=rows)
    return {"exempt": exempt, "n_diff": n_diff, "q_rot_err": qerr, "out_err": oerr, "got": got, "ref": ref}
