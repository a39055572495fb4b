"""The attention entry point for callers that cannot allocate device memory.

vh_paged_decode_attn_noalloc keeps its split-K partial results in a fixed
array compiled into the library instead of a caller-provided workspace.  It
serves callers with no way to allocate: runtimes that only hand kernels
preallocated arenas, plug-ins whose host owns the CUDA context, measurements
that must keep the memory footprint fixed.  Its result must match the
float64 oracle on the same inputs, and the workspace path
(vh_paged_decode_attn + vh_decode_combine), on two calls in a row.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import pytest
import torch

import gpu_harness as H
import oracle
import workloads

pytestmark = pytest.mark.gpu


def _prepared(inp, page_table="inp"):
    """The new token appended and q rotated by the existing calls (on a copy of
    inp's pool); returns (device inputs, q_rot)."""
    v = H.vh()
    g = inp.to("cuda").clone()
    B, Hq, D, P = g.B, g.Hq, g.D, g.P
    cos_sin = torch.empty((g.max_pages_per_seq * P, D), dtype=torch.float32, device="cuda")
    v.vh_rope_table(cos_sin, g.theta)
    q_rot = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    pt = g.page_table if page_table == "inp" else page_table
    v.vh_rope_kv_append(g.q, g.k_new, g.v_new, cos_sin, g.pool[:, 0], g.pool[:, 1], pt, g.seq_lens,
                        g.active, q_rot)
    return g, q_rot


def _with_workspace(g, q_rot, page_table="inp"):
    v = H.vh()
    pt = g.page_table if page_table == "inp" else page_table
    out = torch.full((g.B, g.Hq, g.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = v.alloc_workspace(g.B, g.Hq, g.Hkv, g.D, g.P, device="cuda")
    v.vh_paged_decode_attn(q_rot, g.pool[:, 0], g.pool[:, 1], pt, g.seq_lens, g.active, out, ws)
    v.vh_decode_combine(ws, out, g.Hkv, g.P)
    return out


def _without_workspace(g, q_rot, err, page_table="inp"):
    v = H.vh()
    pt = g.page_table if page_table == "inp" else page_table
    out = torch.full((g.B, g.Hq, g.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    v.vh_paged_decode_attn_noalloc(q_rot, g.pool[:, 0], g.pool[:, 1], pt, g.seq_lens, g.active, out,
                                   err_flag=err)
    return out


def _agree(a, b):
    a, b = a.double().cpu(), b.double().cpu()
    assert torch.isfinite(a).all() and torch.isfinite(b).all()
    assert ((a - b).abs() <= H.ATOL + H.RTOL * b.abs()).all()


def test_noalloc_matches_oracle_and_workspace_path_on_two_calls_in_a_row():
    # two different shapes, so the second call runs over what the first left in the array
    first = workloads.make_inputs("long")
    second = workloads.make_inputs("padded")
    ref1 = oracle.reference_step(first)["out"]
    ref2 = oracle.reference_step(second)["out"]
    g1, q1 = _prepared(first)
    g2, q2 = _prepared(second)
    ws1 = _with_workspace(g1, q1)
    ws2 = _with_workspace(g2, q2)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got1 = _without_workspace(g1, q1, err)
    got2 = _without_workspace(g2, q2, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H.check_out(first, ref1, got1.cpu())
    H.check_out(second, ref2, got2.cpu())
    _agree(got1, ws1)
    _agree(got2, ws2)
    # and once more on the first inputs, after the second call overwrote the array
    again = _without_workspace(g1, q1, err)
    torch.cuda.synchronize()
    H.check_out(first, ref1, again.cpu())


def test_noalloc_contiguous_cache_without_page_table():
    # the same rows stored as one contiguous run of pages per row (row b owns
    # pages b*m .. b*m+m-1 of a token-major pool) and no page table
    inp = workloads.make_case(B=6, Hq=16, Hkv=8, D=128, P=16, seq_lens=[300, 17, 1, 129, 64, 250],
                              active=[1, 1, 1, 1, 0, 1], seed=77)
    ref = oracle.reference_step(inp)["out"]
    m, B = inp.max_pages_per_seq, inp.B
    pool = torch.full((B * m,) + tuple(inp.pool.shape[1:]), 0, dtype=inp.pool.dtype)
    pool.view(torch.int16).fill_(workloads.NAN_BITS)
    for b in range(B):
        if not int(inp.active[b]):
            continue
        n = -(-int(inp.seq_lens[b]) // inp.P)
        pool[b * m:b * m + n] = inp.pool[inp.page_table[b, :n].long()]
    contig = workloads.DecodeInputs(B=B, Hq=inp.Hq, Hkv=inp.Hkv, D=inp.D, P=inp.P, max_pages_per_seq=m,
                                    num_pages=B * m, theta=inp.theta, q=inp.q, k_new=inp.k_new,
                                    v_new=inp.v_new, pool=pool, page_table=inp.page_table,
                                    seq_lens=inp.seq_lens, active=inp.active)
    g, q_rot = _prepared(contig, page_table=None)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _without_workspace(g, q_rot, err, page_table=None)
    ws = _with_workspace(g, q_rot, page_table=None)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H.check_out(inp, ref, got.cpu())
    _agree(got, ws)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    v = H.vh()
    # 4096 rows x 1024 kv heads: the per-(row, kv head) counters alone
    # (4096 * 1024 * 4 bytes = 16 MiB) exceed the 8 MiB array whatever the CTA
    # count, while the shape still fits the kernel's shared-memory plan, so the
    # call is rejected on the host with VH_ESCRATCH.  Every buffer is still
    # allocated at its full size, so even a wrong verdict could only launch
    # over all-padding rows into valid memory.
    B, Hq, Hkv, D, P = 4096, 1024, 1024, 64, 16
    assert B * Hkv * 4 > 8 << 20
    dev = "cuda"
    q_rot = torch.zeros((B, Hq, D), dtype=torch.float32, device=dev)
    pool = torch.zeros((1, 2, P, Hkv, D), dtype=torch.bfloat16, device=dev)
    page_table = torch.zeros((B, 1), dtype=torch.int32, device=dev)
    seq_lens = torch.ones(B, dtype=torch.int32, device=dev)
    active = torch.zeros(B, dtype=torch.int32, device=dev)
    out = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device=dev)
    with pytest.raises(v.VHError) as e:
        v.vh_paged_decode_attn_noalloc(q_rot, pool[:, 0], pool[:, 1], page_table, seq_lens, active, out)
    assert e.value.status == v.VH_ESCRATCH
    assert "scratch" in v.vh_status_string(v.VH_ESCRATCH)
