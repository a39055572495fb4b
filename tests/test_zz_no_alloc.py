"""The attention entry point for callers that cannot allocate device memory.

vh_paged_decode_attn_noalloc keeps its split-K partial results in a fixed
array compiled into the library instead of a caller-provided workspace.  It
serves callers with no way to allocate: runtimes that only hand kernels
preallocated arenas, plug-ins whose host owns the CUDA context, measurements
that must keep the memory footprint fixed.  Its result must match the
workspace path (vh_paged_decode_attn + vh_decode_combine) on the same inputs.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import pytest
import torch

import gpu_harness as H
import workloads

pytestmark = pytest.mark.gpu


def _prepared(name):
    """Inputs with the new token already appended and q rotated (existing calls)."""
    v = H.vh()
    inp = workloads.make_inputs(name, device="cuda")
    B, Hq, D, P = inp.B, inp.Hq, inp.D, inp.P
    cos_sin = torch.empty((inp.max_pages_per_seq * P, D), dtype=torch.float32, device="cuda")
    v.vh_rope_table(cos_sin, inp.theta)
    q_rot = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    v.vh_rope_kv_append(inp.q, inp.k_new, inp.v_new, cos_sin, inp.pool[:, 0], inp.pool[:, 1],
                        inp.page_table, inp.seq_lens, inp.active, q_rot)
    return inp, q_rot


def _with_workspace(inp, q_rot):
    v = H.vh()
    out = torch.full((inp.B, inp.Hq, inp.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = v.alloc_workspace(inp.B, inp.Hq, inp.Hkv, inp.D, inp.P, device="cuda")
    v.vh_paged_decode_attn(q_rot, inp.pool[:, 0], inp.pool[:, 1], inp.page_table, inp.seq_lens,
                           inp.active, out, ws)
    v.vh_decode_combine(ws, out, inp.Hkv, inp.P)
    return out


def _without_workspace(inp, q_rot, err):
    v = H.vh()
    out = torch.full((inp.B, inp.Hq, inp.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    v.vh_paged_decode_attn_noalloc(q_rot, inp.pool[:, 0], inp.pool[:, 1], inp.page_table,
                                   inp.seq_lens, inp.active, out, err_flag=err)
    return out


def _agree(a, b):
    a, b = a.double().cpu(), b.double().cpu()
    assert torch.isfinite(a).all() and torch.isfinite(b).all()
    assert ((a - b).abs() <= H.ATOL + H.RTOL * b.abs()).all()


def test_noalloc_matches_workspace_path_on_two_calls_in_a_row():
    # two different shapes, so the second call runs over what the first left in the array
    first, q1 = _prepared("long")
    second, q2 = _prepared("padded")
    ref1 = _with_workspace(first, q1)
    ref2 = _with_workspace(second, q2)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got1 = _without_workspace(first, q1, err)
    got2 = _without_workspace(second, q2, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _agree(got1, ref1)
    _agree(got2, ref2)
    # and once more on the first inputs, after the second call overwrote the array
    _agree(_without_workspace(first, q1, err), ref1)


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
