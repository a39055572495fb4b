"""Contiguous per-request caches (the Fast AR step) on the GPU, against the
float64 oracle: no page table, a cache of P positions per row (any P up to
1024, here mostly the 11 positions of 10 residual codebooks + 1), the new
token written and read in place.  Both paths (three calls and fused)."""
import pytest
import torch

import gpu_harness as H
import workloads

pytestmark = pytest.mark.gpu


def contig(lens, *, Hq=16, Hkv=8, D=64, P=11, seed=1, **kw):
    return workloads.make_case(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, P=P, seq_lens=lens, seed=seed,
                               device="cuda", layout="CONTIG", **kw)


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("layer", [0, 1, 2, 3])
def test_fastar_workload_layers(layer, path):
    inp = workloads.make_inputs("fastar", layer=layer, device="cuda")
    assert inp.api_page_table is None
    H.full_check(inp, path=path)


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("P", [11, 16, 32, 100])
def test_contiguous_cache_mixed_lengths(P, path):
    g = torch.Generator().manual_seed(P)
    lens = torch.randint(1, P + 1, (48,), generator=g).tolist()
    H.full_check(contig(lens, P=P, seed=P + 1), path=path)


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_contiguous_cache_groups_and_dims(G, D, path):
    inp = contig([1, 5, 11, 9, 2], Hq=2 * G, Hkv=2, D=D, seed=G + D)
    H.full_check(inp, path=path)


@pytest.mark.parametrize("path", H.PATHS)
def test_contiguous_cache_fp16_interleaved_norm_and_padding(path):
    act = [1, 0, 1, 1, 0, 1]
    lens = [11, 1, 3, 8, 1, 10]
    inp = contig(lens, active=act, seed=9, dtype=torch.float16)
    g = torch.Generator().manual_seed(3)
    norm = {"q": (1 + 0.2 * torch.randn(inp.D, generator=g)).float(),
            "k": (1 + 0.2 * torch.randn(inp.D, generator=g)).float(), "eps": 1e-6}
    before = H.bits16(inp.nhd_pool().cpu())
    r = H.full_check(inp, path=path, interleaved=True, norm=norm)
    after = H.bits16(r["got"]["pool_after"])
    for b in (1, 4):  # padding rows: their caches are not touched
        assert torch.equal(after[b], before[b])


@pytest.mark.parametrize("path", H.PATHS)
def test_fast_ar_decode_loop_step_by_step(path):
    # one Fast AR pass: 11 positions, each step appends one token per row and
    # attends over the cache so far; the GPU's cache after a step feeds the next
    # step, and every step is checked against the oracle on that same cache
    B, P = 32, 11
    inp = contig([1] * B, P=P, seed=77)
    for step in range(1, P + 1):
        fresh = contig([step] * B, P=P, seed=1000 + step)
        inp.q, inp.k_new, inp.v_new = fresh.q, fresh.k_new, fresh.v_new
        inp.seq_lens = torch.full((B,), step, dtype=torch.int32, device="cuda")
        r = H.full_check(inp, path=path)
        inp.pool = r["got"]["pool_after"].permute(1, 0, 3, 2, 4).contiguous().to("cuda")
    # all P slots are now written
    assert not torch.isnan(inp.pool.float()).any()
