"""KV-append placement, bit for bit, on the GPU (both paths, all layouts).

After one decode step the pool must differ from the pool before it only in
the appended slots (slot seq_len-1 of each active row): the dummy page 0, the
guard page at the end of the pool, the other requests' pages, the unused
pages and every other slot of a row's pages keep their bits.  In the
appended slot, V is v_new bit for bit and K is the oracle's rotated key
rounded to the element type (up to the fp32-rotation midpoint exemption of
the comparison helper)."""
import pytest
import torch

import gpu_harness as H
import oracle
import workloads

pytestmark = pytest.mark.gpu

CASES = [("tiny", "NHD", torch.bfloat16), ("c64", "NHD", torch.bfloat16), ("padded", "NHD", torch.bfloat16),
         ("long", "NHD", torch.bfloat16), ("c64", "HND", torch.float16), ("padded", "HND", torch.bfloat16),
         ("fastar", "CONTIG", torch.bfloat16), ("fastar", "CONTIG", torch.float16)]


def _slots(inp):
    act = inp.active.cpu().bool()
    lens, pt = inp.seq_lens.cpu(), inp.page_table.cpu()
    out = {}
    for b in torch.nonzero(act).flatten().tolist():
        L = int(lens[b])
        out[b] = (int(pt[b, (L - 1) // inp.P]), (L - 1) % inp.P)
    return out


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("name,layout,dtype", CASES)
def test_only_appended_slots_change(name, layout, dtype, path):
    inp = workloads.make_inputs(name, device="cuda", layout=layout, dtype=dtype)
    before = H.bits16(inp.nhd_pool().contiguous().cpu())       # [NP, 2, P, Hkv, D]
    got = H.run_step(inp, path=path)
    assert got["err"] == 0
    after = H.bits16(got["pool_after"])
    slots = _slots(inp)
    allowed = torch.zeros_like(before, dtype=torch.bool)
    for page, off in slots.values():
        allowed[page, :, off] = True
    changed = before != after
    assert not (changed & ~allowed).any(), "a slot other than an appended one changed"
    if layout != "CONTIG":
        assert torch.equal(after[0], before[0]), "dummy page 0 changed"
        assert torch.equal(after[-1], before[-1]), "guard page changed"
    # V: v_new bit for bit; K: the oracle's rounding of the rotated key
    v_new = H.bits16(inp.v_new.cpu())
    for b, (page, off) in slots.items():
        assert torch.equal(after[page, 1, off], v_new[b])
    ref = oracle.reference_step(inp.to("cpu").as_nhd(), rows=[])
    H.check_append(inp.to("cpu").as_nhd(), ref, got["pool_after"])


@pytest.mark.parametrize("path", H.PATHS)
def test_padding_rows_with_stale_page_ids_write_nothing(path):
    # padding rows whose page-table rows point at live pages of other requests
    # (not at page 0) still must not write anything
    inp = workloads.make_inputs("padded", device="cuda")
    act = inp.active.cpu().bool()
    live_pages = inp.page_table.cpu()[act][:, 0]
    pt = inp.page_table.clone()
    dead = torch.nonzero(~act).flatten()
    pt[dead, 0] = live_pages[: len(dead)].to(pt.device) if len(live_pages) >= len(dead) else live_pages[0].item()
    inp.page_table = pt
    before = H.bits16(inp.pool.cpu())
    got = H.run_step(inp, path=path)
    after = H.bits16(got["pool_after"])
    allowed = torch.zeros_like(before, dtype=torch.bool)
    for page, off in _slots(inp).values():
        allowed[page, :, off] = True
    assert not ((before != after) & ~allowed).any()
