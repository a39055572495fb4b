"""The seeded input generator (no GPU): reproducible draws, the NaN poisoning
of every slot without a cached token, and the head-major page layout holding
exactly the token-major values."""
import torch

import workloads


def _bits(t):
    return t.contiguous().view(torch.int16)


def test_same_seed_same_inputs_and_fp16_uses_the_same_draws():
    a = workloads.make_inputs("tiny")
    b = workloads.make_inputs("tiny")
    assert torch.equal(_bits(a.pool), _bits(b.pool)) and torch.equal(a.page_table, b.page_table)
    h = workloads.make_inputs("tiny", dtype=torch.float16)
    assert h.pool.dtype == torch.float16 and torch.equal(h.page_table, a.page_table)
    live = ~torch.isnan(a.pool.float())
    assert torch.equal(live, ~torch.isnan(h.pool.float()))
    assert torch.allclose(a.pool.float()[live], h.pool.float()[live], rtol=2 ** -7, atol=0)


def test_slots_without_a_cached_token_are_nan():
    inp = workloads.make_inputs("padded")
    nan = torch.isnan(inp.pool.float())
    assert nan[0].all() and nan[-1].all()                  # dummy page and guard page
    for b in range(inp.B):
        L = int(inp.seq_lens[b])
        if not int(inp.active[b]):
            continue
        for j in (0, L - 2):
            if j >= 0:
                assert not nan[int(inp.page_table[b, j // inp.P]), :, j % inp.P].any()
        slot = L - 1                                        # the append target is poisoned
        assert nan[int(inp.page_table[b, slot // inp.P]), :, slot % inp.P].all()


def test_head_major_pages_hold_the_token_major_values():
    a = workloads.make_inputs("tiny")
    b = workloads.make_inputs("tiny", layout="HND")
    assert b.pool.shape == (a.num_pages, 2, a.Hkv, a.P, a.D) and b.pool.is_contiguous()
    assert torch.equal(_bits(b.nhd_pool()), _bits(a.pool))
    assert torch.equal(_bits(b.as_nhd().pool), _bits(a.pool)) and b.as_nhd().layout == "NHD"
    k = b.k_cache()
    assert k.shape == (a.num_pages, a.P, a.Hkv, a.D)
    assert k.stride() == (b.page_stride, b.token_stride, b.head_stride, 1)
    assert (b.token_stride, b.head_stride) == (a.D, a.P * a.D)
    assert (a.token_stride, a.head_stride) == (a.Hkv * a.D, a.D)
    assert a.k_cache().stride() == (a.page_stride, a.token_stride, a.head_stride, 1)
    assert b.v_cache().data_ptr() - b.k_cache().data_ptr() == a.P * a.Hkv * a.D * 2
    c = b.clone()
    assert c.layout == "HND" and torch.equal(_bits(c.pool), _bits(b.pool))


def test_layers_of_one_step_share_the_batch_but_not_the_values():
    # every layer of a multi-layer step sees the same lengths, active rows and
    # page table; its pool and q/k/v values are its own
    a = workloads.make_inputs("fastar", layer=0)
    b = workloads.make_inputs("fastar", layer=3)
    assert torch.equal(a.seq_lens, b.seq_lens) and torch.equal(a.page_table, b.page_table)
    assert not torch.equal(_bits(a.q), _bits(b.q)) and not torch.equal(_bits(a.pool), _bits(b.pool))
    c = workloads.make_inputs("fastar", layer=4)          # the next step: a new draw of everything
    assert c.meta["step_first_layer"] == 4 and not torch.equal(_bits(c.q), _bits(a.q))
    # first layer of a step unchanged by the sharing (the draw of a one-layer workload)
    assert a.meta["step_first_layer"] == 0 and workloads.make_inputs("tiny", layer=5).meta["step_first_layer"] == 5
