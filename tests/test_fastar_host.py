"""The contiguous-cache (Fast AR) inputs on the CPU: the layout the library is
given and the token-major copy the oracle reads hold the same values, and
the oracle's append into a one-page-per-row cache of 11 positions lands in
the row's own cache."""
import torch

import oracle
import workloads


def _bits(t):
    return t.contiguous().view(torch.int16)


def test_contiguous_cache_views_and_strides():
    inp = workloads.make_inputs("fastar")
    B, Hkv, P, D = inp.B, inp.Hkv, inp.P, inp.D
    assert inp.layout == "CONTIG" and inp.pool.shape == (2, B, Hkv, P, D) and inp.api_page_table is None
    k = inp.k_cache()
    assert k.shape == (B, P, Hkv, D)
    assert k.stride() == (inp.page_stride, inp.token_stride, inp.head_stride, 1) == (Hkv * P * D, D, P * D, 1)
    assert inp.v_cache().data_ptr() - k.data_ptr() == B * Hkv * P * D * 2
    n = inp.as_nhd()
    assert torch.equal(_bits(n.pool[:, 0]), _bits(k)) and torch.equal(_bits(n.pool[:, 1]), _bits(inp.v_cache()))
    assert torch.equal(n.page_table.view(-1), torch.arange(B, dtype=torch.int32))


def test_oracle_append_into_a_contiguous_cache():
    inp = workloads.make_case(B=3, Hq=4, Hkv=2, D=16, P=11, seq_lens=[1, 7, 11], seed=4, layout="CONTIG")
    n = inp.as_nhd()
    q_rot, pool, bad = oracle.rope_kv_append(n.q, n.k_new, n.v_new, n.pool, n.page_table, n.seq_lens, n.active,
                                             P=n.P, theta=n.theta)
    assert bad == 0
    changed = (_bits(pool) != _bits(n.pool))
    for b, L in enumerate([1, 7, 11]):
        assert torch.equal(_bits(pool[b, 1, L - 1]), _bits(n.v_new[b]))
        others = changed[b].clone()
        others[:, L - 1] = False
        assert not others.any()
