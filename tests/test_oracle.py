"""Pins of the float64 oracle against things other than itself.

Every check here runs on the CPU.  The pins are closed forms, invariants of
the mathematics, a library routine for a special case (scaled dot-product
attention in float64 for G = 1), an independent pure-Python brute force on
tiny inputs (tests/brute.py) and hand-derived fixtures (tests/golden/).  Each
is chosen so that a plausible slip in the oracle (a dropped term, a wrong
sign or index, a transposed operand, a wrong head map or page lookup) fails
at least one of them.
"""
import json
import math
import os

import pytest
import torch

import brute
import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bits(t):
    return t.contiguous().view(torch.int16).to(torch.int32) & 0xFFFF


def _f64(t_bf16):
    return t_bf16.to(torch.float64)


# ---------------------------------------------------------------- bf16 rounding

@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3F80),
    (-2.0, 0xC000),
    (1.0 + 2 ** -8, 0x3F80),            # midpoint between 0x3F80 (even) and 0x3F81: down
    (1.0 + 3 * 2 ** -8, 0x3F82),        # midpoint between 0x3F81 (odd) and 0x3F82: up
    (1.0 + 2 ** -8 + 2 ** -40, 0x3F81), # just above the midpoint: up
    (1.0 + 2 ** -8 - 2 ** -40, 0x3F80), # just below: down
    (3.0e38, 0x7F62),
    (3.4e38, 0x7F80),                   # beyond the largest finite bf16: inf
    (2 ** -130, 0x0008),                # subnormal
    (0.0, 0x0000),
    (-0.0, 0x8000),
])
def test_bf16_rounding_fixed_points(x, bits):
    assert oracle.bf16_from_double(x) == bits
    assert brute.bf16_round_bits(x) == bits


def test_bf16_rounding_matches_exact_bracketing():
    g = torch.Generator().manual_seed(7)
    xs = (torch.randn(3000, generator=g, dtype=torch.float64) * 4).tolist()
    # add values sitting exactly on midpoints
    for bits in range(0x3F00, 0x3F40):
        a = brute.bf16_bits_to_float(bits)
        b = brute.bf16_bits_to_float(bits + 1)
        xs.append((a + b) / 2)
    for x in xs:
        assert oracle.bf16_from_double(x) == brute.bf16_round_bits(x), x


def test_bf16_rounding_agrees_with_torch_on_float32_values():
    # For values exactly representable in float32 there is no double rounding,
    # so torch's float32 -> bf16 conversion (round to nearest even) applies.
    g = torch.Generator().manual_seed(3)
    xs = torch.randn(4000, generator=g, dtype=torch.float32) * 100
    ref = _bits(xs.to(torch.bfloat16)).tolist()
    got = [oracle.bf16_from_double(float(v)) for v in xs.tolist()]
    assert got == ref


# ---------------------------------------------------------------- RoPE

def _rope_via_oracle(x, pos, theta=10000.0):
    """Rotate one head vector with the oracle (through the q path)."""
    D = len(x)
    q = torch.tensor([[x]], dtype=torch.float32).to(torch.bfloat16)
    k = torch.zeros((1, 1, D), dtype=torch.bfloat16)
    pool = torch.zeros((3, 2, 16, 1, D), dtype=torch.bfloat16)
    q_rot, _, bad = oracle.rope_kv_append(q, k, k, pool, torch.tensor([[1]]), torch.tensor([1]),
                                          torch.tensor([1]), P=16, theta=theta,
                                          positions=torch.tensor([pos]))
    assert bad == 0
    return q_rot[0, 0].tolist()


def test_rope_golden_closed_forms():
    cases = json.load(open(os.path.join(GOLDEN, "closed_forms.json")))["cases"]
    n = 0
    for c in cases:
        if not c["name"].startswith("rope"):
            continue
        got = _rope_via_oracle(c["x"], c["pos"], c["theta"])
        want = [eval(e, {"math": math}) for e in c["expect"]]
        assert got == pytest.approx(want, abs=1e-15), c["name"]
        n += 1
    assert n >= 3


def test_rope_position_zero_is_identity():
    x = torch.randn(64, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    got = _rope_via_oracle(x.float().tolist(), 0)
    assert got == x.double().tolist()


def test_rope_preserves_norm_and_is_relative():
    g = torch.Generator().manual_seed(2)
    D = 64
    x = torch.randn(D, generator=g).to(torch.bfloat16).float().tolist()
    y = torch.randn(D, generator=g).to(torch.bfloat16).float().tolist()
    for pos in (1, 17, 1000, 8191):
        rx = _rope_via_oracle(x, pos)
        assert math.sqrt(sum(v * v for v in rx)) == pytest.approx(math.sqrt(sum(v * v for v in x)), rel=1e-13)
    # <rot_m x, rot_n y> depends only on m - n
    def dot(a, b):
        return math.fsum(p * q for p, q in zip(a, b))
    ref = dot(_rope_via_oracle(x, 5), _rope_via_oracle(y, 2))
    for shift in (1, 100, 4000):
        got = dot(_rope_via_oracle(x, 5 + shift), _rope_via_oracle(y, 2 + shift))
        assert got == pytest.approx(ref, rel=1e-11, abs=1e-11)
    # and it does change with m - n (the rotation is not trivial)
    assert abs(dot(_rope_via_oracle(x, 6), _rope_via_oracle(y, 2)) - ref) > 1e-6


def test_rope_matches_brute_force():
    g = torch.Generator().manual_seed(4)
    for D in (4, 64, 128):
        x = torch.randn(D, generator=g).to(torch.bfloat16).float().tolist()
        for pos in (0, 3, 129, 8191):
            assert _rope_via_oracle(x, pos) == pytest.approx(brute.rope(x, pos, 10000.0), abs=1e-12)


# ---------------------------------------------------------------- append placement

def _small_case(lens, active=None, B=None, Hq=4, Hkv=2, D=16, P=16, seed=0, **kw):
    B = len(lens) if B is None else B
    return workloads.make_case(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, seq_lens=lens, active=active,
                               seed=seed, **kw)


@pytest.mark.parametrize("L,page_idx,off", [(1, 0, 0), (16, 0, 15), (17, 1, 0), (33, 2, 0), (40, 2, 7)])
def test_append_places_token_in_its_slot(L, page_idx, off):
    inp = _small_case([L, 5], P=16)
    q_rot, after, bad = oracle.rope_kv_append(inp.q, inp.k_new, inp.v_new, inp.pool, inp.page_table,
                                              inp.seq_lens, inp.active, P=inp.P, theta=inp.theta)
    assert bad == 0
    page = int(inp.page_table[0, page_idx])
    before_bits = _bits(inp.pool)
    after_bits = _bits(after)
    changed = (before_bits != after_bits)
    # slot of row 0 and slot of row 1 (L=5 -> page 0, offset 4) changed; nothing else
    mask = torch.zeros_like(changed)
    mask[page, :, off] = True
    mask[int(inp.page_table[1, 0]), :, 4] = True
    assert not (changed & ~mask).any()
    # V slot holds v_new bit for bit
    assert torch.equal(after_bits[page, 1, off], _bits(inp.v_new[0]))
    # K slot holds bf16(RNE(rope(k_new))) from the brute force
    pos = L - 1
    for h in range(inp.Hkv):
        kr = brute.rope(inp.k_new[0, h].float().tolist(), pos, inp.theta)
        assert after_bits[page, 0, off, h].tolist() == [brute.bf16_round_bits(v) for v in kr]


@pytest.mark.parametrize("L,page_idx,off", [(8, 0, 7), (9, 1, 0), (24, 2, 7), (25, 3, 0)])
def test_append_places_token_in_its_slot_with_8_token_pages(L, page_idx, off):
    inp = _small_case([L, 3], P=8)
    _, after, bad = oracle.rope_kv_append(inp.q, inp.k_new, inp.v_new, inp.pool, inp.page_table,
                                          inp.seq_lens, inp.active, P=inp.P, theta=inp.theta)
    assert bad == 0
    page = int(inp.page_table[0, page_idx])
    changed = _bits(inp.pool) != _bits(after)
    mask = torch.zeros_like(changed)
    mask[page, :, off] = True
    mask[int(inp.page_table[1, 0]), :, 2] = True
    assert not (changed & ~mask).any()
    assert torch.equal(_bits(after)[page, 1, off], _bits(inp.v_new[0]))


def test_append_skips_padding_rows_and_bad_rows():
    inp = _small_case([9, 1, 7], active=[1, 0, 1])
    # row 2 claims a length beyond its page-table row
    inp.seq_lens[2] = inp.max_pages_per_seq * inp.P + 1
    _, after, bad = oracle.rope_kv_append(inp.q, inp.k_new, inp.v_new, inp.pool, inp.page_table,
                                          inp.seq_lens, inp.active, P=inp.P, theta=inp.theta)
    assert bad == 1
    changed = (_bits(inp.pool) != _bits(after))
    # only row 0's slot (page_table[0][0], offset 8) may change; page 0 untouched
    allowed = torch.zeros_like(changed)
    allowed[int(inp.page_table[0, 0]), :, 8] = True
    assert not (changed & ~allowed).any()
    assert changed[int(inp.page_table[0, 0]), :, 8].any()
    assert not changed[0].any()


# ---------------------------------------------------------------- attention closed forms

def test_golden_attention_cases():
    cases = json.load(open(os.path.join(GOLDEN, "closed_forms.json")))["cases"]
    n = 0
    for c in cases:
        if "seq_len" not in c:
            continue
        D, P, L = c["D"], c["P"], c["seq_len"]
        kc = c["k_cached"] if isinstance(c["k_cached"][0], list) else [c["k_cached"]]
        vc = c["v_cached"] if isinstance(c["v_cached"][0], list) else [c["v_cached"]]
        pool = torch.full((3, 2, P, 1, D), float("nan")).to(torch.bfloat16)
        for j, (kr, vr) in enumerate(zip(kc, vc)):
            pool[1, 0, j, 0] = torch.tensor(kr, dtype=torch.float32).to(torch.bfloat16)
            pool[1, 1, j, 0] = torch.tensor(vr, dtype=torch.float32).to(torch.bfloat16)
        bf = lambda v: torch.tensor([[v]], dtype=torch.float32).to(torch.bfloat16)
        pt = torch.tensor([[1]])
        q_rot, after, bad = oracle.rope_kv_append(bf(c["q"]), bf(c["k_new"]), bf(c["v_new"]), pool, pt,
                                                  torch.tensor([L]), torch.tensor([1]), P=P,
                                                  theta=10000.0, positions=torch.tensor([c["position"]]))
        out = oracle.decode_attn(q_rot, after, pt, torch.tensor([L]), torch.tensor([1]), P=P)
        want = [eval(e, {"math": math}) for e in c["expect"]]
        assert out[0, 0].tolist() == pytest.approx(want, abs=1e-15), c["name"]
        n += 1
    assert n >= 2


def _step(inp, **kw):
    return oracle.reference_step(inp, **kw)


def test_single_key_returns_v_new_exactly():
    inp = _small_case([1, 1, 1], D=64, Hq=8, Hkv=2)
    r = _step(inp)
    G = inp.Hq // inp.Hkv
    for b in range(inp.B):
        for g in range(inp.Hq):
            assert torch.equal(r["out"][b, g], _f64(inp.v_new[b, g // G]))


def test_identical_keys_give_mean_of_values():
    inp = _small_case([37, 20], D=32, Hq=4, Hkv=2, poison=False)
    key = torch.randn(inp.D, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    inp.pool[:, 0] = key  # every cached key equal
    q_rot = torch.randn((inp.B, inp.Hq, inp.D), dtype=torch.float64)
    out = oracle.decode_attn(q_rot, inp.pool, inp.page_table, inp.seq_lens, inp.active, P=inp.P)
    G = inp.Hq // inp.Hkv
    for b in range(inp.B):
        L = int(inp.seq_lens[b])
        for g in range(inp.Hq):
            vs = torch.stack([_f64(inp.pool[int(inp.page_table[b, j // inp.P]), 1, j % inp.P, g // G])
                              for j in range(L)])
            assert torch.allclose(out[b, g], vs.mean(0), rtol=0, atol=1e-14)


def test_tiny_scale_gives_mean_and_peaked_query_selects_value():
    inp = _small_case([23], D=16, Hq=2, Hkv=1, poison=False)
    q_rot = torch.randn((1, 2, inp.D), dtype=torch.float64)
    out = oracle.decode_attn(q_rot, inp.pool, inp.page_table, inp.seq_lens, inp.active, P=inp.P,
                             sm_scale=1e-300)
    vs = torch.stack([_f64(inp.pool[int(inp.page_table[0, j // inp.P]), 1, j % inp.P, 0]) for j in range(23)])
    assert torch.allclose(out[0, 0], vs.mean(0), atol=1e-14)
    # q = alpha * K_j picks V_j
    j = 13
    kj = _f64(inp.pool[int(inp.page_table[0, j // inp.P]), 0, j % inp.P, 0])
    q_rot[0, 0] = 200.0 * kj / kj.norm()
    out = oracle.decode_attn(q_rot, inp.pool, inp.page_table, inp.seq_lens, inp.active, P=inp.P)
    assert torch.allclose(out[0, 0], vs[j], atol=1e-6)


def test_value_linearity_and_key_shift_invariance():
    # integer-valued K and V so that the edits below are exact in bf16
    inp = _small_case([29, 50], D=16, Hq=4, Hkv=2, poison=False)
    g = torch.Generator().manual_seed(9)
    inp.pool.copy_(torch.randint(-8, 9, inp.pool.shape, generator=g).to(torch.bfloat16))
    q_rot = torch.randn((inp.B, inp.Hq, inp.D), generator=g, dtype=torch.float64) * 0.2
    base = oracle.decode_attn(q_rot, inp.pool, inp.page_table, inp.seq_lens, inp.active, P=inp.P)
    p2 = inp.pool.clone()
    p2[:, 1] *= 2
    assert torch.allclose(oracle.decode_attn(q_rot, p2, inp.page_table, inp.seq_lens, inp.active, P=inp.P),
                          2 * base, atol=1e-12)
    u = torch.randint(-4, 5, (inp.Hkv, inp.D), generator=g).to(torch.bfloat16)
    p3 = inp.pool.clone()
    p3[:, 1] += u
    shifted = oracle.decode_attn(q_rot, p3, inp.page_table, inp.seq_lens, inp.active, P=inp.P)
    G = inp.Hq // inp.Hkv
    for hq in range(inp.Hq):
        assert torch.allclose(shifted[:, hq], base[:, hq] + _f64(u[hq // G]), atol=1e-12)
    w = torch.randint(-4, 5, (inp.Hkv, inp.D), generator=g).to(torch.bfloat16)
    p4 = inp.pool.clone()
    p4[:, 0] += w
    assert torch.allclose(oracle.decode_attn(q_rot, p4, inp.page_table, inp.seq_lens, inp.active, P=inp.P),
                          base, atol=1e-12)


def test_physical_page_permutation_invariance():
    inp = workloads.make_inputs("tiny")
    r = _step(inp)
    NP = inp.num_pages
    g = torch.Generator().manual_seed(11)
    perm = torch.randperm(NP, generator=g)       # new physical index of page p is perm[p]
    pool2 = torch.empty_like(inp.pool)
    pool2[perm] = inp.pool
    pt2 = perm[inp.page_table.long()].to(torch.int32)
    inp2 = workloads.DecodeInputs(**{**{k: getattr(inp, k) for k in (
        "B", "Hq", "Hkv", "D", "P", "max_pages_per_seq", "num_pages", "theta", "q", "k_new",
        "v_new", "seq_lens", "active")}, "pool": pool2, "page_table": pt2})
    r2 = _step(inp2)
    assert torch.equal(r["out"], r2["out"])
    assert torch.equal(_bits(r2["pool_after"])[perm], _bits(r["pool_after"]))


def test_gqa_group_of_one_matches_torch_sdpa():
    inp = _small_case([70, 3, 33], D=64, Hq=4, Hkv=4, seed=3)
    r = _step(inp)
    for b in range(inp.B):
        L = int(inp.seq_lens[b])
        idx = [(int(inp.page_table[b, j // inp.P]), j % inp.P) for j in range(L)]
        K = torch.stack([_f64(r["pool_after"][p, 0, o]) for p, o in idx], dim=1)  # [Hkv, L, D]
        V = torch.stack([_f64(r["pool_after"][p, 1, o]) for p, o in idx], dim=1)
        qh = r["q_rot"][b].unsqueeze(1)                                          # [Hq, 1, D]
        ref = torch.nn.functional.scaled_dot_product_attention(qh, K, V).squeeze(1)
        assert torch.allclose(r["out"][b], ref, atol=1e-13, rtol=0)


def test_gqa_head_map_and_identical_q_heads():
    inp = _small_case([45, 18], D=32, Hq=8, Hkv=2, seed=8)
    G = inp.Hq // inp.Hkv
    inp.q[:, 1] = inp.q[:, 0]          # heads 0 and 1 share kv head 0
    inp.q[:, G] = inp.q[:, 0]          # head G uses kv head 1
    r = _step(inp)
    assert torch.equal(r["out"][:, 1], r["out"][:, 0])
    assert not torch.allclose(r["out"][:, G], r["out"][:, 0])
    # the map is contiguous groups: q head g reads kv head g // G (SDPA on that head)
    b, g = 0, G + 2
    L = int(inp.seq_lens[b])
    idx = [(int(inp.page_table[b, j // inp.P]), j % inp.P) for j in range(L)]
    K = torch.stack([_f64(r["pool_after"][p, 0, o, g // G]) for p, o in idx])
    V = torch.stack([_f64(r["pool_after"][p, 1, o, g // G]) for p, o in idx])
    ref = torch.nn.functional.scaled_dot_product_attention(
        r["q_rot"][b, g].view(1, 1, -1), K.unsqueeze(0), V.unsqueeze(0)).view(-1)
    assert torch.allclose(r["out"][b, g], ref, atol=1e-13, rtol=0)


def test_row_output_independent_of_batch_composition():
    inp = _small_case([40, 77, 5], D=32, Hq=4, Hkv=2, seed=12)
    r = _step(inp)
    sub = _small_case([40], D=32, Hq=4, Hkv=2, seed=12)
    # give the single-row batch exactly row 0's data
    sub.q[0] = inp.q[0]
    sub.k_new[0] = inp.k_new[0]
    sub.v_new[0] = inp.v_new[0]
    for j in range(40):
        p0, o0 = int(inp.page_table[0, j // 16]), j % 16
        p1, o1 = int(sub.page_table[0, j // 16]), j % 16
        sub.pool[p1, :, o1] = inp.pool[p0, :, o0]
    r1 = _step(sub)
    assert torch.equal(r1["out"][0], r["out"][0])


def test_padding_rows_are_zero_and_stale_slots_never_leak():
    inp = workloads.make_inputs("padded")
    act = inp.active.bool()
    rows = torch.nonzero(act).flatten()[:6].tolist() + torch.nonzero(~act).flatten()[:4].tolist()
    r = oracle.reference_step(inp, rows=rows)
    out = r["out"][rows]
    assert torch.isfinite(out).all()
    for b in rows:
        if not act[b]:
            assert not r["out"][b].any()
    # page 0 (all NaN) is never written by padding rows
    assert torch.equal(_bits(r["pool_after"][0]), _bits(inp.pool[0]))


# ---------------------------------------------------------------- split combine

@pytest.mark.parametrize("S", [1, 2, 3, 7, 64, 200])
def test_split_combine_equals_unsplit(S):
    inp = workloads.make_inputs("tiny")
    r = _step(inp)
    split = oracle.decode_attn_split(r["q_rot"], r["pool_after"], inp.page_table, inp.seq_lens,
                                     inp.active, P=inp.P, n_splits=S)
    assert torch.allclose(split, r["out"], rtol=0, atol=1e-12)


def test_lse_combine_edge_cases():
    o = torch.tensor([[1.0, 2.0], [5.0, 7.0]], dtype=torch.float64)
    # one empty split carries no weight
    got, lse = oracle.lse_combine(o, torch.tensor([0.3, float("-inf")], dtype=torch.float64))
    assert got.tolist() == [1.0, 2.0] and lse == pytest.approx(0.3)
    # equal lse: plain mean; lse grows by ln 2
    got, lse = oracle.lse_combine(o, torch.tensor([1.5, 1.5], dtype=torch.float64))
    assert got.tolist() == [3.0, 4.5] and lse == pytest.approx(1.5 + math.log(2))
    # weights exp(lse): lse (0, ln 3) gives weights 1/4, 3/4
    got, _ = oracle.lse_combine(o, torch.tensor([0.0, math.log(3)], dtype=torch.float64))
    assert torch.allclose(got, torch.tensor([4.0, 5.75], dtype=torch.float64), atol=1e-15)
    # all empty: zero output
    got, lse = oracle.lse_combine(o, torch.tensor([float("-inf")] * 2, dtype=torch.float64))
    assert got.tolist() == [0.0, 0.0] and lse == float("-inf")


# ---------------------------------------------------------------- brute force

def _nested(t):
    return (t.contiguous().view(torch.int16).to(torch.int32) & 0xFFFF).tolist()


@pytest.mark.parametrize("shape", [
    dict(lens=[17, 5, 33], Hq=4, Hkv=2, D=8, P=16),
    dict(lens=[1, 16, 40], Hq=2, Hkv=1, D=16, P=16),
    dict(lens=[9, 30], Hq=6, Hkv=3, D=4, P=16),
    dict(lens=[70, 12], Hq=4, Hkv=2, D=8, P=64),
    dict(lens=[17, 8, 9, 25], Hq=4, Hkv=2, D=8, P=8),   # 8-token pages: keys cross a page every 8 slots
])
def test_oracle_matches_brute_force(shape):
    inp = _small_case(shape["lens"], Hq=shape["Hq"], Hkv=shape["Hkv"], D=shape["D"], P=shape["P"], seed=21)
    r = _step(inp)
    pool = _nested(inp.pool)
    q_rot, out = brute.step(_nested(inp.q), _nested(inp.k_new), _nested(inp.v_new), pool,
                            inp.page_table.tolist(), inp.seq_lens.tolist(), inp.active.tolist(),
                            inp.P, inp.theta)
    assert torch.allclose(r["q_rot"], torch.tensor(q_rot, dtype=torch.float64), atol=1e-12, rtol=0)
    assert torch.allclose(r["out"], torch.tensor(out, dtype=torch.float64), atol=1e-12, rtol=0)
    assert _nested(r["pool_after"]) == pool


def test_oracle_matches_brute_force_on_tiny_workload_rows():
    inp = workloads.make_inputs("tiny")
    r = _step(inp)
    pool = _nested(inp.pool)
    q_rot, out = brute.step(_nested(inp.q), _nested(inp.k_new), _nested(inp.v_new), pool,
                            inp.page_table.tolist(), inp.seq_lens.tolist(), inp.active.tolist(),
                            inp.P, inp.theta)
    assert torch.allclose(r["out"], torch.tensor(out, dtype=torch.float64), atol=1e-12, rtol=0)
    assert _nested(r["pool_after"]) == pool


# ---------------------------------------------------------------- RMSNorm (fused before RoPE)

def _norm_weights(D, seed):
    g = torch.Generator().manual_seed(seed)
    return (1.0 + 0.1 * torch.randn(D, generator=g)).to(torch.float32)


def _q_path(q_bf16, pos, w, eps):
    B, H, D = q_bf16.shape
    k = torch.zeros((B, 1, D), dtype=torch.bfloat16)
    pool = torch.zeros((3, 2, 16, 1, D), dtype=torch.bfloat16)
    q_rot, _, bad = oracle.rope_kv_append(q_bf16, k, k, pool, torch.ones((B, 1), dtype=torch.int32),
                                          torch.ones(B, dtype=torch.int32), torch.ones(B, dtype=torch.int32),
                                          P=16, theta=10000.0, positions=torch.full((B,), pos), q_norm_w=w,
                                          norm_eps=eps)
    assert bad == 0
    return q_rot


def test_rms_norm_matches_torch_rms_norm():
    g = torch.Generator().manual_seed(30)
    for D in (64, 128):
        q = torch.randn((3, 4, D), generator=g).to(torch.bfloat16)
        w = _norm_weights(D, D)
        got = _q_path(q, 0, w, 1e-6)  # position 0: RoPE is the identity
        ref = torch.nn.functional.rms_norm(q.double(), (D,), weight=w.double(), eps=1e-6)
        assert torch.allclose(got, ref, atol=1e-14, rtol=1e-14)


def test_rms_norm_closed_forms():
    D = 64
    w = _norm_weights(D, 1)
    c = torch.full((1, 1, D), -3.0).to(torch.bfloat16)  # constant vector: rms = |c|
    got = _q_path(c, 0, w, 0.0)[0, 0]
    assert torch.allclose(got, -w.double(), atol=1e-15)
    # invariance to positive scaling (eps = 0), and unit RMS with unit weights
    x = torch.randn((1, 2, D), generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    a = _q_path(x, 0, torch.ones(D), 0.0)
    b = _q_path((x.float() * 4).to(torch.bfloat16), 0, torch.ones(D), 0.0)
    assert torch.allclose(a, b, atol=1e-15)
    assert torch.allclose(a.pow(2).mean(-1), torch.ones((1, 2), dtype=torch.float64), atol=1e-14)
    # RoPE after the norm keeps the unit RMS (a rotation)
    r = _q_path(x, 777, torch.ones(D), 0.0)
    assert torch.allclose(r.pow(2).mean(-1), torch.ones((1, 2), dtype=torch.float64), atol=1e-14)


def test_rms_norm_step_matches_brute_force():
    inp = _small_case([17, 5, 33], Hq=4, Hkv=2, D=8, P=16, seed=31)
    qw, kw = _norm_weights(8, 3), _norm_weights(8, 4)
    r = oracle.reference_step(inp, q_norm_w=qw, k_norm_w=kw, norm_eps=1e-5)
    pool = _nested(inp.pool)
    q_rot, out = brute.step(_nested(inp.q), _nested(inp.k_new), _nested(inp.v_new), pool,
                            inp.page_table.tolist(), inp.seq_lens.tolist(), inp.active.tolist(),
                            inp.P, inp.theta, q_norm_w=qw.double().tolist(), k_norm_w=kw.double().tolist(),
                            eps=1e-5)
    assert torch.allclose(r["q_rot"], torch.tensor(q_rot, dtype=torch.float64), atol=1e-12, rtol=0)
    assert torch.allclose(r["out"], torch.tensor(out, dtype=torch.float64), atol=1e-12, rtol=0)
    assert _nested(r["pool_after"]) == pool
    # and the key fed to RoPE is the normalised key
    kp = r["k_pre"][0, 1]
    ref = torch.nn.functional.rms_norm(inp.k_new[0, 1].double().view(1, -1), (8,), weight=kw.double(), eps=1e-5)
    assert torch.allclose(kp, ref.view(-1), atol=1e-14)


# ---------------------------------------------------------------- fp16 element type

@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3C00),
    (-2.0, 0xC000),
    (1.0 + 2 ** -11, 0x3C00),              # midpoint between 0x3C00 (even) and 0x3C01: down
    (1.0 + 3 * 2 ** -11, 0x3C02),          # midpoint between 0x3C01 (odd) and 0x3C02: up
    (1.0 + 2 ** -11 + 2 ** -40, 0x3C01),   # just above the midpoint: up
    (65504.0, 0x7BFF),                     # largest finite
    (65519.99, 0x7BFF),                    # below the midpoint to 2^16: stays finite
    (65520.0, 0x7C00),                     # the midpoint itself rounds to even = inf
    (2 ** -24, 0x0001),                    # smallest subnormal
    (2 ** -25, 0x0000),                    # half of it: tie to even (zero)
    (3 * 2 ** -25, 0x0002),                # 1.5 quanta: tie to even (2)
    (2 ** -14, 0x0400),                    # smallest normal
    (2 ** -14 - 2 ** -25, 0x0400),         # midpoint below it: rounds up to the even normal
    (0.0, 0x0000),
    (-0.0, 0x8000),
])
def test_f16_rounding_fixed_points(x, bits):
    assert oracle.f16_from_double(x) == bits
    assert brute.f16_round_bits(x) == bits


def test_f16_decode_every_pattern():
    # every finite / infinite binary16 pattern against Python's own half codec
    import struct
    for bits in range(0x10000):
        want = struct.unpack("<e", struct.pack("<H", bits))[0]
        got = oracle.f16_to_double(bits)
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), hex(bits)


def test_f16_rounding_matches_exact_bracketing_and_numpy():
    np = pytest.importorskip("numpy")
    g = torch.Generator().manual_seed(17)
    xs = (torch.randn(2000, generator=g, dtype=torch.float64) * 8).tolist()
    xs += (torch.randn(500, generator=g, dtype=torch.float64) * 2 ** -18).tolist()   # subnormals
    xs += (torch.randn(200, generator=g, dtype=torch.float64) * 3e4).tolist()        # near overflow
    for bits in list(range(0x3C00, 0x3C40)) + list(range(0x0001, 0x0020)) + [0x7BFE]:
        a, b = brute.f16_bits_to_float(bits), brute.f16_bits_to_float(bits + 1)
        xs.append((a + b) / 2)
    for x in xs:
        o = oracle.f16_from_double(x)
        assert o == brute.f16_round_bits(x), x
        # numpy converts float64 -> float16 in one correctly rounded step
        with np.errstate(over="ignore"):
            want = int(np.array([x], dtype=np.float64).astype(np.float16).view(np.uint16)[0])
        assert o == want, x


def _fp16_case(lens, **kw):
    return _small_case(lens, dtype=torch.float16, **kw)


def test_fp16_attention_matches_torch_sdpa_on_fp16_cache():
    inp = _fp16_case([70, 3, 33], D=64, Hq=4, Hkv=4, seed=3)
    r = _step(inp)
    assert r["pool_after"].dtype == torch.float16
    for b in range(inp.B):
        L = int(inp.seq_lens[b])
        idx = [(int(inp.page_table[b, j // inp.P]), j % inp.P) for j in range(L)]
        K = torch.stack([_f64(r["pool_after"][p, 0, o]) for p, o in idx], dim=1)
        V = torch.stack([_f64(r["pool_after"][p, 1, o]) for p, o in idx], dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(r["q_rot"][b].unsqueeze(1), K, V).squeeze(1)
        assert torch.allclose(r["out"][b], ref, atol=1e-13, rtol=0)
    # the appended key is the fp16 rounding of the rotated key (not the bf16 one)
    b = 1
    L = int(inp.seq_lens[b])
    page, off = int(inp.page_table[b, (L - 1) // inp.P]), (L - 1) % inp.P
    want = [oracle.f16_from_double(v) for v in r["k_rot"][b].flatten().tolist()]
    assert _bits(r["pool_after"][page, 0, off]).flatten().tolist() == want
    assert torch.equal(_bits(r["pool_after"][page, 1, off]), _bits(inp.v_new[b]))


def test_fp16_inputs_are_read_as_fp16():
    # the same float32 draws as bf16 and as fp16 give different q_rot (values
    # read in the wrong format would be garbage, not a small difference)
    a = _small_case([20], D=16, seed=5)
    b = _fp16_case([20], D=16, seed=5)
    ra, rb = _step(a), _step(b)
    assert torch.allclose(ra["q_rot"], rb["q_rot"], atol=0.05)
    assert not torch.equal(ra["q_rot"], rb["q_rot"])
    assert torch.equal(rb["q_rot"][0], oracle.rope_kv_append(
        b.q, b.k_new, b.v_new, b.pool, b.page_table, b.seq_lens, b.active, P=b.P,
        theta=b.theta)[0][0])


# ---------------------------------------------------------------- interleaved RoPE

def test_interleaved_rope_is_complex_rotation():
    # GPT-J pairing: (x_2i + i x_2i+1) * exp(i pos theta^(-2i/D)), in complex128
    g = torch.Generator().manual_seed(31)
    D, theta = 64, 10000.0
    for dtype in (torch.bfloat16, torch.float16):
        q = torch.randn((2, 3, D), generator=g).to(dtype)
        k = torch.randn((2, 1, D), generator=g).to(dtype)
        pool = torch.zeros((4, 2, 16, 1, D), dtype=dtype)
        pos = torch.tensor([0, 4097])
        q_rot, _, bad, k_rot = oracle.rope_kv_append(
            q, k, k, pool, torch.tensor([[1], [2]]), torch.tensor([1, 1]), torch.tensor([1, 1]), P=16,
            theta=theta, positions=pos, return_k_rot=True, interleaved=True)
        assert bad == 0
        freq = theta ** (-2.0 * torch.arange(D // 2, dtype=torch.float64) / D)
        for x, got in ((q, q_rot), (k, k_rot)):
            z = torch.view_as_complex(x.to(torch.float64).reshape(2, x.shape[1], D // 2, 2).contiguous())
            rot = torch.polar(torch.ones_like(freq), pos.to(torch.float64).view(2, 1, 1) * freq)
            want = torch.view_as_real(z * rot).reshape(2, x.shape[1], D)
            assert torch.allclose(got, want, atol=1e-12, rtol=0)


def test_interleaved_is_rotate_half_on_deinterleaved_vectors():
    # permuting (2i, 2i+1) -> (i, i + D/2) turns one pairing into the other
    inp = _small_case([40, 7], D=32, Hq=4, Hkv=2, seed=9)
    D = inp.D
    perm = torch.cat([torch.arange(0, D, 2), torch.arange(1, D, 2)])   # new[j] = old[perm[j]]
    r_int = oracle.reference_step(inp, interleaved=True)
    de = inp.clone()
    de.q = inp.q[..., perm].contiguous()
    de.k_new = inp.k_new[..., perm].contiguous()
    de.v_new = inp.v_new[..., perm].contiguous()
    de.pool = inp.pool[..., perm].contiguous()
    r_half = oracle.reference_step(de)
    inv = torch.argsort(perm)
    assert torch.equal(r_half["q_rot"][..., inv], r_int["q_rot"])
    assert torch.equal(_bits(r_half["pool_after"][..., inv]), _bits(r_int["pool_after"]))
    assert torch.allclose(r_half["out"][..., inv], r_int["out"], atol=1e-14, rtol=0)
    # and the two pairings do differ on the same vectors
    assert not torch.allclose(oracle.reference_step(inp)["q_rot"], r_int["q_rot"])


@pytest.mark.parametrize("dtype,interleaved,norm", [
    ("fp16", False, False), ("fp16", True, False), ("bf16", True, False), ("fp16", True, True)])
def test_fp16_and_interleaved_step_matches_brute_force(dtype, interleaved, norm):
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    inp = _small_case([17, 5, 33], Hq=4, Hkv=2, D=8, P=16, seed=23, dtype=tdt)
    qw = kw = None
    if norm:
        qw, kw = _norm_weights(inp.D, 1), _norm_weights(inp.D, 2)
    r = oracle.reference_step(inp, interleaved=interleaved, q_norm_w=qw, k_norm_w=kw)
    pool = _nested(inp.pool)
    q_rot, out = brute.step(_nested(inp.q), _nested(inp.k_new), _nested(inp.v_new), pool,
                            inp.page_table.tolist(), inp.seq_lens.tolist(), inp.active.tolist(),
                            inp.P, inp.theta, dtype=dtype, interleaved=interleaved,
                            q_norm_w=None if qw is None else qw.tolist(),
                            k_norm_w=None if kw is None else kw.tolist())
    assert torch.allclose(r["q_rot"], torch.tensor(q_rot, dtype=torch.float64), atol=1e-12, rtol=0)
    assert torch.allclose(r["out"], torch.tensor(out, dtype=torch.float64), atol=1e-12, rtol=0)
    assert _nested(r["pool_after"]) == pool
