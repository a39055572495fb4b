"""Parity of the CUDA paths (through the C interface) with the float64 oracle.

Both paths are checked: the three calls (RoPE + append, attention, combine)
and the fused one-launch step.  All five serving workloads at full size,
plus edge cases: single-key rows,
exact-tile lengths, the maximum length, padding batches, every GQA group
size, head_dim 64 and 128, several page sizes, head groups split across
CTAs, forced split counts, explicit positions and scale, CUDA-graph replay,
and device-side data-error flags.
"""
import pytest
import torch

import gpu_harness as H
import oracle
import workloads

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- the five workloads

@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("name", ["tiny", "c64", "padded", "long"])
def test_workload_full_parity(name, path):
    inp = workloads.make_inputs(name, device="cuda")
    r = H.full_check(inp, path=path)
    print(f"{name}: out max|d| {r['out_err']:.2e}, q_rot max|d| {r['q_rot_err']:.2e}, "
          f"midpoint-exempt K elements {r['exempt']} (differing {r['n_diff']})")


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("layer", [0, 13, 27])
def test_high_concurrency_layers(layer, path):
    # 256 rows, pages of 64; every row checked (the oracle runs a layer in seconds)
    inp = workloads.make_inputs("high", layer=layer, device="cuda")
    H.full_check(inp, path=path)


@pytest.mark.parametrize("path", H.PATHS)
def test_padded_live_pages_bit_identical_outside_appended_slots(path):
    inp = workloads.make_inputs("padded", device="cuda")
    before = H.bits16(inp.pool.cpu())
    got = H.run_step(inp, path=path)
    after = H.bits16(got["pool_after"])
    changed = before != after
    allowed = torch.zeros_like(changed)
    act = inp.active.cpu().bool()
    lens, pt = inp.seq_lens.cpu(), inp.page_table.cpu()
    for b in torch.nonzero(act).flatten().tolist():
        L = int(lens[b])
        allowed[int(pt[b, (L - 1) // inp.P]), :, (L - 1) % inp.P] = True
    assert not (changed & ~allowed).any()
    assert not changed[0].any(), "dummy page 0 was written"
    assert torch.equal(got["out"][~act], torch.zeros_like(got["out"][~act]))


# ---------------------------------------------------------------- edge cases

def case(lens, *, active=None, Hq=8, Hkv=2, D=128, P=16, seed=1, mps=None, **kw):
    return workloads.make_case(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, P=P, seq_lens=lens, active=active,
                               max_pages_per_seq=mps, seed=seed, device="cuda", **kw)


@pytest.mark.parametrize("path", H.PATHS)
def test_single_key_rows_return_v_new_bit_exactly(path):
    inp = case([1, 1, 1, 1, 1], Hq=16, Hkv=8)
    r = H.full_check(inp, path=path)
    G = inp.Hq // inp.Hkv
    v_new = inp.v_new.cpu()
    for g in range(inp.Hq):
        assert torch.equal(r["got"]["out"][:, g], v_new[:, g // G])


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("lens", [[16, 32, 48, 160], [15, 17, 31, 33], [2, 3, 4, 1000], [4096, 1, 77]])
def test_tile_boundaries(lens, path):
    H.full_check(case(lens, seed=sum(lens)), path=path)


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_gqa_groups_and_head_dims(G, D, path):
    Hkv = 2
    H.full_check(case([37, 300, 129, 1], Hq=G * Hkv, Hkv=Hkv, D=D, seed=G * 10 + D), path=path)


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("P", [8, 16, 32, 64, 128, 256, 512, 1024])
def test_page_sizes(P, path):
    H.full_check(case([1, P - 1, P, P + 1, 3 * P + 5], P=P, Hq=8, Hkv=4, seed=P), path=path)


@pytest.mark.parametrize("path", H.PATHS)
def test_head_groups_split_across_ctas(path):
    # Hkv * D > 1024: several CTAs per tile range, each owning a group of kv heads
    H.full_check(case([200, 513, 17], Hq=32, Hkv=16, D=128, seed=5), path=path)
    H.full_check(case([90, 33], Hq=32, Hkv=32, D=64, seed=6), path=path)
    H.full_check(case([300, 41], Hq=64, Hkv=8, D=128, seed=7), path=path)   # G = 8


@pytest.mark.parametrize("path", H.PATHS)
def test_maximum_length_row(path):
    mps = 64
    H.full_check(case([mps * 16, 5, mps * 16 - 1], mps=mps, seed=7), path=path)


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("num_ctas", [1, 2, 3, 7, 64, 1000])
def test_forced_cta_counts_agree(num_ctas, path):
    inp = workloads.make_inputs("c64", device="cuda")
    H.full_check(inp, num_ctas=num_ctas, path=path)


@pytest.mark.parametrize("path", H.PATHS)
def test_rows_split_into_many_pieces(path):
    # 700 CTAs per head group: rows of up to 512 tiles split into ~70 pieces,
    # so the fused merge takes several rounds of staged pieces (8 per round at
    # G = 4) and the three-call combine several register batches
    inp = workloads.make_inputs("long", device="cuda")
    H.full_check(inp, num_ctas=700, path=path)


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_many_pieces_every_group_and_head_dim(G, D, path):
    # a 3000-token and a 700-token row over 96 CTAs per head group: the long
    # row splits into ~78 pieces, so the fused merge stages them through
    # shared memory in every slice layout (one 2 KB slice per piece, two at
    # G = 8 and head_dim 128; 8 pieces per round at head_dim 128, 4 at 64)
    H.full_check(case([3000, 700, 5], Hq=G * 4, Hkv=4, D=D, seed=200 + G * 10 + D), path=path, num_ctas=96)


@pytest.mark.parametrize("path", H.PATHS)
def test_single_very_long_row(path):
    # one row of 32768 tokens (2048 tiles) with G = 4: every CTA of a head
    # group takes a piece of it, so one CTA merges ~150 pieces
    inp = case([32768], Hq=32, Hkv=8, seed=11)
    H.full_check(inp, path=path)


def test_split_count_changes_only_rounding():
    inp = workloads.make_inputs("long", device="cuda")
    a = H.run_step(inp, num_ctas=1)["out"].double()
    b = H.run_step(inp, num_ctas=500)["out"].double()
    # each side is within ATOL + RTOL |ref| of the oracle, so they agree to twice that
    assert ((a - b).abs() <= 2 * (H.ATOL + H.RTOL * a.abs())).all()


@pytest.mark.parametrize("path", H.PATHS)
def test_explicit_positions_and_scale(path):
    inp = case([40, 300, 2], seed=9)
    pos = torch.tensor([7, 1000, 0], dtype=torch.int32)
    H.full_check(inp, positions=pos, sm_scale=0.05, max_pos=2048, path=path)


@pytest.mark.parametrize("path", H.PATHS)
def test_all_padding_batch(path):
    inp = case([1, 1, 1], active=[0, 0, 0], seed=10)
    r = H.full_check(inp, path=path)
    assert not r["got"]["out"].any()


@pytest.mark.parametrize("path", H.PATHS)
def test_batch_of_one_and_deterministic(path):
    inp = case([777], seed=11)
    a = H.run_step(inp, path=path)
    b = H.run_step(inp, path=path)
    assert torch.equal(a["out"], b["out"])
    if path == "three":
        assert torch.equal(a["q_rot"], b["q_rot"])
    H.full_check(inp, path=path)


@pytest.mark.parametrize("path", H.PATHS)
def test_cuda_graph_replay_matches(path):
    inp = workloads.make_inputs("padded", device="cuda")
    H.full_check(inp, graph=True, path=path)


def test_fused_repeated_calls_reuse_the_workspace():
    # the per-row counters of the fused merge must come back to zero after each call
    inp = workloads.make_inputs("long", device="cuda")
    H.full_check(inp, path="fused", repeat=3)
    H.full_check(inp, path="fused", repeat=2, num_ctas=500)


@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("name", ["tiny", "c64", "padded", "long", "high"])
def test_fused_programmatic_dependent_launch(name, graph):
    # back-to-back fused launches, each a programmatic dependent of the previous one
    inp = workloads.make_inputs(name, device="cuda")
    H.full_check(inp, path="fused", repeat=3, pdl=True, graph=graph)


def test_fused_and_three_call_paths_agree():
    inp = workloads.make_inputs("c64", device="cuda")
    a = H.run_step(inp, path="three")
    b = H.run_step(inp, path="fused")
    assert torch.equal(H.bits16(a["pool_after"]), H.bits16(b["pool_after"]))
    d, r = a["out"].double(), b["out"].double()
    assert ((d - r).abs() <= 2 * (H.ATOL + H.RTOL * r.abs())).all()


@pytest.mark.parametrize("path", H.PATHS)
def test_identical_keys_give_mean_of_values(path):
    inp = case([300, 45], seed=12, poison=True)
    # set every live cached key of kv head 0 to one vector; values stay random
    key = torch.randn(inp.D, device="cuda").to(torch.bfloat16)
    inp.pool[:, 0, :, 0] = torch.where(torch.isnan(inp.pool[:, 0, :, 0].float()), inp.pool[:, 0, :, 0], key)
    H.full_check(inp, path=path)


# ---------------------------------------------------------------- device-side data errors

def _err_run(inp, **kw):
    return H.run_step(inp, **kw)


@pytest.mark.parametrize("path", H.PATHS)
def test_seq_len_out_of_range_is_flagged_and_row_zeroed(path):
    inp = case([50, 60, 70], seed=13)
    inp.seq_lens[1] = inp.max_pages_per_seq * inp.P + 5
    inp.seq_lens[2] = 0
    got = _err_run(inp, path=path)
    assert got["err"] & 1
    assert not got["out"][1:].any()
    # the healthy row is still right
    cpu = inp.to("cpu")
    act = cpu.active.clone()
    act[1:] = 0
    ref = oracle.reference_step(workloads.DecodeInputs(**{**cpu.__dict__, "active": act}))
    H.check_out(workloads.DecodeInputs(**{**cpu.__dict__, "active": act}), ref["out"], got["out"], rows=[0])


@pytest.mark.parametrize("path", H.PATHS)
def test_page_id_out_of_range_is_flagged_without_writes(path):
    inp = case([20, 20], seed=14)
    before = H.bits16(inp.pool.cpu())
    inp.page_table[1, 1] = inp.num_pages + 3   # the page of row 1's new token
    got = _err_run(inp, path=path)
    assert got["err"] & 2
    after = H.bits16(got["pool_after"])
    changed = (before != after).nonzero()
    # only row 0's slot may change
    p0, off0 = int(inp.page_table[0, 1]), 19 % 16
    assert all(int(c[0]) == p0 and int(c[2]) == off0 for c in changed)


@pytest.mark.parametrize("path", H.PATHS)
def test_position_beyond_table_is_flagged(path):
    inp = case([20, 30], seed=15)
    pos = torch.tensor([3, 10_000], dtype=torch.int32)
    got = H.run_step(inp, positions=pos, max_pos=64, path=path)
    assert got["err"] & 4
    if path == "fused":
        assert not got["out"][1].any(), "a row with an invalid position is treated as padding"


@pytest.mark.parametrize("path", H.PATHS)
def test_large_batch_of_short_rows(path):
    # 2048 rows: the prologue scans eight rows per thread; many rows per CTA
    g = torch.Generator().manual_seed(17)
    lens = torch.randint(1, 48, (2048,), generator=g).tolist()
    active = (torch.rand(2048, generator=g) > 0.1).to(torch.int64).tolist()
    lens = [L if a else 1 for L, a in zip(lens, active)]
    inp = workloads.make_case(B=2048, Hq=8, Hkv=4, D=128, P=16, seq_lens=lens, active=active, seed=18,
                              device="cuda", max_pages_per_seq=3)
    H.full_check(inp, path=path)


@pytest.mark.parametrize("path", H.PATHS)
def test_batch_near_the_shared_memory_limit(path):
    # 12,000 rows: every CTA keeps 12 bytes per row (tile count, length,
    # position) in shared memory, 144 KB here, next to its pipeline stages
    g = torch.Generator().manual_seed(19)
    B = 12000
    lens = torch.randint(1, 41, (B,), generator=g).tolist()
    active = (torch.rand(B, generator=g) > 0.1).to(torch.int64).tolist()
    lens = [L if a else 1 for L, a in zip(lens, active)]
    inp = workloads.make_case(B=B, Hq=4, Hkv=2, D=64, P=16, seq_lens=lens, active=active, seed=20,
                              device="cuda", max_pages_per_seq=3)
    H.full_check(inp, path=path)


# ---------------------------------------------------------------- per-head RMSNorm before RoPE

def _norm(D, seed, eps=1e-6):
    g = torch.Generator().manual_seed(seed)
    return {"q": (1.0 + 0.2 * torch.randn(D, generator=g)).float(),
            "k": (1.0 + 0.2 * torch.randn(D, generator=g)).float(), "eps": eps}


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("name", ["tiny", "c64", "long", "high"])
def test_qk_rms_norm_parity(name, path):
    inp = workloads.make_inputs(name, device="cuda")
    H.full_check(inp, path=path, norm=_norm(inp.D, 40 + inp.D))


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_qk_rms_norm_groups_and_dims(G, D, path):
    inp = case([37, 300, 129, 1], Hq=G * 2, Hkv=2, D=D, seed=G * 10 + D + 1)
    H.full_check(inp, path=path, norm=_norm(D, G + D, eps=1e-5))


@pytest.mark.parametrize("path", H.PATHS)
def test_qk_rms_norm_of_q_only(path):
    inp = case([77, 16, 5], seed=41)
    nm = _norm(inp.D, 41)
    H.full_check(inp, path=path, norm={"q": nm["q"], "k": None, "eps": 1e-6})


# ---------------------------------------------------------------- fp16 elements and interleaved RoPE

F16 = torch.float16


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("name", ["tiny", "c64", "padded", "long"])
def test_fp16_workload_parity(name, path):
    inp = workloads.make_inputs(name, device="cuda", dtype=F16)
    r = H.full_check(inp, path=path)
    assert r["got"]["out"].dtype == F16
    print(f"{name} fp16: out max|d| {r['out_err']:.2e}, exempt {r['exempt']} (differing {r['n_diff']})")


@pytest.mark.parametrize("path", H.PATHS)
def test_fp16_high_concurrency_layer(path):
    inp = workloads.make_inputs("high", layer=5, device="cuda", dtype=F16)
    H.full_check(inp, path=path)


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("dtype", [torch.bfloat16, F16])
@pytest.mark.parametrize("name", ["tiny", "c64", "long"])
def test_interleaved_rope_parity(name, dtype, path):
    inp = workloads.make_inputs(name, device="cuda", dtype=dtype)
    H.full_check(inp, path=path, interleaved=True)


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_fp16_groups_and_dims(G, D, interleaved, path):
    inp = case([37, 300, 129, 1, 16], Hq=G * 2, Hkv=2, D=D, seed=G * 7 + D, dtype=F16)
    H.full_check(inp, path=path, interleaved=interleaved)


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("dtype", [torch.bfloat16, F16])
def test_interleaved_rope_with_qk_norm(dtype, path):
    inp = case([200, 33, 1, 64], Hq=16, Hkv=8, seed=51, dtype=dtype)
    H.full_check(inp, path=path, norm=_norm(inp.D, 52), interleaved=True)


@pytest.mark.parametrize("path", H.PATHS)
def test_fp16_single_key_rows_return_v_new_bit_exactly(path):
    inp = case([1, 1, 1], Hq=16, Hkv=8, dtype=F16)
    r = H.full_check(inp, path=path, interleaved=True)
    G = inp.Hq // inp.Hkv
    for g in range(inp.Hq):
        assert torch.equal(H.bits16(r["got"]["out"][:, g]), H.bits16(inp.v_new.cpu()[:, g // G]))


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("num_ctas", [1, 3, 64, 1000])
def test_fp16_forced_cta_counts(num_ctas, path):
    # split rows are merged into fp16 by the combine kernel / the fused merge
    inp = case([1500, 7, 640, 33], Hq=16, Hkv=8, seed=61, dtype=F16)
    H.full_check(inp, path=path, num_ctas=num_ctas)


@pytest.mark.parametrize("graph", [False, True])
def test_fp16_fused_programmatic_dependent_launch(graph):
    inp = workloads.make_inputs("c64", device="cuda", dtype=F16)
    H.full_check(inp, path="fused", pdl=True, graph=graph, interleaved=True)


@pytest.mark.parametrize("path", H.PATHS)
def test_fp16_wide_value_range(path):
    # keys scaled up (large, peaked scores) and values spread from fp16
    # subnormals (below 2^-14) to a few thousand, all exactly representable
    inp = case([90, 300, 17], Hq=8, Hkv=2, seed=71, dtype=F16)
    g = torch.Generator(device="cuda").manual_seed(72)
    scale = torch.exp2(torch.randint(-20, 12, inp.pool[:, 1].shape, generator=g, device="cuda").float())
    nan = torch.isnan(inp.pool.float())
    inp.pool[:, 1] = (inp.pool[:, 1].float() * scale).to(F16)
    inp.pool[:, 0] = (inp.pool[:, 0].float() * 6.0).to(F16)
    inp.pool[nan] = float("nan")                      # keep the stale slots poisoned
    inp.v_new.mul_(1e-6)
    r = H.full_check(inp, path=path)
    assert torch.isfinite(r["got"]["out"].float()).all()


def test_fp16_fused_and_three_call_paths_agree():
    inp = workloads.make_inputs("c64", device="cuda", dtype=F16)
    a = H.run_step(inp, path="three", interleaved=True)
    b = H.run_step(inp, path="fused", interleaved=True)
    assert torch.equal(H.bits16(a["pool_after"]), H.bits16(b["pool_after"]))
    d = (a["out"].double() - b["out"].double()).abs()
    assert (d <= 2e-3 + 1e-2 * a["out"].double().abs()).all()


# ---------------------------------------------------------------- head-major (HND) pages

@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("name", ["tiny", "c64", "padded", "long"])
def test_head_major_pages_workload_parity(name, path):
    inp = workloads.make_inputs(name, device="cuda", layout="HND")
    assert inp.pool.shape[2] == inp.Hkv and inp.head_stride == inp.P * inp.D
    H.full_check(inp, path=path)


@pytest.mark.parametrize("path", H.PATHS)
def test_head_major_pages_high_concurrency_layer(path):
    inp = workloads.make_inputs("high", layer=9, device="cuda", layout="HND")
    H.full_check(inp, path=path)


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_head_major_pages_groups_and_dims(G, D, path):
    inp = case([37, 300, 129, 1, 16], Hq=G * 2, Hkv=2, D=D, seed=G * 5 + D + 3, layout="HND")
    H.full_check(inp, path=path)


@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("P", [16, 64, 256])
def test_head_major_pages_sizes_fp16_interleaved_norm(P, path):
    inp = case([P * 3 + 5, 17, 1, 2 * P], Hq=16, Hkv=8, P=P, seed=P + 80, layout="HND", dtype=torch.float16)
    H.full_check(inp, path=path, interleaved=True, norm=_norm(inp.D, P))


@pytest.mark.parametrize("path", H.PATHS)
def test_head_major_and_token_major_pages_agree_bit_for_bit(path):
    a = workloads.make_inputs("c64", device="cuda")
    b = workloads.make_inputs("c64", device="cuda", layout="HND")
    assert torch.equal(H.bits16(b.nhd_pool().cpu()), H.bits16(a.pool.cpu()))
    ra = H.run_step(a, path=path)
    rb = H.run_step(b, path=path)
    # the same copies land in the same shared-memory rows: identical results
    assert torch.equal(H.bits16(ra["out"]), H.bits16(rb["out"]))
    assert torch.equal(H.bits16(ra["pool_after"]), H.bits16(rb["pool_after"]))


@pytest.mark.parametrize("path", H.PATHS)
def test_head_major_padding_rows_leave_page_zero_alone(path):
    inp = workloads.make_inputs("padded", device="cuda", layout="HND")
    before = H.bits16(inp.nhd_pool().cpu())
    got = H.run_step(inp, path=path)
    assert torch.equal(H.bits16(got["pool_after"][0]), before[0]), "dummy page 0 was written"


# ---------------------------------------------------------------- cached K/V requested before the wait

@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("name", ["tiny", "c64", "padded", "long"])
def test_fused_kv_requested_before_dependency_wait(name, graph):
    # two identical calls in a row on one cache: the only slot the first call
    # writes is the one the second rewrites from k_new / v_new, so the second
    # may request its cached tiles before the first has completed
    inp = workloads.make_inputs(name, device="cuda")
    H.full_check(inp, path="fused", pdl=True, pdl_kv=True, graph=graph, repeat=2)


@pytest.mark.parametrize("layout", ["HND", "CONTIG"])
def test_fused_kv_requested_early_other_layouts(layout):
    name = "fastar" if layout == "CONTIG" else "c64"
    inp = workloads.make_inputs(name, device="cuda", layout=layout, dtype=torch.float16)
    H.full_check(inp, path="fused", pdl=True, pdl_kv=True, graph=True, repeat=3, interleaved=True)


# ---------------------------------------------------------------- batch-size limit of the plan

def test_batch_beyond_the_shared_memory_plan_is_rejected_on_the_host():
    v = H.vh()
    assert v.vh_decode_num_ctas(16384, 16, 8, 128, 16) > 0
    with pytest.raises(v.VHError) as e:
        v.vh_decode_num_ctas(20000, 16, 8, 128, 16)
    assert e.value.status == v.VH_EINVAL
    assert v.lib.vh_decode_workspace_bytes(20000, 16, 8, 128, 16, 0) == 0


@pytest.mark.parametrize("path", H.PATHS)
def test_batch_near_the_plan_limit(path):
    # 16384 one-token and short rows, a quarter of them padding
    g = torch.Generator().manual_seed(90)
    B = 16384
    act = (torch.rand(B, generator=g) > 0.25).int().tolist()
    lens = [int(x) if a else 1 for x, a in zip(torch.randint(1, 40, (B,), generator=g).tolist(), act)]
    inp = workloads.make_case(B=B, Hq=2, Hkv=1, D=64, P=16, seq_lens=lens, active=act, seed=91,
                              device="cuda", max_pages_per_seq=3)
    rows = list(range(0, B, 97))  # the oracle checks a sample of rows; the append is checked everywhere
    H.full_check(inp, path=path, rows=rows)


# ---------------------------------------------------------------- fallback tile copies

@pytest.mark.parametrize("path", H.PATHS)
@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_one_head_box_fallback(layout, path, monkeypatch):
    # the copy path used if the tensor-map encoder rejected the multi-head box
    # order: every tile as one-head 8-token boxes, dimensions in stride order
    monkeypatch.setenv("VH_TMA_BOX_HEADS", "1")
    inp = workloads.make_inputs("c64", device="cuda", layout=layout)
    H.full_check(inp, path=path)
    inp = case([17, 9, 300, 1], Hq=16, Hkv=8, D=64, seed=95, layout=layout, dtype=torch.float16)
    H.full_check(inp, path=path, interleaved=True)


# ---------------------------------------------------------------- launch plan

def test_launch_plan_keeps_two_ctas_per_sm():
    # the attention kernels are planned for two resident CTAs per SM (four kv
    # heads per CTA at head_dim 128, two pipeline stages): a plan whose shared
    # memory grows past half an SM halves the CTA count and the bandwidth
    v = H.vh()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    groups = 8 // 4
    assert v.vh_decode_num_ctas(64, 16, 8, 128, 16) == 2 * sms // groups
    assert v.vh_decode_num_ctas(256, 32, 8, 128, 64) == 2 * sms // groups
