"""The C interface without a GPU: the library loads, exports every function
include/vh.h declares, and rejects bad arguments on the host before any
device work (only argument combinations that fail validation are used, so
nothing here can launch a kernel)."""
import ctypes
import re

import pytest

import paged_len_decode_gb300 as v

FAKE = ctypes.c_void_p(0x10000)       # 16-byte aligned, never dereferenced
ODD = ctypes.c_void_p(0x10008)        # misaligned


def test_every_declared_function_is_exported():
    names = v.header_functions()
    assert set(names) >= {"vh_rope_table", "vh_rope_kv_append", "vh_decode_num_ctas",
                          "vh_decode_workspace_bytes", "vh_paged_decode_attn", "vh_decode_combine",
                          "vh_status_string"}
    for n in names:
        assert hasattr(v.lib, n), n


def test_header_declares_extern_c_and_status_codes():
    text = open(v.HEADER_PATH).read()
    assert 'extern "C"' in text
    for code, val in [("VH_OK", 0), ("VH_EINVAL", -1), ("VH_EALIGN", -2), ("VH_EWORKSPACE", -3),
                      ("VH_ECUDA", -4), ("VH_ENODEV", -5)]:
        assert re.search(rf"#define {code} \(?{val}\)?", text), code
        assert getattr(v, code) == val


def test_status_strings():
    assert v.vh_status_string(0) == "ok"
    assert "aligned" in v.vh_status_string(-2)
    assert v.vh_status_string(12345) == "unknown status"


def attn(**over):
    a = dict(q_rot=FAKE, k=FAKE, vv=FAKE, ps=2 * 16 * 8 * 128, ts=8 * 128, hs=128, npages=100, pt=FAKE, mps=10,
             sl=FAKE, act=FAKE, out=FAKE, scale=0.0, nctas=0, ws=FAKE, wsb=1 << 30, err=None, flags=0,
             B=4, Hq=16, Hkv=8, D=128, P=16)
    a.update(over)
    return v.lib.vh_paged_decode_attn(a["q_rot"], a["k"], a["vv"], a["ps"], a["ts"], a["hs"], a["npages"], a["pt"],
                                      a["mps"], a["sl"], a["act"], a["out"], a["scale"], a["nctas"], a["ws"],
                                      a["wsb"], a["err"], a["flags"], a["B"], a["Hq"], a["Hkv"], a["D"], a["P"],
                                      None)


@pytest.mark.parametrize("over,code", [
    (dict(q_rot=None), v.VH_EINVAL),
    (dict(out=None), v.VH_EINVAL),
    (dict(Hq=12, Hkv=8), v.VH_EINVAL),        # Hq % Hkv != 0
    (dict(Hq=24, Hkv=8), v.VH_EINVAL),        # G = 3
    (dict(D=96), v.VH_EINVAL),
    (dict(P=12), v.VH_EINVAL),               # multi-page rows: P a multiple of 16, or 8
    (dict(P=24), v.VH_EINVAL),
    (dict(B=0), v.VH_EINVAL),
    (dict(B=70000), v.VH_EINVAL),
    (dict(mps=0), v.VH_EINVAL),
    (dict(npages=0), v.VH_EINVAL),
    (dict(nctas=-1), v.VH_EINVAL),
    (dict(scale=float("nan")), v.VH_EINVAL),
    (dict(mps=1 << 22), v.VH_EINVAL),         # lengths beyond 2^24 tokens
    (dict(q_rot=ODD), v.VH_EALIGN),
    (dict(k=ODD), v.VH_EALIGN),
    (dict(ts=8 * 128 + 4), v.VH_EALIGN),      # stride not a multiple of 16 bytes
    (dict(hs=0), v.VH_EINVAL),
    (dict(hs=68), v.VH_EALIGN),               # head stride not a multiple of 16 bytes
    (dict(ws=None), v.VH_EWORKSPACE),
    (dict(ws=ODD), v.VH_EALIGN),
    (dict(flags=v.VH_FLAG_PDL_KV), v.VH_EINVAL),              # not a flag of this call
    (dict(flags=v.VH_FLAG_ROPE_INTERLEAVED), v.VH_EINVAL),    # nor this one (no RoPE here)
    (dict(flags=8), v.VH_EINVAL),
    (dict(flags=v.VH_FLAG_PLAN_THREE_CALL), v.VH_EINVAL),    # a flag of vh_decode_plan only
    (dict(flags=v.VH_FLAG_HOST_IO), v.VH_EINVAL),            # a flag of vh_decode_fused only
    (dict(flags=v.VH_FLAG_PLANNED, ws=None), v.VH_EWORKSPACE),  # the plan lives in the workspace
    (dict(flags=v.VH_FLAG_FP16, q_rot=ODD), v.VH_EALIGN),     # fp16 passes the flag check
])
def test_attention_argument_checks(over, code):
    assert attn(**over) == code


def test_valid_arguments_without_device_report_no_device():
    # all host checks pass; the device query then fails on a GPU-less machine
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert attn() == v.VH_ENODEV


def test_rope_append_argument_checks():
    f = v.lib.vh_rope_kv_append

    def call(**over):
        a = dict(q=FAKE, k=FAKE, vv=FAKE, cs=FAKE, max_pos=4096, pos=None, qw=None, kw=None, eps=1e-6,
                 kc=FAKE, vc=FAKE, ps=2 * 16 * 8 * 128, ts=128, hs=16 * 128, npages=100, pt=FAKE, mps=10,
                 sl=FAKE, act=FAKE, q_rot=FAKE, err=None, flags=0, B=4, Hq=16, Hkv=8, D=128, P=16)
        a.update(over)
        return f(a["q"], a["k"], a["vv"], a["cs"], a["max_pos"], a["pos"], a["qw"], a["kw"], a["eps"], a["kc"],
                 a["vc"], a["ps"], a["ts"], a["hs"], a["npages"], a["pt"], a["mps"], a["sl"], a["act"], a["q_rot"],
                 a["err"], a["flags"], a["B"], a["Hq"], a["Hkv"], a["D"], a["P"], None)

    assert call(cs=None) == v.VH_EINVAL
    assert call(max_pos=0) == v.VH_EINVAL
    assert call(D=80) == v.VH_EINVAL
    assert call(eps=-1.0) == v.VH_EINVAL
    assert call(eps=float("nan")) == v.VH_EINVAL
    assert call(q=ODD) == v.VH_EALIGN
    assert call(q_rot=ODD) == v.VH_EALIGN
    assert call(qw=ODD) == v.VH_EALIGN
    assert call(kw=ODD) == v.VH_EALIGN
    assert call(flags=v.VH_FLAG_PDL) == v.VH_EINVAL
    assert call(flags=16) == v.VH_EINVAL
    assert call(flags=v.VH_FLAG_FP16 | v.VH_FLAG_ROPE_INTERLEAVED, q=ODD) == v.VH_EALIGN
    assert call(hs=-8) == v.VH_EINVAL
    assert call(hs=16 * 128 + 2) == v.VH_EALIGN


def test_fused_argument_checks():
    f = v.lib.vh_decode_fused

    def call(**over):
        a = dict(q=FAKE, k=FAKE, vv=FAKE, cs=FAKE, max_pos=4096, pos=None, qw=None, kw=None, eps=1e-6,
                 kc=FAKE, vc=FAKE, ps=2 * 16 * 8 * 128, ts=8 * 128, hs=128, npages=100, pt=FAKE, mps=10,
                 sl=FAKE, act=FAKE, out=FAKE, scale=0.0, nctas=0, ws=FAKE, wsb=1 << 30, err=None, flags=0,
                 B=4, Hq=16, Hkv=8, D=128, P=16)
        a.update(over)
        return f(a["q"], a["k"], a["vv"], a["cs"], a["max_pos"], a["pos"], a["qw"], a["kw"], a["eps"], a["kc"],
                 a["vc"], a["ps"], a["ts"], a["hs"], a["npages"], a["pt"], a["mps"], a["sl"], a["act"], a["out"], a["scale"],
                 a["nctas"], a["ws"], a["wsb"], a["err"], a["flags"], a["B"], a["Hq"], a["Hkv"], a["D"], a["P"],
                 None)

    assert call(q=None) == v.VH_EINVAL
    assert call(flags=128) == v.VH_EINVAL          # unknown flag
    assert call(flags=v.VH_FLAG_PLAN_THREE_CALL) == v.VH_EINVAL   # a flag of vh_decode_plan only
    assert call(flags=v.VH_FLAG_HOST_IO, q=ODD) == v.VH_EALIGN    # host I/O passes the flag check
    assert call(flags=v.VH_FLAG_PDL_KV, out=ODD) == v.VH_EALIGN
    assert call(flags=v.VH_FLAG_PDL | v.VH_FLAG_FP16 | v.VH_FLAG_ROPE_INTERLEAVED, out=ODD) == v.VH_EALIGN
    assert call(Hq=24) == v.VH_EINVAL
    assert call(eps=-0.5) == v.VH_EINVAL
    assert call(out=ODD) == v.VH_EALIGN
    assert call(kw=ODD) == v.VH_EALIGN
    assert call(ws=None) == v.VH_EWORKSPACE
    assert call(hs=0) == v.VH_EINVAL
    assert call(hs=100) == v.VH_EALIGN


def test_rope_table_and_combine_argument_checks():
    assert v.lib.vh_rope_table(None, 10, 128, 10000.0, None) == v.VH_EINVAL
    assert v.lib.vh_rope_table(FAKE, 10, 128, -1.0, None) == v.VH_EINVAL
    assert v.lib.vh_rope_table(ODD, 10, 128, 10000.0, None) == v.VH_EALIGN
    assert v.lib.vh_decode_combine(None, 0, FAKE, 0, 0, 4, 16, 8, 128, 16, None) == v.VH_EWORKSPACE
    assert v.lib.vh_decode_combine(FAKE, 1 << 30, ODD, 0, 0, 4, 16, 8, 128, 16, None) == v.VH_EALIGN
    assert v.lib.vh_decode_combine(FAKE, 1 << 30, FAKE, 0, 0, 4, 12, 8, 128, 16, None) == v.VH_EINVAL
    assert v.lib.vh_decode_combine(FAKE, 1 << 30, FAKE, 0, v.VH_FLAG_PDL, 4, 16, 8, 128, 16, None) == v.VH_EINVAL
    assert v.lib.vh_decode_combine(FAKE, 1 << 30, ODD, 0, v.VH_FLAG_FP16, 4, 16, 8, 128, 16, None) == v.VH_EALIGN
    assert v.lib.vh_decode_workspace_bytes(4, 12, 8, 128, 16, 10) == 0
    assert v.lib.vh_decode_workspace_bytes(4, 16, 8, 128, 16, 152) > 0


def test_contiguous_cache_arguments():
    # no page table: the rows' pages b * max_pages_per_seq + j must exist
    assert attn(pt=None, npages=3, mps=1) == v.VH_EINVAL          # B = 4 rows, 3 pages
    assert attn(pt=None, npages=8, mps=2, P=11) == v.VH_EINVAL    # pages of 11 tokens need one page per row
    assert attn(P=11, mps=2) == v.VH_EINVAL
    assert attn(P=0) == v.VH_EINVAL
    assert attn(P=1025) == v.VH_EINVAL


def test_contiguous_cache_arguments_pass_host_checks_without_device():
    # valid without a table: on a GPU-less machine the device query is the
    # first check that fails (the fake pointers are never used)
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert attn(pt=None, npages=4, mps=1, P=11) == v.VH_ENODEV


def test_wait_timeout_selftest_arguments():
    assert v.lib.vh_selftest_wait_timeout(None, None) == v.VH_EINVAL
    assert v.lib.vh_selftest_wait_timeout(ctypes.c_void_p(0x10002), None) == v.VH_EALIGN


def test_wait_timeout_selftest_without_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert v.lib.vh_selftest_wait_timeout(FAKE, None) == v.VH_ENODEV


def plan(**over):
    a = dict(pos=None, max_pos=4096, npages=100, pt=FAKE, mps=10, sl=FAKE, act=FAKE, nctas=0, ws=FAKE,
             wsb=1 << 30, err=None, flags=0, B=4, Hq=16, Hkv=8, D=128, P=16)
    a.update(over)
    return v.lib.vh_decode_plan(a["pos"], a["max_pos"], a["npages"], a["pt"], a["mps"], a["sl"], a["act"],
                                a["nctas"], a["ws"], a["wsb"], a["err"], a["flags"], a["B"], a["Hq"], a["Hkv"],
                                a["D"], a["P"], None)


@pytest.mark.parametrize("over,code", [
    (dict(sl=None), v.VH_EINVAL),
    (dict(act=None), v.VH_EINVAL),
    (dict(flags=v.VH_FLAG_PDL), v.VH_EINVAL),          # not a flag of this call
    (dict(flags=64), v.VH_EINVAL),
    (dict(max_pos=0), v.VH_EINVAL),                    # the fused rules need the RoPE table size
    (dict(P=12), v.VH_EINVAL),
    (dict(pt=None, npages=3, mps=1), v.VH_EINVAL),     # contiguous cache: 4 rows, 3 pages
    (dict(nctas=-1), v.VH_EINVAL),
    (dict(Hq=12), v.VH_EINVAL),
    (dict(ws=None), v.VH_EWORKSPACE),
    (dict(ws=ODD), v.VH_EALIGN),
])
def test_plan_argument_checks(over, code):
    assert plan(**over) == code


def test_plans_and_eight_token_pages_pass_host_checks_without_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert plan() == v.VH_ENODEV
    assert plan(max_pos=0, flags=v.VH_FLAG_PLAN_THREE_CALL) == v.VH_ENODEV   # max_pos unused there
    assert plan(P=8) == v.VH_ENODEV
    assert attn(P=8) == v.VH_ENODEV                    # 8-token pages: every tile spans two pages
    assert attn(flags=v.VH_FLAG_PLANNED) == v.VH_ENODEV


def test_noalloc_takes_a_contiguous_cache_without_page_table():
    import torch
    f = v.lib.vh_paged_decode_attn_noalloc

    def call(**over):
        a = dict(q_rot=FAKE, k=FAKE, vv=FAKE, ps=2 * 16 * 8 * 128, ts=8 * 128, npages=100, pt=FAKE, mps=10,
                 sl=FAKE, act=FAKE, out=FAKE, scale=0.0, nctas=0, err=None, B=4, Hq=16, Hkv=8, D=128, P=16)
        a.update(over)
        return f(a["q_rot"], a["k"], a["vv"], a["ps"], a["ts"], a["npages"], a["pt"], a["mps"], a["sl"], a["act"],
                 a["out"], a["scale"], a["nctas"], a["err"], a["B"], a["Hq"], a["Hkv"], a["D"], a["P"], None)

    assert call(pt=None, npages=3, mps=1) == v.VH_EINVAL   # 4 rows need 4 pages
    assert call(q_rot=None) == v.VH_EINVAL
    if not torch.cuda.is_available():
        assert call(pt=None, npages=4, mps=1) == v.VH_ENODEV
