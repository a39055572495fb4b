"""Thin Python binding of libvh.so (the C interface in include/vh.h).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of libvh.so.  Tensors are torch CUDA tensors; the binding checks
dtypes, contiguity and devices, reads shapes and strides, and passes raw
pointers plus the current torch stream.  There is no fallback: if the
library is missing or a call fails, an exception is raised.

The 16-bit element type (bf16 or fp16) is the cache's dtype; q, k_new,
v_new and out must have the same dtype, and VH_FLAG_FP16 is passed for fp16.
`interleaved=True` selects the (2i, 2i+1) RoPE pairing.  page_table=None
selects a contiguous cache (row b owns pages b*m .. b*m+m-1, m = pages / B).

Functions mirror the C entry points by name:
    vh_rope_table, vh_rope_kv_append, vh_decode_num_ctas,
    vh_decode_workspace_bytes, vh_paged_decode_attn, vh_decode_combine,
    vh_decode_fused, vh_decode_plan, vh_paged_decode_attn_noalloc, vh_selftest_wait_timeout,
    vh_status_string
plus `decode_step`, which issues the three calls of one decode step.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvh.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "vh.h")

VH_OK, VH_EINVAL, VH_EALIGN, VH_EWORKSPACE, VH_ECUDA, VH_ENODEV = 0, -1, -2, -3, -4, -5
VH_ESCRATCH = -6
VH_ERR_SEQLEN, VH_ERR_PAGE, VH_ERR_POS, VH_ERR_TIMEOUT = 1, 2, 4, 8
VH_FLAG_PDL, VH_FLAG_FP16, VH_FLAG_ROPE_INTERLEAVED, VH_FLAG_PDL_KV = 1, 2, 4, 8
VH_FLAG_PLANNED, VH_FLAG_PLAN_THREE_CALL, VH_FLAG_HOST_IO = 16, 32, 64
ELEM_DTYPES = (torch.bfloat16, torch.float16)


class VHError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({vh_status_string(status)})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first (paged_len_decode_gb300.build.build())")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, F, D, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                           ctypes.c_double, ctypes.c_size_t)
    lib.vh_selftest_wait_timeout.argtypes = [P, P]
    lib.vh_selftest_wait_timeout.restype = I
    lib.vh_status_string.argtypes = [I]
    lib.vh_status_string.restype = ctypes.c_char_p
    lib.vh_rope_table.argtypes = [P, I, I, D, P]
    lib.vh_rope_table.restype = I
    U = ctypes.c_uint
    lib.vh_rope_kv_append.argtypes = [P, P, P, P, I, P, P, P, F, P, P, I64, I64, I64, I, P, I, P, P, P, P, U,
                                      I, I, I, I, I, P]
    lib.vh_rope_kv_append.restype = I
    lib.vh_decode_num_ctas.argtypes = [I, I, I, I, I]
    lib.vh_decode_num_ctas.restype = I
    lib.vh_decode_workspace_bytes.argtypes = [I, I, I, I, I, I]
    lib.vh_decode_workspace_bytes.restype = SZ
    lib.vh_paged_decode_attn.argtypes = [P, P, P, I64, I64, I64, I, P, I, P, P, P, F, I, P, SZ, P, U,
                                         I, I, I, I, I, P]
    lib.vh_paged_decode_attn.restype = I
    lib.vh_decode_combine.argtypes = [P, SZ, P, I, U, I, I, I, I, I, P]
    lib.vh_decode_combine.restype = I
    lib.vh_paged_decode_attn_noalloc.argtypes = [P, P, P, I64, I64, I, P, I, P, P, P, F, I, P,
                                                 I, I, I, I, I, P]
    lib.vh_paged_decode_attn_noalloc.restype = I
    lib.vh_decode_fused.argtypes = [P, P, P, P, I, P, P, P, F, P, P, I64, I64, I64, I, P, I, P, P, P, F, I, P,
                                    SZ, P, ctypes.c_uint, I, I, I, I, I, P]
    lib.vh_decode_fused.restype = I
    lib.vh_decode_plan.argtypes = [P, I, I, P, I, P, P, I, P, SZ, P, U, I, I, I, I, I, P]
    lib.vh_decode_plan.restype = I
    return lib


lib = _load()


def header_functions() -> list[str]:
    """Names of the functions include/vh.h declares."""
    text = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(vh_\w+)\s*\(", text, flags=re.M)))


def vh_status_string(status: int) -> str:
    return lib.vh_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != VH_OK:
        raise VHError(status, where)


def _ptr(t: torch.Tensor | None, dtype=None, name: str = "") -> ctypes.c_void_p | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _contig(t: torch.Tensor, dtype, name: str) -> ctypes.c_void_p:
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return _ptr(t, dtype, name)


def _io(t: torch.Tensor, dtype, name: str, host_io: bool) -> ctypes.c_void_p:
    """Pointer of a per-step input or output: a CUDA tensor, or with host_io a
    pinned CPU tensor, which the device reads or writes in place."""
    if host_io and t is not None and t.device.type == "cpu":
        if not t.is_pinned():
            raise ValueError(f"{name} must be pinned host memory (or a CUDA tensor)")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        return ctypes.c_void_p(t.data_ptr())
    return _contig(t, dtype, name)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _cache_view(k_cache: torch.Tensor, v_cache: torch.Tensor, bf16_only: bool = False):
    """Pointers and element strides of a [NP, P, Hkv, D] paged cache view.

    Returns (k, v, page_stride, token_stride, head_stride, NP, P, Hkv, D).  The
    view may be token-major (a slice of [NP, 2, P, Hkv, D]) or head-major (a
    slice of [NP, 2, Hkv, P, D], transposed to [NP, P, Hkv, D]); head_dim must
    be contiguous.  With bf16_only (the entry point without a workspace) the
    heads of a slot must also be contiguous."""
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape or v_cache.stride() != k_cache.stride():
        raise ValueError("k_cache / v_cache must be [NP, P, Hkv, D] views with equal strides")
    if k_cache.stride(3) != 1:
        raise ValueError("head_dim must be contiguous in the cache")
    if bf16_only and k_cache.stride(2) != k_cache.shape[3]:
        raise ValueError("the heads of one token slot must be contiguous ([.., Hkv, D] dense)")
    if k_cache.dtype not in (ELEM_DTYPES[:1] if bf16_only else ELEM_DTYPES):
        raise TypeError(f"k_cache must be bfloat16{'' if bf16_only else ' or float16'}, got {k_cache.dtype}")
    NP, P, Hkv, D = k_cache.shape
    return (_ptr(k_cache, k_cache.dtype, "k_cache"), _ptr(v_cache, k_cache.dtype, "v_cache"),
            k_cache.stride(0), k_cache.stride(1), k_cache.stride(2), NP, P, Hkv, D)


def _table(page_table, B: int, NP: int):
    """(pointer, max_pages_per_seq) of the page table; None means a contiguous
    cache whose row b owns pages b * m .. b * m + m - 1, m = NP // B."""
    if page_table is None:
        if NP % B != 0:
            raise ValueError("without a page table the cache must hold a whole number of pages per row")
        return None, NP // B
    return _contig(page_table, torch.int32, "page_table"), page_table.shape[1]


def _elem_flags(k_cache: torch.Tensor, interleaved: bool = False) -> int:
    return (VH_FLAG_FP16 if k_cache.dtype == torch.float16 else 0) | (VH_FLAG_ROPE_INTERLEAVED if interleaved else 0)


def vh_selftest_wait_timeout(err_flag: torch.Tensor, stream=None) -> None:
    """Run the kernels' bounded pipeline wait on a barrier nothing arrives on;
    VH_ERR_TIMEOUT is ORed into err_flag (int32 CUDA tensor) after about a second."""
    _check(lib.vh_selftest_wait_timeout(_contig(err_flag, torch.int32, "err_flag"), _stream(stream)),
           "vh_selftest_wait_timeout")


def vh_rope_table(cos_sin: torch.Tensor, theta: float = 10000.0, stream=None) -> torch.Tensor:
    """Fill cos_sin (float32 [max_pos, D]) with the RoPE table."""
    max_pos, D = cos_sin.shape
    _check(lib.vh_rope_table(_contig(cos_sin, torch.float32, "cos_sin"), max_pos, D, float(theta),
                             _stream(stream)), "vh_rope_table")
    return cos_sin


def _norm_w(t, D, name):
    if t is None:
        return None
    if t.shape != (D,):
        raise ValueError(f"{name} must have shape ({D},)")
    return _contig(t, torch.float32, name)


def vh_rope_kv_append(q, k_new, v_new, cos_sin, k_cache, v_cache, page_table, seq_lens, active,
                      q_rot, positions=None, err_flag=None, q_norm_w=None, k_norm_w=None,
                      norm_eps: float = 1e-6, interleaved: bool = False, stream=None) -> None:
    B, Hq, D = q.shape
    kp, vp, ps, ts, hs, NP, P, Hkv, Dc = _cache_view(k_cache, v_cache)
    et = k_cache.dtype
    if Dc != D or k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) or q_rot.shape != (B, Hq, D):
        raise ValueError("shape mismatch between q, k_new, v_new, q_rot and the cache")
    _check(lib.vh_rope_kv_append(
        _contig(q, et, "q"), _contig(k_new, et, "k_new"),
        _contig(v_new, et, "v_new"), _contig(cos_sin, torch.float32, "cos_sin"),
        cos_sin.shape[0], None if positions is None else _contig(positions, torch.int32, "positions"),
        _norm_w(q_norm_w, D, "q_norm_w"), _norm_w(k_norm_w, D, "k_norm_w"), float(norm_eps),
        kp, vp, ps, ts, hs, NP, *_table(page_table, B, NP),
        _contig(seq_lens, torch.int32, "seq_lens"), _contig(active, torch.int32, "active"),
        _contig(q_rot, torch.float32, "q_rot"),
        None if err_flag is None else _contig(err_flag, torch.int32, "err_flag"),
        _elem_flags(k_cache, interleaved), B, Hq, Hkv, D, P, _stream(stream)), "vh_rope_kv_append")


def vh_decode_num_ctas(B: int, Hq: int, Hkv: int, D: int, page_size: int) -> int:
    n = lib.vh_decode_num_ctas(B, Hq, Hkv, D, page_size)
    if n < 0:
        raise VHError(n, "vh_decode_num_ctas")
    return n


def vh_decode_workspace_bytes(B: int, Hq: int, Hkv: int, D: int, page_size: int, num_ctas: int = 0) -> int:
    n = lib.vh_decode_workspace_bytes(B, Hq, Hkv, D, page_size, num_ctas)
    if n == 0:
        raise VHError(VH_EINVAL, "vh_decode_workspace_bytes")
    return n


def vh_paged_decode_attn(q_rot, k_cache, v_cache, page_table, seq_lens, active, out, workspace,
                         sm_scale: float = 0.0, num_ctas: int = 0, err_flag=None, pdl: bool = False,
                         planned: bool = False, stream=None) -> None:
    B, Hq, D = q_rot.shape
    kp, vp, ps, ts, hs, NP, P, Hkv, Dc = _cache_view(k_cache, v_cache)
    if Dc != D or out.shape != (B, Hq, D):
        raise ValueError("shape mismatch between q_rot, out and the cache")
    _check(lib.vh_paged_decode_attn(
        _contig(q_rot, torch.float32, "q_rot"), kp, vp, ps, ts, hs, NP, *_table(page_table, B, NP),
        _contig(seq_lens, torch.int32, "seq_lens"), _contig(active, torch.int32, "active"),
        _contig(out, k_cache.dtype, "out"), float(sm_scale), int(num_ctas),
        _contig(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        None if err_flag is None else _contig(err_flag, torch.int32, "err_flag"),
        _elem_flags(k_cache) | (VH_FLAG_PDL if pdl else 0) | (VH_FLAG_PLANNED if planned else 0),
        B, Hq, Hkv, D, P, _stream(stream)), "vh_paged_decode_attn")


def vh_decode_combine(workspace, out, Hkv: int, page_size: int, num_ctas: int = 0, stream=None) -> None:
    """Merge split rows into out (bf16 or fp16: the type vh_paged_decode_attn wrote)."""
    B, Hq, D = out.shape
    if out.dtype not in ELEM_DTYPES:
        raise TypeError(f"out must be bfloat16 or float16, got {out.dtype}")
    _check(lib.vh_decode_combine(
        _contig(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _contig(out, out.dtype, "out"), int(num_ctas), VH_FLAG_FP16 if out.dtype == torch.float16 else 0,
        B, Hq, Hkv, D, page_size, _stream(stream)), "vh_decode_combine")


def vh_paged_decode_attn_noalloc(q_rot, k_cache, v_cache, page_table, seq_lens, active, out,
                                 sm_scale: float = 0.0, num_ctas: int = 0, err_flag=None,
                                 stream=None) -> None:
    """Attention plus combine into `out` with the library's fixed scratch array,
    for callers that cannot allocate a workspace (see include/vh.h).
    page_table=None selects a contiguous token-major cache (row b owns pages
    b*m .. b*m+m-1, m = pages / B)."""
    B, Hq, D = q_rot.shape
    kp, vp, ps, ts, _hs, NP, P, Hkv, Dc = _cache_view(k_cache, v_cache, bf16_only=True)
    if Dc != D or out.shape != (B, Hq, D):
        raise ValueError("shape mismatch between q_rot, out and the cache")
    _check(lib.vh_paged_decode_attn_noalloc(
        _contig(q_rot, torch.float32, "q_rot"), kp, vp, ps, ts, NP, *_table(page_table, B, NP),
        _contig(seq_lens, torch.int32, "seq_lens"), _contig(active, torch.int32, "active"),
        _contig(out, torch.bfloat16, "out"), float(sm_scale), int(num_ctas),
        None if err_flag is None else _contig(err_flag, torch.int32, "err_flag"),
        B, Hq, Hkv, D, P, _stream(stream)), "vh_paged_decode_attn_noalloc")


def vh_decode_fused(q, k_new, v_new, cos_sin, k_cache, v_cache, page_table, seq_lens, active, out,
                    workspace, positions=None, sm_scale: float = 0.0, num_ctas: int = 0, err_flag=None,
                    pdl: bool = False, q_norm_w=None, k_norm_w=None, norm_eps: float = 1e-6,
                    interleaved: bool = False, pdl_kv: bool = False, planned: bool = False,
                    host_io: bool = False, stream=None) -> torch.Tensor:
    """One whole decode step in one launch (RoPE, append, attention, merge).
    `workspace` must be zero-filled before its first use (alloc_workspace does that).
    pdl=True sets VH_FLAG_PDL, pdl_kv=True VH_FLAG_PDL_KV (see include/vh.h for
    when each is allowed); planned=True (VH_FLAG_PLANNED) takes the work list
    from the plan vh_decode_plan wrote into `workspace`; host_io=True
    (VH_FLAG_HOST_IO) lets q, k_new, v_new, positions, seq_lens, active,
    page_table and out be pinned CPU tensors that the kernel reads and writes
    in place."""
    B, Hq, D = q.shape
    kp, vp, ps, ts, hs, NP, P, Hkv, Dc = _cache_view(k_cache, v_cache)
    et = k_cache.dtype
    if Dc != D or k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) or out.shape != (B, Hq, D):
        raise ValueError("shape mismatch between q, k_new, v_new, out and the cache")
    h = host_io
    if page_table is None:
        pt, mps = _table(None, B, NP)
    else:
        pt, mps = _io(page_table, torch.int32, "page_table", h), page_table.shape[1]
    _check(lib.vh_decode_fused(
        _io(q, et, "q", h), _io(k_new, et, "k_new", h),
        _io(v_new, et, "v_new", h), _contig(cos_sin, torch.float32, "cos_sin"),
        cos_sin.shape[0], None if positions is None else _io(positions, torch.int32, "positions", h),
        _norm_w(q_norm_w, D, "q_norm_w"), _norm_w(k_norm_w, D, "k_norm_w"), float(norm_eps),
        kp, vp, ps, ts, hs, NP, pt, mps,
        _io(seq_lens, torch.int32, "seq_lens", h), _io(active, torch.int32, "active", h),
        _io(out, et, "out", h), float(sm_scale), int(num_ctas),
        _contig(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        None if err_flag is None else _contig(err_flag, torch.int32, "err_flag"),
        (VH_FLAG_PDL if pdl else 0) | (VH_FLAG_PDL_KV if pdl_kv else 0) | _elem_flags(k_cache, interleaved)
        | (VH_FLAG_PLANNED if planned else 0) | (VH_FLAG_HOST_IO if host_io else 0), B, Hq, Hkv, D, P,
        _stream(stream)), "vh_decode_fused")
    return out


def vh_decode_plan(seq_lens, active, page_table, workspace, *, Hq: int, Hkv: int, D: int, page_size: int,
                   num_pages: int, max_pages_per_seq: int | None = None, positions=None, max_pos: int = 0,
                   num_ctas: int = 0, err_flag=None, fp16: bool = False, three_call: bool = False,
                   stream=None) -> None:
    """Write the step's attention work list into `workspace` (see include/vh.h):
    for vh_decode_fused(planned=True), or with three_call=True for
    vh_paged_decode_attn(planned=True).  page_table=None: contiguous cache with
    max_pages_per_seq pages per row (default num_pages // B)."""
    B = seq_lens.shape[0]
    if page_table is None:
        pt, mps = None, (max_pages_per_seq if max_pages_per_seq is not None else num_pages // B)
    else:
        pt, mps = _contig(page_table, torch.int32, "page_table"), page_table.shape[1]
    _check(lib.vh_decode_plan(
        None if positions is None else _contig(positions, torch.int32, "positions"), int(max_pos), int(num_pages),
        pt, mps, _contig(seq_lens, torch.int32, "seq_lens"), _contig(active, torch.int32, "active"), int(num_ctas),
        _contig(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        None if err_flag is None else _contig(err_flag, torch.int32, "err_flag"),
        (VH_FLAG_FP16 if fp16 else 0) | (VH_FLAG_PLAN_THREE_CALL if three_call else 0),
        B, Hq, Hkv, D, page_size, _stream(stream)), "vh_decode_plan")


def alloc_workspace(B: int, Hq: int, Hkv: int, D: int, page_size: int, num_ctas: int = 0,
                    device=None) -> torch.Tensor:
    """Zero-filled device scratch for the attention calls (torch allocation)."""
    n = vh_decode_workspace_bytes(B, Hq, Hkv, D, page_size, num_ctas)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def decode_step(q, k_new, v_new, cos_sin, k_cache, v_cache, page_table, seq_lens, active, q_rot,
                out, workspace, positions=None, sm_scale: float = 0.0, num_ctas: int = 0,
                err_flag=None, q_norm_w=None, k_norm_w=None, norm_eps: float = 1e-6,
                interleaved: bool = False, planned: bool = False, stream=None) -> torch.Tensor:
    """One decode step of one layer: (RMSNorm +) RoPE + append, attention, combine.
    planned=True: the attention takes its work list from the plan vh_decode_plan
    (three_call=True) wrote into `workspace`."""
    vh_rope_kv_append(q, k_new, v_new, cos_sin, k_cache, v_cache, page_table, seq_lens, active,
                      q_rot, positions=positions, err_flag=err_flag, q_norm_w=q_norm_w,
                      k_norm_w=k_norm_w, norm_eps=norm_eps, interleaved=interleaved, stream=stream)
    # the attention launch depends programmatically on the append kernel just
    # before it, which writes neither lengths, flags nor the page table
    vh_paged_decode_attn(q_rot, k_cache, v_cache, page_table, seq_lens, active, out, workspace,
                         sm_scale=sm_scale, num_ctas=num_ctas, err_flag=err_flag, pdl=True, planned=planned,
                         stream=stream)
    vh_decode_combine(workspace, out, k_cache.shape[2], k_cache.shape[1], num_ctas=num_ctas,
                      stream=stream)
    return out
