"""Float64 CPU oracle of the paged q_len=1 decode step (ctypes over oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  Nothing here imports or links the
CUDA library, and the CUDA library never calls into this package.

All functions take CPU torch tensors: bf16 / fp16 tensors are read as their
bit patterns (the element type is taken from the tensor's dtype), float64
tensors are used as is.  See oracle.c for what each step
computes and which passage it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2, OpenMP, strict IEEE) into liboracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
                        "-fno-fast-math", _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_bf16_from_double.argtypes = [D]
            lib.oracle_bf16_from_double.restype = ctypes.c_uint16
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = D
            lib.oracle_f16_from_double.argtypes = [D]
            lib.oracle_f16_from_double.restype = ctypes.c_uint16
            lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_double.restype = D
            lib.oracle_num_threads.restype = I
            lib.oracle_set_num_threads.argtypes = [I]
            lib.oracle_rope_kv_append.argtypes = [P, P, P, P, P, P, D, P, P, I64, I64, P, I, I, P, P, P, P,
                                                  P, I, I, I, I, I, D, I, I]
            lib.oracle_rope_kv_append.restype = I
            lib.oracle_decode_attn.argtypes = [P, P, P, I64, I64, P, I, P, P, P, P, D, P, I,
                                               I, I, I, I, I, I]
            lib.oracle_decode_attn.restype = None
            lib.oracle_decode_attn_split.argtypes = [P, P, P, I64, I64, P, I, P, P, P, D, I,
                                                     I, I, I, I, I, I]
            lib.oracle_decode_attn_split.restype = None
            lib.oracle_lse_combine.argtypes = [P, P, I, I, P]
            lib.oracle_lse_combine.restype = D
            _lib = lib
    return _lib


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    assert t.device.type == "cpu" and t.is_contiguous()
    return ctypes.c_void_p(t.data_ptr())


def _i32(t: torch.Tensor) -> torch.Tensor:
    return t.detach().to("cpu", torch.int32).contiguous()


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(n)


def bf16_from_double(x: float) -> int:
    """bf16 bit pattern nearest to x (ties to even), one rounding step."""
    return int(_load().oracle_bf16_from_double(float(x)))


def bf16_to_double(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(bits & 0xFFFF))


def f16_from_double(x: float) -> int:
    """IEEE binary16 bit pattern nearest to x (ties to even), one rounding step."""
    return int(_load().oracle_f16_from_double(float(x)))


def f16_to_double(bits: int) -> float:
    return float(_load().oracle_f16_to_double(bits & 0xFFFF))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return 1
    assert t.dtype == torch.bfloat16, t.dtype
    return 0


def rope_kv_append(q, k_new, v_new, pool, page_table, seq_lens, active, *, P, theta,
                   positions=None, num_pages=None, return_k_rot=False, in_place=False,
                   q_norm_w=None, k_norm_w=None, norm_eps=1e-6, return_k_pre=False,
                   interleaved=False):
    """RoPE + append on a copy of `pool` ([NP, 2, P, Hkv, D] bf16 or fp16, the
    type of q, k_new and v_new), or on `pool` itself when in_place (a
    contiguous CPU tensor).

    Returns (q_rot float64 [B, Hq, D], pool_after bf16, n_bad), plus the
    unrounded rotated keys float64 [B, Hkv, D] if return_k_rot, plus the keys
    fed to RoPE if return_k_pre.  Rows with active == 0 keep q_rot = 0 and
    write nothing.  q_norm_w / k_norm_w (length-D weights, or None) switch on
    the per-head RMSNorm before RoPE.  interleaved pairs elements (2i, 2i+1)
    instead of (i, i + D/2).
    """
    lib = _load()
    dt = _dtype_code(q)
    assert k_new.dtype == q.dtype and v_new.dtype == q.dtype and pool.dtype == q.dtype
    B, Hq, D = q.shape
    Hkv = k_new.shape[1]
    if in_place:
        assert pool.device.type == "cpu" and pool.is_contiguous()
        pool_after = pool
    else:
        pool_after = pool.detach().to("cpu").contiguous().clone()
    NP = pool_after.shape[0]
    bits = pool_after.view(torch.int16)
    q_rot = torch.zeros((B, Hq, D), dtype=torch.float64)
    k_rot = torch.zeros((B, Hkv, D), dtype=torch.float64)
    k_pre = torch.zeros((B, Hkv, D), dtype=torch.float64)
    qw = None if q_norm_w is None else torch.as_tensor(q_norm_w).detach().to("cpu", torch.float64).contiguous()
    kw = None if k_norm_w is None else torch.as_tensor(k_norm_w).detach().to("cpu", torch.float64).contiguous()
    qb = q.detach().to("cpu").contiguous().view(torch.int16)
    kb = k_new.detach().to("cpu").contiguous().view(torch.int16)
    vb = v_new.detach().to("cpu").contiguous().view(torch.int16)
    pt = _i32(page_table)
    sl = _i32(seq_lens)
    ac = _i32(active)
    pos = _i32(positions) if positions is not None else None
    page_stride = 2 * P * Hkv * D
    token_stride = Hkv * D
    k_ptr = bits.data_ptr()
    v_ptr = bits.data_ptr() + P * Hkv * D * 2
    bad = lib.oracle_rope_kv_append(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(pos), _ptr(qw), _ptr(kw),
                                    float(norm_eps), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
                                    page_stride, token_stride, _ptr(pt), pt.shape[1],
                                    NP if num_pages is None else num_pages,
                                    _ptr(sl), _ptr(ac), _ptr(q_rot), _ptr(k_rot), _ptr(k_pre),
                                    B, Hq, Hkv, D, P, float(theta), dt, int(bool(interleaved)))
    res = (q_rot, pool_after, int(bad))
    if return_k_rot:
        res = res + (k_rot,)
    if return_k_pre:
        res = res + (k_pre,)
    return res


def decode_attn(q_rot, pool, page_table, seq_lens, active, *, P, sm_scale=0.0, rows=None,
                return_lse=False):
    """Softmax attention of every (or the listed) row over its paged keys.

    q_rot: float64 [B, Hq, D]; pool: bf16 or fp16 [NP, 2, P, Hkv, D].
    Returns float64 out [B, Hq, D] (rows not listed stay zero), and the
    natural-log lse [B, Hq] if return_lse.
    """
    lib = _load()
    B, Hq, D = q_rot.shape
    Hkv = pool.shape[3]
    qr = q_rot.detach().to("cpu", torch.float64).contiguous()
    bits = pool.detach().to("cpu").contiguous().view(torch.int16)
    pt = _i32(page_table)
    sl = _i32(seq_lens)
    ac = _i32(active)
    out = torch.zeros((B, Hq, D), dtype=torch.float64)
    lse = torch.full((B, Hq), float("-inf"), dtype=torch.float64)
    rw = _i32(torch.as_tensor(rows)) if rows is not None else None
    lib.oracle_decode_attn(_ptr(qr), ctypes.c_void_p(bits.data_ptr()),
                           ctypes.c_void_p(bits.data_ptr() + P * Hkv * D * 2),
                           2 * P * Hkv * D, Hkv * D, _ptr(pt), pt.shape[1], _ptr(sl), _ptr(ac),
                           _ptr(out), _ptr(lse), float(sm_scale), _ptr(rw),
                           0 if rw is None else rw.numel(), B, Hq, Hkv, D, P, _dtype_code(pool))
    return (out, lse) if return_lse else out


def decode_attn_split(q_rot, pool, page_table, seq_lens, active, *, P, n_splits, sm_scale=0.0):
    """The same attention as decode_attn, as n_splits segments merged by LSE."""
    lib = _load()
    B, Hq, D = q_rot.shape
    Hkv = pool.shape[3]
    qr = q_rot.detach().to("cpu", torch.float64).contiguous()
    bits = pool.detach().to("cpu").contiguous().view(torch.int16)
    pt = _i32(page_table)
    sl = _i32(seq_lens)
    ac = _i32(active)
    out = torch.zeros((B, Hq, D), dtype=torch.float64)
    lib.oracle_decode_attn_split(_ptr(qr), ctypes.c_void_p(bits.data_ptr()),
                                 ctypes.c_void_p(bits.data_ptr() + P * Hkv * D * 2),
                                 2 * P * Hkv * D, Hkv * D, _ptr(pt), pt.shape[1], _ptr(sl),
                                 _ptr(ac), _ptr(out), float(sm_scale), int(n_splits),
                                 B, Hq, Hkv, D, P, _dtype_code(pool))
    return out


def lse_combine(o_parts: torch.Tensor, lse_parts: torch.Tensor):
    """Merge S partials of one head: o_parts float64 [S, D], lse_parts [S]."""
    lib = _load()
    op = o_parts.detach().to("cpu", torch.float64).contiguous()
    lp = lse_parts.detach().to("cpu", torch.float64).contiguous()
    S, D = op.shape
    o = torch.zeros(D, dtype=torch.float64)
    lse = lib.oracle_lse_combine(_ptr(op), _ptr(lp), S, D, _ptr(o))
    return o, float(lse)


def reference_step(inp, positions=None, rows=None, sm_scale=0.0, q_norm_w=None, k_norm_w=None,
                   norm_eps=1e-6, interleaved=False):
    """Whole step on one layer's inputs (any object with the DecodeInputs fields).

    Returns dict(q_rot, k_rot, k_pre, pool_after, out, n_bad): (RMSNorm +) RoPE
    + append, then attention over the appended cache.  k_rot is the rotated key
    before its rounding to the cache type, k_pre the key fed to RoPE.
    """
    q_rot, pool_after, bad, k_rot, k_pre = rope_kv_append(
        inp.q, inp.k_new, inp.v_new, inp.pool, inp.page_table, inp.seq_lens, inp.active, P=inp.P,
        theta=inp.theta, positions=positions, num_pages=inp.num_pages, return_k_rot=True,
        q_norm_w=q_norm_w, k_norm_w=k_norm_w, norm_eps=norm_eps, return_k_pre=True,
        interleaved=interleaved)
    out = decode_attn(q_rot, pool_after, inp.page_table, inp.seq_lens, inp.active, P=inp.P,
                      rows=rows, sm_scale=sm_scale)
    return {"q_rot": q_rot, "k_rot": k_rot, "k_pre": k_pre, "pool_after": pool_after, "out": out,
            "n_bad": bad}
