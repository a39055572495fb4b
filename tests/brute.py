"""Pure-Python brute force of the decode step, for tiny inputs only.

A second, independent implementation used to pin the C oracle: plain lists,
`math` functions, an exact bf16 rounding built on `fractions.Fraction`, and
no code shared with the oracle or the CUDA library.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction


def bf16_bits_to_float(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (bits & 0xFFFF) << 16))[0]


def f16_bits_to_float(bits: int) -> float:
    """IEEE binary16 bit pattern -> float, by Python's own half-precision codec."""
    return struct.unpack("<e", struct.pack("<H", bits & 0xFFFF))[0]


def f16_round_bits(x: float) -> int:
    """Nearest binary16 to the double x, ties to the even bit pattern.

    The same exact-rational bracketing as bf16_round_bits, over the 0x7BFF
    finite magnitudes (largest 65504); at or beyond 65520 (the midpoint to
    the next power of two) the result is infinity."""
    if math.isnan(x):
        return 0x7E00
    if x == 0.0:
        return 0x8000 if math.copysign(1.0, x) < 0 else 0
    sign = 0x8000 if x < 0 else 0
    fx = Fraction(abs(x))
    if fx >= 65520:
        return sign | 0x7C00
    lo, hi = 0, 0x7BFF
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if Fraction(f16_bits_to_float(mid)) <= fx:
            lo = mid
        else:
            hi = mid - 1
    t = lo
    if t == 0x7BFF:
        return sign | t
    a, b = Fraction(f16_bits_to_float(t)), Fraction(f16_bits_to_float(t + 1))
    da, db = fx - a, b - fx
    if da < db:
        r = t
    elif db < da:
        r = t + 1
    else:
        r = t if t % 2 == 0 else t + 1
    return sign | r


# element codecs by type name
DECODE = {"bf16": bf16_bits_to_float, "fp16": f16_bits_to_float}


def _bf16_value(bits: int) -> Fraction:
    return Fraction(bf16_bits_to_float(bits))


def bf16_round_bits(x: float) -> int:
    """Nearest bf16 to the double x, ties to the even bit pattern.

    Brackets x between the two bf16 neighbours obtained by truncating its
    float32 image, then compares exact rational distances (no floating-point
    rounding in the decision)."""
    if math.isnan(x):
        return 0x7FC0
    if x == 0.0:
        return 0x8000 if math.copysign(1.0, x) < 0 else 0
    sign = 0x8000 if x < 0 else 0
    ax = abs(x)
    fx = Fraction(ax)
    max_bf16 = Fraction((2 ** 8 - 1) * 2 ** (127 - 7))
    if fx >= max_bf16 + (Fraction(2) ** (127 - 8)):  # at or beyond the midpoint to "2^128"
        return sign | 0x7F80
    # find the bf16 bit pattern t (sign cleared) with value(t) <= ax < value(t+1)
    lo, hi = 0, 0x7F7F
    while lo < hi:                      # largest t with value(t) <= ax
        mid = (lo + hi + 1) // 2
        if _bf16_value(mid) <= fx:
            lo = mid
        else:
            hi = mid - 1
    t = lo
    if t == 0x7F7F:
        return sign | t
    a, b = _bf16_value(t), _bf16_value(t + 1)
    da, db = fx - a, b - fx
    if da < db:
        r = t
    elif db < da:
        r = t + 1
    else:
        r = t if t % 2 == 0 else t + 1
    return sign | r


def rms_norm(x: list[float], w, eps: float) -> list[float]:
    """w_d * x_d / sqrt(mean(x^2) + eps); w None: unchanged."""
    if w is None:
        return list(x)
    r = 1.0 / math.sqrt(math.fsum(v * v for v in x) / len(x) + eps)
    return [wd * (v * r) for wd, v in zip(w, x)]


def rope(x: list[float], pos: float, theta: float, interleaved: bool = False) -> list[float]:
    """RoPE with angle pos * theta^(-2i/D) for pair i: (i, i + D/2) in the
    rotate-half form, (2i, 2i + 1) in the interleaved form."""
    D = len(x)
    h = D // 2
    y = list(x)
    for i in range(h):
        a = pos * theta ** (-2.0 * i / D)
        c, s = math.cos(a), math.sin(a)
        u, v = (2 * i, 2 * i + 1) if interleaved else (i, i + h)
        y[u] = x[u] * c - x[v] * s
        y[v] = x[v] * c + x[u] * s
    return y


def step(q, k_new, v_new, pool, page_table, seq_lens, active, P, theta, sm_scale=None,
         positions=None, q_norm_w=None, k_norm_w=None, eps=1e-6, dtype="bf16", interleaved=False):
    """Whole step on nested lists of bf16 (or, dtype "fp16", fp16) bit patterns.

    q: [B][Hq][D], k_new/v_new: [B][Hkv][D], pool: [NP][2][P][Hkv][D] (bits, mutated
    in place), page_table: [B][MPS], seq_lens/active: [B].
    Returns (q_rot [B][Hq][D] floats, out [B][Hq][D] floats).
    """
    B = len(q)
    Hq = len(q[0])
    D = len(q[0][0])
    Hkv = len(k_new[0])
    G = Hq // Hkv
    scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(D)
    dec = DECODE[dtype]
    enc = f16_round_bits if dtype == "fp16" else bf16_round_bits
    q_rot = [[[0.0] * D for _ in range(Hq)] for _ in range(B)]
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        if not active[b]:
            continue
        L = seq_lens[b]
        pos = positions[b] if positions is not None else L - 1
        for g in range(Hq):
            q_rot[b][g] = rope(rms_norm([dec(v) for v in q[b][g]], q_norm_w, eps), pos, theta, interleaved)
        slot = L - 1
        page = page_table[b][slot // P]
        off = slot % P
        for h in range(Hkv):
            kr = rope(rms_norm([dec(v) for v in k_new[b][h]], k_norm_w, eps), pos, theta, interleaved)
            pool[page][0][off][h] = [enc(v) for v in kr]
            pool[page][1][off][h] = list(v_new[b][h])
    for b in range(B):
        if not active[b]:
            continue
        L = seq_lens[b]
        for g in range(Hq):
            h = g // G
            scores = []
            for j in range(L):
                page = page_table[b][j // P]
                krow = [dec(v) for v in pool[page][0][j % P][h]]
                scores.append(scale * math.fsum(a * c for a, c in zip(q_rot[b][g], krow)))
            m = max(scores)
            w = [math.exp(s - m) for s in scores]
            tot = math.fsum(w)
            o = [0.0] * D
            for j in range(L):
                page = page_table[b][j // P]
                vrow = [dec(v) for v in pool[page][1][j % P][h]]
                for d in range(D):
                    o[d] += w[j] * vrow[d]
            out[b][g] = [v / tot for v in o]
    return q_rot, out
