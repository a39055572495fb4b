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


def rope(x: list[float], pos: float, theta: float) -> list[float]:
    """Rotate-half RoPE: pair (i, i + D/2), angle pos * theta^(-2i/D)."""
    D = len(x)
    h = D // 2
    y = list(x)
    for i in range(h):
        a = pos * theta ** (-2.0 * i / D)
        c, s = math.cos(a), math.sin(a)
        y[i] = x[i] * c - x[i + h] * s
        y[i + h] = x[i + h] * c + x[i] * s
    return y


def step(q, k_new, v_new, pool, page_table, seq_lens, active, P, theta, sm_scale=None,
         positions=None, q_norm_w=None, k_norm_w=None, eps=1e-6):
    """Whole step on nested lists of bf16 bit patterns.

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
    q_rot = [[[0.0] * D for _ in range(Hq)] for _ in range(B)]
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        if not active[b]:
            continue
        L = seq_lens[b]
        pos = positions[b] if positions is not None else L - 1
        for g in range(Hq):
            q_rot[b][g] = rope(rms_norm([bf16_bits_to_float(v) for v in q[b][g]], q_norm_w, eps), pos, theta)
        slot = L - 1
        page = page_table[b][slot // P]
        off = slot % P
        for h in range(Hkv):
            kr = rope(rms_norm([bf16_bits_to_float(v) for v in k_new[b][h]], k_norm_w, eps), pos, theta)
            pool[page][0][off][h] = [bf16_round_bits(v) for v in kr]
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
                krow = [bf16_bits_to_float(v) for v in pool[page][0][j % P][h]]
                scores.append(scale * math.fsum(a * c for a, c in zip(q_rot[b][g], krow)))
            m = max(scores)
            w = [math.exp(s - m) for s in scores]
            tot = math.fsum(w)
            o = [0.0] * D
            for j in range(L):
                page = page_table[b][j // P]
                vrow = [bf16_bits_to_float(v) for v in pool[page][1][j % P][h]]
                for d in range(D):
                    o[d] += w[j] * vrow[d]
            out[b][g] = [v / tot for v in o]
    return q_rot, out
