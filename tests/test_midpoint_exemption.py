"""Host check of the append comparison's midpoint exemption (no GPU).

The GPU kernels rotate the new key in fp32 (fp32 cos/sin from the RoPE
table, products and a difference, possibly fused into an FMA) and round to
the element type; the oracle rotates in float64 and rounds once.  The two
may pick different neighbours only where the float64 value sits within the
fp32 error of a rounding midpoint.  Here the fp32 rotation is emulated on
the CPU with each contraction order the compiler may choose, and every
element where it rounds differently from the oracle must fall inside the
exemption window that the GPU parity tests grant (gpu_harness.midpoint_mask),
for bf16 and fp16 and both RoPE pairings.
"""
import pytest
import torch

import gpu_harness as H
import oracle
import workloads


def _table_row(pos, D, theta):
    i = torch.arange(D // 2, dtype=torch.float64)
    a = pos.view(-1, 1).double() * theta ** (-2.0 * i / D)
    return torch.cos(a).float().double(), torch.sin(a).float().double()   # fp32 values, held exactly


def _f32(x):
    return x.float().double()


def _emulated(k, c, s, interleaved, order):
    """fp32 rotation of keys k [B, H, D] (float64 holding exact 16-bit values)."""
    D = k.shape[-1]
    if interleaved:
        x, y = k[..., 0::2], k[..., 1::2]
    else:
        x, y = k[..., : D // 2], k[..., D // 2:]
    c, s = c.unsqueeze(1), s.unsqueeze(1)
    if order == "plain":
        rx, ry = _f32(_f32(x * c) - _f32(y * s)), _f32(_f32(y * c) + _f32(x * s))
    elif order == "fma_first":
        rx, ry = _f32(x * c - _f32(y * s)), _f32(y * c + _f32(x * s))
    else:
        rx, ry = _f32(_f32(x * c) - y * s), _f32(_f32(y * c) + x * s)
    if interleaved:
        return torch.stack([rx, ry], dim=-1).flatten(-2)
    return torch.cat([rx, ry], dim=-1)


@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_fp32_rotation_differs_from_float64_only_inside_the_window(dtype, interleaved):
    # one-token rows (each appends to slot 0 of its own page) at random
    # positions up to 9000, so the angles vary as in long rows
    B, Hkv, D, P = 384, 8, 128, 16
    g = torch.Generator().manual_seed(5)
    pos = torch.randint(0, 9000, (B,), generator=g)
    inp = workloads.make_case(B=B, Hq=Hkv, Hkv=Hkv, D=D, P=P, seq_lens=[1] * B, seed=6, dtype=dtype,
                              poison=False)
    q_rot, pool, bad, k_rot, k_pre = oracle.rope_kv_append(
        inp.q, inp.k_new, inp.v_new, inp.pool, inp.page_table, inp.seq_lens, inp.active, P=P,
        theta=inp.theta, positions=pos, return_k_rot=True, return_k_pre=True, interleaved=interleaved)
    assert bad == 0
    want = H.bits16(pool[inp.page_table[:, 0].long(), 0, 0])
    mask = H.midpoint_mask(k_rot, k_pre, H.MIDPOINT_REL, dtype=dtype, interleaved=interleaved)
    c, s = _table_row(pos, D, inp.theta)
    k = inp.k_new.double()
    n_diff = 0
    kp = k_pre.abs()
    if interleaved:
        pair = kp[..., 0::2] + kp[..., 1::2]
        scale = torch.stack([pair, pair], dim=-1).flatten(-2)
    else:
        pair = kp[..., : D // 2] + kp[..., D // 2:]
        scale = torch.cat([pair, pair], dim=-1)
    for order in ("plain", "fma_first", "fma_second"):
        val = _emulated(k, c, s, interleaved, order).float().to(dtype)
        got = H.bits16(val)
        diff = got != want
        assert not (diff & ~mask).any(), f"{order}: {int((diff & ~mask).sum())} differences outside the window"
        # the value test the GPU comparison applies to differing elements
        g_, x_ = val.double()[diff], k_rot[diff]
        mag = torch.maximum(g_.abs(), x_.abs())
        bits, qmin = H._GRID[dtype]
        e = torch.frexp(torch.where(mag > 0, mag, torch.ones_like(mag))).exponent
        step = torch.ldexp(torch.ones_like(mag), (e - bits).clamp(min=qmin))
        assert ((g_ - x_).abs() <= H.MIDPOINT_REL * scale[diff] + step).all()
        n_diff += int(diff.sum())
    # the window is narrow: a small share of all elements
    assert int(mask.sum()) < 0.01 * mask.numel()
    print(f"{dtype} interleaved={interleaved}: window {int(mask.sum())} of {mask.numel()}, differing {n_diff}")
