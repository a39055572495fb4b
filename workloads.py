"""Seeded synthetic inputs for the paged q_len=1 decode step.

This module only draws inputs: batch shapes, sequence lengths, page tables,
KV pools and the new q/k/v rows. It holds none of the method's arithmetic
(no RoPE, no softmax, no append), so both the float64 oracle and the CUDA
library can take their inputs from it without sharing any code.

The five workloads are the serving shapes of the Talker decode step:
  * "tiny"    -- 4 rows, 8 q / 2 kv heads, head_dim 64, pages of 16 tokens,
                 lengths {17, 64, 129, 200}, a 64-page pool;
  * "c64"     -- 64 concurrent rows (the c=64 serving load), 16 q / 8 kv heads,
                 head_dim 128, pages of 16, lengths uniform in [200, 1200];
  * "padded"  -- a captured batch of 64 with 37 live rows and 27 padding rows
                 (active == 0, seq_len 1, page-table row all page 0);
  * "long"    -- 16 rows, 32 q / 8 kv heads, lengths uniform in [2048, 8192];
  * "high"    -- 256 rows, 32 q / 8 kv heads, pages of 64 tokens, lengths
                 log-uniform in [256, 4096], values N(0, 0.5), 28 layers that
                 each own a separate KV pool (the layers of one decode step
                 share the batch: lengths, active rows and page table);
  * "fastar"  -- the Fast AR step: 64 rows, 16 q / 8 kv heads, head_dim 64,
                 a contiguous per-request cache of 11 positions (10 residual
                 codebooks + 1) per layer, 4 layers, every row at its last
                 step (length 11).

Layout of one layer's pool (the paged KV layout of the vox-serve "Adding a
Model" page, section "1. The model code", with the layer axis dropped because
every layer here owns its own pool):  bf16 (or fp16) [num_pages, 2,
page_size, num_kv_heads, head_dim], K at [:, 0] and V at [:, 1]; on request
the same values are stored head-major, [num_pages, 2, num_kv_heads,
page_size, head_dim] (the other layout generic paged attention offers).

Recipe (seed = 20260000 + 100 * workload_index + layer, torch.Generator; for
the layers of one step of a multi-layer workload, steps 1-3 come from the
seed of the step's first layer, so every layer sees the same batch, and the
values of steps 4-5 from the layer's own seed):
  1. seq_lens: integers uniform in [lo, hi], or floor(exp(U(ln lo, ln hi)))
     clamped to [lo, hi] for the log-uniform workload; "tiny" uses its fixed
     list.  A length counts the token being appended (position = len - 1).
  2. active rows: all rows, or (padded workload) a seeded random subset;
     padding rows get seq_len 1 and a page-table row of zeros.
  3. pages: page 0 is the reserved dummy page and the last page is a guard
     page.  Live pages are a seeded permutation of 1 .. num_pages - 2,
     handed out to the active rows in row order and logical page order.
  4. pool values: randn * sigma rounded to the element type; every slot that holds no
     cached token (page 0, the guard page, unused pages, the tail of each
     row's last page and the slot the new token will be appended to) is
     filled with a quiet-NaN bit pattern, so a read of a stale slot shows up
     in the output.
  5. q ~ N(0, 1); k_new, v_new ~ N(0, sigma); all bf16, or all fp16 when
     fp16 is asked for (the same float32 draws, rounded to fp16 instead).

The generator runs on any torch device; large pools are drawn on the GPU and
copied to the host where the oracle needs them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

# 0x7FC0 is a quiet NaN both as bf16 (exponent all ones, mantissa 0x40) and
# as fp16 (exponent 0x1F, mantissa 0x3C0), so one pattern poisons either type.
NAN_BITS = 0x7FC0
SEED_BASE = 20260000


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    Hq: int
    Hkv: int
    D: int
    P: int
    len_lo: int
    len_hi: int
    dist: str = "uniform"          # "fixed" | "uniform" | "loguniform"
    fixed_lens: tuple = ()
    n_active: int | None = None     # None: all rows active
    sigma: float = 1.0
    layers: int = 1
    pool_pages: int = 0             # minimum pool size (0: just what is needed)
    theta: float = 10000.0
    layout: str = "NHD"             # default cache layout (see make_case)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def max_pages_per_seq(self) -> int:
        return -(-self.len_hi // self.P)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", 0, B=4, Hq=8, Hkv=2, D=64, P=16, len_lo=17, len_hi=200,
                 dist="fixed", fixed_lens=(17, 64, 129, 200), pool_pages=64),
        Workload("c64", 1, B=64, Hq=16, Hkv=8, D=128, P=16, len_lo=200, len_hi=1200),
        Workload("padded", 2, B=64, Hq=16, Hkv=8, D=128, P=16, len_lo=100, len_hi=800,
                 n_active=37),
        Workload("long", 3, B=16, Hq=32, Hkv=8, D=128, P=16, len_lo=2048, len_hi=8192),
        Workload("high", 4, B=256, Hq=32, Hkv=8, D=128, P=64, len_lo=256, len_hi=4096,
                 dist="loguniform", sigma=0.5, layers=28),
        Workload("fastar", 5, B=64, Hq=16, Hkv=8, D=64, P=11, len_lo=11, len_hi=11,
                 dist="fixed", fixed_lens=(11,) * 64, layers=4, layout="CONTIG"),
    ]
}


@dataclass
class DecodeInputs:
    """One layer's inputs.  Tensors live on `device`; q, k_new, v_new and pool
    are all torch.bfloat16 or all torch.float16."""
    B: int
    Hq: int
    Hkv: int
    D: int
    P: int
    max_pages_per_seq: int
    num_pages: int
    theta: float
    q: torch.Tensor            # [B, Hq, D] bf16 / fp16
    k_new: torch.Tensor        # [B, Hkv, D]
    v_new: torch.Tensor        # [B, Hkv, D]
    pool: torch.Tensor         # NHD: [NP, 2, P, Hkv, D]; HND: [NP, 2, Hkv, P, D] (K at [:,0], V at [:,1]);
                               # CONTIG: [2, B, Hkv, P, D] (K at [0], V at [1])
    page_table: torch.Tensor   # [B, MPS] int32
    seq_lens: torch.Tensor     # [B] int32
    active: torch.Tensor       # [B] int32
    meta: dict = field(default_factory=dict)
    layout: str = "NHD"        # "NHD": token-major pages; "HND": head-major pages;
                               # "CONTIG": one contiguous cache per row, no page table

    # element strides of the pool, as the C interface takes them
    @property
    def page_stride(self) -> int:
        return self.P * self.Hkv * self.D * (1 if self.layout == "CONTIG" else 2)

    @property
    def token_stride(self) -> int:
        return self.Hkv * self.D if self.layout == "NHD" else self.D

    @property
    def head_stride(self) -> int:
        return self.D if self.layout == "NHD" else self.P * self.D

    @property
    def api_page_table(self):
        """The page table the library gets: None for contiguous caches."""
        return None if self.layout == "CONTIG" else self.page_table

    def k_cache(self) -> torch.Tensor:
        """K as a [NP, P, Hkv, D] view (strided unless token-major)."""
        if self.layout == "CONTIG":
            return self.pool[0].transpose(1, 2)
        return self.pool[:, 0] if self.layout == "NHD" else self.pool[:, 0].transpose(1, 2)

    def v_cache(self) -> torch.Tensor:
        if self.layout == "CONTIG":
            return self.pool[1].transpose(1, 2)
        return self.pool[:, 1] if self.layout == "NHD" else self.pool[:, 1].transpose(1, 2)

    def nhd_pool(self) -> torch.Tensor:
        """The pool in token-major order [NP, 2, P, Hkv, D] (a view, or the pool itself)."""
        if self.layout == "CONTIG":
            return self.pool.permute(1, 0, 3, 2, 4)
        return self.pool if self.layout == "NHD" else self.pool.transpose(2, 3)

    def _fields(self, fn) -> "DecodeInputs":
        kw = {k: getattr(self, k) for k in ("B", "Hq", "Hkv", "D", "P", "max_pages_per_seq",
                                            "num_pages", "theta", "layout")}
        for k in ("q", "k_new", "v_new", "pool", "page_table", "seq_lens", "active"):
            kw[k] = fn(getattr(self, k))
        return DecodeInputs(meta=dict(self.meta), **kw)

    def to(self, device) -> "DecodeInputs":
        return self._fields(lambda t: t.to(device))

    def clone(self) -> "DecodeInputs":
        return self._fields(lambda t: t.clone())

    def as_nhd(self) -> "DecodeInputs":
        """The same inputs with a token-major (contiguous) copy of the pool."""
        d = self._fields(lambda t: t)
        d.pool = self.nhd_pool().contiguous()
        d.layout = "NHD"
        return d


def draw_lengths(w: Workload, gen: torch.Generator, n: int) -> torch.Tensor:
    if w.dist == "fixed":
        return torch.tensor(w.fixed_lens, dtype=torch.int64)
    if w.dist == "uniform":
        return torch.randint(w.len_lo, w.len_hi + 1, (n,), generator=gen, dtype=torch.int64)
    if w.dist == "loguniform":
        u = torch.rand(n, generator=gen, dtype=torch.float64)
        x = torch.exp(math.log(w.len_lo) + u * (math.log(w.len_hi) - math.log(w.len_lo)))
        return torch.floor(x).to(torch.int64).clamp(w.len_lo, w.len_hi)
    raise ValueError(w.dist)


def make_case(*, B: int, Hq: int, Hkv: int, D: int, P: int, seq_lens, active=None,
              max_pages_per_seq: int | None = None, sigma: float = 1.0, seed: int = 0,
              device="cpu", pool_pages: int = 0, theta: float = 10000.0,
              poison: bool = True, page_order: str = "random",
              dtype: torch.dtype = torch.bfloat16, layout: str = "NHD",
              value_seed: int | None = None) -> DecodeInputs:
    """Draw one layer of inputs for explicit shapes and lengths.

    `seq_lens` and `active` are Python sequences (or int64 tensors) of length B.
    Padding rows (active == 0) get seq_len 1 and an all-zero page-table row
    unless the caller passes other lengths for them on purpose.
    `page_order` is "random" (seeded permutation) or "linear" (pages 1, 2, ...).
    `dtype` (torch.bfloat16 or torch.float16) is the type of q, k, v and the pool.
    `value_seed` (if given) seeds the pool and q/k/v values instead of `seed`,
    which then fixes only the page permutation.
    `layout` "HND" stores the same pool values head-major ([NP, 2, Hkv, P, D]);
    "CONTIG" makes one cache of P positions per row (row b owns page b, no
    page permutation) stored as [2, B, Hkv, P, D], with an identity page
    table kept for the oracle.
    """
    assert dtype in (torch.bfloat16, torch.float16)
    assert layout in ("NHD", "HND", "CONTIG")
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    lens = torch.as_tensor(seq_lens, dtype=torch.int64).clone()
    assert lens.numel() == B
    act = torch.ones(B, dtype=torch.int64) if active is None else torch.as_tensor(active, dtype=torch.int64).clone()
    mps = max_pages_per_seq if max_pages_per_seq is not None else max(1, -(-int(lens.max()) // P))
    npages_row = [(-(-int(lens[b]) // P)) if act[b] else 0 for b in range(B)]
    used = sum(npages_row)
    if layout == "CONTIG":
        assert mps == 1, "a contiguous cache holds one page of P positions per row"
        NP = B
        page_table = torch.arange(B, dtype=torch.int64).view(B, 1)
    else:
        NP = max(pool_pages, used + 2)
        if page_order == "random":
            perm = torch.randperm(NP - 2, generator=gen) + 1
        else:
            perm = torch.arange(1, NP - 1)
        page_table = torch.zeros(B, mps, dtype=torch.int64)
        nxt = 0
        for b in range(B):
            n = npages_row[b]
            assert n <= mps, "a row needs more pages than max_pages_per_seq"
            page_table[b, :n] = perm[nxt:nxt + n]
            nxt += n

    # Values are drawn on the target device from a seed derived from the CPU generator.
    dev = torch.device(device)
    dgen = torch.Generator(device=dev)
    vseed = int(torch.randint(0, 2**62, (1,), generator=gen))
    if value_seed is not None:
        vgen = torch.Generator(device="cpu")
        vgen.manual_seed(value_seed)
        vseed = int(torch.randint(0, 2**62, (1,), generator=vgen))
    dgen.manual_seed(vseed)
    pool = (torch.randn((NP, 2, P, Hkv, D), generator=dgen, device=dev, dtype=torch.float32) * sigma).to(dtype)
    q = torch.randn((B, Hq, D), generator=dgen, device=dev, dtype=torch.float32).to(dtype)
    k_new = (torch.randn((B, Hkv, D), generator=dgen, device=dev, dtype=torch.float32) * sigma).to(dtype)
    v_new = (torch.randn((B, Hkv, D), generator=dgen, device=dev, dtype=torch.float32) * sigma).to(dtype)

    if poison:
        live = torch.zeros((NP, P), dtype=torch.bool)
        for b in range(B):
            if not act[b]:
                continue
            # cached tokens are slots 0 .. L-2; slot L-1 receives the new token
            j = torch.arange(int(lens[b]) - 1)
            live[page_table[b, j // P], j % P] = True
        bits = pool.view(torch.int16)
        dead = (~live).to(dev)
        bits.masked_fill_(dead.view(NP, 1, P, 1, 1).expand_as(bits), NAN_BITS)

    if layout == "HND":
        pool = pool.transpose(2, 3).contiguous()
    elif layout == "CONTIG":
        pool = pool.permute(1, 0, 3, 2, 4).contiguous()
    return DecodeInputs(
        B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, max_pages_per_seq=mps, num_pages=NP, theta=theta, layout=layout,
        q=q, k_new=k_new, v_new=v_new, pool=pool,
        page_table=page_table.to(torch.int32).to(dev),
        seq_lens=lens.to(torch.int32).to(dev), active=act.to(torch.int32).to(dev),
        meta={"seed": seed, "sigma": sigma},
    )


def step_structure(name: str, first_layer: int = 0):
    """(seq_lens, active, page-permutation seed) of the step whose first layer
    is `first_layer` (steps 1-2 of the recipe)."""
    w = WORKLOADS[name]
    gen = torch.Generator(device="cpu")
    gen.manual_seed(SEED_BASE + 100 * w.index + first_layer)
    lens = draw_lengths(w, gen, w.B)
    if w.n_active is not None:
        rows = torch.randperm(w.B, generator=gen)[: w.n_active]
        act = torch.zeros(w.B, dtype=torch.int64)
        act[rows] = 1
        lens = torch.where(act.bool(), lens, torch.ones_like(lens))
    else:
        act = torch.ones(w.B, dtype=torch.int64)
    sub_seed = int(torch.randint(0, 2**31 - 1, (1,), generator=gen))
    return lens, act, sub_seed


def make_inputs(name: str, layer: int = 0, device="cpu", dtype: torch.dtype = torch.bfloat16,
                layout: str | None = None) -> DecodeInputs:
    """Inputs of one layer of a named workload (see the module docstring).

    For a workload of L > 1 layers, layer l belongs to the step whose first
    layer is l - l % L: the lengths, active rows and page table are those of
    that first layer, the pool and q/k/v values the layer's own."""
    w = WORKLOADS[name]
    seed = SEED_BASE + 100 * w.index + layer
    first = layer - layer % w.layers
    lens, act, sub_seed = step_structure(name, first)
    inp = make_case(B=w.B, Hq=w.Hq, Hkv=w.Hkv, D=w.D, P=w.P, seq_lens=lens, active=act,
                    max_pages_per_seq=w.max_pages_per_seq, sigma=w.sigma, seed=sub_seed,
                    device=device, pool_pages=w.pool_pages, theta=w.theta, dtype=dtype,
                    layout=layout or w.layout, value_seed=None if layer == first else seed)
    inp.meta.update({"workload": name, "layer": layer, "workload_seed": seed, "step_first_layer": first})
    return inp


def kv_bytes(inp: DecodeInputs) -> int:
    """K+V bytes one decode call must read: sum over active rows of L*Hkv*D*2*(element size)."""
    lens = inp.seq_lens.cpu().to(torch.int64)
    act = inp.active.cpu().to(torch.int64)
    return int((lens * act).sum()) * inp.Hkv * inp.D * 2 * inp.pool.element_size()
