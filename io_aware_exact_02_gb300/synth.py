"""Seeded synthetic inputs for the attention workloads.

This module holds no attention arithmetic: it only draws random tensors.  It
is the one piece shared by the CUDA path's callers (tests, benchmark) and the
oracle's callers, so that both sides see the same bf16 bits.

Recipe (one torch generator per call, seeded with ``seed``; draw order Q, K,
[heavy-row permutation], V, dO; each tensor is ``randn(B, H, N, d)`` in fp32,
multiplied by ``qkv_scale`` (Q, K, V only), then rounded to bf16 with
round-to-nearest-even):

* iid N(0, 1) Q, K, V, dO -- the shapes the CMU 11-868 FlashAttention post
  quotes for the three-step attention (slide page 5: N from 1K to 8K, d from
  64 to 128);
* ``qkv_scale=0.5`` for the causal LM-training shape (exact in bf16: a power
  of two);
* ``heavy_frac=0.01``: after K is drawn, a permutation of the B*H*N key rows
  is drawn from the same generator and the first floor(0.01*B*H*N) rows of K
  (over all heads) are multiplied by 8 (exact in bf16).  These rows give
  heavy-tailed scores, so the running maximum of the online softmax keeps
  growing inside a row.

On a CUDA device the draws come from a CUDA generator with the same seed:
the same distribution, different bits from the CPU draw.  Parity tests
always draw on the CPU and copy to the device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    qkv_scale: float = 1.0
    heavy_frac: float = 0.0
    heavy_factor: float = 8.0
    scale: float = field(default=float("nan"))

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d) if math.isnan(self.scale) else self.scale

    @property
    def BH(self) -> int:
        return self.B * self.H

    def describe(self) -> str:
        s = "B=%d H=%d N=%d d=%d %s" % (self.B, self.H, self.N, self.d,
                                        "causal" if self.causal else "non-causal")
        if self.qkv_scale != 1.0:
            s += " qkv*%g" % self.qkv_scale
        if self.heavy_frac:
            s += " %g%% K rows x%g" % (100 * self.heavy_frac, self.heavy_factor)
        return s


# The five workloads: a tiny case, the forward sweep at the slides' sizes, a
# causal LM-training shape, a long-context stress case and a many-head
# backward-bound shape.
TINY = Workload("tiny", 1, 1, 128, 64, False)
SWEEP = [Workload("sweep_N%d_d%d" % (n, d), 8, 16, n, d, False)
         for d in (64, 128) for n in (1024, 2048, 4096, 8192)]
CAUSAL_LM = Workload("causal_lm", 4, 32, 4096, 128, True, qkv_scale=0.5)
LONG = Workload("long", 1, 16, 16384, 128, True, heavy_frac=0.01)
SMALL_BATCH = Workload("small_batch", 16, 12, 1024, 64, False)
HEADLINE = Workload("sweep_N8192_d128", 8, 16, 8192, 128, False)

ALL = [TINY, *SWEEP, CAUSAL_LM, LONG, SMALL_BATCH]


def by_name(name: str) -> Workload:
    for w in ALL:
        if w.name == name:
            return w
    raise KeyError(name)


def draw(B: int, H: int, N: int, d: int, seed: int = 0, qkv_scale: float = 1.0,
         heavy_frac: float = 0.0, heavy_factor: float = 8.0, device="cpu",
         with_dout: bool = True):
    """Draw (q, k, v, dout) as contiguous bf16 tensors of shape (B, H, N, d)."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    shape = (B, H, N, d)

    def randn():
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32)

    q = (randn() * qkv_scale).to(torch.bfloat16)
    k32 = randn() * qkv_scale
    if heavy_frac > 0.0:
        rows = B * H * N
        perm = torch.randperm(rows, generator=g, device=device)
        n_heavy = int(math.floor(heavy_frac * rows))
        k32 = k32.reshape(rows, d)
        k32[perm[:n_heavy]] *= heavy_factor
        k32 = k32.reshape(shape)
    k = k32.to(torch.bfloat16)
    v = (randn() * qkv_scale).to(torch.bfloat16)
    dout = randn().to(torch.bfloat16) if with_dout else None
    return q, k, v, dout


def draw_workload(w: Workload, seed: int = 0, device="cpu", with_dout: bool = True):
    return draw(w.B, w.H, w.N, w.d, seed=seed, qkv_scale=w.qkv_scale,
                heavy_frac=w.heavy_frac, heavy_factor=w.heavy_factor, device=device,
                with_dout=with_dout)


@dataclass(frozen=True)
class GqaWorkload:
    """A general-form workload: H_q query heads over H_kv key/value heads,
    N_q query rows per head against N_kv keys (causal aligned bottom-right)."""
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nkv: int
    d: int
    causal: bool

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# One-token decode over a 32K-key cache with 4 query heads per K/V head, and
# a causal GQA prefill at the LM-training shape's size.
DECODE = GqaWorkload("decode_B8_Hq32_Hkv8_Nkv32768_d128", 8, 32, 8, 1, 32768, 128, True)
GQA_PREFILL = GqaWorkload("gqa_prefill_B4_Hq32_Hkv8_N4096_d128", 4, 32, 8, 4096, 4096, 128, True)
GQA_ALL = [DECODE, GQA_PREFILL]


def gqa_by_name(name: str) -> GqaWorkload:
    for w in GQA_ALL:
        if w.name == name:
            return w
    raise KeyError(name)


def draw_gqa(w: GqaWorkload, seed: int = 0, device="cpu"):
    """(q, k, v) bf16: q (B, Hq, Nq, d), k and v (B, Hkv, Nkv, d), drawn in
    that order from one generator seeded with ``seed``, iid N(0, 1)."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    q = torch.randn((w.B, w.Hq, w.Nq, w.d), generator=g, device=device).to(torch.bfloat16)
    k = torch.randn((w.B, w.Hkv, w.Nkv, w.d), generator=g, device=device).to(torch.bfloat16)
    v = torch.randn((w.B, w.Hkv, w.Nkv, w.d), generator=g, device=device).to(torch.bfloat16)
    return q, k, v


@dataclass(frozen=True)
class BlockSparseWorkload:
    """Square attention with a 0/1 mask over (128-query block, 128-key block)
    pairs shared by every head (the block-sparse extension of FlashAttention
    in cs2680 Lecture 9's reading guide)."""
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    density: float

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def n_blocks(self) -> int:
        return -(-self.N // 128)


# The headline square shape with a quarter of the blocks active.
BLOCKSPARSE = BlockSparseWorkload("blocksparse_B8_H16_N8192_d128_density0.25", 8, 16, 8192, 128,
                                  False, 0.25)
BLOCKSPARSE_ALL = [BLOCKSPARSE]


def blocksparse_by_name(name: str) -> BlockSparseWorkload:
    for w in BLOCKSPARSE_ALL:
        if w.name == name:
            return w
    raise KeyError(name)


def draw_block_mask(n_blocks: int, density: float, seed: int = 0, diagonal: bool = True):
    """(n_blocks, n_blocks) uint8 on the CPU: each block is 1 with probability
    ``density`` (torch.rand < density from a CPU generator seeded with
    ``seed``); with ``diagonal`` the diagonal blocks are 1 as well, so that
    every query block sees keys under a causal mask."""
    g = torch.Generator()
    g.manual_seed(int(seed))
    m = (torch.rand((n_blocks, n_blocks), generator=g) < density).to(torch.uint8)
    if diagonal:
        m.fill_diagonal_(1)
    return m


def draw_outliers(B: int, H: int, N: int, d: int, seed: int = 0, frac: float = 0.001,
                  magnitude: float = 10.0, device="cpu"):
    """(q, k, v) bf16 with simulated outliers, the data on which incoherent
    processing pays off (CMU 11-868 FlashAttention post, slide page 24; the
    post gives no recipe, so this is the plainest one).  For each of Q, K, V
    in turn: x = randn(B, H, N, d); m = rand(B, H, N, d) < frac; entries
    where m holds are replaced by magnitude * randn(B, H, N, d); all from one
    generator seeded with ``seed``, in that order, then rounded to bf16."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = []
    for _ in range(3):
        x = torch.randn((B, H, N, d), generator=g, device=device)
        m = torch.rand((B, H, N, d), generator=g, device=device) < frac
        big = torch.randn((B, H, N, d), generator=g, device=device) * magnitude
        out.append(torch.where(m, big, x).to(torch.bfloat16))
    return tuple(out)
