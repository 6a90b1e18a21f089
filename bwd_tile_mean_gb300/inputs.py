"""Seeded synthetic problems for tile-top-k block-sparse video attention.

This module only describes problem shapes and draws random inputs. It holds
none of the method's arithmetic, so both the CUDA path and the CPU oracle
may be fed from it.

Shapes follow the pages' workloads:

* the 3D video tile is 4x8x8 = 256 tokens, with padded tiles zero-filled
  after their valid tokens (FastVideo test_vsa256_backward.py, ``_BLOCK``,
  ``_BLOCK_SIZE_3D`` and ``_zero_pad_tail``);
* q, k, v and dO are N(0, 1) drawn in that order from one seed, and the
  padded tails of q, k and v are zeroed (same page, ``_make_inputs``);
* the varlen GQA case uses 128x128 blocks, 12 query heads over 3 KV heads
  and head_dim 128 (Ascend test_npu_block_sparse_attention_backward.py,
  module constants ``TND_GQA_*``).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch

LAYOUTS = ("bhsd", "bshd", "tnd")
DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclass
class Problem:
    """One attention problem: sizes, tile fill and sparsity parameters.

    For the padded video layouts (``bhsd``/``bshd``) every batch entry has
    ``nQ`` query tiles and ``nKV`` key/value tiles; ``q_var``/``kv_var`` give
    the valid tokens of each tile (shared over batch and heads). For the
    varlen layout (``tnd``) sequences are packed along T and ``q_lens`` /
    ``kv_lens`` give each sequence's length; tiles are cut at sequence ends.
    """

    name: str
    layout: str
    B: int
    Hq: int
    Hkv: int
    D: int
    tile_q: int
    tile_kv: int
    nQ: int
    nKV: int
    dtype: str = "bf16"
    q_var: Optional[np.ndarray] = None
    kv_var: Optional[np.ndarray] = None
    q_lens: Optional[List[int]] = None
    kv_lens: Optional[List[int]] = None
    topk: Optional[int] = None          # None: an explicit block mask is used
    gate: Optional[str] = None          # None | "randn01" | "uniform_token_head"
    seed: int = 42
    mask_p: float = 0.5                 # Bernoulli rate of an explicit mask
    backward: bool = True
    note: str = ""
    scale: float = field(init=False)

    def __post_init__(self):
        assert self.layout in LAYOUTS and self.dtype in DTYPES
        self.scale = float(np.float32(1.0 / math.sqrt(self.D)))
        if self.layout != "tnd":
            self.q_var = np.asarray(self.q_var, dtype=np.int32)
            self.kv_var = np.asarray(self.kv_var, dtype=np.int32)
            assert self.q_var.shape == (self.nQ,) and self.kv_var.shape == (self.nKV,)

    # sizes -------------------------------------------------------------
    @property
    def varlen(self) -> bool:
        return self.layout == "tnd"

    @property
    def Sq(self) -> int:
        return sum(self.q_lens) if self.varlen else self.nQ * self.tile_q

    @property
    def Skv(self) -> int:
        return sum(self.kv_lens) if self.varlen else self.nKV * self.tile_kv

    @property
    def cu_q(self) -> Optional[np.ndarray]:
        return None if not self.varlen else np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    @property
    def cu_kv(self) -> Optional[np.ndarray]:
        return None if not self.varlen else np.concatenate([[0], np.cumsum(self.kv_lens)]).astype(np.int32)

    @property
    def max_q(self) -> int:
        return max(self.q_lens) if self.varlen else self.Sq

    @property
    def max_kv(self) -> int:
        return max(self.kv_lens) if self.varlen else self.Skv

    @property
    def cap(self) -> int:
        """Per-Q-tile capacity of the block index (selected KV tiles)."""
        return min(self.topk, self.nKV) if self.topk is not None else self.nKV

    def tile_var(self, q_side: bool, b: int, t: int) -> int:
        T = self.tile_q if q_side else self.tile_kv
        if self.varlen:
            n = (self.q_lens if q_side else self.kv_lens)[b]
            return max(0, min(T, n - t * T))
        return int((self.q_var if q_side else self.kv_var)[t])

    def shape(self, q_side: bool, heads: Optional[int] = None) -> tuple:
        H = heads if heads is not None else (self.Hq if q_side else self.Hkv)
        S = self.Sq if q_side else self.Skv
        if self.layout == "bhsd":
            return (self.B, H, S, self.D)
        if self.layout == "bshd":
            return (self.B, S, H, self.D)
        return (S, H, self.D)

    def lse_shape(self) -> tuple:
        return (self.Hq, self.Sq) if self.varlen else (self.B, self.Hq, self.Sq)

    def rows(self):
        """Every existing query row as (b, h, s), s within batch entry b."""
        out = []
        for b in range(self.B):
            n = self.q_lens[b] if self.varlen else self.Sq
            for h in range(self.Hq):
                out.extend((b, h, s) for s in range(n))
        return np.asarray(out, dtype=np.int32).reshape(-1, 3)

    def kv_tiles(self):
        return np.asarray([(b, hk, j) for b in range(self.B) for hk in range(self.Hkv)
                           for j in range(self.nKV)], dtype=np.int32).reshape(-1, 3)


# ---------------------------------------------------------------- tensors

def _valid_rows(p: Problem, q_side: bool) -> torch.Tensor:
    """Boolean [S] per batch layout: True on a tile's valid slots."""
    T = p.tile_q if q_side else p.tile_kv
    var = torch.as_tensor(p.q_var if q_side else p.kv_var, dtype=torch.int64)
    slot = torch.arange(T).view(1, -1)
    return (slot < var.view(-1, 1)).reshape(-1)


def _zero_tails(p: Problem, x: torch.Tensor, q_side: bool) -> torch.Tensor:
    if p.varlen:
        return x
    valid = _valid_rows(p, q_side).to(x.device)
    if p.layout == "bhsd":
        return x * valid.view(1, 1, -1, 1).to(x.dtype)
    return x * valid.view(1, -1, 1, 1).to(x.dtype)


def make_tensors(p: Problem, device="cpu") -> Dict[str, torch.Tensor]:
    """q, k, v, dO (and gate) for problem p, drawn from p.seed in that order.

    Draws happen on ``device`` with a generator seeded from ``p.seed``;
    padded tails of q, k, v are zeroed.
    """
    dt = DTYPES[p.dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(p.seed)
    sq, skv = p.shape(True), p.shape(False)
    t = {}
    t["q"] = _zero_tails(p, torch.randn(sq, generator=gen, device=device, dtype=dt), True)
    t["k"] = _zero_tails(p, torch.randn(skv, generator=gen, device=device, dtype=dt), False)
    t["v"] = _zero_tails(p, torch.randn(skv, generator=gen, device=device, dtype=dt), False)
    t["dO"] = torch.randn(sq, generator=gen, device=device, dtype=dt)
    if p.gate == "randn01":
        t["gate"] = (torch.randn(sq, generator=gen, device=device, dtype=dt) * 0.1).to(dt)
    elif p.gate == "uniform_token_head":
        g = torch.rand(sq[:-1] + (1,), generator=gen, device=device, dtype=torch.float32)
        t["gate"] = g.expand(sq).to(dt).contiguous()
    return t


def make_mask(p: Problem) -> np.ndarray:
    """Explicit Bernoulli(mask_p) block mask [B, Hq, nQ, nKV] (uint8), drawn
    from a CPU generator seeded with p.seed + 1 after the lengths."""
    gen = torch.Generator().manual_seed(p.seed + 1)
    m = torch.rand((p.B, p.Hq, p.nQ, p.nKV), generator=gen) < p.mask_p
    return m.to(torch.uint8).numpy()


# ---------------------------------------------------------------- problems

def _video_tile_fill(grid, tile=(4, 8, 8)):
    """Valid tokens of each 4x8x8 tile of a T x H x W latent grid, tiles in
    raster order (T-tile, H-tile, W-tile); edge tiles hold fewer tokens."""
    out = []
    nt = [math.ceil(g / t) for g, t in zip(grid, tile)]
    for a in range(nt[0]):
        ta = min(tile[0], grid[0] - a * tile[0])
        for b in range(nt[1]):
            tb = min(tile[1], grid[1] - b * tile[1])
            for c in range(nt[2]):
                tc = min(tile[2], grid[2] - c * tile[2])
                out.append(ta * tb * tc)
    return np.asarray(out, dtype=np.int32)


def varlen_lengths(batch: int, q_range, kv_range, seed: int):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randint(q_range[0], q_range[1] + 1, (batch,), generator=gen).tolist()
    kv = torch.randint(kv_range[0], kv_range[1] + 1, (batch,), generator=gen).tolist()
    return q, kv


def tnd_problem(name, q_lens, kv_lens, Hq, Hkv, dtype="fp16", tile=128, seed=42, mask_p=0.5,
                topk=None, gate=None, note=""):
    nQ = math.ceil(max(q_lens) / tile)
    nKV = math.ceil(max(kv_lens) / tile)
    return Problem(name, "tnd", len(q_lens), Hq, Hkv, 128, tile, tile, nQ, nKV, dtype=dtype,
                   q_lens=list(q_lens), kv_lens=list(kv_lens), seed=seed, mask_p=mask_p, topk=topk,
                   gate=gate, note=note)


def config(n: int) -> Problem:
    """The five workloads (1: tiny VSA-256, 2: GQA varlen, 3: video DiT,
    4: gated + ragged tiles, 5: long-video forward only) and 6, the
    long-video grid taken literally (1,024 tiles, ragged, forward only)."""
    if n == 1:
        return Problem("tiny-vsa256", "bhsd", 1, 2, 2, 128, 256, 256, 3, 4,
                       q_var=[256] * 3, kv_var=[256, 173, 79, 256], topk=2,
                       note="B1 H2 D128 bf16, 3 Q x 4 KV tiles, topk 2")
    if n == 2:
        ql, kl = varlen_lengths(13, (7, 360), (11, 540), seed=42)
        return tnd_problem("gqa-varlen-tnd", ql, kl, 12, 3, dtype="fp16", seed=42,
                           note="13 seqs, Hq12 Hkv3 D128 fp16, [128,128] blocks, Bernoulli(0.5) mask")
    if n == 3:
        nt = 20 * 48 * 80 // 256
        return Problem("video-dit-76800", "bshd", 1, 40, 40, 128, 256, 256, nt, nt,
                       q_var=[256] * nt, kv_var=[256] * nt, topk=30,
                       note="grid 20x48x80 -> 300 tiles, 76,800 tokens, H40 D128 bf16 BSHD, topk 30")
    if n == 4:
        kv_var = _video_tile_fill((21, 45, 80))
        return Problem("gated-ragged", "bshd", 1, 24, 24, 128, 256, 256, 180, 360,
                       q_var=kv_var[:180], kv_var=kv_var, topk=16, gate="uniform_token_head",
                       note="KV grid 21x45x80 -> 360 tiles (75,600 tokens), Q = first 180 tiles, "
                            "H24 D128 bf16, topk 16, gate U(0,1) per token and head")
    if n == 5:
        return Problem("long-video-fwd", "bshd", 1, 24, 24, 128, 256, 256, 480, 480,
                       q_var=[256] * 480, kv_var=[256] * 480, topk=24, backward=False,
                       note="480 full tiles, 122,880 tokens, H24 D128 bf16 BSHD, topk 24, forward only")
    if n == 6:
        # the long-video grid taken literally: 32 x 60 x 128 tiled 4 x 8 x 8 is
        # 8 x 8 x 16 = 1,024 tiles (H = 60 leaves a last row of half tiles:
        # 896 tiles of 256 tokens, 128 of 128), 245,760 tokens
        var = _video_tile_fill((32, 60, 128))
        return Problem("long-video-literal-fwd", "bshd", 1, 24, 24, 128, 256, 256, len(var), len(var),
                       q_var=var, kv_var=var, topk=24, backward=False,
                       note="grid 32x60x128 -> 1,024 tiles (128 half tiles), 245,760 tokens, H24 D128 bf16 BSHD, "
                            "topk 24, forward only")
    raise ValueError(n)


def page_cases() -> List[Problem]:
    """The video-tile cases of the FastVideo VSA-256 backward test page
    (kv_var / q_var vectors, topk and seeds as printed there), each in both
    padded layouts."""
    specs = [
        ("p-basic", [256, 173, 79, 256], [256] * 3, 2, 42, None),
        ("p-gated", [256, 200, 256, 91], [256] * 3, 2, 7, "randn01"),
        ("p-partial-q", [256, 128, 256], [256, 61, 199], 2, 11, None),
        ("p-cross", [256, 143, 256, 256, 88], [256] * 2, 3, 13, None),
    ]
    out = []
    for name, kv, qv, topk, seed, gate in specs:
        for layout in ("bhsd", "bshd"):
            out.append(Problem(f"{name}-{layout}", layout, 1, 2, 2, 128, 256, 256, len(qv), len(kv),
                               q_var=qv, kv_var=kv, topk=topk, seed=seed, gate=gate))
    return out
