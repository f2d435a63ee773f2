"""Seeded synthetic inputs for the UltraQuant KV-cache path.

This module only draws random numbers and lays out page tables.  It holds none
of the method's arithmetic, so both the CUDA path and the CPU oracle can take
their inputs from it.

Shapes and distributions follow the five decode workloads (all head_dim 128):
  tiny       B1  Hkv1 Hq4  ctx 1024, identity pages, fp32 K/V, outlier ch 3 & 77
  gqa8k      B16 Hkv8 Hq64 ctx 8192, shuffled pages
  mixed      B64 Hkv8 Hq64 seq_len ~ U[8192, 65536], 1% of tokens x8
  prefix128k B4  Hkv8 Hq64 ctx 131072, first 98304 tokens shared via the table
  append64k  B8  Hkv8 Hq64 32768 cached + 32768 appended tokens, then decode
K, V ~ N(0,1) with, per kv head, outlier channels scaled x20 in the original
(pre-rotation) basis, the same channels for K and V; q ~ N(0,1).  Values are
drawn in fp32 and cast to bf16 (round to nearest even) unless the workload
keeps fp32.  Draws are made in fixed token blocks with their own seeds, so any
token range of any sequence can be regenerated on its own.
"""
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

BLOCK = 2048  # tokens per independently seeded draw


def _mix(*xs: int) -> int:
    h = 0x243F6A8885A308D3
    for x in xs:
        h = (h ^ (int(x) & 0xFFFFFFFFFFFFFFFF)) * 0x100000001B3 & 0xFFFFFFFFFFFFFFFF
        h ^= h >> 29
    return h & 0x7FFFFFFFFFFFFFFF


@dataclass
class Workload:
    name: str
    B: int
    Hkv: int
    Hq: int
    D: int
    ps: int
    seq_lens: List[int]
    seed: int
    kv_fp32: bool = False
    shuffled: bool = True
    outlier_channels: Optional[List[List[int]]] = None
    n_outlier: int = 8
    outlier_scale: float = 20.0
    token_outlier_frac: float = 0.0
    token_outlier_scale: float = 8.0
    shared_prefix: int = 0          # tokens shared by all sequences via the block table
    extra_tokens: int = 0           # room for tokens appended after the initial context
    block_table: np.ndarray = field(default=None, repr=False)
    num_pages: int = 0

    def __post_init__(self):
        if self.outlier_channels is None:
            g = np.random.default_rng(_mix(self.seed, 7))
            self.outlier_channels = [sorted(g.choice(self.D, self.n_outlier, replace=False).tolist())
                                     for _ in range(self.Hkv)]
        self._layout()

    # ---------------------------------------------------------------- pages
    def _layout(self):
        ps = self.ps
        cap = [(L + self.extra_tokens + ps - 1) // ps for L in self.seq_lens]
        shared = self.shared_prefix // ps
        assert self.shared_prefix % ps == 0
        own = [c - shared for c in cap]
        total = shared + sum(own)
        self.max_pages = max(cap) if cap else 1
        perm = np.arange(total)
        if self.shuffled:
            perm = np.random.default_rng(_mix(self.seed, 11)).permutation(total)
        bt = np.zeros((self.B, self.max_pages), np.int32)
        nxt = shared
        for b in range(self.B):
            logical = list(range(shared)) + list(range(nxt, nxt + own[b]))
            nxt += own[b]
            bt[b, :len(logical)] = perm[logical]
        self.block_table = bt
        self.num_pages = int(total)

    def slots(self, b: int, start: int, n: int) -> np.ndarray:
        """Physical slots of tokens [start, start+n) of sequence b."""
        j = np.arange(start, start + n)
        return self.block_table[b, j // self.ps].astype(np.int64) * self.ps + j % self.ps

    # ----------------------------------------------------------------- draws
    def _kv_block(self, b: int, blk: int, device) -> torch.Tensor:
        """fp32 [2][BLOCK][Hkv][D] draw (K then V) of token block blk of seq b."""
        src_b = 0 if (blk + 1) * BLOCK <= self.shared_prefix else b
        gen = torch.Generator(device=device)
        gen.manual_seed(_mix(self.seed, 1, src_b, blk))
        x = torch.randn((2, BLOCK, self.Hkv, self.D), generator=gen, device=device, dtype=torch.float32)
        ch = torch.zeros((self.Hkv, self.D), device=device, dtype=torch.float32) + 1.0
        for h, chans in enumerate(self.outlier_channels):
            ch[h, chans] = self.outlier_scale
        x = x * ch
        if self.token_outlier_frac > 0:
            u = torch.rand((BLOCK,), generator=gen, device=device)
            tok = torch.where(u < self.token_outlier_frac, self.token_outlier_scale, 1.0)
            x = x * tok.view(1, BLOCK, 1, 1)
        return x

    def kv(self, b: int, start: int, n: int, device="cpu"):
        """K, V of tokens [start, start+n) of sequence b: [n][Hkv][D] each."""
        assert self.shared_prefix % BLOCK == 0
        if n <= 0:
            dt = torch.float32 if self.kv_fp32 else torch.bfloat16
            e = torch.empty((0, self.Hkv, self.D), dtype=dt, device=device)
            return e, e.clone()
        parts = []
        blk0, blk1 = start // BLOCK, (start + n - 1) // BLOCK
        for blk in range(blk0, blk1 + 1):
            parts.append(self._kv_block(b, blk, device))
        x = torch.cat(parts, dim=1)[:, start - blk0 * BLOCK: start - blk0 * BLOCK + n]
        if not self.kv_fp32:
            x = x.to(torch.bfloat16)
        return x[0].contiguous(), x[1].contiguous()

    def q(self, step: int = 0, device="cpu") -> torch.Tensor:
        gen = torch.Generator(device=device)
        gen.manual_seed(_mix(self.seed, 2, step))
        return torch.randn((self.B, self.Hq, self.D), generator=gen, device=device,
                           dtype=torch.float32).to(torch.bfloat16)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def total_tokens(self) -> int:
        return int(sum(self.seq_lens))


def make(name: str, **over) -> Workload:
    """The named workload; keyword arguments override fields (for small cases)."""
    if name == "tiny":
        w = dict(B=1, Hkv=1, Hq=4, D=128, ps=16, seq_lens=[1024], seed=0, kv_fp32=True,
                 shuffled=False, outlier_channels=[[3, 77]])
    elif name == "gqa8k":
        w = dict(B=16, Hkv=8, Hq=64, D=128, ps=16, seq_lens=[8192] * 16, seed=1002)
    elif name == "mixed":
        g = np.random.default_rng(_mix(1003, 5))
        w = dict(B=64, Hkv=8, Hq=64, D=128, ps=16,
                 seq_lens=g.integers(8192, 65536, size=64, endpoint=True).tolist(), seed=1003,
                 token_outlier_frac=0.01)
    elif name == "prefix128k":
        w = dict(B=4, Hkv=8, Hq=64, D=128, ps=16, seq_lens=[131072] * 4, seed=1004,
                 shared_prefix=98304)
    elif name == "append64k":
        w = dict(B=8, Hkv=8, Hq=64, D=128, ps=16, seq_lens=[32768] * 8, seed=1005,
                 extra_tokens=32768 + 16)
    else:
        raise KeyError(name)
    w.update(over)
    return Workload(name=name, **w)


NAMES = ["tiny", "gqa8k", "mixed", "prefix128k", "append64k"]
