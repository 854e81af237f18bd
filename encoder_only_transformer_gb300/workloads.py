"""Seeded synthetic inputs for the attention block.

This module holds no arithmetic of the method: it only draws sequence lengths
and fused-Wqkv rows from seeded torch CPU generators, so that the oracle and
the CUDA path are fed identical inputs.  The shapes follow the ModernBERT-base
model the pages describe (12 heads x 64, up to 8192 tokens per sequence,
22 layers, layer i global iff i % 3 == 0); no page names a dataset for this
path.

Recipe: ``g = torch.Generator('cpu').manual_seed(seed)``; sequence lengths are
drawn first with ``torch.randint(lo, hi + 1, (1,), generator=g)``; then
``qkv = torch.randn(T, 2304, generator=g) * sigma`` rounded to bf16.
"""
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

WIDTH = 2304          # 3 * 12 heads * 64
OUT_WIDTH = 768
N_LAYERS = 22


@dataclass
class Workload:
    name: str
    seed: int
    sigma: float
    lengths: List[int]
    kinds: List[str]
    qkv: torch.Tensor = field(repr=False)          # bf16 [T, 2304], CPU
    cu_seqlens: torch.Tensor = field(repr=False)   # int32 [n+1], CPU

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def n_seqs(self) -> int:
        return len(self.lengths)

    @property
    def max_seqlen(self) -> int:
        return max(self.lengths) if self.lengths else 0


def cu_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def draw_qkv(g: torch.Generator, T: int, sigma: float, sigma_qk: Optional[float] = None) -> torch.Tensor:
    """randn(T, 2304) * sigma rounded to bf16; with sigma_qk the Q and K
    columns (0 .. 1535) are drawn with that spread instead, V keeping sigma."""
    x = torch.randn(T, WIDTH, generator=g, dtype=torch.float32)
    if sigma != 1.0:
        x.mul_(sigma)
    if sigma_qk is not None:
        x[:, :2 * OUT_WIDTH].mul_(sigma_qk / sigma)
    return x.to(torch.bfloat16)


def custom(lengths, seed: int, sigma: float = 1.0, kinds=("global", "local"),
           name: Optional[str] = None, sigma_qk: Optional[float] = None) -> Workload:
    g = torch.Generator().manual_seed(seed)
    lengths = [int(L) for L in lengths]
    cu = cu_from_lengths(lengths)
    qkv = draw_qkv(g, int(cu[-1]), sigma, sigma_qk)
    return Workload(name or f"custom{lengths}", seed, sigma, lengths, list(kinds), qkv, cu)


def spiked(lengths, seed: int, every: int, factor: float) -> Workload:
    """N(0, 1) rows whose K columns (768 .. 1535, every head) are multiplied
    by `factor` on every `every`-th packed row: a few keys whose scores are
    far above (or below) the rest for many queries."""
    g = torch.Generator().manual_seed(seed)
    lengths = [int(L) for L in lengths]
    cu = cu_from_lengths(lengths)
    T = int(cu[-1])
    x = torch.randn(T, WIDTH, generator=g, dtype=torch.float32)
    x[::every, OUT_WIDTH:2 * OUT_WIDTH].mul_(factor)
    return Workload(f"spiked{lengths}x{factor}", seed, 1.0, lengths, ["global", "local"],
                    x.to(torch.bfloat16), cu)


def towering_keys(lengths, seed: int, heads: int = 6, first: float = 0.05,
                  later: float = 40.0) -> Workload:
    """N(0, 1) rows; in the first sequence and heads 0 .. heads-1 the K rows
    of the first 128 keys are multiplied by `first` and every later K row by
    `later`: scores that stay small over a query's first key tile and rise
    hundreds of binary orders of magnitude above it afterwards."""
    g = torch.Generator().manual_seed(seed)
    lengths = [int(L) for L in lengths]
    cu = cu_from_lengths(lengths)
    x = torch.randn(int(cu[-1]), WIDTH, generator=g, dtype=torch.float32)
    L0 = lengths[0] if lengths else 0
    for h in range(heads):
        cols = slice(OUT_WIDTH + 64 * h, OUT_WIDTH + 64 * h + 64)
        x[0:min(128, L0), cols] *= first
        x[128:L0, cols] *= later
    return Workload(f"towering{lengths}", seed, 1.0, lengths, ["global"], x.to(torch.bfloat16), cu)


def aligned_keys(lengths, seed: int, first: float = 0.2, later: float = 2.0,
                 noise: float = 0.3, first_rows: int = 128) -> Workload:
    """Per head one random direction u (norm 8): every Q row is u plus
    N(0, noise^2) noise, every K row `first` (the first `first_rows` keys of
    each sequence) or `later` times u plus noise; V ~ N(0, 1).  A key near
    the query's own position then scores close to |q| |k| / 8, so the
    scores of later key tiles rise far above those of the first ones while
    staying close to the Cauchy-Schwarz bound of the norms."""
    g = torch.Generator().manual_seed(seed)
    lengths = [int(L) for L in lengths]
    cu = cu_from_lengths(lengths)
    T = int(cu[-1])
    x = torch.randn(T, WIDTH, generator=g, dtype=torch.float32)
    for h in range(12):
        u = torch.randn(64, generator=g)
        u *= 8.0 / u.norm()
        qc = slice(64 * h, 64 * h + 64)
        kc = slice(OUT_WIDTH + 64 * h, OUT_WIDTH + 64 * h + 64)
        x[:, qc] = u + noise * torch.randn(T, 64, generator=g)
        scale = torch.full((T, 1), later)
        for b in cu[:-1].tolist():
            scale[b:b + first_rows] = first
        x[:, kc] = scale * (u + noise * torch.randn(T, 64, generator=g))
    return Workload(f"aligned{lengths}", seed, 1.0, lengths, ["global"], x.to(torch.bfloat16), cu)


def band_probe(lengths, magnitude: float = 16.0) -> Workload:
    """Q = K = 0 and, in head h, V[t, h*64 + d] = magnitude when
    (t + h) % 64 == d, else 0 (t the packed row): no randomness.  Every key
    puts its magnitude into one column of each head, so a key the softmax
    admits in error, or leaves out, moves that column of the query's output
    by about magnitude / (number of admitted keys)."""
    lengths = [int(L) for L in lengths]
    cu = cu_from_lengths(lengths)
    T = int(cu[-1])
    x = torch.zeros(T, WIDTH, dtype=torch.float32)
    t = torch.arange(T)
    for h in range(12):
        x[t, 2 * OUT_WIDTH + h * 64 + (t + h) % 64] = magnitude
    return Workload(f"band_probe{lengths}", 0, 0.0, lengths, ["global", "local"],
                    x.to(torch.bfloat16), cu)


def _uniform_lengths(g, n, lo, hi):
    return [int(torch.randint(lo, hi + 1, (1,), generator=g)) for _ in range(n)]


def _fill_lengths(g, total, lo, hi):
    """Draw L ~ U{lo..hi} until the next draw would overflow `total`; the last
    sequence takes the remainder."""
    out, acc = [], 0
    while True:
        L = int(torch.randint(lo, hi + 1, (1,), generator=g))
        if acc + L > total:
            if total - acc > 0:
                out.append(total - acc)
            return out
        out.append(L)
        acc += L


def layer_kind(i: int) -> str:
    """Layer i of the 22-layer schedule is global iff i % 3 == 0."""
    return "global" if i % 3 == 0 else "local"


def config(k: int, layer: int = 0) -> Workload:
    """The five synthetic workloads.

    1: one sequence of 300 tokens, sigma 1, seed 1.
    2: 8 sequences, L ~ U{64..512}, sigma 1, seed 2.
    3: one sequence of 8192 tokens, sigma 1, seed 3.
    4: 65536 tokens, L ~ U{128..8192} filled to the total, sigma 0.5, seed 4.
    5: 32 x 8192 tokens; layer i of 22 uses seed 1000 + i and is global iff
       i % 3 == 0.
    """
    if k == 1:
        g = torch.Generator().manual_seed(1)
        lengths = [300]
        sigma, kinds, seed = 1.0, ["local", "global"], 1
    elif k == 2:
        g = torch.Generator().manual_seed(2)
        lengths = _uniform_lengths(g, 8, 64, 512)
        sigma, kinds, seed = 1.0, ["local", "global"], 2
    elif k == 3:
        g = torch.Generator().manual_seed(3)
        lengths = [8192]
        sigma, kinds, seed = 1.0, ["global", "local"], 3
    elif k == 4:
        g = torch.Generator().manual_seed(4)
        lengths = _fill_lengths(g, 65536, 128, 8192)
        sigma, kinds, seed = 0.5, ["local", "global"], 4
    elif k == 5:
        seed = 1000 + layer
        g = torch.Generator().manual_seed(seed)
        lengths = [8192] * 32
        sigma, kinds = 1.0, [layer_kind(layer)]
    else:
        raise ValueError(f"no workload {k}")
    cu = cu_from_lengths(lengths)
    qkv = draw_qkv(g, int(cu[-1]), sigma)
    return Workload(f"config{k}" + (f"_layer{layer}" if k == 5 else ""), seed, sigma,
                    lengths, kinds, qkv, cu)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 view of a bf16 CPU tensor (no conversion)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_rows(cu_seqlens, per_seq: int, seed: int) -> np.ndarray:
    """A seeded, sorted sample of packed row indices: `per_seq` rows from each
    sequence (all of them when it is shorter), always including its first and
    last rows."""
    g = torch.Generator().manual_seed(seed)
    cu = [int(x) for x in cu_seqlens]
    rows = []
    for s in range(len(cu) - 1):
        b, e = cu[s], cu[s + 1]
        L = e - b
        if L <= 0:
            continue
        if L <= per_seq:
            rows.extend(range(b, e))
            continue
        pick = torch.randperm(L, generator=g)[:per_seq - 2].tolist()
        sel = set(pick) | {0, L - 1}
        rows.extend(b + i for i in sorted(sel))
    return np.asarray(sorted(rows), dtype=np.int64)
