"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module only draws random numbers and lays out page tables; it holds
none of the cache's arithmetic (no quantisation, no attention).  Both the
CUDA path and the CPU oracle receive the same BF16 bits from here.

Value recipe (one seeded ``torch.Generator`` per stream, fp32 draws rounded
to BF16 with round-to-nearest-even by torch):
  * K, V, Q ~ N(0, 1);
  * optional outliers: an independent Bernoulli(p) per element multiplies it
    by a factor (1% x20 in the tiny-decode and append workloads);
  * optional per-(kv_head, channel) factors exp(N(0, 1)), drawn separately for
    K and V (the long-context workload's channel outliers);
  * optional all-zero 16-blocks: an independent Bernoulli(p) per block sets
    its 16 values to +0.0, applied last.
Shapes follow the page's workloads (Accelerating Long-Context and Agentic
Inference with NVFP4 KV Cache, A4: 32K / 160K / 1M contexts, GQA head_dim
128) and the shared 3,200-token agent prefix with 512-token chunks of the
prefix-caching page.

Each sequence's K/V come from their own generator, seeded from the workload
seed and the sequence index, so one sequence can be regenerated alone (for a
sampled oracle check of a huge cache) on the device that made it.  torch's
CPU and CUDA generators give different streams, so a check regenerates on
the same device the product inputs were drawn on.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

HEAD_DIM = 128
BLOCK = 16


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + int(stream) * 7_919 + 12_345) % (2**63 - 1))
    return g


def _normal(shape, seed, stream, device, chunk_elems=1 << 26) -> torch.Tensor:
    """N(0,1) fp32 draws rounded to BF16; generated in chunks to bound fp32 scratch."""
    g = _gen(seed, stream, device)
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        out[s:e] = torch.randn(e - s, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out.view(*shape)


@dataclasses.dataclass
class ValueRecipe:
    outlier_p: float = 0.0
    outlier_scale: float = 20.0
    channel_lognormal: bool = False
    zero_block_p: float = 0.0


def draw_kv(n_tokens: int, num_kv_heads: int, seed: int, stream: int, device, recipe: ValueRecipe,
            which: int, factors: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One BF16 tensor [n_tokens][num_kv_heads][128] of K (which=0) or V (which=1)."""
    shape = (n_tokens, num_kv_heads, HEAD_DIM)
    if recipe.outlier_p == 0.0 and not recipe.channel_lognormal and recipe.zero_block_p == 0.0:
        return _normal(shape, seed, 2 * stream + which, device)
    g = _gen(seed, 2 * stream + which, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if recipe.outlier_p > 0.0:
        hit = torch.rand(shape, generator=g, device=device) < recipe.outlier_p
        x = torch.where(hit, x * recipe.outlier_scale, x)
    if recipe.channel_lognormal:
        assert factors is not None
        x = x * factors.to(device)[None, :, :]
    x = x.to(torch.bfloat16)
    if recipe.zero_block_p > 0.0:
        zb = torch.rand((n_tokens, num_kv_heads, HEAD_DIM // BLOCK), generator=g, device=device) < recipe.zero_block_p
        x = x.view(n_tokens, num_kv_heads, HEAD_DIM // BLOCK, BLOCK)
        x = torch.where(zb[..., None], torch.zeros((), dtype=x.dtype, device=device), x)
        x = x.view(shape)
    return x


@dataclasses.dataclass
class DecodeWorkload:
    """A batch of cached sequences, their page table, and one decode query.

    block_table rows are padded with -1 past each sequence's last page.
    Sequences listed in ``shared_prefix_tokens`` > 0 all start with the same
    physical pages (prefix-cache reuse) and the same prefix K/V.
    """

    name: str
    seed: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    page_size: int
    num_pages: int
    seq_lens: torch.Tensor          # int32 [B] (cpu)
    block_table: torch.Tensor       # int32 [B][max_pages] (cpu)
    recipe: ValueRecipe
    shared_prefix_tokens: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(HEAD_DIM)

    def channel_factors(self, which: int) -> Optional[torch.Tensor]:
        if not self.recipe.channel_lognormal:
            return None
        g = _gen(self.seed, 1_000_000 + which, "cpu")
        return torch.exp(torch.randn((self.num_kv_heads, HEAD_DIM), generator=g, dtype=torch.float32))

    def q(self, device) -> torch.Tensor:
        return _normal((self.batch, self.num_q_heads, HEAD_DIM), self.seed, 999_999, device)

    def _draw(self, n, stream, device, which):
        return draw_kv(n, self.num_kv_heads, self.seed, stream, device, self.recipe, which,
                       self.channel_factors(which))

    def prefix_kv(self, device):
        """K, V of the shared prefix, [shared_prefix_tokens][Hkv][128]."""
        n = self.shared_prefix_tokens
        return self._draw(n, 500_000, device, 0), self._draw(n, 500_000, device, 1)

    def private_kv(self, b: int, device):
        """K, V of sequence b's own tokens (those after the shared prefix)."""
        n = int(self.seq_lens[b]) - self.shared_prefix_tokens
        return self._draw(n, b, device, 0), self._draw(n, b, device, 1)

    def seq_kv(self, b: int, device):
        """K, V of sequence b's whole cached context, [n][Hkv][128]."""
        k, v = self.private_kv(b, device)
        if self.shared_prefix_tokens:
            pk, pv = self.prefix_kv(device)
            k, v = torch.cat([pk, k]), torch.cat([pv, v])
        return k, v

    def slots(self, b: int, start: int = 0, end: Optional[int] = None) -> torch.Tensor:
        """int64 slot of each token position in [start, end) of sequence b."""
        end = int(self.seq_lens[b]) if end is None else end
        t = torch.arange(start, end, dtype=torch.int64)
        pages = self.block_table[b].to(torch.int64)[t // self.page_size]
        return pages * self.page_size + t % self.page_size


def _place_pages(gen: torch.Generator, num_pages: int, counts: List[int], shared: int = 0):
    """Physical pages for sequences needing `counts[i]` pages; the first `shared`
    pages of each sequence are common, the rest private, all seeded-permuted."""
    perm = torch.randperm(num_pages, generator=gen).to(torch.int32)
    shared_pages = perm[:shared]
    pos = shared
    rows = []
    for c in counts:
        own = perm[pos:pos + c - shared]
        pos += c - shared
        rows.append(torch.cat([shared_pages, own]))
    assert pos <= num_pages
    width = max(counts) if counts else 1
    bt = torch.full((len(counts), max(width, 1)), -1, dtype=torch.int32)
    for i, r in enumerate(rows):
        bt[i, :r.numel()] = r
    return bt


def make_decode(name: str, seed: int, seq_lens: List[int], num_q_heads: int, num_kv_heads: int, page_size: int,
                num_pages: Optional[int] = None, recipe: Optional[ValueRecipe] = None,
                shared_prefix_tokens: int = 0, extra_pages: int = 0) -> DecodeWorkload:
    recipe = recipe or ValueRecipe()
    counts = [max(1, -(-int(n) // page_size)) if n > 0 else 0 for n in seq_lens]
    shared = shared_prefix_tokens // page_size
    assert shared * page_size == shared_prefix_tokens
    need = shared + sum(max(0, c - shared) for c in counts)
    num_pages = num_pages or need + extra_pages
    gen = _gen(seed, 77, "cpu")
    bt = _place_pages(gen, num_pages, counts, shared)
    return DecodeWorkload(name, seed, len(seq_lens), num_q_heads, num_kv_heads, page_size, num_pages,
                          torch.tensor(seq_lens, dtype=torch.int32), bt, recipe, shared_prefix_tokens)


# ------------------------------------------------------------------ named workloads

def tiny_decode() -> DecodeWorkload:
    """Batch 2, lengths 256 and 300, 4 query heads on 1 KV head, pages of 16
    placed by a seeded permutation into a 64-page pool; 1% x20 outliers."""
    return make_decode("tiny-decode b2 lens256/300 q4kv1 p16", 1001, [256, 300], 4, 1, 16, num_pages=64,
                       recipe=ValueRecipe(outlier_p=0.01))


@dataclasses.dataclass
class AppendWorkload:
    """New tokens written through a random slot mapping."""

    name: str
    seed: int
    num_tokens: int
    num_kv_heads: int
    page_size: int
    num_pages: int
    recipe: ValueRecipe

    def kv(self, device):
        return (draw_kv(self.num_tokens, self.num_kv_heads, self.seed, 0, device, self.recipe, 0),
                draw_kv(self.num_tokens, self.num_kv_heads, self.seed, 0, device, self.recipe, 1))

    def slot_mapping(self) -> torch.Tensor:
        gen = _gen(self.seed, 78, "cpu")
        perm = torch.randperm(self.num_pages * self.page_size, generator=gen)
        return perm[:self.num_tokens].to(torch.int64)


def append_65k() -> AppendWorkload:
    """65,536 tokens x 8 KV heads, 64-token pages in a 2,048-page pool;
    1% x20 outliers and 0.1% all-zero 16-blocks."""
    return AppendWorkload("append t65536 kv8 p64", 1002, 65_536, 8, 64, 2_048,
                          ValueRecipe(outlier_p=0.01, zero_block_p=0.001))


def decode_32k() -> DecodeWorkload:
    """Batch 64 x 32,768 cached tokens, 64 query / 8 KV heads, pages of 64
    under a randomly permuted block table (the page's 32K iso-concurrency shape)."""
    return make_decode("decode b64 s32768 q64kv8 p64", 1003, [32_768] * 64, 64, 8, 64)


def decode_1m() -> DecodeWorkload:
    """Batch 2 x 1,048,576 cached tokens, 40 query / 8 KV heads, pages of 64,
    K and V scaled per (kv_head, channel) by exp(N(0,1))."""
    return make_decode("decode b2 s1048576 q40kv8 p64", 1004, [1_048_576] * 2, 40, 8, 64,
                       recipe=ValueRecipe(channel_lognormal=True))


def agent_lengths(n: int, seed: int, stream: int) -> List[int]:
    """Lognormal lengths around 16K (sigma 1), clipped to [2,048, 163,840],
    then raised to at least 3,201 so every sequence extends the shared prefix."""
    g = _gen(seed, stream, "cpu")
    z = torch.randn(n, generator=g, dtype=torch.float64)
    L = torch.exp(z + math.log(16_384)).round().clamp(2_048, 163_840).to(torch.int64)
    return [max(int(x), 3_201) for x in L]


@dataclasses.dataclass
class AgentMixWorkload:
    """128 decode sequences sharing one 3,200-token prefix (50 pages of 64),
    plus 8 extend requests whose cached prefixes share the same pages and
    that each bring a 512-token BF16 chunk."""

    decode: DecodeWorkload          # 128 decode sequences + 8 extend prefixes as one table
    num_decode: int
    extend_prefix_lens: List[int]
    chunk_tokens: int

    def extend_rows(self) -> List[int]:
        return list(range(self.num_decode, self.num_decode + len(self.extend_prefix_lens)))

    def chunk_kv(self, r: int, device):
        w = self.decode
        return (draw_kv(self.chunk_tokens, w.num_kv_heads, w.seed, 300_000 + r, device, w.recipe, 0),
                draw_kv(self.chunk_tokens, w.num_kv_heads, w.seed, 300_000 + r, device, w.recipe, 1))

    def chunk_q(self, r: int, device) -> torch.Tensor:
        """Queries of extend request r's chunk, BF16 [chunk_tokens][num_q_heads][128]."""
        w = self.decode
        return _normal((self.chunk_tokens, w.num_q_heads, HEAD_DIM), w.seed, 400_000 + r, device)

    def chunk_slots(self, r: int) -> torch.Tensor:
        """Slots of extend request r's chunk (positions prefix .. prefix+chunk)."""
        row = self.num_decode + r
        p = self.extend_prefix_lens[r]
        return self.decode.slots(row, p, p + self.chunk_tokens)


def agent_mix(num_decode: int = 128, num_extend: int = 8, chunk_tokens: int = 512) -> AgentMixWorkload:
    seed = 1005
    dec = agent_lengths(num_decode, seed, 11)
    ext = agent_lengths(num_extend, seed, 12)
    # Extend rows reserve pages for prefix + chunk; their seq_lens cover the prefix only.
    lens = dec + [p + chunk_tokens for p in ext]
    w = make_decode("agent-mix 128 seqs shared 3200 q32kv8 p64 + 8 extends of 512", seed, lens, 32, 8, 64,
                    shared_prefix_tokens=3_200)
    w.seq_lens[num_decode:] = torch.tensor(ext, dtype=torch.int32)
    return AgentMixWorkload(w, num_decode, ext, chunk_tokens)
