"""Seeded synthetic inputs for fp8 paged decode attention.

This module is shared by both sides of every parity check: the CUDA path and
the fp64 oracle read the same tensors made here. It holds no attention
arithmetic: it draws random numbers, quantises them to the cache's storage
type with PyTorch's own cast, and lays them out in the paged cache format.

Shapes of the pages' kernel-latency table (vLLM pull request
lishuoshuo-amd/vllm#3, section "Kernel latency, accuracy runs and kernel
error": 40/8 and 32/8 heads, head size 128, contexts 1024 and 4096, 16 to 256
sequences, fp8 cache, 16-token blocks) plus a ragged-length batch and a GQA-8,
64-token-block batch.

Recipe (the same for every config, all draws from one ``torch.Generator``
seeded with ``seed`` on the chosen device, in this order):

1. ragged configs only: ``seq_lens`` ~ U{lo..hi} inclusive;
2. ``q``: N(0, 1) in fp32, rounded to bf16, shape ``[S, H, D]``;
3. K then V: N(0, 1) in fp32, rounded to bf16, divided by the per-tensor
   scale in fp32, clamped to +-448 and cast to ``float8_e4m3fn``
   (round-to-nearest-even), drawn in storage order of
   ``[NB, Hk, D/16, bs, 16]`` (K) and ``[NB, Hk, D, bs]`` (V);
4. a random permutation of the ``NB`` physical blocks; sequence s takes the
   next ``ceil(L_s / bs)`` entries of it as its pages, in order. Table
   entries past a sequence's last page hold 0. The pool holds
   ``ceil(pool_factor * sum_s ceil(L_s / bs))`` blocks; blocks no sequence
   uses keep their random contents.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

FP8 = torch.float8_e4m3fn
FP8_MAX = 448.0


@dataclass(frozen=True)
class Config:
    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_size: int = 128
    block_size: int = 16
    ctx: int | None = None
    ctx_range: tuple[int, int] | None = None
    pool_factor: float = 1.0
    k_scale: float = 0.05
    v_scale: float = 0.05
    seed: int = 0

    @property
    def gqa(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def max_ctx(self) -> int:
        return self.ctx if self.ctx is not None else self.ctx_range[1]

    @property
    def max_num_blocks_per_seq(self) -> int:
        return max(1, math.ceil(self.max_ctx / self.block_size))

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_size)

    def with_(self, **kw) -> "Config":
        d = dict(self.__dict__)
        d.update(kw)
        return Config(**d)


# The five benchmark-shaped batches. The first is the small case the oracle
# finishes in seconds; the third (256 sequences at 4096 tokens) is the
# headline throughput workload.
CONFIGS: dict[str, Config] = {
    c.name: c
    for c in [
        Config("32q8kv-16seq-ctx1024-bs16", 16, 32, 8, ctx=1024, pool_factor=1.0),
        Config("40q8kv-64seq-ctx1024-bs16", 64, 40, 8, ctx=1024, pool_factor=1.25),
        Config("32q8kv-256seq-ctx4096-bs16", 256, 32, 8, ctx=4096, pool_factor=1.0),
        Config("40q8kv-256seq-ctx1to4000-bs16", 256, 40, 8, ctx_range=(1, 4000), pool_factor=1.0),
        Config("64q8kv-128seq-ctx8192-bs64", 128, 64, 8, block_size=64, ctx=8192, pool_factor=2.0),
    ]
}
SMALL = "32q8kv-16seq-ctx1024-bs16"
HEADLINE = "32q8kv-256seq-ctx4096-bs16"


@dataclass
class Batch:
    cfg: Config
    q: torch.Tensor              # bf16 [S, H, D]
    k_cache: torch.Tensor        # float8_e4m3fn [NB, Hk, D/16, bs, 16]
    v_cache: torch.Tensor        # float8_e4m3fn [NB, Hk, D, bs]
    block_tables: torch.Tensor   # int32 [S, MB]
    seq_lens: torch.Tensor       # int32 [S]
    seq_lens_host: list[int] = field(default_factory=list)

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    def to(self, device) -> "Batch":
        return Batch(self.cfg, self.q.to(device), self.k_cache.to(device), self.v_cache.to(device),
                     self.block_tables.to(device), self.seq_lens.to(device), list(self.seq_lens_host))

    def raw(self) -> dict:
        """Host numpy views of the raw bit patterns (the oracle's input form)."""
        return dict(
            q=self.q.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16),
            k_cache=self.k_cache.detach().cpu().contiguous().view(torch.uint8).numpy(),
            v_cache=self.v_cache.detach().cpu().contiguous().view(torch.uint8).numpy(),
            block_tables=self.block_tables.detach().cpu().contiguous().numpy(),
            seq_lens=self.seq_lens.detach().cpu().contiguous().numpy(),
        )

    def pages_used(self) -> int:
        bs = self.cfg.block_size
        return sum((L + bs - 1) // bs for L in self.seq_lens_host)


def quantized_normal(shape, scale: float, gen: torch.Generator, device, chunk: int = 1 << 26) -> torch.Tensor:
    """N(0,1) -> bf16 -> /scale (fp32) -> clamp +-448 -> e4m3 (torch cast, RNE)."""
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=FP8, device=device)
    for off in range(0, n, chunk):
        m = min(chunk, n - off)
        x = torch.randn(m, generator=gen, device=device, dtype=torch.float32)
        x = x.to(torch.bfloat16).to(torch.float32) / scale
        out[off:off + m] = x.clamp_(-FP8_MAX, FP8_MAX).to(FP8)
    return out.view(shape)


def make_batch(cfg: Config, device="cpu", seed: int | None = None) -> Batch:
    device = torch.device(device)
    seed = cfg.seed if seed is None else seed
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    S, H, Hk, D, bs = cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.head_size, cfg.block_size
    if H % Hk or D % 16 or bs % 16:
        raise ValueError("config outside the cache format: %s" % (cfg,))
    if cfg.ctx_range is not None:
        lo, hi = cfg.ctx_range
        lens = torch.randint(lo, hi + 1, (S,), generator=gen, device=device, dtype=torch.int64)
        lens_host = [int(x) for x in lens.cpu().tolist()]
    else:
        lens_host = [int(cfg.ctx)] * S
    pages = [(L + bs - 1) // bs for L in lens_host]
    needed = sum(pages)
    NB = max(1, math.ceil(cfg.pool_factor * needed))
    MB = cfg.max_num_blocks_per_seq

    q = torch.randn(S, H, D, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    k_cache = quantized_normal((NB, Hk, D // 16, bs, 16), cfg.k_scale, gen, device)
    v_cache = quantized_normal((NB, Hk, D, bs), cfg.v_scale, gen, device)
    perm = torch.randperm(NB, generator=gen, device=device).to(torch.int32).cpu()

    tables = _fill_tables(S, MB, pages, perm)
    seq_lens = torch.tensor(lens_host, dtype=torch.int32)
    return Batch(cfg, q, k_cache, v_cache, tables.to(device), seq_lens.to(device), lens_host)


def _fill_tables(S: int, MB: int, pages, perm: torch.Tensor) -> torch.Tensor:
    """Block table [S, MB] int32: sequence s takes the next pages[s] entries of
    perm (a permutation of the pool), in order; the rest of its row is 0."""
    tables = torch.zeros(S, MB, dtype=torch.int32)
    counts = torch.tensor(pages, dtype=torch.int64)
    total = int(counts.sum())
    if total:
        rows = torch.repeat_interleave(torch.arange(S), counts)
        starts = torch.cumsum(counts, 0) - counts
        cols = torch.arange(total) - torch.repeat_interleave(starts, counts)
        tables[rows, cols] = perm[:total]
    return tables


def make_custom(num_seqs, num_heads, num_kv_heads, seq_lens, *, block_size=16, head_size=128,
                pool_factor=1.0, k_scale=0.05, v_scale=0.05, seed=0, device="cpu",
                max_num_blocks_per_seq=None) -> Batch:
    """A batch with explicit per-sequence lengths (edge cases, ragged tails)."""
    lens_host = [int(x) for x in seq_lens]
    assert len(lens_host) == num_seqs
    cfg = Config("custom", num_seqs, num_heads, num_kv_heads, head_size=head_size, block_size=block_size,
                 ctx=max(lens_host + [1]), pool_factor=pool_factor, k_scale=k_scale, v_scale=v_scale, seed=seed)
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    S, H, Hk, D, bs = num_seqs, num_heads, num_kv_heads, head_size, block_size
    pages = [(L + bs - 1) // bs for L in lens_host]
    needed = sum(pages)
    NB = max(1, math.ceil(pool_factor * needed))
    MB = max_num_blocks_per_seq or max(1, max(pages + [1]))
    if MB != cfg.max_num_blocks_per_seq:
        cfg = cfg.with_(ctx=MB * bs)
    q = torch.randn(S, H, D, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    k_cache = quantized_normal((NB, Hk, D // 16, bs, 16), k_scale, gen, device)
    v_cache = quantized_normal((NB, Hk, D, bs), v_scale, gen, device)
    perm = torch.randperm(NB, generator=gen, device=device).to(torch.int32).cpu()
    tables = _fill_tables(S, MB, pages, perm)
    seq_lens_t = torch.tensor(lens_host, dtype=torch.int32)
    return Batch(cfg, q, k_cache, v_cache, tables.to(device), seq_lens_t.to(device), lens_host)


def algorithmic_bytes(cfg: Config, seq_lens_host) -> int:
    """Bytes one decode call must move at minimum.

    K and V pages touched (whole 16-token-multiple pages, each byte once for
    all query heads of its group), q in, out written (both bf16), the block
    table rows and seq_lens.
    """
    bs, D, Hk = cfg.block_size, cfg.head_size, cfg.num_kv_heads
    pages = sum((int(L) + bs - 1) // bs for L in seq_lens_host)
    kv = pages * bs * D * Hk * 2
    qo = 2 * cfg.num_seqs * cfg.num_heads * D * 2
    tables = cfg.num_seqs * cfg.max_num_blocks_per_seq * 4 + cfg.num_seqs * 4
    return kv + qo + tables
