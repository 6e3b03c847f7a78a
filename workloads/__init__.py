"""Seeded synthetic inputs for paged-attention decode.

This module is shared by the oracle tests and the CUDA-path tests/benchmark.
It only draws inputs (queries, paged K/V caches, block tables, sequence
lengths); it holds none of the attention arithmetic.

The workloads stand in for the ones the pages describe: single-sequence
decode up to 100K tokens with block_size 16 and grouped-query attention
("vllm/_custom_ops.py" commit 900ae0b, section 1; "paged_attention_v2_pytorch.py"
commit 15ef28e, "Before": 6250 blocks of 16 tokens for 100K).  There is no
dataset: every value is drawn from a seeded generator.

Recipe (all configs): values are drawn in fp32 from N(0, 1) and cast to the
storage dtype with round-to-nearest-even; the block pool is ``pool_factor``
times the blocks in use (or a fixed size); each sequence's blocks are
distinct pool slots taken from one seeded permutation, so blocks are
scattered at random; block-table slots past a sequence's last block hold -1.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

F16 = 0
BF16 = 1
TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16}
DTYPE_NAME = {F16: "f16", BF16: "bf16"}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    partition_size: int
    dtype: int
    seq_len_kind: str              # "fixed" | "uniform" | "lognormal" | "list"
    seq_len: int = 0               # fixed length / upper bound / clip max
    seq_len_min: int = 1
    lognormal_median: float = 0.0
    lognormal_sigma: float = 0.0
    seq_lens: tuple = ()           # for kind == "list"
    pool_factor: float = 1.25      # pool = ceil(pool_factor * used blocks) ...
    pool_blocks: int = 0           # ... unless a fixed pool size is given
    outlier_frac: float = 0.0      # fraction of K channels scaled by outlier_scale
    outlier_scale: float = 1.0
    q_len: int = 1                 # new tokens per sequence (query [S, q_len, H, D] when > 1)
    seed: int = 20261202

    @property
    def group_size(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads the build is measured on.
TINY = Workload("tiny", 1, 8, 2, 128, 16, 512, F16, "fixed", seq_len=1000, pool_blocks=128,
                seed=20261202)
BATCH = Workload("batch_decode", 32, 32, 8, 128, 16, 512, BF16, "uniform", seq_len=8192,
                 seq_len_min=1, seed=20261203)
LONG = Workload("long_100k", 1, 32, 4, 128, 16, 512, BF16, "fixed", seq_len=100000,
                seed=20261204)
LONG_1024 = LONG.with_(name="long_100k_p1024", partition_size=1024)
RAGGED = Workload("ragged_serving", 64, 64, 8, 128, 32, 512, BF16, "lognormal", seq_len=32768,
                  seq_len_min=16, lognormal_median=2048.0, lognormal_sigma=1.0,
                  outlier_frac=0.05, outlier_scale=8.0, seed=20261205)
STRESS = Workload("stress", 8, 64, 8, 128, 16, 1024, F16, "fixed", seq_len=131072,
                  pool_blocks=70000, seed=20261206)

# Batch decode checking 4 speculated tokens per sequence (several new tokens per call).
BATCH_SPEC4 = BATCH.with_(name="batch_decode_spec4", q_len=4)

# Batch decode checking 16 speculated tokens per sequence: 64 query rows per KV head.
SPEC_VERIFY16 = BATCH.with_(name="spec_verify_16", q_len=16)
# Chunked prefill: 2 sequences, each adding a 2048-token chunk (already written
# to the cache) after a 30,720-token prefix; 32 query / 8 KV heads.
CHUNKED_PREFILL = Workload("chunked_prefill", 2, 32, 8, 128, 16, 512, BF16, "fixed",
                           seq_len=32768, q_len=2048, seed=20261207)
# The same step with fp16 storage (run by the two-query-tile kernel).
CHUNKED_PREFILL_F16 = CHUNKED_PREFILL.with_(name="chunked_prefill_f16", dtype=F16)

# Batch decode with one query head per KV head (G = 1, 8 / 8 heads): the same
# K/V bytes as batch_decode, one eighth of an MMA n-tile of query rows.
BATCH_G1 = BATCH.with_(name="batch_decode_g1", num_heads=8)

# The stress shape at 2 of its 8 sequences, its pool cut to match (1.07 GB of
# K/V, still well above L2): the case ncu captures in several passes, which
# keeps a capture's device footprint small.
STRESS_2SEQ = STRESS.with_(name="stress_2seq", num_seqs=2, pool_blocks=17500)

ALL = {w.name: w for w in (TINY, BATCH, BATCH_G1, LONG, LONG_1024, RAGGED, STRESS, STRESS_2SEQ, BATCH_SPEC4,
                           SPEC_VERIFY16, CHUNKED_PREFILL, CHUNKED_PREFILL_F16)}


def draw_seq_lens(w: Workload) -> list:
    g = torch.Generator().manual_seed(w.seed * 7 + 1)
    if w.seq_len_kind == "fixed":
        return [w.seq_len] * w.num_seqs
    if w.seq_len_kind == "list":
        return [int(x) for x in w.seq_lens]
    if w.seq_len_kind == "uniform":
        return torch.randint(w.seq_len_min, w.seq_len + 1, (w.num_seqs,), generator=g).tolist()
    if w.seq_len_kind == "lognormal":
        z = torch.randn(w.num_seqs, generator=g, dtype=torch.float64)
        x = torch.exp(math.log(w.lognormal_median) + w.lognormal_sigma * z)
        x = torch.round(x).clamp(w.seq_len_min, w.seq_len)
        return [int(v) for v in x.tolist()]
    raise ValueError(w.seq_len_kind)


def blocks_for(seq_len: int, block_size: int) -> int:
    return -(-seq_len // block_size)


@dataclasses.dataclass
class Inputs:
    workload: Workload
    query: torch.Tensor          # [S, H, D] (or [S, Q, H, D] for q_len Q > 1) dtype
    key_cache: torch.Tensor      # [num_blocks, KV, bs, D] dtype
    value_cache: torch.Tensor    # [num_blocks, KV, bs, D] dtype
    block_tables: torch.Tensor   # [S, max_blocks] int32 (-1 padding)
    seq_lens: torch.Tensor       # [S] int32
    outlier_channels: list

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.seq_lens.numel() else 0

    @property
    def kv_bytes(self) -> int:
        """K and V bytes the decode must read: sum_b L_b * KV * D * 2 * elem."""
        w = self.workload
        return int(self.seq_lens.sum().item()) * w.num_kv_heads * w.head_dim * 2 * 2

    def to(self, device) -> "Inputs":
        return dataclasses.replace(
            self, query=self.query.to(device), key_cache=self.key_cache.to(device),
            value_cache=self.value_cache.to(device), block_tables=self.block_tables.to(device),
            seq_lens=self.seq_lens.to(device))


def _randn(shape, gen, device, dtype):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def make_inputs(w: Workload, device="cpu", seq_lens: Optional[Sequence[int]] = None,
                max_blocks: Optional[int] = None) -> Inputs:
    """Draw the inputs of workload ``w`` on ``device`` (torch's seeded generator there).

    ``seq_lens`` overrides the drawn lengths; ``max_blocks`` widens the table.
    """
    device = torch.device(device)
    lens = list(seq_lens) if seq_lens is not None else draw_seq_lens(w)
    S = len(lens)
    bs = w.block_size
    used = [blocks_for(L, bs) for L in lens]
    width = max(max(used) if used else 1, 1)
    if max_blocks is not None:
        width = max(width, int(max_blocks))
    if w.seq_len_kind in ("uniform", "lognormal", "fixed") and seq_lens is None:
        width = max(width, blocks_for(w.seq_len, bs))
    total_used = sum(used)
    pool = w.pool_blocks if w.pool_blocks else max(1, math.ceil(w.pool_factor * total_used))
    if pool < total_used:
        raise ValueError(f"pool of {pool} blocks is smaller than the {total_used} blocks in use")

    gcpu = torch.Generator().manual_seed(w.seed)
    perm = torch.randperm(pool, generator=gcpu).to(torch.int32)
    table = torch.full((S, width), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(used):
        table[b, :n] = perm[pos:pos + n]
        pos += n

    outliers = []
    if w.outlier_frac > 0:
        n_out = int(round(w.outlier_frac * w.head_dim))
        outliers = sorted(torch.randperm(w.head_dim, generator=gcpu)[:n_out].tolist())

    gdev = torch.Generator(device=device).manual_seed(w.seed + 1)
    dt = TORCH_DTYPE[w.dtype]
    H, KV, D = w.num_heads, w.num_kv_heads, w.head_dim
    query = _randn((S, H, D) if w.q_len == 1 else (S, w.q_len, H, D), gdev, device, dt)
    if outliers:
        k32 = torch.randn((pool, KV, bs, D), generator=gdev, device=device, dtype=torch.float32)
        idx = torch.tensor(outliers, device=device)
        k32[..., idx] *= w.outlier_scale
        key_cache = k32.to(dt)
        del k32
    else:
        key_cache = _randn((pool, KV, bs, D), gdev, device, dt)
    value_cache = _randn((pool, KV, bs, D), gdev, device, dt)
    return Inputs(w, query, key_cache, value_cache, table.to(device),
                  torch.tensor(lens, dtype=torch.int32).to(device), outliers)


def poison_unreferenced(inp: Inputs, value: float) -> None:
    """Fill every cache slot the decode must never read with ``value`` (in place).

    That is: pool blocks no sequence references, and the rows past seq_len in
    each sequence's last block.  Used to show that masked slots are never read
    into the result.
    """
    w = inp.workload
    bs = w.block_size
    tables = inp.block_tables.cpu()
    lens = inp.seq_lens.cpu().tolist()
    referenced = torch.zeros(inp.key_cache.shape[0], dtype=torch.bool)
    for b, L in enumerate(lens):
        n = blocks_for(L, bs)
        if n:
            referenced[tables[b, :n].long()] = True
    dev = inp.key_cache.device
    unref = (~referenced).nonzero().flatten().to(dev)
    for cache in (inp.key_cache, inp.value_cache):
        cache[unref] = value
        for b, L in enumerate(lens):
            n = blocks_for(L, bs)
            if n and L % bs:
                cache[int(tables[b, n - 1]), :, L % bs:, :] = value


def relabel_blocks(inp: Inputs, seed: int) -> Inputs:
    """Same logical sequences, physical blocks moved to new pool slots.

    new_cache[perm[i]] = old_cache[i] and new_table = perm[old_table], so
    every sequence reads the same K/V rows from different physical ids.
    """
    pool = inp.key_cache.shape[0]
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(pool, generator=g)
    dev = inp.key_cache.device
    permd = perm.to(dev)
    kc = torch.empty_like(inp.key_cache)
    vc = torch.empty_like(inp.value_cache)
    kc[permd] = inp.key_cache
    vc[permd] = inp.value_cache
    tab = inp.block_tables.cpu().long()
    new_tab = torch.where(tab >= 0, perm[tab.clamp(min=0)], tab).to(torch.int32)
    return dataclasses.replace(inp, key_cache=kc, value_cache=vc, block_tables=new_tab.to(dev))


def to_oracle_arrays(inp: Inputs):
    """CPU numpy views for the oracle: raw uint16 patterns and int32 tables."""
    import numpy as np

    def u16(t):
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    return dict(query=u16(inp.query), key_cache=u16(inp.key_cache),
                value_cache=u16(inp.value_cache),
                block_tables=inp.block_tables.cpu().numpy().astype(np.int32),
                seq_lens=inp.seq_lens.cpu().numpy().astype(np.int32),
                scale=inp.workload.scale, dtype=inp.workload.dtype)
