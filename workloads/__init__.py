"""Seeded synthetic decode workloads for paged KV caches.

This module only draws inputs: query vectors, per-token key/value vectors,
sequence lengths, a shuffled pool of physical block ids dealt into block
tables, and the slot of every token.  It holds none of the attention or
cache-conversion arithmetic, so both the CUDA path and the CPU oracle can
consume its output without sharing any of the method.

Layouts (all row-major):

* ``q``: ``[num_seqs, num_q_heads, head_dim]``
* ``block_tables``: ``int32 [num_seqs, max_blocks_per_seq]``; entries past a
  sequence's last block hold ``UNUSED_TABLE_ENTRY``, an id outside the pool,
  so that a reader that strays past the end is caught.
* token key/value vectors ``[T, num_kv_heads, head_dim]`` with their slots
  ``int64 [T]``, slot = block_id * block_size + offset: token position ``p``
  of sequence ``i`` lives in block ``block_tables[i][p // block_size]`` at
  offset ``p % block_size`` (the addressing of "PagedAttention por dentro",
  section "La tabla de páginas (block table)").

The history tokens (positions ``< seq_len - 1``) are written before the step;
the step's new token (position ``seq_len - 1``) is written by the step itself.

Named configurations follow the five decode workloads of the benchmark:
``tiny_mha``, ``llama3_8b``, ``llama70b_128``, ``long_split_kv`` and
``prefix_fp8``.  Seeds are ``1234 + index`` with the index in that order.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

UNUSED_TABLE_ENTRY = 0x7FFFFFFF

CACHE_DTYPES = ("f32", "bf16", "fp8_e4m3")
_TORCH_SRC = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    cache_dtype: str          # "f32" | "bf16" | "fp8_e4m3"
    q_dtype: str              # "f32" | "bf16" (also the output dtype)
    src_dtype: str            # dtype of the key/value vectors written to the cache
    q: torch.Tensor
    seq_lens: torch.Tensor    # int32 [B]
    block_tables: torch.Tensor  # int32 [B, max_blocks_per_seq]
    hist_k: torch.Tensor      # [T_hist, Hkv, d]
    hist_v: torch.Tensor
    hist_slots: torch.Tensor  # int64 [T_hist]
    new_k: torch.Tensor       # [T_new, Hkv, d] (one token per non-empty sequence)
    new_v: torch.Tensor
    new_slots: torch.Tensor   # int64 [T_new]
    scale: float
    kv_scale: float = 1.0
    partition_tokens: int = 0
    shared_prefix_blocks: int = 0
    notes: dict = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.num_seqs else 0

    @property
    def gqa_group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def all_tokens(self):
        """History and new tokens together: (k, v, slots)."""
        return (torch.cat([self.hist_k, self.new_k]), torch.cat([self.hist_v, self.new_v]),
                torch.cat([self.hist_slots, self.new_slots]))


def _normal(gen: torch.Generator, shape, dtype: torch.dtype) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(dtype)


def make_workload(name: str, seq_lens: Sequence[int], num_q_heads: int, num_kv_heads: int,
                  head_dim: int, block_size: int = 16, cache_dtype: str = "bf16",
                  seed: int = 0, num_blocks: Optional[int] = None, pool_slack: float = 1.0,
                  prefix_tokens: int = 0, max_blocks_per_seq: Optional[int] = None,
                  partition_tokens: int = 0, kv_scale: Optional[float] = None,
                  identity_tables: bool = False) -> Workload:
    """Draw one decode workload.

    ``prefix_tokens`` (a multiple of ``block_size``) makes every sequence's
    first ``prefix_tokens // block_size`` table entries point at the same
    physical blocks, whose tokens are drawn once.  ``identity_tables`` deals
    block ids in order instead of shuffling the pool (the contiguous control).
    For an fp8 cache with ``kv_scale=None`` the scale is the largest key/value
    magnitude divided by 448, the largest finite e4m3 value.
    """
    if cache_dtype not in CACHE_DTYPES:
        raise ValueError(cache_dtype)
    if num_q_heads % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    if prefix_tokens % block_size:
        raise ValueError("prefix_tokens must be a multiple of block_size")
    gen = torch.Generator().manual_seed(seed)
    lens = [int(x) for x in seq_lens]
    B = len(lens)
    q_dtype = "f32" if cache_dtype == "f32" else "bf16"
    src_dtype = q_dtype
    tdt = _TORCH_SRC[src_dtype]

    nb = [(L + block_size - 1) // block_size for L in lens]
    pblocks = prefix_tokens // block_size
    for L in lens:
        if prefix_tokens and L <= prefix_tokens:
            raise ValueError("with a shared prefix every sequence must extend past it")
    unique_blocks = pblocks + sum(n - pblocks for n in nb) if prefix_tokens else sum(nb)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(unique_blocks * pool_slack))
    if num_blocks < unique_blocks:
        raise ValueError("pool too small")
    mb = max(1, max(nb) if nb else 1)
    if max_blocks_per_seq is not None:
        if max_blocks_per_seq < mb:
            raise ValueError("max_blocks_per_seq too small")
        mb = max_blocks_per_seq

    # the placement has its own stream so that token values do not depend on it
    perm_gen = torch.Generator().manual_seed(seed + 7919)
    perm = (torch.arange(num_blocks, dtype=torch.int64) if identity_tables
            else torch.randperm(num_blocks, generator=perm_gen))
    tables = torch.full((B, mb), UNUSED_TABLE_ENTRY, dtype=torch.int32)
    cursor = 0
    prefix_ids = perm[:pblocks]
    cursor = pblocks
    for i, n in enumerate(nb):
        if pblocks:
            tables[i, :pblocks] = prefix_ids.to(torch.int32)
        own = n - pblocks if pblocks else n
        tables[i, (pblocks if pblocks else 0):n] = perm[cursor:cursor + own].to(torch.int32)
        cursor += own

    q = _normal(gen, (B, num_q_heads, head_dim), tdt)

    # Token positions whose vectors are drawn: the shared prefix once (owned by
    # sequence 0), then every sequence's own history, then the new tokens.
    hist_pos = []  # (sequence, position)
    for i, L in enumerate(lens):
        start = prefix_tokens if (pblocks and i > 0) else 0
        for p in range(start, max(L - 1, 0)):
            hist_pos.append((i, p))
    new_pos = [(i, L - 1) for i, L in enumerate(lens) if L >= 1]

    def slots_for(pos):
        if not pos:
            return torch.zeros(0, dtype=torch.int64)
        seq = torch.tensor([i for i, _ in pos], dtype=torch.int64)
        p = torch.tensor([pp for _, pp in pos], dtype=torch.int64)
        blk = tables.to(torch.int64)[seq, p // block_size]
        return blk * block_size + p % block_size

    hist_slots = slots_for(hist_pos)
    new_slots = slots_for(new_pos)
    hist_k = _normal(gen, (len(hist_pos), num_kv_heads, head_dim), tdt)
    hist_v = _normal(gen, (len(hist_pos), num_kv_heads, head_dim), tdt)
    new_k = _normal(gen, (len(new_pos), num_kv_heads, head_dim), tdt)
    new_v = _normal(gen, (len(new_pos), num_kv_heads, head_dim), tdt)

    if cache_dtype == "fp8_e4m3" and kv_scale is None:
        amax = max(float(t.abs().max()) if t.numel() else 0.0
                   for t in (hist_k, hist_v, new_k, new_v))
        kv_scale = (amax if amax > 0 else 1.0) / 448.0
    if kv_scale is None:
        kv_scale = 1.0

    return Workload(
        name=name, num_seqs=B, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=block_size, num_blocks=num_blocks,
        cache_dtype=cache_dtype, q_dtype=q_dtype, src_dtype=src_dtype, q=q,
        seq_lens=torch.tensor(lens, dtype=torch.int32), block_tables=tables,
        hist_k=hist_k, hist_v=hist_v, hist_slots=hist_slots, new_k=new_k, new_v=new_v,
        new_slots=new_slots, scale=1.0 / math.sqrt(head_dim), kv_scale=float(kv_scale),
        partition_tokens=partition_tokens, shared_prefix_blocks=pblocks,
        notes={"seed": seed, "unique_blocks": unique_blocks})


# ------------------------------------------------------------------ named configs
def tiny_mha(seed: int = 1234) -> Workload:
    """4 sequences of 1, 17, 33 and 100 tokens, 4 q heads = 4 kv heads,
    head_dim 64, fp32, block_size 16, a 64-block shuffled pool."""
    return make_workload("tiny_mha", [1, 17, 33, 100], 4, 4, 64, 16, "f32", seed=seed,
                         num_blocks=64)


def llama3_8b(seed: int = 1235, num_seqs: int = 64, block_size: int = 16,
              identity_tables: bool = False) -> Workload:
    """Llama-3-8B-shaped decode layer: 32 q / 8 kv heads, head_dim 128, bf16,
    seq_lens uniform in [128, 2048], 16384-block shuffled pool.  Other block
    sizes keep the pool's token capacity (262,144 tokens); identity tables
    deal the pool in order (the contiguous control)."""
    gen = torch.Generator().manual_seed(seed + 100_000)
    lens = torch.randint(128, 2049, (num_seqs,), generator=gen).tolist()
    return make_workload("llama3_8b", lens, 32, 8, 128, block_size, "bf16", seed=seed,
                         num_blocks=16384 * 16 // block_size, identity_tables=identity_tables)


def llama70b_128(seed: int = 1236, num_seqs: int = 128, sigma: float = 1.0) -> Workload:
    """Llama-70B-shaped decode layer at 128 requests: 64 q / 8 kv heads,
    head_dim 128, bf16, seq_lens log-normal with median 800 (sigma 1.0)
    clipped to [16, 8192], pool 1.1x the blocks needed, shuffled."""
    gen = torch.Generator().manual_seed(seed + 100_000)
    z = torch.randn(num_seqs, generator=gen, dtype=torch.float64)
    lens = torch.exp(math.log(800.0) + sigma * z).round().clamp(16, 8192).to(torch.int64).tolist()
    return make_workload("llama70b_128", lens, 64, 8, 128, 16, "bf16", seed=seed, pool_slack=1.1)


def long_split_kv(seed: int = 1237, num_seqs: int = 8, seq_len: int = 32768) -> Workload:
    """Long-context split-KV: 8 sequences of 32768 tokens, 32 q / 8 kv heads,
    head_dim 128, bf16, exactly the needed 16384 blocks shuffled, KV
    partitions of 512 tokens."""
    return make_workload("long_split_kv", [seq_len] * num_seqs, 32, 8, 128, 16, "bf16",
                         seed=seed, partition_tokens=512)


def prefix_fp8(seed: int = 1238, num_seqs: int = 256, prefix_tokens: int = 2048) -> Workload:
    """Prefix sharing with an fp8-e4m3 cache: 256 sequences whose tables all
    start with the same 2048-token prefix blocks, then unique suffixes of
    uniform 1..512 tokens; 32 q / 8 kv heads, head_dim 128, per-tensor scale."""
    gen = torch.Generator().manual_seed(seed + 100_000)
    suffix = torch.randint(1, 513, (num_seqs,), generator=gen).tolist()
    lens = [prefix_tokens + s for s in suffix]
    return make_workload("prefix_fp8", lens, 32, 8, 128, 16, "fp8_e4m3", seed=seed,
                         prefix_tokens=prefix_tokens)


CONFIGS = {
    "tiny_mha": tiny_mha,
    "llama3_8b": llama3_8b,
    "llama70b_128": llama70b_128,
    "long_split_kv": long_split_kv,
    "prefix_fp8": prefix_fp8,
}


def chunk_queries(w: Workload, q_lens: Sequence[int], seed: int = 0):
    """Query rows for several query tokens per sequence (a prefill chunk, or
    the tokens a speculative step verifies): sequence s gets ``q_lens[s]``
    rows, ``1 <= q_lens[s] <= seq_lens[s]`` (0 allowed), seeded N(0, 1) in the
    workload's query dtype.  Returns ``(q [total, Hq, d], q_start int32
    [B + 1])``: sequence s owns rows ``q_start[s] .. q_start[s+1]-1``, its last
    ``q_lens[s]`` positions (the cache already holds their K and V)."""
    lens = w.seq_lens.tolist()
    if len(q_lens) != len(lens):
        raise ValueError("one query count per sequence")
    for T, L in zip(q_lens, lens):
        if T < 0 or T > L:
            raise ValueError("0 <= q_lens[s] <= seq_lens[s]")
    gen = torch.Generator().manual_seed(seed)
    total = int(sum(q_lens))
    q = _normal(gen, (total, w.num_q_heads, w.head_dim), _TORCH_SRC[w.q_dtype])
    q_start = torch.zeros(len(lens) + 1, dtype=torch.int32)
    q_start[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
    return q, q_start


# ------------------------------------------------------------------ multi-token configs
def verify4_llama3_8b(seed: int = 1301):
    """Speculative verification on the Llama-3-8B-shaped batch: 64
    sequences, L ~ U[128, 2048], the last 4 positions of each are query
    tokens (3 drafted + 1)."""
    w = llama3_8b(seed=seed)
    q, q_start = chunk_queries(w, [4] * w.num_seqs, seed=seed + 1)
    return w, q, q_start


def prefill_chunk512(seed: int = 1302, num_seqs: int = 8):
    """Chunked prefill at the default chunk size: 8 sequences of Llama-3-8B
    heads whose next 512-token chunk lands at L ~ U[1024, 4096] (the chunk is
    the last 512 positions, already in the cache)."""
    gen = torch.Generator().manual_seed(seed)
    lens = torch.randint(1024, 4097, (num_seqs,), generator=gen).tolist()
    w = make_workload("prefill_chunk512", lens, 32, 8, 128, 16, "bf16", seed=seed)
    q, q_start = chunk_queries(w, [512] * num_seqs, seed=seed + 1)
    return w, q, q_start


MULTI_CONFIGS = {
    "verify4_llama3_8b": verify4_llama3_8b,
    "prefill_chunk512": prefill_chunk512,
}


def poison_bits(cache_dtype: str) -> int:
    """Byte pattern that fills a fresh cache: a NaN in every float type, so a
    reader of a never-written slot poisons its result."""
    return {"f32": 0xFF, "bf16": 0xFF, "fp8_e4m3": 0xFF}[cache_dtype]


def cache_shape(w: Workload):
    return (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)


def cache_torch_dtype(cache_dtype: str) -> torch.dtype:
    """Storage dtype of a cache: fp32 as float32, bf16 as bfloat16, fp8 codes
    as uint8."""
    return {"f32": torch.float32, "bf16": torch.bfloat16, "fp8_e4m3": torch.uint8}[cache_dtype]
