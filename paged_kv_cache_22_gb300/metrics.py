"""Byte accounting for the decode step's bandwidth metric (host-side only).

The KV size of one token is ``2 * layers * kv_heads * head_dim * elem_bytes``
(K and V), the formula of "Capítulo 2 — KV cache, jerarquía de memoria,
continuous batching y PagedAttention", section "Una fórmula útil para estimar
memoria", and of "KV cache: la memoria de trabajo que sostiene la inferencia
LLM", section "El precio: cuánto pesa la mochila".  The kernels here serve one
layer, so a step reads ``layers = 1`` worth of it per cached token.

Algorithmic bytes of one decode call (what the kernel must move at minimum)::

    sum_i L_i * 2 * Hkv * d * e_cache      K and V of every valid token
  + B * Hq * d * e_q                       q
  + B * Hq * d * e_q                       out
  + sum_i ceil(L_i / bs) * 4               block-table entries used
  + 4 * B                                  seq_lens

and of one cache write of T tokens::

    2 * T * Hkv * d * (e_src + e_cache) + 8 * T
"""
from __future__ import annotations

from typing import Iterable

ELEM_BYTES = {"f32": 4, "bf16": 2, "fp8_e4m3": 1}


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    return 2 * layers * kv_heads * head_dim * elem_bytes


def block_bytes(block_tokens: int, layers: int, kv_heads: int, head_dim: int,
                elem_bytes: int) -> int:
    return block_tokens * kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes)


def blocks_for_tokens(tokens: int, block_size: int) -> int:
    return -(-int(tokens) // int(block_size))


def attended_tokens(L: int, window: int = 0, sinks: int = 0) -> int:
    """Tokens a sequence of length L attends: all of them, or with a sliding
    window its first `sinks` and last `window` tokens."""
    if window <= 0 or L <= window:
        return L
    return min(sinks, L - window) + window


def blocks_read(L: int, block_size: int, window: int = 0, sinks: int = 0) -> int:
    """Blocks whose table entry and K/V a decode reads: every block, or with a
    window the blocks holding sink tokens and the window's blocks."""
    nb = blocks_for_tokens(L, block_size)
    if window <= 0 or L <= window:
        return nb
    ws = L - window
    nsb, wsb = blocks_for_tokens(min(sinks, ws), block_size), ws // block_size
    return nb - (wsb - nsb) if wsb > nsb else nb


def decode_bytes(seq_lens: Iterable[int], num_q_heads: int, num_kv_heads: int, head_dim: int,
                 cache_dtype: str, q_dtype: str, block_size: int, window: int = 0,
                 sinks: int = 0) -> int:
    lens = [int(x) for x in seq_lens]
    e_c, e_q = ELEM_BYTES[cache_dtype], ELEM_BYTES[q_dtype]
    kv = sum(attended_tokens(L, window, sinks) for L in lens) * kv_bytes_per_token(1, num_kv_heads, head_dim, e_c)
    qo = 2 * len(lens) * num_q_heads * head_dim * e_q
    tables = 4 * sum(blocks_read(L, block_size, window, sinks) for L in lens)
    return kv + qo + tables + 4 * len(lens)


def reshape_bytes(num_tokens: int, num_kv_heads: int, head_dim: int, src_dtype: str,
                  cache_dtype: str) -> int:
    per = num_kv_heads * head_dim * (ELEM_BYTES[src_dtype] + ELEM_BYTES[cache_dtype])
    return 2 * num_tokens * per + 8 * num_tokens


def unique_kv_bytes(seq_lens: Iterable[int], shared_prefix_tokens: int, num_kv_heads: int,
                    head_dim: int, cache_dtype: str) -> int:
    """KV bytes counting a prefix shared by every sequence once."""
    lens = [int(x) for x in seq_lens]
    per = kv_bytes_per_token(1, num_kv_heads, head_dim, ELEM_BYTES[cache_dtype])
    if not lens:
        return 0
    uniq = shared_prefix_tokens + sum(L - shared_prefix_tokens for L in lens)
    return uniq * per


def cascade_bytes(seq_lens: Iterable[int], prefix_tokens: int, num_q_heads: int, num_kv_heads: int,
                  head_dim: int, cache_dtype: str, q_dtype: str, block_size: int) -> int:
    """Algorithmic bytes of a decode call that reads a prefix shared by every
    sequence once: the prefix tokens any sequence attends, each sequence's
    tokens past the prefix, q, out, the table entries read (the prefix's
    once) and seq_lens.  The prefix partial result the cascade writes and
    reads back is traffic of the method, not counted here."""
    lens = [int(x) for x in seq_lens]
    if not lens:
        return 0
    e_c, e_q = ELEM_BYTES[cache_dtype], ELEM_BYTES[q_dtype]
    per = kv_bytes_per_token(1, num_kv_heads, head_dim, e_c)
    pre = min(prefix_tokens, max(lens))
    kv = (pre + sum(max(L - prefix_tokens, 0) for L in lens)) * per
    qo = 2 * len(lens) * num_q_heads * head_dim * e_q
    pb = blocks_for_tokens(prefix_tokens, block_size)
    tables = 4 * (blocks_for_tokens(pre, block_size)
                  + sum(max(blocks_for_tokens(L, block_size) - pb, 0) for L in lens))
    return kv + qo + tables + 4 * len(lens)


def multi_bytes(seq_lens: Iterable[int], q_lens: Iterable[int], num_q_heads: int, num_kv_heads: int,
                head_dim: int, cache_dtype: str, q_dtype: str, block_size: int) -> int:
    """Algorithmic bytes of one multi-token attention call: each sequence's K
    and V up to its last position once per kv head (the chunk's last token
    attends all of them), q and out of every query row, the table entries
    read, seq_lens and the query offsets."""
    lens = [int(x) for x in seq_lens]
    rows = sum(int(t) for t in q_lens)
    e_c, e_q = ELEM_BYTES[cache_dtype], ELEM_BYTES[q_dtype]
    kv = sum(lens) * kv_bytes_per_token(1, num_kv_heads, head_dim, e_c)
    qo = 2 * rows * num_q_heads * head_dim * e_q
    tables = 4 * sum(blocks_for_tokens(L, block_size) for L in lens)
    return kv + qo + tables + 4 * len(lens) + 4 * (len(lens) + 1)


def multi_flops(seq_lens: Iterable[int], q_lens: Iterable[int], num_q_heads: int, head_dim: int) -> int:
    """Multiply-add work of one multi-token attention call, 2 FLOP each: q.K
    and P.V over the positions every query row attends (query token i of a
    chunk of T attends L - T + i + 1 positions): 4 * d FLOP per (row, head,
    position)."""
    total = 0
    for L, T in zip(seq_lens, q_lens):
        L, T = int(L), int(T)
        attended = T * (L - T) + T * (T + 1) // 2  # sum over i of (L - T + i + 1)
        total += attended
    return 4 * head_dim * num_q_heads * total
