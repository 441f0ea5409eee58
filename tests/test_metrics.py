"""Byte and FLOP accounting behind the benchmark's numbers, checked against
brute-force counts over every (row, head, position) and block, and the
seeded query generator's contract (host only)."""
from __future__ import annotations

import pytest
import torch

import workloads
from paged_kv_cache_22_gb300 import metrics


def _brute_multi(lens, q_lens, Hq, Hkv, d, e_c, e_q, bs):
    kv = sum(L * 2 * Hkv * d * e_c for L in lens)  # every position once per kv head
    rows = sum(q_lens)
    qo = 2 * rows * Hq * d * e_q
    tables = 4 * sum(-(-L // bs) for L in lens)
    flops = 0
    for L, T in zip(lens, q_lens):
        for i in range(T):
            for _ in range(Hq):
                flops += (L - T + i + 1) * 4 * d  # q.K and P.V, 2 FLOP per multiply-add
    return kv + qo + tables + 4 * len(lens) + 4 * (len(lens) + 1), flops


@pytest.mark.parametrize("lens,q_lens", [([10, 1, 300], [3, 1, 17]), ([64], [64]), ([5, 7], [0, 7])])
def test_multi_bytes_and_flops_match_brute_force(lens, q_lens):
    b, f = _brute_multi(lens, q_lens, 8, 2, 64, 2, 2, 16)
    assert metrics.multi_bytes(lens, q_lens, 8, 2, 64, "bf16", "bf16", 16) == b
    assert metrics.multi_flops(lens, q_lens, 8, 64) == f


def test_multi_with_one_token_is_decode_bytes():
    """T = 1 everywhere: the multi-token count is decode's plus the offsets
    array (B + 1 int32)."""
    lens = [5, 40, 1000]
    dec = metrics.decode_bytes(lens, 32, 8, 128, "bf16", "bf16", 16)
    assert metrics.multi_bytes(lens, [1, 1, 1], 32, 8, 128, "bf16", "bf16", 16) == dec + 4 * (len(lens) + 1)


def test_cascade_bytes_count_the_prefix_once():
    """Shared prefix of P tokens: its K/V once, every sequence's own tokens
    past it, q, out, the prefix's table entries once and each sequence's own."""
    lens, P, bs = [2048 + 10, 2048 + 1, 2048 + 300], 2048, 16
    per = 2 * 8 * 128 * 1  # fp8, 8 kv heads, d 128
    kv = (P + 10 + 1 + 300) * per
    qo = 2 * 3 * 32 * 128 * 2
    tables = 4 * (P // bs + sum(-(-L // bs) - P // bs for L in lens))
    assert metrics.cascade_bytes(lens, P, 32, 8, 128, "fp8_e4m3", "bf16", bs) == kv + qo + tables + 4 * 3
    # a sequence ending inside the prefix reads no block of its own
    short = metrics.cascade_bytes([100], P, 32, 8, 128, "fp8_e4m3", "bf16", bs)
    assert short == 100 * per + 2 * 32 * 128 * 2 + 4 * (-(-100 // bs)) + 4


def test_window_bytes_count_only_kept_tokens():
    L, W, S, bs = 1000, 64, 4, 16
    kept = S + W
    per = 2 * 8 * 128 * 2
    blocks = 1 + (-(-L // bs) - (L - W) // bs)  # the sink block, then the window's blocks
    assert metrics.attended_tokens(L, W, S) == kept
    assert metrics.blocks_read(L, bs, W, S) == blocks
    assert metrics.decode_bytes([L], 32, 8, 128, "bf16", "bf16", bs, W, S) == \
        kept * per + 2 * 32 * 128 * 2 + 4 * blocks + 4


def test_chunk_queries_contract():
    w = workloads.make_workload("cq", [5, 40, 3], 8, 2, 64, 16, "bf16", seed=1)
    q, q_start = workloads.chunk_queries(w, [2, 0, 3], seed=2)
    assert q.shape == (5, 8, 64) and q.dtype == torch.bfloat16
    assert q_start.tolist() == [0, 2, 2, 5] and q_start.dtype == torch.int32
    q2, _ = workloads.chunk_queries(w, [2, 0, 3], seed=2)
    assert torch.equal(q, q2)  # seeded
    with pytest.raises(ValueError):
        workloads.chunk_queries(w, [6, 0, 0])  # more query tokens than positions
    with pytest.raises(ValueError):
        workloads.chunk_queries(w, [1, 1])  # one count per sequence
