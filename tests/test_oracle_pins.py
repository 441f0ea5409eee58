"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each test checks the oracle against something it cannot agree with by
construction: a value printed by the source pages (fixtures under
``tests/golden``), a closed form, an invariant of softmax attention, or a
library routine that the special case reduces to (torch's scaled dot-product
attention in fp64, torch's bf16 and float8_e4m3fn conversions).
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import empty_cache_np, oracle_caches, oracle_decode, to_np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _records(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                kind, *vals = line.split()
                out.append((kind, [int(v) for v in vals]))
    return out


# ---------------------------------------------------------------- worked examples
def test_pages_block_table_example_gather():
    """Table [7, 2, 11]: tokens 0..15 come from block 7, 16..31 from 2, 32..47
    from 11, each at offset (token - range start)."""
    recs = _records("block_table_examples.txt")
    table = next(v for k, v in recs if k == "table")
    ranges = [v for k, v in recs if k == "token_range"]
    bs, NB, Hkv, d = 16, 12, 1, 4
    # every slot carries its own (block, offset) as data, in fp32
    kc = np.zeros((NB, Hkv, bs, d), dtype=np.float32)
    for b in range(NB):
        for o in range(bs):
            kc[b, 0, o, :] = [b, o, -b, -o]
    vc = kc + 0.5
    L = 48
    ko, vo = oracle.gather_kv(kc, vc, np.array([table], dtype=np.int32),
                              np.array([L], dtype=np.int32))
    for first, last, phys in ranges:
        for p in range(first, last + 1):
            assert ko[p, 0, 0] == phys and ko[p, 0, 1] == p - first
            assert vo[p, 0, 0] == phys + 0.5


def test_pages_token_counts_through_generator():
    """Block counts and the table position of a token follow the pages'
    worked numbers (200 -> entry 12, 273 -> 18 blocks, 500 -> 32 blocks)."""
    recs = _records("block_table_examples.txt")
    for kind, v in recs:
        if kind == "tokens_to_blocks":
            tokens, bs, blocks = v
            w = workloads.make_workload("t", [tokens], 1, 1, 8, bs, "f32", seed=1)
            valid = (w.block_tables[0] != workloads.UNUSED_TABLE_ENTRY).sum().item()
            assert valid == blocks
        elif kind == "token_to_table_index":
            tok, bs, idx = v
            w = workloads.make_workload("t", [tok + 1], 1, 1, 8, bs, "f32", seed=2)
            # the new token sits at position `tok`; its slot's block is entry `idx`
            slot = int(w.new_slots[0])
            assert slot // bs == int(w.block_tables[0, idx]) and slot % bs == tok % bs
        elif kind == "blocks_all_layers":
            tokens, bs, layers, blocks = v
            from paged_kv_cache_22_gb300.metrics import blocks_for_tokens
            assert blocks_for_tokens(tokens, bs) * layers == blocks


def test_pages_kv_byte_figures():
    from paged_kv_cache_22_gb300 import metrics
    seen = 0
    for kind, v in _records("kv_bytes_examples.txt"):
        if kind == "kv_bytes_per_token":
            layers, kvh, d, e, want = v
            assert metrics.kv_bytes_per_token(layers, kvh, d, e) == want
        elif kind == "block_bytes":
            bt, layers, kvh, d, e, want = v
            assert metrics.block_bytes(bt, layers, kvh, d, e) == want
        elif kind == "seq_bytes":
            tokens, layers, kvh, d, e, want = v
            assert tokens * metrics.kv_bytes_per_token(layers, kvh, d, e) == want
        seen += 1
    assert seen >= 8


# ---------------------------------------------------------------- element types
def test_bf16_encode_matches_torch_rne():
    gen = torch.Generator().manual_seed(7)
    x = torch.randn(4000, generator=gen) * torch.exp(torch.randn(4000, generator=gen) * 6)
    # exact ties: 1 + (2k+1) * 2^-8 lies halfway between two bf16 values
    ties = torch.tensor([1 + (2 * k + 1) * 2.0 ** -8 for k in range(64)], dtype=torch.float32)
    x = torch.cat([x, ties, -ties, torch.tensor([0.0, -0.0, 3.4e38, -3.4e38, 1e-40, float("inf")])])
    ours = oracle.bf16_encode(x.numpy())
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_decode_is_exact_widening():
    bits = np.arange(0, 1 << 16, 97, dtype=np.uint16)
    ours = oracle.bf16_decode(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(ours[~both_nan], ref[~both_nan])


def test_fp8_decode_all_256_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.fp8_e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_fp8_encode_roundtrip_ties_and_saturation():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.fp8_e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.fp8_e4m3_encode(vals), codes)
    # midpoints between neighbouring positive codes go to the even code
    pos = np.arange(0, 0x7E, dtype=np.uint8)
    lo, hi = oracle.fp8_e4m3_decode(pos), oracle.fp8_e4m3_decode(pos + 1)
    mids = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (lo + hi) / 2)  # exactly representable
    enc = oracle.fp8_e4m3_encode(mids)
    want = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint8)
    assert np.array_equal(enc, want)
    sat = oracle.fp8_e4m3_encode(np.array([448.0, 449.0, 500.0, 1e9, np.inf, -1e9, -np.inf],
                                          dtype=np.float32))
    assert list(sat) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert oracle.fp8_e4m3_encode(np.array([np.nan], dtype=np.float32))[0] in (0x7F, 0xFF)


def test_fp8_encode_matches_torch_in_range():
    gen = torch.Generator().manual_seed(11)
    x = torch.randn(20000, generator=gen) * torch.exp(torch.randn(20000, generator=gen) * 2.5)
    x = x[x.abs() <= 448]
    ours = oracle.fp8_e4m3_encode(x.numpy())
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------- cache write
@pytest.mark.parametrize("cache_dtype", ["f32", "bf16", "fp8_e4m3"])
def test_reshape_and_cache_layout_and_skip(cache_dtype):
    """Token t with slot s lands at [s // bs, h, s % bs, :] of the
    [num_blocks, kv_heads, block_size, head_dim] cache; slot -1 is skipped."""
    T, Hkv, d, bs, NB = 5, 3, 8, 4, 6
    gen = torch.Generator().manual_seed(3)
    src_dtype = torch.float32 if cache_dtype == "f32" else torch.bfloat16
    k = torch.randn(T, Hkv, d, generator=gen).to(src_dtype)
    v = torch.randn(T, Hkv, d, generator=gen).to(src_dtype)
    slots = np.array([0, 23, -1, 9, 14], dtype=np.int64)
    dt = {"f32": np.float32, "bf16": np.uint16, "fp8_e4m3": np.uint8}[cache_dtype]
    kc = np.zeros((NB, Hkv, bs, d), dtype=dt)
    vc = np.zeros_like(kc)
    kv_scale = 0.0625
    oracle.reshape_and_cache(to_np(k), to_np(v), kc, vc, slots, kv_scale)
    kf, vf = k.float(), v.float()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = s // bs, s % bs
        if cache_dtype == "f32":
            want_k, want_v = kf[t].numpy(), vf[t].numpy()
        elif cache_dtype == "bf16":
            want_k = kf[t].to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            want_v = vf[t].to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        else:  # torch's e4m3 conversion of x / kv_scale (all values well in range)
            want_k = (kf[t] / kv_scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            want_v = (vf[t] / kv_scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(kc[blk, :, off, :], want_k)
        assert np.array_equal(vc[blk, :, off, :], want_v)
    written = {(s // bs, s % bs) for s in slots if s >= 0}
    for b in range(NB):
        for o in range(bs):
            if (b, o) not in written:
                assert not kc[b, :, o, :].any()


# ---------------------------------------------------------------- attention
def _sdpa_contiguous(q, K, V, scale):
    """torch scaled_dot_product_attention in fp64; K, V [Hkv, L, d]."""
    qt = torch.from_numpy(q)[:, None, :]  # [Hq, 1, d]
    out = torch.nn.functional.scaled_dot_product_attention(
        qt, torch.from_numpy(K), torch.from_numpy(V), scale=scale, enable_gqa=True)
    return out[:, 0, :].numpy()


@pytest.mark.parametrize("cache_dtype,Hq,Hkv,d", [("f32", 4, 4, 64), ("bf16", 32, 8, 128),
                                                   ("bf16", 8, 1, 64), ("fp8_e4m3", 16, 2, 128)])
def test_contiguous_case_matches_torch_sdpa(cache_dtype, Hq, Hkv, d):
    """With identity block tables the paged cache is the contiguous baseline;
    the oracle must agree with torch SDPA (fp64) on the decoded cache."""
    lens = [1, 16, 17, 75]
    w = workloads.make_workload("c", lens, Hq, Hkv, d, 16, cache_dtype, seed=5,
                                identity_tables=True, num_blocks=sum(-(-L // 16) for L in lens))
    kc, vc = oracle_caches(w)
    out = oracle_decode(w, kc, vc)
    if cache_dtype == "f32":
        Kall, Vall = kc.astype(np.float64), vc.astype(np.float64)
    elif cache_dtype == "bf16":
        Kall = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16).double().numpy()
        Vall = torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16).double().numpy()
    else:
        Kall = torch.from_numpy(kc).view(torch.float8_e4m3fn).double().numpy() * w.kv_scale
        Vall = torch.from_numpy(vc).view(torch.float8_e4m3fn).double().numpy() * w.kv_scale
    q = w.q.double().numpy()
    start = 0
    for i, L in enumerate(lens):
        nb = -(-L // 16)
        K = Kall[start:start + nb].transpose(1, 0, 2, 3).reshape(Hkv, nb * 16, d)[:, :L]
        V = Vall[start:start + nb].transpose(1, 0, 2, 3).reshape(Hkv, nb * 16, d)[:, :L]
        ref = _sdpa_contiguous(q[i], np.ascontiguousarray(K), np.ascontiguousarray(V), w.scale)
        np.testing.assert_allclose(out[i], ref, rtol=0, atol=1e-12)
        start += nb


def test_block_permutation_invariance_is_exact():
    lens = [5, 40, 100, 1]
    ident = workloads.make_workload("p", lens, 8, 2, 64, 16, "bf16", seed=9, identity_tables=True,
                                    num_blocks=20)
    shuf = workloads.make_workload("p", lens, 8, 2, 64, 16, "bf16", seed=9, num_blocks=20)
    # same draws, different placement: q, tokens equal; tables differ
    assert torch.equal(ident.q, shuf.q) and torch.equal(ident.hist_k, shuf.hist_k)
    assert not torch.equal(ident.block_tables, shuf.block_tables)
    a, b = oracle_decode(ident), oracle_decode(shuf)
    assert np.array_equal(a, b)


def _single_seq(L, Hq, Hkv, d, seed=0, cache_dtype="f32"):
    return workloads.make_workload("s", [L], Hq, Hkv, d, 16, cache_dtype, seed=seed)


def test_length_one_returns_own_value_exactly():
    w = _single_seq(1, 4, 2, 64, seed=21)
    out = oracle_decode(w)
    v = w.new_v.double().numpy()[0]  # [Hkv, d]
    g = w.gqa_group
    for qh in range(4):
        assert np.array_equal(out[0, qh], v[qh // g])


def _cache_with_tokens(K, V, bs=16, dtype=np.float32):
    """Identity-table cache holding K, V [L, Hkv, d] (fp32)."""
    L, Hkv, d = K.shape
    nb = -(-L // bs)
    kc = np.zeros((nb, Hkv, bs, d), dtype=dtype)
    vc = np.zeros_like(kc)
    for p in range(L):
        kc[p // bs, :, p % bs, :] = K[p]
        vc[p // bs, :, p % bs, :] = V[p]
    return kc, vc, np.arange(nb, dtype=np.int32)[None, :]


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(0)
    L, Hkv, d = 37, 2, 16
    K = np.repeat(rng.standard_normal((1, Hkv, d)), L, axis=0).astype(np.float32)
    V = rng.standard_normal((L, Hkv, d)).astype(np.float32)
    kc, vc, tbl = _cache_with_tokens(K, V)
    q = rng.standard_normal((1, 4, d)).astype(np.float32)
    out = oracle.paged_attention_decode(q, kc, vc, tbl, np.array([L], np.int32), 0.25)
    for qh in range(4):
        np.testing.assert_allclose(out[0, qh], V[:, qh // 2].astype(np.float64).mean(0),
                                   rtol=0, atol=1e-13)


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(1)
    L, Hkv, d = 50, 1, 32
    K = rng.standard_normal((L, Hkv, d)).astype(np.float32)
    V = rng.standard_normal((L, Hkv, d)).astype(np.float32)
    kc, vc, tbl = _cache_with_tokens(K, V)
    q = np.zeros((1, 1, d), dtype=np.float32)
    out = oracle.paged_attention_decode(q, kc, vc, tbl, np.array([L], np.int32), 0.3)
    np.testing.assert_allclose(out[0, 0], V[:, 0].astype(np.float64).mean(0), rtol=0, atol=1e-13)


def test_two_tokens_closed_form():
    """out = v0 + (v1 - v0) * sigmoid(s1 - s0), s_t = scale * q.k_t."""
    rng = np.random.default_rng(2)
    d = 8
    K = rng.standard_normal((2, 1, d)).astype(np.float32)
    V = rng.standard_normal((2, 1, d)).astype(np.float32)
    kc, vc, tbl = _cache_with_tokens(K, V)
    q = rng.standard_normal((1, 1, d)).astype(np.float32)
    scale = 0.7
    out = oracle.paged_attention_decode(q, kc, vc, tbl, np.array([2], np.int32), scale)
    Kd, Vd, qd = K.astype(np.float64), V.astype(np.float64), q.astype(np.float64)
    s0 = scale * float(Kd[0, 0] @ qd[0, 0])
    s1 = scale * float(Kd[1, 0] @ qd[0, 0])
    sig = 1.0 / (1.0 + math.exp(-(s1 - s0)))
    np.testing.assert_allclose(out[0, 0], Vd[0, 0] + (Vd[1, 0] - Vd[0, 0]) * sig, rtol=0,
                               atol=1e-14)


def test_affine_in_values_and_convex_hull():
    rng = np.random.default_rng(3)
    L, d = 29, 16
    K = rng.standard_normal((L, 1, d)).astype(np.float32)
    # values on the bf16 grid, so that 2 * V - 3 is exact in fp32
    V = torch.from_numpy(rng.standard_normal((L, 1, d)).astype(np.float32)).bfloat16().float()
    V = V.numpy()
    q = rng.standard_normal((1, 1, d)).astype(np.float32)
    lens = np.array([L], np.int32)
    kc, vc, tbl = _cache_with_tokens(K, V)
    base = oracle.paged_attention_decode(q, kc, vc, tbl, lens, 0.5)[0, 0]
    a, b = np.float32(2.0), np.float32(-3.0)  # exact in fp32 for these values
    kc2, vc2, _ = _cache_with_tokens(K, a * V + b)
    aff = oracle.paged_attention_decode(q, kc2, vc2, tbl, lens, 0.5)[0, 0]
    np.testing.assert_allclose(aff, 2.0 * base - 3.0, rtol=0, atol=1e-12)
    assert np.all(base <= V[:, 0].max(0) + 1e-12) and np.all(base >= V[:, 0].min(0) - 1e-12)


def test_score_shift_invariance():
    """A key component shared by every token adds the same constant to every
    score; the output must not move."""
    rng = np.random.default_rng(4)
    L, d = 20, 8
    K = rng.standard_normal((L, 1, d)).astype(np.float32)
    K[:, 0, 0] = 1.5
    V = rng.standard_normal((L, 1, d)).astype(np.float32)
    kc, vc, tbl = _cache_with_tokens(K, V)
    lens = np.array([L], np.int32)
    q1 = rng.standard_normal((1, 1, d)).astype(np.float32)
    q2 = q1.copy()
    q2[0, 0, 0] += 7.0
    o1 = oracle.paged_attention_decode(q1, kc, vc, tbl, lens, 0.4)
    o2 = oracle.paged_attention_decode(q2, kc, vc, tbl, lens, 0.4)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def test_empty_sequence_gives_zero_row_and_threads_agree():
    w = workloads.make_workload("e", [0, 5, 0, 33], 4, 2, 64, 16, "bf16", seed=12)
    out1 = oracle_decode(w, threads=1)
    out4 = oracle_decode(w, threads=4)
    assert not out1[0].any() and not out1[2].any()
    assert np.array_equal(out1, out4)


@pytest.mark.parametrize("P", [16, 32, 48, 512])
def test_split_merge_equals_unsplit(P):
    w = workloads.make_workload("m", [1, 16, 100, 333, 0], 8, 2, 64, 16, "bf16", seed=13)
    kc, vc = oracle_caches(w)
    full = oracle_decode(w, kc, vc)
    maxp = max(1, -(-w.max_seq_len // P))
    o, m, l = oracle.partition_attention(to_np(w.q), kc, vc, to_np(w.block_tables),
                                         to_np(w.seq_lens), w.scale, w.kv_scale, P, maxp)
    merged = oracle.split_kv_reduce(o, m, l, to_np(w.seq_lens), P)
    np.testing.assert_allclose(merged, full, rtol=0, atol=1e-12)
    # partitions past the end are empty (-inf, 0); a single partition is the full result
    lens = w.seq_lens.numpy()
    for i, L in enumerate(lens):
        npart = -(-int(L) // P)
        assert np.all(np.isneginf(m[i, :, npart:])) and not l[i, :, npart:].any()
        if npart == 1:
            np.testing.assert_allclose(o[i, :, 0], full[i], rtol=0, atol=1e-13)


def test_reduce_closed_form_equal_maxima():
    """With equal partition maxima the merge is the l-weighted mean of the
    partition outputs."""
    rng = np.random.default_rng(6)
    d = 4
    o = rng.standard_normal((1, 1, 3, d))
    m = np.full((1, 1, 3), 0.75)
    l = np.array([[[2.0, 5.0, 1.0]]])
    out = oracle.split_kv_reduce(o, m, l, np.array([40], np.int32), 16)
    want = (2 * o[0, 0, 0] + 5 * o[0, 0, 1] + 1 * o[0, 0, 2]) / 8.0
    np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-14)


def test_fp8_attention_reads_code_times_scale():
    """An fp8 cache is read as code value * kv_scale: scaling kv_scale by 2
    doubles every value, which (with q halved) leaves scores unchanged and
    doubles the output."""
    w = workloads.make_workload("f", [7, 40], 8, 2, 128, 16, "fp8_e4m3", seed=14)
    kc, vc = oracle_caches(w)
    q = to_np(w.q)
    o1 = oracle.paged_attention_decode(q, kc, vc, to_np(w.block_tables), to_np(w.seq_lens),
                                       w.scale, w.kv_scale)
    o2 = oracle.paged_attention_decode(q, kc, vc, to_np(w.block_tables), to_np(w.seq_lens),
                                       w.scale / 2, w.kv_scale * 2)
    np.testing.assert_allclose(o2, 2 * o1, rtol=0, atol=1e-12)


def test_poisoned_unused_slots_never_reach_the_output():
    """Fresh caches are NaN everywhere; only written slots are read, so the
    oracle output stays finite (tokens past seq_len in a last block and
    table entries past the last block are never touched)."""
    w = workloads.make_workload("n", [3, 17, 31], 4, 4, 64, 16, "f32", seed=15, num_blocks=16)
    kc, vc = oracle_caches(w)
    assert np.isnan(kc).any()
    assert np.isfinite(oracle_decode(w, kc, vc)).all()


# ---------------------------------------------------------------- workload generator
@pytest.mark.parametrize("name", ["tiny_mha", "llama3_8b", "prefix_fp8"])
def test_generator_invariants(name):
    kw = {"llama3_8b": {"num_seqs": 16}, "prefix_fp8": {"num_seqs": 12}}.get(name, {})
    w = workloads.CONFIGS[name](**kw)
    k, v, slots = w.all_tokens()
    s = slots.numpy()
    assert len(np.unique(s)) == len(s), "one writer per slot"
    assert s.min() >= 0 and s.max() < w.num_blocks * w.block_size
    tbl = w.block_tables.numpy()
    lens = w.seq_lens.numpy()
    used = set()
    for i, L in enumerate(lens):
        nb = -(-int(L) // w.block_size)
        row = tbl[i, :nb]
        assert np.all((row >= 0) & (row < w.num_blocks))
        assert np.all(tbl[i, nb:] == workloads.UNUSED_TABLE_ENTRY)
        own = row[w.shared_prefix_blocks:]
        assert not (set(own.tolist()) & used), "private blocks are not shared"
        used |= set(own.tolist())
    if w.shared_prefix_blocks:
        assert np.all(tbl[:, :w.shared_prefix_blocks] == tbl[0, :w.shared_prefix_blocks])
        assert not (set(tbl[0, :w.shared_prefix_blocks].tolist()) & used)
    assert len(w.new_slots) == int((lens > 0).sum())


def test_config_shapes():
    w = workloads.tiny_mha()
    assert w.seq_lens.tolist() == [1, 17, 33, 100] and w.num_blocks == 64
    assert (w.num_q_heads, w.num_kv_heads, w.head_dim, w.cache_dtype) == (4, 4, 64, "f32")
    w = workloads.llama70b_128()
    lens = w.seq_lens.numpy()
    assert lens.min() >= 16 and lens.max() <= 8192 and len(lens) == 128
    assert w.num_blocks == math.ceil(1.1 * sum(-(-int(L) // 16) for L in lens))


# ---------------------------------------------------------------- block copies
def _pool(rng, nb, hkv=2, bs=16, d=64):
    k = rng.integers(0, 1 << 16, size=(nb, hkv, bs, d), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(nb, hkv, bs, d), dtype=np.uint16)
    return k, v


def test_copy_on_write_keeps_the_shared_block_and_diverges_the_copy():
    """Two sequences share their first block; the branch about to write gets
    a copy first.  Through the (independent) gather: right after the copy both
    sequences read the same tokens; after the write into the copy only the
    writer's token changes, and the other sequence still reads the original."""
    rng = np.random.default_rng(7)
    kc, vc = _pool(rng, 8)
    tables = np.array([[3, 5], [3, 6]], dtype=np.int32)  # block 3 shared
    lens = np.array([20, 20], dtype=np.int32)
    before_k, before_v = oracle.gather_kv(kc, vc, tables, lens)
    oracle.copy_blocks(kc, vc, kc, vc, np.array([[3, 1]]))  # COW: 3 -> fresh block 1
    tables_b = tables.copy()
    tables_b[1, 0] = 1
    k1, v1 = oracle.gather_kv(kc, vc, tables_b, lens)
    assert np.array_equal(k1, before_k) and np.array_equal(v1, before_v)
    # sequence 1 writes token 4 (inside its copy, slot 1*16 + 4)
    new = rng.standard_normal((1, 2, 64)).astype(np.float32)
    oracle.reshape_and_cache(new, new, kc, vc, np.array([1 * 16 + 4]), 1.0)
    k2, v2 = oracle.gather_kv(kc, vc, tables_b, lens)
    diff = np.nonzero(np.any(k2 != before_k, axis=(1, 2)))[0]
    assert diff.tolist() == [20 + 4], "only the writer's token changes"
    k_a, _ = oracle.gather_kv(kc, vc, tables[:1], lens[:1])
    assert np.array_equal(k_a, before_k[:20]), "the shared block is untouched"


def test_swap_out_and_back_to_other_ids_preserves_every_token():
    """Swap a sequence's blocks to a host pool and back into different device
    blocks; with the table rewritten to the new ids the gather is unchanged."""
    rng = np.random.default_rng(8)
    kc, vc = _pool(rng, 12)
    host_k, host_v = np.zeros((4, 2, 16, 64), np.uint16), np.zeros((4, 2, 16, 64), np.uint16)
    table = np.array([[9, 2, 7]], dtype=np.int32)
    lens = np.array([40], dtype=np.int32)
    ref_k, ref_v = oracle.gather_kv(kc, vc, table, lens)
    oracle.copy_blocks(host_k, host_v, kc, vc, np.array([[9, 0], [2, 1], [7, 2]]))
    oracle.copy_blocks(kc, vc, host_k, host_v, np.array([[0, 4], [1, 10], [2, 0]]))
    got_k, got_v = oracle.gather_kv(kc, vc, np.array([[4, 10, 0]], dtype=np.int32), lens)
    assert np.array_equal(got_k, ref_k) and np.array_equal(got_v, ref_v)


def test_copy_blocks_rejects_ids_outside_the_pools():
    rng = np.random.default_rng(9)
    kc, vc = _pool(rng, 4)
    snap = kc.copy()
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(kc, vc, kc, vc, np.array([[0, 4]]))
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(kc, vc, kc, vc, np.array([[-1, 2]]))
    assert np.array_equal(kc, snap)


# ---------------------------------------------------------------- sliding window and sinks
def _window_case(seed=31):
    w = workloads.make_workload("win", [1, 5, 17, 40, 70], 8, 2, 64, 16, "f32", seed=seed)
    kc, vc = oracle_caches(w)
    return w, kc, vc


def _decode(w, kc, vc, tables=None, **kw):
    return oracle.paged_attention_decode(to_np(w.q), kc, vc, to_np(w.block_tables if tables is None else tables),
                                         to_np(w.seq_lens), w.scale, w.kv_scale, 1, **kw)


def test_window_covering_every_token_is_plain_attention():
    w, kc, vc = _window_case()
    plain = _decode(w, kc, vc)
    assert np.array_equal(_decode(w, kc, vc, window=70), plain)
    assert np.array_equal(_decode(w, kc, vc, window=20, sinks=50), plain)  # sinks + window >= L


def test_window_of_one_returns_the_last_value():
    w, kc, vc = _window_case()
    got = _decode(w, kc, vc, window=1)
    k_all, v_all = oracle.gather_kv(kc, vc, to_np(w.block_tables), to_np(w.seq_lens))
    cu = np.concatenate([[0], np.cumsum(w.seq_lens.numpy())])
    g = w.num_q_heads // w.num_kv_heads
    for s in range(w.num_seqs):
        last = v_all[cu[s + 1] - 1].astype(np.float64)  # [Hkv, d]
        assert np.array_equal(got[s], np.repeat(last, g, axis=0))


@pytest.mark.parametrize("window,sinks", [(8, 0), (8, 4), (20, 3), (33, 16)])
def test_window_equals_brute_force_over_the_kept_tokens(window, sinks):
    """numpy fp64 softmax over exactly the kept positions (first `sinks`,
    last `window`) of the gathered sequence; the hole between the sinks and
    the window lies inside one block for some lengths."""
    w, kc, vc = _window_case()
    got = _decode(w, kc, vc, window=window, sinks=sinks)
    k_all, v_all = oracle.gather_kv(kc, vc, to_np(w.block_tables), to_np(w.seq_lens))
    lens = w.seq_lens.numpy()
    cu = np.concatenate([[0], np.cumsum(lens)])
    q = w.q.numpy().astype(np.float64)
    g = w.num_q_heads // w.num_kv_heads
    for s in range(w.num_seqs):
        L = int(lens[s])
        keep = [p for p in range(L) if L <= window or p < sinks or p >= L - window]
        K = k_all[cu[s]:cu[s + 1]].astype(np.float64)[keep]  # [n, Hkv, d]
        V = v_all[cu[s]:cu[s + 1]].astype(np.float64)[keep]
        for qh in range(w.num_q_heads):
            sc = w.scale * (K[:, qh // g] @ q[s, qh])
            p = np.exp(sc - sc.max())
            ref = (p[:, None] * V[:, qh // g]).sum(0) / p.sum()
            assert np.abs(got[s, qh] - ref).max() < 1e-12


def test_window_never_reads_blocks_outside_the_kept_tokens():
    """Blocks holding no kept token may have been freed: their table entries
    point outside the pool, and the result does not change."""
    w, kc, vc = _window_case()
    window, sinks, bs = 16, 4, w.block_size
    ref = _decode(w, kc, vc, window=window, sinks=sinks)
    tables = w.block_tables.clone()
    for s, L in enumerate(w.seq_lens.tolist()):
        for j in range(-(-L // bs)):
            toks = range(j * bs, min(L, (j + 1) * bs))
            if not any(L <= window or p < sinks or p >= L - window for p in toks):
                tables[s, j] = w.num_blocks + 7
    assert not torch.equal(tables, w.block_tables)
    assert np.array_equal(_decode(w, kc, vc, tables=tables, window=window, sinks=sinks), ref)


# ------------------------------------------------------------------ multi-token queries
def _multi_case(cache_dtype="f32", seed=41, lens=(1, 5, 17, 40, 70), q_lens=(1, 3, 17, 8, 33), Hq=8, Hkv=2,
                d=64, identity=False):
    kw = dict(identity_tables=True, num_blocks=sum(-(-L // 16) for L in lens)) if identity else {}
    w = workloads.make_workload("mq", list(lens), Hq, Hkv, d, 16, cache_dtype, seed=seed, **kw)
    q, q_start = workloads.chunk_queries(w, list(q_lens), seed=seed + 1)
    kc, vc = oracle_caches(w)
    return w, q, q_start, kc, vc


def _multi(w, q, q_start, kc, vc, tables=None):
    return oracle.paged_attention_multi(to_np(q), to_np(q_start), kc, vc,
                                        to_np(w.block_tables if tables is None else tables),
                                        to_np(w.seq_lens), w.scale, w.kv_scale, 2)


def test_multi_with_one_query_token_is_decode():
    """T = 1 for every sequence: the query token is the last position, which
    is exactly decode."""
    w, _, _, kc, vc = _multi_case()
    q_start = torch.arange(w.num_seqs + 1, dtype=torch.int32)
    got = _multi(w, w.q, q_start, kc, vc)
    assert np.array_equal(got, oracle_decode(w, kc, vc))


def test_multi_last_token_of_each_chunk_is_decode_of_its_query():
    """The last query token of a chunk sits at position L - 1 and sees the
    whole sequence: the decode of that query row."""
    w, q, q_start, kc, vc = _multi_case(seed=43)
    got = _multi(w, q, q_start, kc, vc)
    last = q[q_start[1:].long() - 1]  # [B, Hq, d]
    ref = oracle.paged_attention_decode(to_np(last), kc, vc, to_np(w.block_tables), to_np(w.seq_lens),
                                        w.scale, w.kv_scale, 1)
    assert np.array_equal(got[q_start[1:].numpy() - 1], ref)


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16", "fp8_e4m3"])
def test_multi_contiguous_case_matches_torch_sdpa_with_bottom_right_causal_mask(cache_dtype):
    """Identity tables make the paged cache contiguous; torch SDPA in fp64
    with an explicit mask (query token i of T may see key j iff
    j <= L - T + i) on the decoded cache must agree."""
    lens, q_lens = (1, 16, 17, 75), (1, 16, 5, 30)
    Hq, Hkv, d = 8, 2, 64
    w, q, q_start, kc, vc = _multi_case(cache_dtype, seed=47, lens=lens, q_lens=q_lens, Hq=Hq, Hkv=Hkv, d=d,
                                        identity=True)
    got = _multi(w, q, q_start, kc, vc)
    if cache_dtype == "f32":
        Kall, Vall = kc.astype(np.float64), vc.astype(np.float64)
    elif cache_dtype == "bf16":
        Kall = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16).double().numpy()
        Vall = torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16).double().numpy()
    else:
        Kall = torch.from_numpy(kc).view(torch.float8_e4m3fn).double().numpy() * w.kv_scale
        Vall = torch.from_numpy(vc).view(torch.float8_e4m3fn).double().numpy() * w.kv_scale
    qd = q.double()
    start = 0
    for s, (L, T) in enumerate(zip(lens, q_lens)):
        nb = -(-L // 16)
        K = torch.from_numpy(Kall[start:start + nb].transpose(1, 0, 2, 3).reshape(Hkv, nb * 16, d)[:, :L].copy())
        V = torch.from_numpy(Vall[start:start + nb].transpose(1, 0, 2, 3).reshape(Hkv, nb * 16, d)[:, :L].copy())
        rows = qd[int(q_start[s]):int(q_start[s + 1])].transpose(0, 1)  # [Hq, T, d]
        mask = torch.arange(L)[None, :] <= (L - T + torch.arange(T))[:, None]  # [T, L]
        ref = torch.nn.functional.scaled_dot_product_attention(rows, K, V, attn_mask=mask, scale=w.scale,
                                                               enable_gqa=True)  # [Hq, T, d]
        np.testing.assert_allclose(got[int(q_start[s]):int(q_start[s + 1])], ref.transpose(0, 1).numpy(),
                                   rtol=0, atol=1e-12)
        start += nb


def test_multi_is_causal_inside_the_chunk():
    """Changing the cache at positions after a query token's own position
    leaves its output unchanged; changing its own position changes it (the
    token attends itself)."""
    w, q, q_start, kc, vc = _multi_case(seed=53, lens=(40,), q_lens=(12,))
    base = _multi(w, q, q_start, kc, vc)
    L, T, bs = 40, 12, w.block_size
    for pos in (L - T + 3, L - 1):  # a position inside the chunk
        k2, v2 = kc.copy(), vc.copy()
        blk = int(w.block_tables[0, pos // bs])
        k2[blk, :, pos % bs, :] += 0.5
        v2[blk, :, pos % bs, :] -= 0.25
        got = _multi(w, q, q_start, k2, v2)
        i_pos = pos - (L - T)  # the query token sitting at `pos`
        assert np.array_equal(got[:i_pos], base[:i_pos])  # earlier tokens never see it
        assert not np.allclose(got[i_pos], base[i_pos])   # the token at pos attends itself


def test_multi_equal_keys_give_running_means_of_values():
    """With every key equal the softmax is uniform: query token i of a chunk
    of T returns the mean of V over positions 0 .. L - T + i."""
    rng = np.random.default_rng(7)
    L, T, Hkv, d, Hq = 37, 9, 2, 16, 4
    K = np.repeat(rng.standard_normal((1, Hkv, d)).astype(np.float32), L, axis=0)
    V = rng.standard_normal((L, Hkv, d)).astype(np.float32)
    kc, vc, tables = _cache_with_tokens(K, V)
    q = rng.standard_normal((T, Hq, d)).astype(np.float32)
    out = oracle.paged_attention_multi(q, np.array([0, T], np.int32), kc, vc, tables,
                                       np.array([L], np.int32), 0.3, 1.0, 1)
    g = Hq // Hkv
    for i in range(T):
        mean = V[:L - T + i + 1].astype(np.float64).mean(axis=0)  # [Hkv, d]
        for qh in range(Hq):
            np.testing.assert_allclose(out[i, qh], mean[qh // g], rtol=0, atol=1e-12)


def test_multi_block_permutation_invariance_and_empty_chunks():
    """Placement of the blocks does not matter; a sequence with no query
    token contributes no row."""
    lens, q_lens = [5, 40, 100, 1], [2, 0, 33, 1]
    ident = workloads.make_workload("p", lens, 8, 2, 64, 16, "bf16", seed=9, identity_tables=True, num_blocks=20)
    shuf = workloads.make_workload("p", lens, 8, 2, 64, 16, "bf16", seed=9, num_blocks=20)
    q, q_start = workloads.chunk_queries(ident, q_lens, seed=3)
    a = _multi(ident, q, q_start, *oracle_caches(ident))
    b = _multi(shuf, q, q_start, *oracle_caches(shuf))
    assert a.shape == (sum(q_lens), 8, 64)
    assert np.array_equal(a, b)


def test_multi_rejects_bad_query_ranges():
    w, q, q_start, kc, vc = _multi_case()
    bad = q_start.clone()
    bad[1] = bad[0] + int(w.seq_lens[0]) + 1  # more query tokens than positions
    bad[2:] += int(bad[1]) - int(q_start[1])
    qq = torch.zeros((int(bad[-1]), w.num_q_heads, w.head_dim), dtype=q.dtype)
    with pytest.raises(Exception):
        _multi(w, qq, bad, kc, vc)
