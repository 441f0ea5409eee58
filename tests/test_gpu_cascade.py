"""Parity of cascade decode (pkv_cascade_decode: the shared prefix attended
once for the whole batch, then each sequence's own blocks, merged by
log-sum-exp) with the oracle's plain decode: the cascade only reorders the
sum, so the reference is the same softmax over each sequence's tokens."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import oracle_caches, oracle_decode, to_np
from tests.test_gpu_parity import TOL, assert_close, gpu_caches

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_22_gb300 as m
    m.library()
    return m


def run_cascade(pkv, w, kc, vc, prefix_blocks, seq_lens=None, tables=None):
    q = w.q.to(DEV)
    out = torch.full_like(q, float("nan"))
    lens = w.seq_lens if seq_lens is None else seq_lens
    pkv.cascade_decode(out, q, kc, vc, (w.block_tables if tables is None else tables).to(DEV), lens.to(DEV),
                       prefix_blocks, w.scale, w.kv_scale, max_seq_len=max(int(lens.max()), 1))
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def plain_ref(w, okc, ovc, seq_lens=None):
    lens = w.seq_lens if seq_lens is None else seq_lens
    return oracle.paged_attention_decode(to_np(w.q), okc, ovc, to_np(w.block_tables), to_np(lens),
                                         w.scale, w.kv_scale, 4)


# (name, suffix lengths, Hq, Hkv, d, block size, cache dtype, prefix tokens)
CASES = [
    ("bf16_g4", [1, 5, 16, 17, 40, 300], 32, 8, 128, 16, "bf16", 64),
    ("bf16_g8_bs8", [3, 9, 100], 16, 2, 128, 8, "bf16", 40),
    ("bf16_g1", [2, 31, 77], 4, 4, 128, 16, "bf16", 32),
    ("bf16_g2_bs32", [7, 64, 65], 8, 4, 128, 32, "bf16", 96),
    ("bf16_d64", [4, 19, 130], 16, 4, 64, 16, "bf16", 48),
    ("bf16_g16", [1, 33], 32, 2, 128, 16, "bf16", 16),
    ("fp8_g4", [1, 5, 40, 511], 32, 8, 128, 16, "fp8_e4m3", 128),
    ("fp8_d64_g8", [12, 70], 16, 2, 64, 16, "fp8_e4m3", 32),
    ("bf16_many_rows", [int(x) for x in np.random.default_rng(3).integers(1, 90, 37)], 32, 8, 128, 16, "bf16",
     80),
    # long prefixes over few rows: the prefix pass cuts them into many pieces,
    # the last one shorter
    ("bf16_long_prefix", [3, 50], 32, 8, 128, 16, "bf16", 1024),
    ("fp8_odd_prefix", [7, 20, 1], 32, 8, 128, 16, "fp8_e4m3", 37 * 16),
    ("bf16_bs8_odd_prefix", [5], 16, 2, 128, 8, "bf16", 29 * 8),
    # at least 128 rows (sequences x g) per kv head: the prefix pass runs on
    # the tcgen05 kernel (128-row tiles, pieces merged by the last one)
    ("bf16_rows160", [int(x) for x in np.random.default_rng(5).integers(1, 60, 40)], 32, 8, 128, 16, "bf16",
     256),
    ("bf16_rows300_g8_bs8", [int(x) for x in np.random.default_rng(6).integers(1, 40, 40)], 64, 8, 128, 8,
     "bf16", 37 * 8),
    ("bf16_rows_d64", [int(x) for x in np.random.default_rng(7).integers(1, 50, 33)], 16, 4, 64, 16,
     "bf16", 96),
    ("fp8_rows160", [int(x) for x in np.random.default_rng(8).integers(1, 80, 40)], 32, 8, 128, 16, "fp8_e4m3",
     512),
    ("fp8_rows_long_prefix", [int(x) for x in np.random.default_rng(9).integers(1, 30, 32)], 32, 8, 128, 16,
     "fp8_e4m3", 2048),
]

# cascade batches with at least 128 rows per kv head run the prefix pass on
# the tcgen05 kernel unless it is switched off; every case runs both ways
KERNELS = ["tcgen05", "mma_sync"]


def make_case(case, seed):
    name, suffix, Hq, Hkv, d, bs, dt, ptok = case
    lens = [ptok + s for s in suffix]
    return workloads.make_workload(name, lens, Hq, Hkv, d, bs, dt, seed=seed, prefix_tokens=ptok)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_cascade_matches_plain_decode(pkv, case, kernel):
    w = make_case(case, 71)
    kc, vc = gpu_caches(pkv, w)
    okc, ovc = oracle_caches(w)
    ref = plain_ref(w, okc, ovc)
    P = w.shared_prefix_blocks
    # the whole shared prefix, a part of it, and none (plain decode)
    with pkv.tcgen05(kernel == "tcgen05"):
        for pb in sorted({P, max(P // 2, 1), 1, 0}):
            got = run_cascade(pkv, w, kc, vc, pb)
            assert_close(got, ref, TOL[w.cache_dtype], f"{case[0]} prefix_blocks={pb}")
    assert pkv.get_device_error() == 0


# sequence counts of the edge-case tests: a few rows (mma.sync prefix pass)
# and, repeating the lengths, at least 128 rows per kv head (tcgen05)
REPEATS = [1, 32]


@pytest.mark.parametrize("repeat", REPEATS)
def test_sequences_shorter_than_the_prefix(pkv, repeat):
    """Sequences that end inside the prefix, at its end or are empty attend
    only their own tokens of it; their suffix is empty, so their row is the
    prefix partial alone."""
    w = make_case(("short", [5, 9, 1, 30, 2] * repeat, 32, 8, 128, 16, "bf16", 128), 72)
    lens = torch.tensor([3, 128, 0, 77, 129] * repeat, dtype=torch.int32)
    kc, vc = gpu_caches(pkv, w)
    okc, ovc = oracle_caches(w)
    got = run_cascade(pkv, w, kc, vc, w.shared_prefix_blocks, seq_lens=lens)
    ref = plain_ref(w, okc, ovc, seq_lens=lens)
    assert_close(got, ref, TOL["bf16"], "short sequences")
    assert np.all(got[2::5] == 0.0)
    assert pkv.get_device_error() == 0


@pytest.mark.parametrize("repeat", REPEATS)
def test_prefix_tail_nobody_attends_is_never_used(pkv, repeat):
    """Every sequence ends inside the prefix: the prefix tokens past the
    longest one are NaN in both caches and must not reach any output."""
    w = make_case(("tail", [4, 4, 4] * repeat, 16, 4, 128, 16, "bf16", 96), 73)
    lens = torch.tensor([20, 51, 7] * repeat, dtype=torch.int32)
    kc, vc = gpu_caches(pkv, w)
    okc, ovc = oracle_caches(w)
    bs = w.block_size
    nan_bf16 = torch.tensor(float("nan"), dtype=torch.bfloat16)
    for p in range(51, 96):
        blk, off = int(w.block_tables[0, p // bs]), p % bs
        kc[blk, :, off, :] = nan_bf16
        vc[blk, :, off, :] = nan_bf16
    got = run_cascade(pkv, w, kc, vc, w.shared_prefix_blocks, seq_lens=lens)
    ref = plain_ref(w, okc, ovc, seq_lens=lens)
    assert_close(got, ref, TOL["bf16"], "prefix tail")
    assert pkv.get_device_error() == 0


@pytest.mark.parametrize("repeat", REPEATS)
def test_table_that_disagrees_on_the_prefix_is_flagged(pkv, repeat):
    """A sequence whose table names another block for a prefix block it
    attends is flagged; entries past a short sequence's end are not
    compared."""
    w = make_case(("mismatch", [10, 20, 30] * repeat, 32, 8, 128, 16, "bf16", 64), 74)
    kc, vc = gpu_caches(pkv, w)
    okc, ovc = oracle_caches(w)
    lens = torch.tensor([74, 20, 94] * repeat, dtype=torch.int32)  # sequence 1 ends in prefix block 1
    tables = w.block_tables.clone()
    tables[1, 2] = workloads.UNUSED_TABLE_ENTRY  # past its end: not read, not compared
    tables[1, 3] = workloads.UNUSED_TABLE_ENTRY
    assert pkv.get_device_error() == 0
    got = run_cascade(pkv, w, kc, vc, w.shared_prefix_blocks, seq_lens=lens, tables=tables)
    assert pkv.get_device_error() == 0
    ref = oracle.paged_attention_decode(to_np(w.q), okc, ovc, to_np(tables), to_np(lens), w.scale, 1.0, 4)
    assert_close(got, ref, TOL["bf16"], "short table")
    tables[2, 1] = tables[2, 5]  # sequence 2 attends prefix block 1
    run_cascade(pkv, w, kc, vc, w.shared_prefix_blocks, seq_lens=lens, tables=tables)
    assert pkv.get_device_error() & pkv.DEVERR_BAD_BLOCK_ID


def test_workspace_size_formula(pkv):
    # the balanced decode's workspace, then the prefix partial [B * Hq] rows of
    # d + 4 fp32 values, then one such partial per piece when there are
    # several (pieces fill one wave of 12 warps per SM over (kv head,
    # 16-row block) pairs, at most 32); each region 256-byte aligned
    B, Hq, Hkv, d, L = 256, 32, 8, 128, 2560

    def up(x):
        return (x + 255) // 256 * 256
    dec = pkv.decode_workspace_bytes(B, Hq, Hkv, d, L, 0)
    assert dec > 0
    pairs = Hkv * -(-B * (Hq // Hkv) // 16)
    pieces = max(1, min(pkv.library().pkv_device_sm_count() * 12 // pairs, 32))
    row_bytes = B * Hq * (d + 4) * 4
    want = up(dec) + up(row_bytes) + (up(pieces * row_bytes) if pieces > 1 else 0)
    assert pkv.cascade_workspace_bytes(B, Hq, Hkv, d, L) == want


def test_invalid_calls(pkv):
    w = make_case(("inv", [3, 4], 8, 2, 64, 16, "f32", 32), 75)
    kc, vc = gpu_caches(pkv, w)
    q = w.q.to(DEV)
    out = torch.empty_like(q)
    with pytest.raises(pkv.PkvError):  # fp32 caches: no tensor-core prefix pass
        pkv.cascade_decode(out, q, kc, vc, w.block_tables.to(DEV), w.seq_lens.to(DEV), 2, w.scale)
    wb = make_case(("inv2", [3, 4], 8, 2, 64, 16, "bf16", 32), 76)
    kb, vb = gpu_caches(pkv, wb)
    qb = wb.q.to(DEV)
    ob = torch.empty_like(qb)
    for pb in (-1, wb.block_tables.shape[1] + 1):
        with pytest.raises(pkv.PkvError):
            pkv.cascade_decode(ob, qb, kb, vb, wb.block_tables.to(DEV), wb.seq_lens.to(DEV), pb, wb.scale)


def test_prefix_fp8_full_size(pkv):
    """The full-size shared-prefix fp8 workload (256 sequences, a 2048-token
    prefix): every output row against the oracle's plain decode."""
    w = workloads.CONFIGS["prefix_fp8"]()
    kc, vc = gpu_caches(pkv, w)
    okc, ovc = oracle_caches(w)
    ref = oracle_decode(w, okc, ovc, threads=os.cpu_count() or 4)
    got = run_cascade(pkv, w, kc, vc, w.shared_prefix_blocks)  # the prefix pass the benchmark times (tcgen05)
    assert_close(got, ref, TOL[w.cache_dtype], "prefix_fp8 cascade")
    with pkv.tcgen05(False):
        got = run_cascade(pkv, w, kc, vc, w.shared_prefix_blocks)
    assert_close(got, ref, TOL[w.cache_dtype], "prefix_fp8 cascade (mma.sync prefix pass)")
    assert pkv.get_device_error() == 0
