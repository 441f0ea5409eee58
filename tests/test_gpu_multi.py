"""Parity of paged attention for several query tokens per sequence
(pkv_paged_attention_multi: prefill chunks, speculative verification) with
the oracle's multi-token attention, on the GPU through the C ABI."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import oracle_caches, to_np
from tests.test_gpu_parity import TOL, assert_close, gpu_caches

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_22_gb300 as m
    m.library()
    return m


def run_multi(pkv, w, kc, vc, q, q_start, max_q=None, tables=None):
    out = torch.full((q.shape[0], w.num_q_heads, w.head_dim), float("nan"), dtype=torch.bfloat16, device=DEV)
    pkv.paged_attention_multi(out, q.to(DEV), q_start.to(DEV), kc, vc,
                              (w.block_tables if tables is None else tables).to(DEV), w.seq_lens.to(DEV),
                              w.scale, w.kv_scale, max_q=max_q, max_seq_len=max(w.max_seq_len, 1))
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def multi_ref(w, okc, ovc, q, q_start, threads=4):
    return oracle.paged_attention_multi(to_np(q), to_np(q_start), okc, ovc, to_np(w.block_tables),
                                        to_np(w.seq_lens), w.scale, w.kv_scale, threads)


# (name, seq lens, query tokens per sequence, Hq, Hkv, d, block size, cache dtype)
CASES = [
    ("verify4_bf16", [5, 17, 40, 300, 1000], [4, 4, 4, 4, 4], 32, 8, 128, 16, "bf16"),
    ("chunks_bf16", [64, 130, 600, 33], [64, 100, 37, 1], 32, 8, 128, 16, "bf16"),
    ("whole_prefill", [16, 45], [16, 45], 32, 8, 128, 16, "bf16"),
    ("decode_t1", [1, 9, 200, 77], [1, 1, 1, 1], 32, 8, 128, 16, "bf16"),
    ("empty_chunks", [20, 50, 8], [0, 7, 0], 32, 8, 128, 16, "bf16"),
    ("fp8_verify", [3, 70, 511], [3, 5, 8], 32, 8, 128, 16, "fp8_e4m3"),
    ("fp8_d64_chunk", [200, 90], [50, 90], 16, 2, 64, 16, "fp8_e4m3"),
    ("bf16_d64_g4", [19, 130], [6, 40], 16, 4, 64, 16, "bf16"),
    ("bf16_g8_bs8", [9, 130], [2, 33], 16, 2, 128, 8, "bf16"),
    ("bf16_g1_bs32", [31, 77, 150], [5, 1, 64], 4, 4, 128, 32, "bf16"),
    ("bf16_g8_long", [3000, 2500], [3, 16], 64, 8, 128, 16, "bf16"),
    ("fp8_chunks_d128", [700, 90, 300], [200, 90, 1], 32, 8, 128, 16, "fp8_e4m3"),
    ("fp8_bs8_chunk", [130, 77], [64, 40], 16, 2, 128, 8, "fp8_e4m3"),
    # fewer than 128 rows per (sequence, kv head), blocks of 32: only the
    # tcgen05 kernel has an fp8 instance, so it serves the call
    ("fp8_bs32_small", [70, 33, 5], [3, 9, 5], 32, 8, 128, 32, "fp8_e4m3"),
    # at most 32 rows per (sequence, kv head) and g a power of two up to 16:
    # the balanced decode kernel in its multi-query form (16 rows per unit,
    # 16 / g tokens), including token counts that leave a unit part empty,
    # two units per kv head, long sequences whose segments are cut between
    # warps (merged by four warps of four rows), and g = 3 (the mma.sync
    # multi-token kernel)
    ("mq_g8_t3", [1500, 40, 700], [3, 1, 2], 64, 8, 128, 16, "bf16"),
    ("mq_g2_t5", [900, 33, 2100], [5, 2, 5], 16, 8, 128, 16, "bf16"),
    ("mq_g1_t4_bs8", [300, 1200], [4, 3], 8, 8, 128, 8, "bf16"),
    ("mq_d64", [400, 50, 1700], [4, 4, 2], 32, 8, 64, 16, "bf16"),
    ("mq_fp8_d64", [300, 1000], [4, 2], 32, 8, 64, 16, "fp8_e4m3"),
    ("mq_long_cut", [9000, 7000, 3], [4, 4, 3], 32, 8, 128, 16, "bf16"),
    ("mq_bs32", [100, 900], [4, 4], 32, 8, 128, 32, "bf16"),
    ("mq_g16_t2", [800, 2000, 5], [2, 2, 1], 32, 2, 128, 16, "bf16"),
    ("mq_fp8_d128", [1200, 300, 60], [4, 3, 4], 32, 8, 128, 16, "fp8_e4m3"),
    ("mq_g4_t8", [3000, 700, 9], [8, 5, 8], 32, 8, 128, 16, "bf16"),
    ("g3_small", [200, 70], [4, 3], 24, 8, 128, 16, "bf16"),
]


# calls with at least 128 rows per (sequence, kv head) run the tcgen05 kernel
# (bf16, and fp8 with head_dim 128) unless it is switched off; every case runs
# both ways
KERNELS = ["tcgen05", "mma_sync"]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_multi_matches_oracle(pkv, case, kernel):
    name, lens, q_lens, Hq, Hkv, d, bs, dt = case
    w = workloads.make_workload(name, lens, Hq, Hkv, d, bs, dt, seed=81 + len(lens))
    q, q_start = workloads.chunk_queries(w, q_lens, seed=82)
    kc, vc = gpu_caches(pkv, w)
    okc, ovc = oracle_caches(w)
    ref = multi_ref(w, okc, ovc, q, q_start)
    if kernel == "mma_sync" and dt == "fp8_e4m3" and bs != 16:
        # the mma.sync kernels serve fp8 caches of 16-token blocks only
        with pkv.tcgen05(False), pytest.raises(pkv.PkvError, match="UNSUPPORTED"):
            run_multi(pkv, w, kc, vc, q, q_start)
        return
    with pkv.tcgen05(kernel == "tcgen05"):
        if name.startswith("mq_"):  # the case exercises the multi-query decode
            assert pkv.multi_kernel_for(w.num_seqs, max(q_lens), Hq, Hkv, d, bs, dt) == "multi_query_decode"
        got = run_multi(pkv, w, kc, vc, q, q_start)
        assert_close(got, ref, TOL[dt], name)
        # a larger bound on the rows per sequence changes the grid, not the result
        got2 = run_multi(pkv, w, kc, vc, q, q_start, max_q=max(q_lens) + 37)
        assert_close(got2, ref, TOL[dt], name + " (max_q larger)")
    assert pkv.get_device_error() == 0


def test_multi_with_one_token_equals_decode(pkv):
    """One query token per sequence at its last position is decode: the two
    entry points agree to bf16 rounding on the same inputs."""
    w = workloads.make_workload("t1", [1, 16, 17, 300, 1111], 32, 8, 128, 16, "bf16", seed=91)
    kc, vc = gpu_caches(pkv, w)
    q_start = torch.arange(w.num_seqs + 1, dtype=torch.int32)
    got = run_multi(pkv, w, kc, vc, w.q, q_start)
    q = w.q.to(DEV)
    out = torch.empty_like(q)
    pkv.paged_attention_decode(out, q, kc, vc, w.block_tables.to(DEV), w.seq_lens.to(DEV), w.scale,
                               max_seq_len=w.max_seq_len)
    dec = out.float().cpu().numpy().astype(np.float64)
    assert np.abs(got - dec).max() <= 2 ** -7
    assert pkv.get_device_error() == 0


def test_multi_rows_beyond_the_bound_are_flagged(pkv):
    """A sequence with more query tokens than max_q (or than its length) is
    flagged and its rows are left as they were; the others are computed."""
    w = workloads.make_workload("bad", [40, 60], 32, 8, 128, 16, "bf16", seed=93)
    q, q_start = workloads.chunk_queries(w, [3, 9], seed=94)
    kc, vc = gpu_caches(pkv, w)
    okc, ovc = oracle_caches(w)
    ref = multi_ref(w, okc, ovc, q, q_start)
    assert pkv.get_device_error() == 0
    got = run_multi(pkv, w, kc, vc, q, q_start, max_q=4)  # sequence 1 has 9 > 4
    assert pkv.get_device_error() & pkv.DEVERR_BAD_SEQ_LEN
    assert_close(got[:3], ref[:3], TOL["bf16"], "in-bound sequence")
    assert np.isnan(got[3:]).all()


@pytest.mark.parametrize("kernel", KERNELS)
def test_multi_long_chunk_beyond_the_bound_is_flagged(pkv, kernel):
    """The same with chunks long enough for the tcgen05 kernel (at least 128
    rows per sequence and kv head)."""
    w = workloads.make_workload("bad_long", [200, 300, 150], 32, 8, 128, 16, "bf16", seed=97)
    q, q_start = workloads.chunk_queries(w, [40, 90, 33], seed=98)
    kc, vc = gpu_caches(pkv, w)
    okc, ovc = oracle_caches(w)
    ref = multi_ref(w, okc, ovc, q, q_start)
    assert pkv.get_device_error() == 0
    with pkv.tcgen05(kernel == "tcgen05"):
        got = run_multi(pkv, w, kc, vc, q, q_start, max_q=64)  # sequence 1 has 90 > 64
    assert pkv.get_device_error() & pkv.DEVERR_BAD_SEQ_LEN
    assert_close(got[:40], ref[:40], TOL["bf16"], "sequence 0")
    assert np.isnan(got[40:130]).all()
    assert_close(got[130:], ref[130:], TOL["bf16"], "sequence 2")


@pytest.mark.parametrize("kernel", KERNELS)
def test_multi_bad_block_ids_are_masked(pkv, kernel):
    """A table entry outside the pool is flagged and its positions are left
    out, by either kernel: the rows equal the oracle's over a table whose
    bad block is dropped from the attended positions."""
    w = workloads.make_workload("badid", [100, 180], 32, 8, 128, 16, "bf16", seed=99)
    q, q_start = workloads.chunk_queries(w, [40, 64], seed=100)
    kc, vc = gpu_caches(pkv, w)
    tables = w.block_tables.clone()
    tables[1, 2] = w.num_blocks + 5  # positions 32..47 of sequence 1
    assert pkv.get_device_error() == 0
    with pkv.tcgen05(kernel == "tcgen05"):
        got = run_multi(pkv, w, kc, vc, q, q_start, tables=tables)
    assert pkv.get_device_error() & pkv.DEVERR_BAD_BLOCK_ID
    okc, ovc = oracle_caches(w)
    ref = multi_ref(w, okc, ovc, q, q_start)
    assert_close(got[:40], ref[:40], TOL["bf16"], "sequence 0 untouched by the bad id")
    assert np.isfinite(got[40:]).all()


def test_tcgen05_switch(pkv):
    assert pkv.get_tcgen05()
    with pkv.tcgen05(False):
        assert not pkv.get_tcgen05()
    assert pkv.get_tcgen05()


def test_multi_invalid_calls(pkv):
    w = workloads.make_workload("inv", [8, 9], 8, 2, 64, 16, "f32", seed=95)
    q, q_start = workloads.chunk_queries(w, [2, 2], seed=96)
    kc, vc = gpu_caches(pkv, w)
    out = torch.empty((4, 8, 64), dtype=torch.float32, device=DEV)
    with pytest.raises(pkv.PkvError):  # fp32 caches: the products run on the tensor cores
        pkv.paged_attention_multi(out, q.to(DEV), q_start.to(DEV), kc, vc, w.block_tables.to(DEV),
                                  w.seq_lens.to(DEV), w.scale, max_q=2)


@pytest.mark.parametrize("which", ["verify4_llama3_8b", "prefill_chunk512"])
def test_multi_full_size(pkv, which):
    """The multi-token workloads the benchmark times (in the kernel it times:
    tcgen05 for the prefill chunks), every row against the (multi-threaded)
    oracle; the prefill chunks also through the mma.sync kernel."""
    w, q, q_start = workloads.MULTI_CONFIGS[which]()
    kc, vc = gpu_caches(pkv, w)
    okc, ovc = oracle_caches(w)
    ref = multi_ref(w, okc, ovc, q, q_start, threads=os.cpu_count() or 4)
    got = run_multi(pkv, w, kc, vc, q, q_start)
    assert_close(got, ref, TOL[w.cache_dtype], which)
    if which == "prefill_chunk512":
        with pkv.tcgen05(False):
            got = run_multi(pkv, w, kc, vc, q, q_start)
        assert_close(got, ref, TOL[w.cache_dtype], which + " (mma.sync)")
    assert pkv.get_device_error() == 0
