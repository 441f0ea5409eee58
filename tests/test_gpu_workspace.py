"""One decode workspace reused across calls of different sizes.

The balanced decode keeps one merge counter per (sequence, kv-head unit)
segment at the start of the workspace, in a region of at least 1 MiB, and its
partial results after that region.  A batch with more than 262,144 segments
needs a larger counter region, which covers bytes where a smaller call left
partials.  The library must clear that region itself, so that a workspace
zero-filled once serves any sequence of calls: large batch, then a small one
(and a multi-token call, whose partials also start at 1 MiB), then the large
batch again, each compared with the oracle.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import oracle_caches, oracle_decode, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = {"f32": 1e-5, "bf16": 1e-2, "fp8_e4m3": 5e-2}


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_22_gb300 as m
    m.library()
    return m


def _caches(pkv, w):
    shape = workloads.cache_shape(w)
    dt = workloads.cache_torch_dtype(w.cache_dtype)
    kc = torch.full(shape, float("nan"), dtype=dt, device=DEV)
    vc = torch.full(shape, float("nan"), dtype=dt, device=DEV)
    k, v, slots = w.all_tokens()
    pkv.kv_reshape_and_cache(k.to(DEV), v.to(DEV), kc, vc, slots.to(DEV), w.kv_scale)
    return kc, vc


def _decode(pkv, w, kc, vc, ws):
    q = w.q.to(DEV)
    out = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode(out, q, kc, vc, w.block_tables.to(DEV), w.seq_lens.to(DEV), w.scale,
                               w.kv_scale, max_seq_len=w.max_seq_len, workspace=ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def _close(got, ref, tol, what):
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = float(np.abs(got - ref).max())
    assert err <= tol, f"{what}: max |gpu - oracle| = {err:.3g} > {tol}"


def test_large_small_large_batches_share_one_workspace(pkv):
    # 8,500 sequences x 32 kv-head units = 272,000 segments: a counter region
    # of 1,088,000 bytes.  The last 300 sequences span 4 blocks each, so the
    # segments cut between warps -- whose counters are read -- include ones
    # at indices past 262,144, in the bytes beyond the first 1 MiB.
    lens = [1] * 8200 + [64] * 300
    big = workloads.make_workload("big", lens, 32, 32, 64, 16, "bf16", seed=501)
    assert big.num_seqs * 32 * 4 > (1 << 20)
    # two long sequences: ~19 warps per segment, so most warps of the grid
    # write partial slots, starting at 1 MiB
    small = workloads.make_workload("small", [5000, 4000], 32, 32, 64, 16, "bf16", seed=502)
    ws = pkv.DecodeWorkspace(torch.device(DEV))

    bkc, bvc = _caches(pkv, big)
    okc, ovc = oracle_caches(big)
    ref_big = oracle_decode(big, okc, ovc)
    _close(_decode(pkv, big, bkc, bvc, ws), ref_big, TOL["bf16"], "large batch, fresh workspace")

    skc, svc = _caches(pkv, small)
    sokc, sovc = oracle_caches(small)
    _close(_decode(pkv, small, skc, svc, ws), oracle_decode(small, sokc, sovc), TOL["bf16"], "small batch")

    # a multi-token call on the same workspace, on the kernel that cuts each
    # sequence's K/V range (its partials also start at 1 MiB)
    q, q_start = workloads.chunk_queries(small, [300, 200], seed=503)
    out = torch.full(q.shape, float("nan"), dtype=q.dtype, device=DEV)
    with pkv.tcgen05(False):
        pkv.paged_attention_multi(out, q.to(DEV), q_start.to(DEV), skc, svc, small.block_tables.to(DEV),
                                  small.seq_lens.to(DEV), small.scale, max_q=300, workspace=ws)
    torch.cuda.synchronize()
    ref_multi = oracle.paged_attention_multi(to_np(q), to_np(q_start), sokc, sovc, to_np(small.block_tables),
                                             to_np(small.seq_lens), small.scale, small.kv_scale, 4)
    _close(out.float().cpu().numpy().astype(np.float64), ref_multi, TOL["bf16"], "multi-token call")

    for rep in range(2):
        _close(_decode(pkv, big, bkc, bvc, ws), ref_big, TOL["bf16"], f"large batch again ({rep})")
    assert pkv.get_device_error() == 0
