"""The allocation-free decode entry point, through the C ABI.

pkv_paged_attention_decode_noalloc serves callers that cannot allocate
device memory: a plugin inside a serving runtime that has reserved all of
the GPU's memory for its own pool, plain C code that is handed tensor
pointers but no allocator, or a latency-critical loop that must not touch
one.  It keeps its scratch in a fixed array the library reserves on each GPU,
and that array keeps the previous call's contents.  Every output is compared
with the oracle, call after call, in an order where a later call's merge
counters lie on bytes where an earlier call left partial results (so the
clearing at the start of each call is exercised).  This file is collected
last so that a stop-at-first-failure run has already run everything else.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import workloads
from tests._util import oracle_caches, oracle_decode

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = {"f32": 1e-5, "bf16": 1e-2, "fp8_e4m3": 5e-2}


def _noalloc_fn(pkv):
    fn = pkv.library().pkv_paged_attention_decode_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    fn.argtypes = [vp, vp, ctypes.c_int, i32, i32, vp, vp, ctypes.POINTER(pkv.CacheDesc), vp, i32,
                   vp, i32, f32, f32, vp]
    fn.restype = ctypes.c_int
    return fn


def _setup(pkv, w):
    shape = workloads.cache_shape(w)
    cdt = workloads.cache_torch_dtype(w.cache_dtype)
    kc = torch.zeros(shape, dtype=cdt, device=DEV)
    vc = torch.zeros_like(kc)
    k, v, slots = w.all_tokens()
    pkv.kv_reshape_and_cache(k.to(DEV), v.to(DEV), kc, vc, slots.to(DEV), w.kv_scale)
    return kc, vc


# In this order on the one scratch array: "long" cuts its 16 segments between
# most warps of the grid, so partial slots fill the scratch from byte 256 on;
# "wide" has 32,000 segments, whose counters (128,000 bytes) cover those
# slots, and its cut segments are among the last ones.
CASES = [
    ("long_gqa4_bf16", [6000, 5000], 32, 8, 128, 16, "bf16"),
    ("wide_gqa4_bf16", [1] * 3700 + [48] * 300, 32, 8, 64, 16, "bf16"),
    ("gqa8_fp8", [5, 700, 1500], 64, 8, 128, 16, "fp8_e4m3"),
    ("mha_f32", [1, 17, 33, 100], 4, 4, 64, 16, "f32"),
    ("long_again", [6000, 5000], 32, 8, 128, 16, "bf16"),
]


def test_noalloc_matches_oracle_call_after_call():
    import paged_kv_cache_22_gb300 as pkv
    fn = _noalloc_fn(pkv)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for i, (name, lens, Hq, Hkv, d, bs, dt) in enumerate(CASES):
        w = workloads.make_workload(name, lens, Hq, Hkv, d, bs, dt, seed=99 + i)
        kc, vc = _setup(pkv, w)
        okc, ovc = oracle_caches(w)
        ref = oracle_decode(w, okc, ovc, threads=4)
        q, tables, seq_lens = w.q.to(DEV), w.block_tables.to(DEV), w.seq_lens.to(DEV)
        desc = pkv.CacheDesc(w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim,
                             {"f32": 0, "bf16": 1, "fp8_e4m3": 2}[dt])
        qdt = 0 if dt == "f32" else 1
        for call in range(2):
            out = torch.full_like(q, float("nan"))
            st = fn(out.data_ptr(), q.data_ptr(), qdt, w.num_seqs, w.num_q_heads, kc.data_ptr(),
                    vc.data_ptr(), ctypes.byref(desc), tables.data_ptr(), w.max_blocks_per_seq,
                    seq_lens.data_ptr(), w.max_seq_len, w.scale, w.kv_scale, stream)
            assert st == 0, f"{name} call {call}: status {st}"
            torch.cuda.synchronize()
            got = out.float().cpu().numpy().astype(np.float64)
            assert np.isfinite(got).all(), f"{name} call {call}: unwritten output"
            err = float(np.abs(got - ref).max())
            assert err <= TOL[dt], f"{name} call {call}: max |noalloc - oracle| = {err}"
    assert pkv.get_device_error() == 0


def test_noalloc_refuses_problems_beyond_its_scratch():
    import paged_kv_cache_22_gb300 as pkv
    fn = _noalloc_fn(pkv)
    # 4M (sequence, kv-head) segments need 16 MiB of counters alone: refused
    # on the host before anything is enqueued (the pointers are never used)
    desc = pkv.CacheDesc(1024, 16, 8, 128, 1)
    p = ctypes.c_void_p(0x10000)
    st = fn(p, p, 1, 1 << 19, 32, p, p, ctypes.byref(desc), p, 1, p, 16, 0.1, 1.0, None)
    assert st == 4  # PKV_ERR_WORKSPACE
