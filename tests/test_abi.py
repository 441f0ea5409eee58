"""The C ABI without a GPU: the library loads, exports every entry point
that include/pkv.h declares, and rejects invalid arguments on the host before
touching the device."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_22_gb300 import build
    build.build()
    import paged_kv_cache_22_gb300 as pkv
    return pkv.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pkv_kv_reshape_and_cache", "pkv_paged_attention_decode", "pkv_split_kv_reduce",
                     "pkv_gather_kv", "pkv_decode_workspace_bytes", "pkv_get_device_error"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in pkv.h but not exported"


def test_status_strings(lib):
    assert lib.pkv_status_string(0) == b"PKV_OK"
    assert lib.pkv_status_string(4) == b"PKV_ERR_WORKSPACE"
    assert lib.pkv_status_string(99) == b"PKV_ERR_UNKNOWN"


def _desc(nb=8, bs=16, hkv=2, d=128, dt=1):
    import paged_kv_cache_22_gb300 as pkv
    return pkv.CacheDesc(nb, bs, hkv, d, dt)


def test_host_validation_rejects_before_launch(lib):
    INVALID, UNSUPPORTED = 1, 2
    p = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    d = _desc()
    # head_dim 96 is outside the supported set
    bad = _desc(d=96)
    assert lib.pkv_paged_attention_decode(p, p, 1, 4, 8, p, p, ctypes.byref(bad), p, 4, p, 64,
                                          1.0, 1.0, 0, p, 1 << 20, None) == INVALID
    # Hq not a multiple of Hkv
    assert lib.pkv_paged_attention_decode(p, p, 1, 4, 3, p, p, ctypes.byref(d), p, 4, p, 64,
                                          1.0, 1.0, 0, p, 1 << 20, None) == INVALID
    # partition not a multiple of the block size
    assert lib.pkv_paged_attention_decode(p, p, 1, 4, 8, p, p, ctypes.byref(d), p, 4, p, 64,
                                          1.0, 1.0, 24, p, 1 << 20, None) == INVALID
    # q type must match the cache (bf16 cache -> bf16 q)
    assert lib.pkv_paged_attention_decode(p, p, 0, 4, 8, p, p, ctypes.byref(d), p, 4, p, 64,
                                          1.0, 1.0, 0, p, 1 << 20, None) == UNSUPPORTED
    # null cache descriptor, negative counts
    assert lib.pkv_paged_attention_decode(p, p, 1, 4, 8, p, p, None, p, 4, p, 64, 1.0, 1.0, 0, p,
                                          1 << 20, None) == INVALID
    assert lib.pkv_kv_reshape_and_cache(p, p, 1, -1, p, p, ctypes.byref(d), p, 1.0, None) == INVALID
    # fp8 needs a positive scale
    f8 = _desc(dt=2)
    assert lib.pkv_kv_reshape_and_cache(p, p, 1, 4, p, p, ctypes.byref(f8), p, 0.0, None) == INVALID
    # misaligned buffers
    odd = ctypes.c_void_p(0x1004)
    assert lib.pkv_kv_reshape_and_cache(odd, p, 1, 4, p, p, ctypes.byref(d), p, 1.0, None) == INVALID
    # empty work is a no-op
    assert lib.pkv_paged_attention_decode(None, None, 1, 0, 8, None, None, ctypes.byref(d), None, 4,
                                          None, 0, 1.0, 1.0, 0, None, 0, None) == 0
    assert lib.pkv_kv_reshape_and_cache(None, None, 1, 0, None, None, ctypes.byref(d), None, 1.0,
                                        None) == 0
    assert lib.pkv_split_kv_reduce(p, 1, p, p, p, p, 2, 8, 96, 64, 4, None) == UNSUPPORTED


def test_partition_workspace_size_formula(lib):
    # fp32 partials [B, Hq, P, d] + m and l [B, Hq, P], each region 256-byte aligned
    B, Hq, Hkv, d, L, pt = 8, 32, 8, 128, 32768, 512
    P = L // pt
    rows = B * Hq * P

    def up(x):
        return (x + 255) // 256 * 256
    want = (1 << 20) + up(rows * d * 4) + 2 * up(rows * 4)  # counters first
    assert lib.pkv_decode_workspace_bytes(B, Hq, Hkv, d, L, pt) == want
    assert lib.pkv_decode_workspace_bytes(B, Hq, 3, d, L, pt) == 0  # invalid GQA split


def test_decode_engine_switch(lib):
    import paged_kv_cache_22_gb300 as pkv
    assert pkv.get_decode_engine() == "tensor_cores"  # the default
    with pkv.decode_engine("cuda_cores"):
        assert pkv.get_decode_engine() == "cuda_cores"
        assert lib.pkv_get_decode_engine() == pkv.ENGINE_CUDA_CORES
    assert pkv.get_decode_engine() == "tensor_cores"
    assert lib.pkv_set_decode_engine(7) == 1  # unknown engine: invalid argument, no change
    assert pkv.get_decode_engine() == "tensor_cores"


def test_cascade_workspace_size_without_a_device(lib):
    # the balanced decode's share depends on the device's SM count: without a
    # device both sizes are 0 (the formula is checked on the GPU)
    B, Hq, Hkv, d, L = 256, 32, 8, 128, 2560
    if lib.pkv_decode_workspace_bytes(B, Hq, Hkv, d, L, 0) == 0:
        assert lib.pkv_cascade_workspace_bytes(B, Hq, Hkv, d, L) == 0
    assert lib.pkv_cascade_workspace_bytes(B, Hq, 3, d, L) == 0  # invalid GQA split


def test_cascade_rejects_bad_prefix_before_launch(lib):
    from paged_kv_cache_22_gb300 import CacheDesc
    INVALID, UNSUPPORTED = 1, 2
    desc = CacheDesc(num_blocks=8, block_size=16, num_kv_heads=2, head_dim=64, dtype=1)
    p = ctypes.c_void_p(256)
    for pb in (-1, 5):  # the table has 4 entries per sequence
        st = lib.pkv_cascade_decode(p, p, 1, 2, 8, p, p, ctypes.byref(desc), p, 4, p, 64, pb, 0.125, 1.0,
                                    p, 1 << 24, None)
        assert st == INVALID
    desc.dtype = 0  # fp32 caches
    st = lib.pkv_cascade_decode(p, p, 0, 2, 8, p, p, ctypes.byref(desc), p, 4, p, 64, 2, 0.125, 1.0,
                                p, 1 << 24, None)
    assert st == UNSUPPORTED


def test_multi_rejects_bad_arguments_before_launch(lib):
    from paged_kv_cache_22_gb300 import CacheDesc
    INVALID, UNSUPPORTED = 1, 2
    p = ctypes.c_void_p(256)
    desc = CacheDesc(num_blocks=8, block_size=16, num_kv_heads=2, head_dim=64, dtype=1)
    # negative sizes
    assert lib.pkv_paged_attention_multi(p, p, 1, p, -1, 4, 2, 8, p, p, ctypes.byref(desc), p, 4, p, 64,
                                         0.125, 1.0, p, 1 << 24, None) == INVALID
    assert lib.pkv_paged_attention_multi(p, p, 1, p, 2, 4, -1, 8, p, p, ctypes.byref(desc), p, 4, p, 64,
                                         0.125, 1.0, p, 1 << 24, None) == INVALID
    # rows but no bound on rows per sequence
    assert lib.pkv_paged_attention_multi(p, p, 1, p, 2, 4, 0, 8, p, p, ctypes.byref(desc), p, 4, p, 64,
                                         0.125, 1.0, p, 1 << 24, None) == INVALID
    # no query rows: nothing to do
    assert lib.pkv_paged_attention_multi(p, p, 1, p, 2, 0, 0, 8, p, p, ctypes.byref(desc), p, 4, p, 64,
                                         0.125, 1.0, p, 1 << 24, None) == 0
    # fp32 caches / fp32 q: the products run on the tensor cores
    desc.dtype = 0
    assert lib.pkv_paged_attention_multi(p, p, 0, p, 2, 4, 2, 8, p, p, ctypes.byref(desc), p, 4, p, 64,
                                         0.125, 1.0, p, 1 << 24, None) == UNSUPPORTED
    desc.dtype = 1
    assert lib.pkv_paged_attention_multi(p, p, 0, p, 2, 4, 2, 8, p, p, ctypes.byref(desc), p, 4, p, 64,
                                         0.125, 1.0, p, 1 << 24, None) == UNSUPPORTED


def test_bindings_reject_mismatched_out_and_caches_before_any_device_work():
    """The Python entry points check that out matches q and that the two
    caches agree, before anything touches the device (CPU tensors here)."""
    import torch

    import paged_kv_cache_22_gb300 as pkv
    kc = torch.zeros((8, 2, 16, 64), dtype=torch.bfloat16)
    q = torch.zeros((2, 8, 64), dtype=torch.bfloat16)
    tables = torch.zeros((2, 4), dtype=torch.int32)
    lens = torch.ones(2, dtype=torch.int32)
    bad_outs = [torch.zeros((2, 8, 64), dtype=torch.float32), torch.zeros((2, 8, 32), dtype=torch.bfloat16)]
    for out in bad_outs:
        with pytest.raises(ValueError):
            pkv.paged_attention_decode(out, q, kc, kc, tables, lens, 0.125)
        with pytest.raises(ValueError):
            pkv.cascade_decode(out, q, kc, kc, tables, lens, 1, 0.125)
        with pytest.raises(ValueError):
            pkv.paged_attention_multi(out, q, torch.tensor([0, 1, 2], dtype=torch.int32), kc, kc, tables, lens,
                                      0.125, max_q=1)
    with pytest.raises(ValueError):  # V cache of another type
        pkv.paged_attention_decode(q.clone(), q, kc, kc.to(torch.uint8), tables, lens, 0.125)


def test_multi_kernel_switch_without_a_device(lib):
    """The tcgen05 kernels (multi-token calls, cascade prefix pass) are on by default; the
    switch only records the choice (no device work)."""
    import paged_kv_cache_22_gb300 as pkv
    assert pkv.get_tcgen05()
    with pkv.tcgen05(False):
        assert not pkv.get_tcgen05()
        assert lib.pkv_get_tcgen05() == 0
    assert pkv.get_tcgen05()


def test_multi_kernel_choice_without_a_device(lib):
    """Which kernel a multi-token call runs, decided on the host: 128-row tcgen05 tiles once a
    (sequence, kv head) holds 128 query rows, the multi-query decode (16 rows per unit) for at
    most 32 rows and a power-of-two group, the mma.sync kernel otherwise."""
    import paged_kv_cache_22_gb300 as pkv

    def k(max_q, hq, hkv=8, d=128, bs=16, dt="bf16", seqs=64):
        return pkv.multi_kernel_for(seqs, max_q, hq, hkv, d, bs, dt)

    # speculative verify on Llama-3-8B heads (g = 4): 4 tokens = 16 rows, 8 tokens = 32 rows
    assert k(4, 32) == "multi_query_decode"
    assert k(8, 32) == "multi_query_decode"
    assert k(9, 32) == "mma_sync"            # 36 rows: beyond two units
    assert k(32, 32) == "tcgen05"            # 128 rows
    assert k(1, 8) == "multi_query_decode"   # g = 1
    assert k(2, 128) == "multi_query_decode"  # g = 16: one token per unit
    assert k(4, 24) == "mma_sync"            # g = 3: rows of a unit would mix kv heads' tokens
    assert k(4, 32, d=64) == "multi_query_decode"
    assert k(4, 32, d=64, bs=32) is None     # bf16, head_dim 64: blocks of 16 only
    assert k(4, 32, dt="fp8_e4m3") == "multi_query_decode"
    assert k(4, 32, dt="fp8_e4m3", bs=32) == "tcgen05"  # no mma.sync fp8 instance for 32-token blocks
    assert k(512, 32) == "tcgen05"
    assert k(512, 32, d=64, dt="fp8_e4m3") == "mma_sync"  # tcgen05 on fp8 caches: head_dim 128 only
    assert k(512, 32, d=64) == "tcgen05"
    assert k(4, 32, seqs=0) == "multi_query_decode"  # an empty batch is valid (nothing is launched)
    with pkv.tcgen05(False):
        assert k(512, 32) == "mma_sync"
        assert k(4, 32, dt="fp8_e4m3", bs=32) is None
        assert k(4, 32) == "multi_query_decode"
    assert k(4, 32, dt="f32") is None        # the products run on the tensor cores
    assert k(0, 32) is None and k(4, 30) is None  # max_q 0; Hq not a multiple of Hkv
