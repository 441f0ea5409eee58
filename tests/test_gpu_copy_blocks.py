"""Parity of pkv_copy_blocks (copy-on-write within a pool, swap to a pinned
host pool and back) with the oracle's block copy: byte for byte."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_22_gb300 as m
    m.library()
    return m


def random_pool(nb, hkv, bs, d, dtype, seed, device):
    """A pool of random bytes (any bit pattern: the copy is byte-exact)."""
    g = torch.Generator().manual_seed(seed)
    n = nb * hkv * bs * d * torch.tensor([], dtype=dtype).element_size()
    raw = torch.randint(0, 256, (n,), generator=g, dtype=torch.uint8)
    t = raw.view(dtype).view(nb, hkv, bs, d)
    return t.to(device) if device == DEV else t.pin_memory()


def oracle_view(t: torch.Tensor) -> np.ndarray:
    return to_np(t)


def same_bytes(a: np.ndarray, b: np.ndarray) -> bool:
    """Byte equality (random fp32 bit patterns include NaNs, which never
    compare equal as floats)."""
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))


def cow_pairs(nb, n, seed):
    """n (src, dst) pairs: distinct destinations that are nobody's source."""
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(nb, generator=g)
    src, dst = perm[:n], perm[n:2 * n]
    return torch.stack([src, dst], 1).to(torch.int64)


@pytest.mark.parametrize("dtype,hkv,bs,d", [(torch.bfloat16, 8, 16, 128), (torch.uint8, 8, 16, 128),
                                              (torch.float32, 4, 16, 64), (torch.bfloat16, 2, 8, 128),
                                              (torch.bfloat16, 8, 32, 128)])
def test_copy_on_write_within_pool(pkv, dtype, hkv, bs, d):
    nb = 300
    kc = random_pool(nb, hkv, bs, d, dtype, 1, DEV)
    vc = random_pool(nb, hkv, bs, d, dtype, 2, DEV)
    pairs = cow_pairs(nb, 97, 3)
    ok, ov = oracle_view(kc), oracle_view(vc)
    oracle.copy_blocks(ok, ov, ok, ov, pairs.numpy())
    pkv.copy_blocks(kc, vc, kc, vc, pairs.to(DEV))
    assert pkv.get_device_error() == 0
    assert same_bytes(oracle_view(kc), ok) and same_bytes(oracle_view(vc), ov)


def test_swap_out_to_pinned_host_and_back(pkv):
    nb, host_nb, hkv, bs, d = 200, 64, 8, 16, 128
    kc = random_pool(nb, hkv, bs, d, torch.bfloat16, 4, DEV)
    vc = random_pool(nb, hkv, bs, d, torch.bfloat16, 5, DEV)
    hk = torch.zeros((host_nb, hkv, bs, d), dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    out_pairs = torch.stack([torch.arange(10, 60), torch.arange(0, 50)], 1).to(torch.int64)
    ok, ov, ohk, ohv = oracle_view(kc), oracle_view(vc), oracle_view(hk), oracle_view(hv)
    oracle.copy_blocks(ohk, ohv, ok, ov, out_pairs.numpy())
    pkv.copy_blocks(hk, hv, kc, vc, out_pairs.to(DEV))  # device -> pinned host
    torch.cuda.synchronize()
    assert same_bytes(oracle_view(hk), ohk) and same_bytes(oracle_view(hv), ohv)
    # back into other device blocks, the pairs themselves in pinned memory
    in_pairs = torch.stack([torch.arange(0, 50), torch.arange(150, 200)], 1).to(torch.int64).pin_memory()
    oracle.copy_blocks(ok, ov, ohk, ohv, in_pairs.numpy())
    pkv.copy_blocks(kc, vc, hk, hv, in_pairs)
    assert pkv.get_device_error() == 0
    assert same_bytes(oracle_view(kc), ok) and same_bytes(oracle_view(vc), ov)


def test_bad_block_id_is_skipped_and_flagged(pkv):
    nb = 40
    kc = random_pool(nb, 2, 16, 64, torch.bfloat16, 6, DEV)
    vc = random_pool(nb, 2, 16, 64, torch.bfloat16, 7, DEV)
    good = torch.tensor([[1, 2], [3, 4]], dtype=torch.int64)
    bad = torch.tensor([[5, nb], [-1, 6]], dtype=torch.int64)
    ok, ov = oracle_view(kc), oracle_view(vc)
    oracle.copy_blocks(ok, ov, ok, ov, good.numpy())
    pkv.copy_blocks(kc, vc, kc, vc, torch.cat([good, bad]).to(DEV))
    assert pkv.get_device_error() & pkv.DEVERR_BAD_BLOCK_ID
    assert same_bytes(oracle_view(kc), ok) and same_bytes(oracle_view(vc), ov)


def test_copy_then_decode_reads_the_copy(pkv):
    """After a copy-on-write, a decode through the rewritten table gives the
    same result as through the shared block (the tables only change where
    the block lives)."""
    w = workloads.make_workload("cow", [40, 70], 8, 2, 128, 16, "bf16", seed=21, num_blocks=64)
    shape = workloads.cache_shape(w)
    kc = torch.zeros(shape, dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    k, v, s = w.all_tokens()
    pkv.kv_reshape_and_cache(k.to(DEV), v.to(DEV), kc, vc, s.to(DEV), 1.0)
    tables = w.block_tables.clone()
    used = set(tables[tables != workloads.UNUSED_TABLE_ENTRY].tolist())
    free = [b for b in range(w.num_blocks) if b not in used]
    src = int(tables[1, 2])
    pkv.copy_blocks(kc, vc, kc, vc, torch.tensor([[src, free[0]]], dtype=torch.int64, device=DEV))
    q = w.q.to(DEV)
    out_a, out_b = torch.empty_like(q), torch.empty_like(q)
    lens = w.seq_lens.to(DEV)
    pkv.paged_attention_decode(out_a, q, kc, vc, tables.to(DEV), lens, w.scale, max_seq_len=w.max_seq_len)
    tables[1, 2] = free[0]
    pkv.paged_attention_decode(out_b, q, kc, vc, tables.to(DEV), lens, w.scale, max_seq_len=w.max_seq_len)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    assert pkv.get_device_error() == 0


def test_empty_and_invalid_calls(pkv):
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16, device=DEV)
    pkv.copy_blocks(kc, kc, kc, kc, torch.zeros((0, 2), dtype=torch.int64, device=DEV))
    other = torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(pkv.PkvError):
        pkv.copy_blocks(other, other, kc, kc, torch.tensor([[0, 1]], dtype=torch.int64, device=DEV))
