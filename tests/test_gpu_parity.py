"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Cache writes and the gather are compared byte for byte; attention outputs
within the stated max-abs tolerances: 1e-5 for fp32 caches, 1e-2 for bf16 and
5e-2 for fp8-e4m3 (the oracle reads the same rounded cache contents; its own
cache write is checked bit-exact against the GPU's first).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import empty_cache_np, oracle_caches, oracle_decode, to_np

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-2, "fp8_e4m3": 5e-2}
DEV = "cuda"


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_22_gb300 as m
    m.library()
    return m


@pytest.fixture(params=["tensor_cores", "cuda_cores"])
def engine(request, pkv):
    """Runs a test once per decode engine (bf16 and fp8 caches; fp32 caches
    take the CUDA cores under both)."""
    with pkv.decode_engine(request.param):
        yield request.param


def gpu_caches(pkv, w: workloads.Workload, include_new: bool = True):
    shape = workloads.cache_shape(w)
    dt = workloads.cache_torch_dtype(w.cache_dtype)
    nbytes = int(np.prod(shape)) * torch.tensor([], dtype=dt).element_size()
    raw_k = torch.full((nbytes,), workloads.poison_bits(w.cache_dtype), dtype=torch.uint8, device=DEV)
    raw_v = raw_k.clone()
    kc, vc = raw_k.view(dt).view(shape), raw_v.view(dt).view(shape)
    if w.hist_slots.numel():
        pkv.kv_reshape_and_cache(w.hist_k.to(DEV), w.hist_v.to(DEV), kc, vc, w.hist_slots.to(DEV),
                                 w.kv_scale)
    if include_new and w.new_slots.numel():
        pkv.kv_reshape_and_cache(w.new_k.to(DEV), w.new_v.to(DEV), kc, vc, w.new_slots.to(DEV),
                                 w.kv_scale)
    return kc, vc


def run_decode(pkv, w, kc, vc, partition_tokens=0, max_seq_len=None):
    q = w.q.to(DEV)
    out = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode(out, q, kc, vc, w.block_tables.to(DEV), w.seq_lens.to(DEV), w.scale,
                               w.kv_scale, max_seq_len=max_seq_len or max(w.max_seq_len, 1),
                               partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def assert_close(got, ref, tol, what=""):
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref).max() if got.size else 0.0
    assert err <= tol, f"{what}: max |gpu - oracle| = {err:.3g} > {tol}"


def check_caches_equal(kc, vc, okc, ovc):
    gk, gv = to_np(kc), to_np(vc)
    assert gk.view(np.uint8).tobytes() == okc.view(np.uint8).tobytes(), "K cache bytes differ"
    assert gv.view(np.uint8).tobytes() == ovc.view(np.uint8).tobytes(), "V cache bytes differ"


# ------------------------------------------------------------------ cache write
@pytest.mark.parametrize("cache_dtype,src", [("f32", "f32"), ("bf16", "bf16"), ("fp8_e4m3", "bf16"),
                                             ("bf16", "f32"), ("fp8_e4m3", "f32"), ("f32", "bf16")])
@pytest.mark.parametrize("d", [64, 128])
def test_reshape_and_cache_bit_exact(pkv, cache_dtype, src, d):
    gen = torch.Generator().manual_seed(100 + d)
    T, Hkv, bs, NB = 77, 4, 16, 40
    sdt = torch.float32 if src == "f32" else torch.bfloat16
    k = (torch.randn(T, Hkv, d, generator=gen) * 3).to(sdt)
    v = (torch.randn(T, Hkv, d, generator=gen) * 3).to(sdt)
    slots = torch.randperm(NB * bs, generator=gen)[:T].to(torch.int64)
    slots[::7] = -1  # padding tokens are skipped
    kv_scale = 0.02 if cache_dtype == "fp8_e4m3" else 1.0  # drives some values into saturation
    shape = (NB, Hkv, bs, d)
    w = workloads.Workload("rc", 0, Hkv, Hkv, d, bs, NB, cache_dtype, "f32", src, None, None, None,
                           k, v, slots, k[:0], v[:0], slots[:0], 1.0, kv_scale)
    okc, ovc = empty_cache_np(w), empty_cache_np(w)
    oracle.reshape_and_cache(to_np(k), to_np(v), okc, ovc, to_np(slots), kv_scale)
    dt = workloads.cache_torch_dtype(cache_dtype)
    nbytes = int(np.prod(shape)) * torch.tensor([], dtype=dt).element_size()
    kc = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV).view(dt).view(shape)
    vc = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV).view(dt).view(shape)
    pkv.kv_reshape_and_cache(k.to(DEV), v.to(DEV), kc, vc, slots.to(DEV), kv_scale)
    torch.cuda.synchronize()
    check_caches_equal(kc, vc, okc, ovc)
    assert pkv.get_device_error() == 0


def test_reshape_and_cache_bad_slot_sets_error(pkv):
    w = workloads.make_workload("bad", [5], 2, 2, 64, 16, "bf16", seed=3, num_blocks=4)
    kc, vc = gpu_caches(pkv, w, include_new=False)
    assert pkv.get_device_error() == 0
    before = kc.clone()
    slots = torch.tensor([4 * 16 + 3], dtype=torch.int64, device=DEV)  # one past the pool
    pkv.kv_reshape_and_cache(w.new_k.to(DEV), w.new_v.to(DEV), kc, vc, slots)
    assert pkv.get_device_error() & pkv.DEVERR_BAD_SLOT
    assert torch.equal(before.view(torch.int16), kc.view(torch.int16))


# ------------------------------------------------------------------ gather
@pytest.mark.parametrize("cache_dtype", ["f32", "bf16", "fp8_e4m3"])
def test_gather_bit_exact(pkv, cache_dtype):
    d = 64 if cache_dtype == "f32" else 128
    w = workloads.make_workload("g", [1, 16, 17, 250, 0, 31], 8, 4, d, 16, cache_dtype, seed=21)
    kc, vc = gpu_caches(pkv, w)
    okc, ovc = oracle_caches(w)
    check_caches_equal(kc, vc, okc, ovc)
    ko, vo = pkv.gather_kv(kc, vc, w.block_tables.to(DEV), w.seq_lens.to(DEV), w.max_seq_len)
    rk, rv = oracle.gather_kv(okc, ovc, to_np(w.block_tables), to_np(w.seq_lens))
    torch.cuda.synchronize()
    assert to_np(ko).tobytes() == rk.tobytes() and to_np(vo).tobytes() == rv.tobytes()


# ------------------------------------------------------------------ attention, small cases
SMALL = [
    # name, lens, Hq, Hkv, d, bs, dtype
    ("mha_f32_d64", [1, 17, 33, 100], 4, 4, 64, 16, "f32"),
    ("gqa4_bf16", [1, 2, 15, 16, 17, 128, 255, 700], 32, 8, 128, 16, "bf16"),
    ("gqa8_bf16", [3, 64, 333, 1000], 64, 8, 128, 16, "bf16"),
    ("gqa2_bf16_d64", [5, 40, 129], 4, 2, 64, 16, "bf16"),
    ("mqa_g16_bf16", [7, 90, 200], 16, 1, 128, 16, "bf16"),
    ("g3_bf16", [9, 50], 6, 2, 128, 16, "bf16"),
    ("gqa4_fp8", [1, 16, 40, 517], 32, 8, 128, 16, "fp8_e4m3"),
    ("gqa8_fp8_d64", [2, 100, 300], 16, 2, 64, 16, "fp8_e4m3"),
    ("gqa4_f32_d128", [1, 33, 300], 8, 2, 128, 16, "f32"),
    ("bs8_bf16", [1, 8, 9, 300], 32, 8, 128, 8, "bf16"),
    ("bs32_bf16", [1, 32, 33, 300], 32, 8, 128, 32, "bf16"),
    ("bs32_g8_bf16", [5, 70, 400], 16, 2, 128, 32, "bf16"),
    ("bs8_g1_bf16", [3, 100], 4, 4, 128, 8, "bf16"),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
@pytest.mark.parametrize("partition_tokens", [0, 64, 512])
def test_decode_small(pkv, engine, case, partition_tokens):
    name, lens, Hq, Hkv, d, bs, dt = case
    if partition_tokens % bs:
        pytest.skip("partition must be a multiple of the block size")
    if dt == "f32" and engine == "cuda_cores":
        pytest.skip("fp32 caches take the CUDA cores under either engine")
    w = workloads.make_workload(name, lens, Hq, Hkv, d, bs, dt, seed=len(name) * 7 + Hq)
    kc, vc = gpu_caches(pkv, w)
    okc, ovc = oracle_caches(w)
    check_caches_equal(kc, vc, okc, ovc)
    ref = oracle_decode(w, okc, ovc)
    got = run_decode(pkv, w, kc, vc, partition_tokens)
    assert_close(got, ref, TOL[dt], name)
    assert pkv.get_device_error() == 0


def test_tiny_mha_config(pkv):
    w = workloads.tiny_mha()
    kc, vc = gpu_caches(pkv, w)
    okc, ovc = oracle_caches(w)
    check_caches_equal(kc, vc, okc, ovc)
    ref = oracle_decode(w, okc, ovc)
    for pt in (0, 16):
        assert_close(run_decode(pkv, w, kc, vc, pt), ref, TOL["f32"], f"tiny pt={pt}")


def test_length_one_and_zero(pkv, engine):
    w = workloads.make_workload("z", [0, 1, 0, 1, 37], 8, 2, 128, 16, "bf16", seed=5)
    kc, vc = gpu_caches(pkv, w)
    for pt in (0, 16):
        got = run_decode(pkv, w, kc, vc, pt)
        assert not got[0].any() and not got[2].any()
        # length 1: own value, up to one bf16 rounding of the output (exact here)
        nv = w.new_v.float().numpy()  # new tokens in sequence order for non-empty sequences
        assert np.array_equal(got[1], np.repeat(nv[0], 4, axis=0))
        assert np.array_equal(got[3], np.repeat(nv[1], 4, axis=0))


def test_block_permutation_invariance(pkv):
    lens = [3, 70, 300, 17]
    a = workloads.make_workload("p", lens, 32, 8, 128, 16, "bf16", seed=9, identity_tables=True,
                                num_blocks=40)
    b = workloads.make_workload("p", lens, 32, 8, 128, 16, "bf16", seed=9, num_blocks=40)
    ka, va = gpu_caches(pkv, a)
    kb, vb = gpu_caches(pkv, b)
    for pt in (0, 32):
        ga, gb = run_decode(pkv, a, ka, va, pt), run_decode(pkv, b, kb, vb, pt)
        assert np.array_equal(ga, gb), "same tokens, different placement: identical results"


def test_split_invariance(pkv, engine):
    w = workloads.make_workload("si", [1, 48, 511, 512, 513, 2000], 32, 8, 128, 16, "bf16", seed=33)
    kc, vc = gpu_caches(pkv, w)
    ref = oracle_decode(w)
    outs = [run_decode(pkv, w, kc, vc, pt) for pt in (0, 16, 512, 2048)]
    for o in outs:
        assert_close(o, ref, TOL["bf16"])
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 2e-2


@pytest.mark.parametrize("dt", ["bf16", "fp8_e4m3"])
def test_poisoned_tail_and_table_never_read(pkv, engine, dt):
    """Caches start NaN everywhere and unused table entries are out of the
    pool: a read past seq_len or past the last block would show up as a NaN
    output or a device error (the tensor-core path masks the V rows past the
    end in registers: a NaN times a zero weight would still be NaN)."""
    w = workloads.make_workload("poison", [1, 15, 17, 31, 33, 100], 16, 4, 128, 16, dt, seed=44,
                                max_blocks_per_seq=20)
    kc, vc = gpu_caches(pkv, w)
    for pt in (0, 16, 64):
        got = run_decode(pkv, w, kc, vc, pt)
        assert np.isfinite(got).all()
    assert pkv.get_device_error() == 0


def test_bad_block_id_sets_error_and_does_not_fault(pkv):
    w = workloads.make_workload("badid", [40, 40], 8, 2, 128, 16, "bf16", seed=45)
    kc, vc = gpu_caches(pkv, w)
    assert pkv.get_device_error() == 0
    tables = w.block_tables.clone()
    tables[1, 1] = w.num_blocks + 5  # outside the pool
    q = w.q.to(DEV)
    out = torch.zeros_like(q)
    pkv.paged_attention_decode(out, q, kc, vc, tables.to(DEV), w.seq_lens.to(DEV), w.scale,
                               max_seq_len=40)
    assert pkv.get_device_error() & pkv.DEVERR_BAD_BLOCK_ID
    ref = oracle_decode(w)
    assert_close(out[0].float().cpu().numpy().astype(np.float64), ref[0], TOL["bf16"], "clean row")


def test_seq_len_beyond_hint_sets_error(pkv):
    w = workloads.make_workload("hint", [100, 20], 8, 2, 128, 16, "bf16", seed=46)
    kc, vc = gpu_caches(pkv, w)
    run_decode(pkv, w, kc, vc, 0, max_seq_len=50)
    assert pkv.get_device_error() & pkv.DEVERR_BAD_SEQ_LEN


# ------------------------------------------------------------------ segments cut between warps
# Batches with more tiles than warps in the balanced grid: segments are cut
# between warps at every length, merged by the last piece to finish, and the
# merge counters must come back to zero call after call.
MEDIUM = [
    ("many_short", [37, 5, 16, 1, 90, 17] * 40, 32, 8, 128, "bf16"),
    ("skewed", [3000, 20, 1, 700, 4096, 33, 2500, 64] * 4, 32, 8, 128, "bf16"),
    ("g8_mixed", [16, 512, 1500, 3, 800, 2047] * 6, 64, 8, 128, "bf16"),
    ("fp8_mixed", [300, 1200, 17, 2100] * 10, 32, 8, 128, "fp8_e4m3"),
]


@pytest.mark.parametrize("case", MEDIUM, ids=[c[0] for c in MEDIUM])
def test_decode_medium_cut_segments(pkv, engine, case):
    name, lens, Hq, Hkv, d, dt = case
    w = workloads.make_workload(name, lens, Hq, Hkv, d, 16, dt, seed=len(lens) + Hq)
    tiles = sum(-(-L // 16) for L in lens) * Hkv * ((Hq // Hkv) // min(8, Hq // Hkv))
    kc, vc = gpu_caches(pkv, w)
    ref = oracle_decode(w, threads=8)
    for rep in range(3):  # counters must come back to zero call after call
        got = run_decode(pkv, w, kc, vc, 0)
        assert_close(got, ref, TOL[dt], f"{name} rep {rep} ({tiles} tiles)")
    assert pkv.get_device_error() == 0


# ------------------------------------------------------------------ fused step
@pytest.mark.parametrize("pt", [0, 64])
def test_decode_step_equals_write_then_decode(pkv, pt):
    w = workloads.make_workload("step", [1, 40, 700, 2000, 0, 333] * 6, 32, 8, 128, 16, "bf16",
                                seed=61)
    kc1, vc1 = gpu_caches(pkv, w, include_new=False)
    kc2, vc2 = kc1.clone(), vc1.clone()
    q, tb, ln = w.q.to(DEV), w.block_tables.to(DEV), w.seq_lens.to(DEV)
    nk, nv, ns = w.new_k.to(DEV), w.new_v.to(DEV), w.new_slots.to(DEV)
    o1 = torch.full_like(q, float("nan"))
    pkv.kv_reshape_and_cache(nk, nv, kc1, vc1, ns)
    pkv.paged_attention_decode(o1, q, kc1, vc1, tb, ln, w.scale, max_seq_len=w.max_seq_len,
                               partition_tokens=pt)
    o2 = torch.full_like(q, float("nan"))
    for _ in range(2):
        pkv.decode_step(nk, nv, ns, o2, q, kc2, vc2, tb, ln, w.scale, max_seq_len=w.max_seq_len,
                        partition_tokens=pt)
    torch.cuda.synchronize()
    assert torch.equal(kc1.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert_close(o2.float().cpu().numpy().astype(np.float64), oracle_decode(w), TOL["bf16"])
    assert pkv.get_device_error() == 0


def test_decode_step_validates_everything_before_enqueueing(pkv):
    w = workloads.make_workload("stepbad", [5, 9], 8, 2, 128, 16, "bf16", seed=62)
    kc, vc = gpu_caches(pkv, w, include_new=False)
    before = kc.clone()
    q = w.q.to(DEV)
    out = torch.zeros_like(q)
    with pytest.raises(pkv.PkvError):  # partition not a multiple of the block size
        pkv.decode_step(w.new_k.to(DEV), w.new_v.to(DEV), w.new_slots.to(DEV), out, q, kc, vc,
                        w.block_tables.to(DEV), w.seq_lens.to(DEV), w.scale, partition_tokens=24)
    torch.cuda.synchronize()
    assert torch.equal(before.view(torch.int16), kc.view(torch.int16))


# ------------------------------------------------------------------ split-KV reduce alone
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_split_kv_reduce_matches_oracle(pkv, out_dtype):
    gen = torch.Generator().manual_seed(77)
    B, Hq, P, d, pt = 5, 8, 9, 128, 64
    lens = torch.tensor([0, 1, 64, 65, 576], dtype=torch.int32)
    o = torch.randn(B, Hq, P, d, generator=gen)
    m = torch.randn(B, Hq, P, generator=gen) * 4
    l = torch.rand(B, Hq, P, generator=gen) * 30 + 0.5
    out = torch.full((B, Hq, d), float("nan"), dtype=out_dtype, device=DEV)
    pkv.split_kv_reduce(out, o.to(DEV), m.to(DEV), l.to(DEV), lens.to(DEV), pt)
    torch.cuda.synchronize()
    ref = oracle.split_kv_reduce(o.double().numpy(), m.double().numpy(), l.double().numpy(),
                                 lens.numpy(), pt)
    tol = 1e-5 if out_dtype == torch.float32 else 1e-2
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, tol, "reduce")


# ------------------------------------------------------------------ named configs
def _config(name):
    return workloads.CONFIGS[name]()


@pytest.mark.parametrize("name,pt", [("llama3_8b", 0), ("llama70b_128", 0), ("long_split_kv", 0),
                                     ("long_split_kv", 512), ("prefix_fp8", 0),
                                     ("llama3_8b", 512)])
def test_named_config_full_size(pkv, name, pt):
    """The full-size workloads in the launch configuration the benchmark
    times; every output row is checked against the (multi-threaded) oracle."""
    w = _config(name)
    kc, vc = gpu_caches(pkv, w)
    got = run_decode(pkv, w, kc, vc, pt)
    okc, ovc = oracle_caches(w)
    # spot-check the cache write bit-exactly on a sample of blocks
    sel = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(1))[:256]
    assert to_np(kc[sel.to(DEV)]).tobytes() == okc[sel.numpy()].tobytes()
    assert to_np(vc[sel.to(DEV)]).tobytes() == ovc[sel.numpy()].tobytes()
    import os
    ref = oracle_decode(w, okc, ovc, threads=os.cpu_count() or 4)
    assert_close(got, ref, TOL[w.cache_dtype], name)
    assert pkv.get_device_error() == 0


# ------------------------------------------------------------------ tensor-core specifics
@pytest.mark.parametrize("dt", ["bf16", "fp8_e4m3"])
def test_large_query_entries(pkv, engine, dt):
    """fp8 caches run q.K with fp16 operands (largest finite 65504): q entries
    far beyond that must still give the oracle's answer.  q is scaled by 2^19
    (exact in bf16) and the softmax scale by 2^-19, so the scores are those of
    an ordinary workload."""
    base = workloads.make_workload("bigq", [7, 100, 333], 16, 4, 128, 16, dt, seed=47)
    f = 2.0 ** 19
    w = dataclasses.replace(base, q=(base.q.float() * f).to(torch.bfloat16), scale=base.scale / f)
    kc, vc = gpu_caches(pkv, w)
    ref = oracle_decode(w)
    for pt in (0, 64):
        assert_close(run_decode(pkv, w, kc, vc, pt), ref, TOL[dt], f"partition_tokens {pt}")
    assert pkv.get_device_error() == 0


ROUNDING = [
    ("gqa4", [1, 2, 17, 300, 1000], 32, 8, 128, 16, "bf16"),
    ("gqa8", [3, 64, 900], 64, 8, 128, 16, "bf16"),
    ("bs8", [9, 300], 32, 8, 128, 8, "bf16"),
    ("bs32", [33, 300], 32, 8, 128, 32, "bf16"),
    ("d64", [5, 129, 400], 8, 2, 64, 16, "bf16"),
    ("fp8", [4, 77, 600], 32, 8, 128, 16, "fp8_e4m3"),
]


@pytest.mark.parametrize("pt", [0, 64])
@pytest.mark.parametrize("case", ROUNDING, ids=[c[0] for c in ROUNDING])
def test_outputs_are_correctly_rounded(pkv, engine, case, pt):
    """Accuracy of the contractions beyond the max-abs bound: the share of bf16
    outputs equal to the oracle's exact result rounded to bf16, and the
    largest distance in bf16 steps.  P reaches P.V as a head plus a remainder
    (bf16 + bf16 for bf16 caches, fp16 + fp16 for fp8 caches), about 16 or
    more significant bits per weight, so nearly every output rounds like the
    exact value."""
    name, lens, Hq, Hkv, d, bs, dt = case
    w = workloads.make_workload(name, lens, Hq, Hkv, d, bs, dt, seed=48 + len(lens))
    kc, vc = gpu_caches(pkv, w)
    ref = oracle_decode(w)
    got = run_decode(pkv, w, kc, vc, pt)
    rounded = oracle.bf16_decode(oracle.bf16_encode(ref))
    exact_share = float(np.mean(got == rounded))
    # one bf16 step at |ref|, floored at 2^-16: near zero the fp32 sums keep
    # an absolute error of a few 1e-8 that no relative bound covers
    step = np.full_like(ref, 2.0 ** -16)
    big = np.abs(ref) >= 2.0 ** -9
    step[big] = 2.0 ** (np.floor(np.log2(np.abs(ref[big]))) - 7)
    steps = float(np.max(np.abs(got - ref) / step))
    want = 0.99
    assert exact_share >= want, f"{name}: {exact_share:.4f} of outputs correctly rounded (< {want})"
    assert steps <= 1.0, f"{name}: an output is {steps:.2f} bf16 steps from the exact value"


# ------------------------------------------------------------------ out-of-pool tables at scale
@pytest.mark.parametrize("dt", ["bf16", "fp8_e4m3"])
def test_out_of_pool_tables_in_half_the_batch(pkv, dt):
    """The first half of a full-size batch has tables pointing outside the
    pool: those tiles are skipped (flagged, never read), so the warps of the
    balanced split holding them finish at once while the rest stream.  Every
    clean row must still match the oracle, call after call (the merge
    counters come back to zero)."""
    import os
    n_bad, n_good = 40, 40
    w = workloads.make_workload("halfbad", [2048] * (n_bad + n_good), 32, 8, 128, 16, dt, seed=91)
    kc, vc = gpu_caches(pkv, w)
    okc, ovc = oracle_caches(w)
    tables = w.block_tables.clone()
    used = tables[:n_bad] != workloads.UNUSED_TABLE_ENTRY
    tables[:n_bad][used] = w.num_blocks + 5
    ref = oracle.paged_attention_decode(to_np(w.q[n_bad:]), okc, ovc, to_np(w.block_tables[n_bad:]),
                                        to_np(w.seq_lens[n_bad:]), w.scale, w.kv_scale,
                                        os.cpu_count() or 4)
    q = w.q.to(DEV)
    for rep in range(3):
        out = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode(out, q, kc, vc, tables.to(DEV), w.seq_lens.to(DEV), w.scale,
                                   w.kv_scale, max_seq_len=w.max_seq_len)
        assert pkv.get_device_error() == pkv.DEVERR_BAD_BLOCK_ID
        got = out[n_bad:].float().cpu().numpy().astype(np.float64)
        assert_close(got, ref, TOL[dt], f"clean rows, call {rep}")


# ------------------------------------------------------------------ sliding window and sinks
WINDOWS = [(8, 0), (8, 4), (20, 3), (33, 16), (1, 0), (4096, 0), (200, 4)]
WIN_CASES = [
    ("w_bf16", [1, 5, 17, 40, 70, 300, 1000], 32, 8, 128, 16, "bf16"),
    ("w_fp8", [3, 33, 500], 32, 8, 128, 16, "fp8_e4m3"),
    ("w_f32", [2, 19, 260], 8, 2, 64, 16, "f32"),
    ("w_bs8_g8", [9, 130], 16, 2, 128, 8, "bf16"),
]


def window_ref(w, window, sinks, tables=None):
    okc, ovc = oracle_caches(w)
    return oracle.paged_attention_decode(to_np(w.q), okc, ovc, to_np(w.block_tables if tables is None else tables),
                                         to_np(w.seq_lens), w.scale, w.kv_scale, 4, window=window, sinks=sinks)


@pytest.mark.parametrize("pt", [0, 64])
@pytest.mark.parametrize("case", WIN_CASES, ids=[c[0] for c in WIN_CASES])
def test_sliding_window_matches_oracle(pkv, engine, case, pt):
    name, lens, Hq, Hkv, d, bs, dt = case
    if dt == "f32" and engine == "cuda_cores":
        pytest.skip("fp32 caches take the CUDA cores under either engine")
    if pt % bs:
        pytest.skip("partition must be a multiple of the block size")
    w = workloads.make_workload(name, lens, Hq, Hkv, d, bs, dt, seed=61 + len(lens))
    kc, vc = gpu_caches(pkv, w)
    q = w.q.to(DEV)
    for window, sinks in WINDOWS:
        out = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode(out, q, kc, vc, w.block_tables.to(DEV), w.seq_lens.to(DEV), w.scale,
                                   w.kv_scale, max_seq_len=w.max_seq_len, partition_tokens=pt,
                                   window=window, sinks=sinks)
        got = out.float().cpu().numpy().astype(np.float64)
        assert_close(got, window_ref(w, window, sinks), TOL[dt], f"{name} window {window} sinks {sinks}")
    assert pkv.get_device_error() == 0


@pytest.mark.parametrize("pt", [0, 32])
def test_sliding_window_never_reads_blocks_left_out(pkv, engine, pt):
    """Blocks holding no attended token may have been freed: their table
    entries point outside the pool and the caches there are NaN; nothing is
    flagged and the output is the oracle's."""
    w = workloads.make_workload("wfree", [100, 333, 1000, 47], 32, 8, 128, 16, "bf16", seed=66,
                                max_blocks_per_seq=70)
    kc, vc = gpu_caches(pkv, w)
    window, sinks, bs = 64, 4, w.block_size
    tables = w.block_tables.clone()
    for s, L in enumerate(w.seq_lens.tolist()):
        for j in range(-(-L // bs)):
            toks = range(j * bs, min(L, (j + 1) * bs))
            if not any(L <= window or p < sinks or p >= L - window for p in toks):
                tables[s, j] = w.num_blocks + 9
    ref = window_ref(w, window, sinks)
    q = w.q.to(DEV)
    out = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode(out, q, kc, vc, tables.to(DEV), w.seq_lens.to(DEV), w.scale,
                               max_seq_len=w.max_seq_len, partition_tokens=pt, window=window, sinks=sinks)
    assert pkv.get_device_error() == 0
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, TOL["bf16"], "window with freed blocks")


# ------------------------------------------------------------------ failure path of the bounded waits
def test_bounded_wait_gives_up_and_the_context_stays_usable(pkv):
    """A wait on an mbarrier whose bytes never arrive (no copy is issued, so
    none is left in flight) gives up after its probe limit, sets
    DEVERR_WAIT_TIMEOUT and returns; the next decode still matches the
    oracle and raises nothing."""
    assert pkv.get_device_error() == 0
    pkv.selftest_wait_timeout()
    assert pkv.get_device_error() == pkv.DEVERR_WAIT_TIMEOUT
    w = workloads.make_workload("after_timeout", [1, 40, 300], 32, 8, 128, 16, "bf16", seed=111)
    kc, vc = gpu_caches(pkv, w)
    assert_close(run_decode(pkv, w, kc, vc), oracle_decode(w), TOL["bf16"], "decode after the timeout")
    assert pkv.get_device_error() == 0


@pytest.mark.parametrize("Hq,Hkv,dt", [(8, 8, "bf16"), (24, 8, "bf16"), (8, 8, "fp8_e4m3"), (4, 4, "f32"),
                                       (40, 8, "bf16")])
def test_one_head_units_with_cut_segments(pkv, engine, Hq, Hkv, dt):
    """Group sizes whose units hold one query head (g = 1, 3, 5): a few long
    sequences, so most segments are cut between warps and merged from their
    partial slots."""
    d = 64 if dt == "f32" else 128
    w = workloads.make_workload(f"g{Hq // Hkv}_{dt}", [6000, 3000, 17, 4500], Hq, Hkv, d, 16, dt, seed=121)
    kc, vc = gpu_caches(pkv, w)
    okc, ovc = oracle_caches(w)
    ref = oracle_decode(w, okc, ovc, threads=4)
    assert_close(run_decode(pkv, w, kc, vc), ref, TOL[dt], f"g={Hq // Hkv} {dt}")
    assert pkv.get_device_error() == 0
