"""Plain fp64 CPU oracle for paged decode attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this package; the product path
(``paged_kv_cache_22_gb300``) never does, and the two share no code.

The arithmetic lives in ``pkv_oracle.c`` (plain loops, double precision),
compiled with gcc into ``_build/liboracle.so`` on first use.  This module only
marshals numpy arrays into it.  Array conventions:

* fp32 tensors are ``np.float32``; bf16 tensors are their raw bit patterns as
  ``np.uint16``; fp8-e4m3 tensors are their codes as ``np.uint8``.
* caches are ``[num_blocks, num_kv_heads, block_size, head_dim]``;
  ``q`` is ``[num_seqs, num_q_heads, head_dim]``;
  ``block_tables`` is ``int32 [num_seqs, max_blocks_per_seq]``;
  ``seq_lens`` is ``int32 [num_seqs]``; ``slot_mapping`` is ``int64``.

Which passage of the source pages each routine follows is stated in the C
file's header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, BF16, FP8_E4M3 = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, no vector intrinsics)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            c_int, c_f, c_d, vp = ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_void_p
            lib.orc_bf16_decode.restype = c_d
            lib.orc_bf16_decode.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_encode.restype = ctypes.c_uint16
            lib.orc_bf16_encode.argtypes = [c_f]
            lib.orc_fp8_e4m3_decode.restype = c_d
            lib.orc_fp8_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.orc_fp8_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_fp8_e4m3_encode.argtypes = [c_f]
            lib.orc_reshape_and_cache.restype = c_int
            lib.orc_reshape_and_cache.argtypes = [vp, vp, c_int, c_int, c_int, c_int, vp, vp,
                                                  c_int, c_int, c_int, vp, c_f]
            lib.orc_copy_blocks.restype = c_int
            lib.orc_copy_blocks.argtypes = [vp, vp, c_int, vp, vp, c_int, c_int, c_int, c_int, c_int,
                                            vp, c_int]
            lib.orc_gather_kv.restype = c_int
            lib.orc_gather_kv.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int,
                                          vp, c_int, vp, vp, c_int]
            lib.orc_paged_attention_decode_window.restype = c_int
            lib.orc_paged_attention_decode_window.argtypes = [vp, vp, c_int, c_int, c_int, vp, vp,
                                                              c_int, c_int, c_int, c_int, c_int, vp,
                                                              c_int, vp, c_d, c_d, c_int, c_int,
                                                              c_int]
            lib.orc_paged_attention_decode.restype = c_int
            lib.orc_paged_attention_decode.argtypes = [vp, vp, c_int, c_int, c_int, vp, vp, c_int,
                                                       c_int, c_int, c_int, c_int, vp, c_int, vp,
                                                       c_d, c_d, c_int]
            lib.orc_partition_attention.restype = c_int
            lib.orc_paged_attention_multi.argtypes = [vp, vp, c_int, vp, c_int, c_int, vp, vp, c_int,
                                                      c_int, c_int, c_int, c_int, vp, c_int, vp,
                                                      c_d, c_d, c_int]
            lib.orc_partition_attention.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, vp, vp,
                                                    c_int, c_int, c_int, c_int, c_int, vp, c_int,
                                                    vp, c_d, c_d, c_int, c_int, c_int]
            lib.orc_split_kv_reduce.restype = c_int
            lib.orc_split_kv_reduce.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int,
                                                c_int]
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise OracleError(f"oracle {what} failed with code {rc}")


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.uint8:
        return FP8_E4M3
    raise TypeError(f"unsupported oracle array dtype {a.dtype}")


# ---------------------------------------------------------------- element types
def bf16_decode(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.orc_bf16_decode(int(b)) for b in flat]).reshape(np.shape(bits))


def bf16_encode(x: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    return np.array([lib.orc_bf16_encode(float(v)) for v in flat],
                    dtype=np.uint16).reshape(np.shape(x))


def fp8_e4m3_decode(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.orc_fp8_e4m3_decode(int(c)) for c in flat]).reshape(np.shape(codes))


def fp8_e4m3_encode(x: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    return np.array([lib.orc_fp8_e4m3_encode(float(v)) for v in flat],
                    dtype=np.uint8).reshape(np.shape(x))


# ---------------------------------------------------------------- cache write / gather
def reshape_and_cache(k: np.ndarray, v: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                      slot_mapping: np.ndarray, kv_scale: float = 1.0) -> None:
    """Scatter k, v ``[T, Hkv, d]`` into the caches in place (slot < 0 skipped)."""
    lib = _load()
    T, Hkv, d = k.shape
    NB, Hkv2, bs, d2 = k_cache.shape
    if (Hkv, d) != (Hkv2, d2) or v.shape != k.shape or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    _check(lib.orc_reshape_and_cache(_ptr(k), _ptr(v), dtype_code(k), T, Hkv, d, _ptr(k_cache),
                                     _ptr(v_cache), dtype_code(k_cache), NB, bs, _ptr(slots),
                                     float(kv_scale)), "reshape_and_cache")


def gather_kv(k_cache: np.ndarray, v_cache: np.ndarray, block_tables: np.ndarray,
              seq_lens: np.ndarray):
    """Contiguous ``[sum(seq_lens), Hkv, d]`` copies of every sequence's K and V."""
    lib = _load()
    NB, Hkv, bs, d = k_cache.shape
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    cu = np.zeros(len(lens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lens)
    k_out = np.zeros((int(cu[-1]), Hkv, d), dtype=k_cache.dtype)
    v_out = np.zeros_like(k_out)
    _check(lib.orc_gather_kv(_ptr(k_out), _ptr(v_out), _ptr(k_cache), _ptr(v_cache),
                             dtype_code(k_cache), NB, Hkv, bs, d, _ptr(tables), tables.shape[1],
                             _ptr(lens), _ptr(cu), len(lens)), "gather_kv")
    return k_out, v_out


def copy_blocks(k_dst: np.ndarray, v_dst: np.ndarray, k_src: np.ndarray, v_src: np.ndarray,
                pairs: np.ndarray) -> None:
    """In place: block ``pairs[i, 0]`` of the source pool replaces block
    ``pairs[i, 1]`` of the destination pool, K and V, pairs in order."""
    lib = _load()
    if k_dst.dtype != k_src.dtype or k_dst.shape[1:] != k_src.shape[1:]:
        raise ValueError("pools differ in block geometry or element type")
    NB_d, Hkv, bs, d = k_dst.shape
    pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    _check(lib.orc_copy_blocks(_ptr(k_dst), _ptr(v_dst), NB_d, _ptr(k_src), _ptr(v_src),
                               k_src.shape[0], dtype_code(k_src), Hkv, bs, d, _ptr(pr), pr.shape[0]),
           "copy_blocks")


# ---------------------------------------------------------------- attention
def paged_attention_decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                           block_tables: np.ndarray, seq_lens: np.ndarray, scale: float,
                           kv_scale: float = 1.0, threads: int = 1, window: int = 0,
                           sinks: int = 0) -> np.ndarray:
    """fp64 ``[B, Hq, d]`` decode attention over each sequence's paged K/V.
    ``window > 0``: a sequence of length L attends only its first ``sinks``
    and last ``window`` tokens."""
    lib = _load()
    B, Hq, d = q.shape
    NB, Hkv, bs, d2 = k_cache.shape
    if d != d2:
        raise ValueError("head_dim mismatch")
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((B, Hq, d), dtype=np.float64)
    _check(lib.orc_paged_attention_decode_window(
        _ptr(out), _ptr(q), dtype_code(q), B, Hq, _ptr(k_cache), _ptr(v_cache), dtype_code(k_cache),
        NB, Hkv, bs, d, _ptr(tables), tables.shape[1], _ptr(lens), float(scale), float(kv_scale),
        int(window), int(sinks), int(threads)), "paged_attention_decode")
    return out


def paged_attention_multi(q: np.ndarray, q_start: np.ndarray, k_cache: np.ndarray,
                          v_cache: np.ndarray, block_tables: np.ndarray, seq_lens: np.ndarray,
                          scale: float, kv_scale: float = 1.0, threads: int = 1) -> np.ndarray:
    """fp64 ``[total, Hq, d]`` attention of several query tokens per sequence:
    sequence s owns rows ``q_start[s] .. q_start[s+1]-1`` of ``q [total, Hq,
    d]``, its last positions; query token i attends positions
    ``0 .. seq_lens[s] - T + i`` (causal inside the chunk)."""
    lib = _load()
    total, Hq, d = q.shape
    NB, Hkv, bs, d2 = k_cache.shape
    if d != d2:
        raise ValueError("head_dim mismatch")
    starts = np.ascontiguousarray(q_start, dtype=np.int32)
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = lens.shape[0]
    if starts.shape[0] != B + 1 or int(starts[-1]) != total:
        raise ValueError("q_start must have num_seqs + 1 entries ending at the number of query rows")
    out = np.zeros((total, Hq, d), dtype=np.float64)
    _check(lib.orc_paged_attention_multi(
        _ptr(out), _ptr(q), dtype_code(q), _ptr(starts), B, Hq, _ptr(k_cache), _ptr(v_cache),
        dtype_code(k_cache), NB, Hkv, bs, d, _ptr(tables), tables.shape[1], _ptr(lens), float(scale),
        float(kv_scale), int(threads)), "paged_attention_multi")
    return out


def partition_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                        block_tables: np.ndarray, seq_lens: np.ndarray, scale: float,
                        kv_scale: float, partition_tokens: int, max_partitions: int,
                        threads: int = 1):
    """Per-partition ``(o [B,Hq,P,d], m [B,Hq,P], l [B,Hq,P])`` in fp64."""
    lib = _load()
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    o = np.zeros((B, Hq, max_partitions, d), dtype=np.float64)
    m = np.zeros((B, Hq, max_partitions), dtype=np.float64)
    l = np.zeros((B, Hq, max_partitions), dtype=np.float64)
    _check(lib.orc_partition_attention(_ptr(o), _ptr(m), _ptr(l), _ptr(q), dtype_code(q), B, Hq,
                                       _ptr(k_cache), _ptr(v_cache), dtype_code(k_cache), NB, Hkv,
                                       bs, d, _ptr(tables), tables.shape[1], _ptr(lens),
                                       float(scale), float(kv_scale), int(partition_tokens),
                                       int(max_partitions), int(threads)), "partition_attention")
    return o, m, l


def split_kv_reduce(o_part: np.ndarray, m_part: np.ndarray, l_part: np.ndarray,
                    seq_lens: np.ndarray, partition_tokens: int) -> np.ndarray:
    """Log-sum-exp merge of partition partials into fp64 ``[B, Hq, d]``."""
    lib = _load()
    B, Hq, P, d = o_part.shape
    o = np.ascontiguousarray(o_part, dtype=np.float64)
    m = np.ascontiguousarray(m_part, dtype=np.float64)
    l = np.ascontiguousarray(l_part, dtype=np.float64)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((B, Hq, d), dtype=np.float64)
    _check(lib.orc_split_kv_reduce(_ptr(out), _ptr(o), _ptr(m), _ptr(l), _ptr(lens), B, Hq, d,
                                   int(partition_tokens), P), "split_kv_reduce")
    return out
