"""GB300 (sm_103a) paged KV-cache decode: a thin Python binding over libpkv.so.

Every function here only marshals torch tensors into the C ABI declared in
``include/pkv.h`` (pointers, sizes, the current CUDA stream); all work runs in
the library's CUDA kernels.  There is no CPU fallback: if ``libpkv.so`` has
not been built, every call raises.

Entry points (same names as the C ABI, without the ``pkv_`` prefix):

* :func:`kv_reshape_and_cache` -- write new K/V tokens into their slots;
* :func:`paged_attention_decode` -- one decode step of attention over the
  paged cache (balanced split with an in-kernel merge, or fixed partitions
  followed by :func:`split_kv_reduce`);
* :func:`decode_step` -- both of the above for one decode step, the decode
  overlapping its prologue with the cache write;
* :func:`split_kv_reduce` -- log-sum-exp merge of partition partials;
* :func:`gather_kv` -- contiguous copy of every sequence's cached tokens;
* :func:`copy_blocks` -- whole-block copies between pools (copy-on-write of a
  shared block, swap to pinned host memory and back);
* :func:`decode_workspace_bytes`, :func:`get_device_error`;
* :func:`set_decode_engine` / :func:`get_decode_engine` (and the
  :func:`decode_engine` context manager) -- tensor cores (default) or CUDA
  cores for the contractions of bf16 and fp8 decodes;
* :func:`set_tcgen05` / :func:`get_tcgen05` (and the :func:`tcgen05`
  context manager) -- whether multi-token calls and cascade prefix passes
  with 128-row tiles take the tcgen05 kernels.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from typing import Optional

import torch

__all__ = [
    "PkvError", "CacheDesc", "kv_reshape_and_cache", "paged_attention_decode", "decode_step",
    "split_kv_reduce", "cascade_decode", "cascade_workspace_bytes", "paged_attention_multi",
    "multi_workspace_bytes", "multi_kernel_for", "MULTI_KERNELS",
    "gather_kv", "copy_blocks", "decode_workspace_bytes", "get_device_error", "library", "library_path",
    "DecodeWorkspace", "F32", "BF16", "FP8_E4M3", "DEVERR_BAD_BLOCK_ID", "DEVERR_BAD_SLOT",
    "DEVERR_BAD_SEQ_LEN", "DEVERR_WAIT_TIMEOUT", "DEVERR_SMEM_ALIGN", "set_decode_engine",
    "get_decode_engine", "decode_engine", "ENGINE_TENSOR_CORES", "ENGINE_CUDA_CORES",
    "set_tcgen05", "get_tcgen05", "tcgen05", "selftest_wait_timeout",
]

F32, BF16, FP8_E4M3 = 0, 1, 2
DEVERR_BAD_BLOCK_ID, DEVERR_BAD_SLOT, DEVERR_BAD_SEQ_LEN, DEVERR_WAIT_TIMEOUT = 0x1, 0x2, 0x4, 0x8
DEVERR_SMEM_ALIGN = 0x10
ENGINE_TENSOR_CORES, ENGINE_CUDA_CORES = 0, 1
_ENGINES = {"tensor_cores": ENGINE_TENSOR_CORES, "cuda_cores": ENGINE_CUDA_CORES}

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libpkv.so")
_lib = None
_lock = threading.Lock()

_STATUS = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED", 3: "PKV_ERR_CUDA",
           4: "PKV_ERR_WORKSPACE"}


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_STATUS.get(status, status)}")
        self.status = status


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int)]


def library() -> ctypes.CDLL:
    """Load libpkv.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(library_path):
            raise RuntimeError(f"{library_path} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(library_path)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        desc = ctypes.POINTER(CacheDesc)
        sigs = {
            "pkv_kv_reshape_and_cache": [vp, vp, ctypes.c_int, i32, vp, vp, desc, vp, f32, vp],
            "pkv_decode_workspace_bytes": [i32, i32, i32, i32, i32, i32],
            "pkv_paged_attention_decode": [vp, vp, ctypes.c_int, i32, i32, vp, vp, desc, vp, i32, vp,
                                           i32, f32, f32, i32, vp, sz, vp],
            "pkv_paged_attention_decode_window": [vp, vp, ctypes.c_int, i32, i32, vp, vp, desc, vp, i32,
                                                  vp, i32, f32, f32, i32, i32, i32, vp, sz, vp],
            "pkv_split_kv_reduce": [vp, ctypes.c_int, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp],
            "pkv_gather_kv": [vp, vp, vp, vp, desc, vp, i32, vp, vp, i32, i32, vp],
            "pkv_decode_step": [vp, vp, ctypes.c_int, i32, vp, vp, vp, desc, vp, vp, ctypes.c_int, i32,
                                i32, vp, i32, vp, i32, f32, f32, i32, vp, sz, vp],
            "pkv_cascade_workspace_bytes": [i32, i32, i32, i32, i32],
            "pkv_cascade_decode": [vp, vp, ctypes.c_int, i32, i32, vp, vp, desc, vp, i32, vp, i32, i32,
                                   f32, f32, vp, sz, vp],
            "pkv_multi_workspace_bytes": [i32, i32, i32, i32, i32, i32],
            "pkv_paged_attention_multi": [vp, vp, ctypes.c_int, vp, i32, i32, i32, i32, vp, vp, desc, vp, i32,
                                          vp, i32, f32, f32, vp, sz, vp],
            "pkv_get_device_error": [ctypes.POINTER(ctypes.c_uint32), vp],
            "pkv_copy_blocks": [vp, vp, desc, vp, vp, desc, vp, i32, vp],
            "pkv_status_string": [ctypes.c_int],
            "pkv_device_sm_count": [],
            "pkv_set_decode_engine": [ctypes.c_int],
            "pkv_get_decode_engine": [],
            "pkv_get_tcgen05": [],
            "pkv_selftest_wait_timeout": [vp],
            "pkv_multi_kernel_for": [i32, i32, i32, desc],
        }
        for name, args in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.pkv_decode_workspace_bytes.restype = sz
        lib.pkv_cascade_workspace_bytes.restype = sz
        lib.pkv_multi_workspace_bytes.restype = sz
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_set_tcgen05.argtypes = [i32]
        lib.pkv_set_tcgen05.restype = None
        _lib = lib
        return lib


# ------------------------------------------------------------------ marshalling
_CACHE_DT = {torch.float32: F32, torch.bfloat16: BF16, torch.uint8: FP8_E4M3}


def _dt(t: torch.Tensor) -> int:
    try:
        return _CACHE_DT[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on the CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _desc(k_cache: torch.Tensor, cache_dtype: Optional[int]) -> CacheDesc:
    if k_cache.dim() != 4:
        raise ValueError("caches are [num_blocks, num_kv_heads, block_size, head_dim]")
    nb, hkv, bs, d = k_cache.shape
    dt = _dt(k_cache) if cache_dtype is None else cache_dtype
    return CacheDesc(nb, bs, hkv, d, dt)


def _same_layout(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor) -> None:
    """The library writes `out` in q's type and shape and reads both caches
    with one descriptor: catch mismatches before anything is enqueued."""
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError(f"out must match q: got {tuple(out.shape)} {out.dtype}, q is {tuple(q.shape)} {q.dtype}")
    if v_cache.shape != k_cache.shape or v_cache.dtype != k_cache.dtype:
        raise ValueError("k_cache and v_cache must have the same shape and dtype")


def _check(status: int, what: str) -> None:
    if status != 0:
        raise PkvError(status, what)


# ------------------------------------------------------------------ entry points
def set_decode_engine(engine) -> None:
    """Run the contractions of bf16 / fp8 decodes on ``"tensor_cores"``
    (default) or ``"cuda_cores"`` (also accepts the ENGINE_* integers);
    process-wide, for calls issued afterwards."""
    code = _ENGINES.get(engine, engine)
    _check(library().pkv_set_decode_engine(int(code)), "set_decode_engine")


def get_decode_engine() -> str:
    code = library().pkv_get_decode_engine()
    return {v: k for k, v in _ENGINES.items()}[code]


@contextlib.contextmanager
def decode_engine(engine):
    """Temporarily select a decode engine (see :func:`set_decode_engine`)."""
    prev = get_decode_engine()
    set_decode_engine(engine)
    try:
        yield
    finally:
        set_decode_engine(prev)


def set_tcgen05(enable: bool) -> None:
    """Let :func:`paged_attention_multi` and the prefix pass of
    :func:`cascade_decode` run the tcgen05 kernels when their tiles can hold
    128 query rows (default True), or keep every call on the mma.sync
    kernels; process-wide."""
    library().pkv_set_tcgen05(1 if enable else 0)


def get_tcgen05() -> bool:
    return bool(library().pkv_get_tcgen05())


@contextlib.contextmanager
def tcgen05(enable: bool):
    """Temporarily set :func:`set_tcgen05`."""
    prev = get_tcgen05()
    set_tcgen05(enable)
    try:
        yield
    finally:
        set_tcgen05(prev)


def kv_reshape_and_cache(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor,
                         v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                         kv_scale: float = 1.0, stream=None) -> None:
    """Scatter ``k, v [T, Hkv, d]`` into the caches at ``slot_mapping`` (int64).

    A uint8 cache holds fp8-e4m3 codes written as ``e4m3(x / kv_scale)``."""
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    if k.dtype not in (torch.float32, torch.bfloat16) or v.dtype != k.dtype:
        raise TypeError("k and v must both be float32 or bfloat16")
    desc = _desc(k_cache, None)
    _check(library().pkv_kv_reshape_and_cache(
        _ptr(k), _ptr(v), _dt(k), int(k.shape[0]), _ptr(k_cache), _ptr(v_cache),
        ctypes.byref(desc), _ptr(slot_mapping), float(kv_scale), _stream(stream)),
        "kv_reshape_and_cache")


def decode_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                           max_seq_len: int, partition_tokens: int = 0) -> int:
    return int(library().pkv_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                    max_seq_len, partition_tokens))


class DecodeWorkspace:
    """A device workspace (torch-allocated) that grows on demand.

    It is zero-filled when (re)allocated.  The library keeps it valid from
    then on: every call leaves its merge counters zero, and a call whose
    counter region reaches past the part that is always kept zero clears
    that region itself."""

    def __init__(self, device=None):
        self.device = device
        self.buf: Optional[torch.Tensor] = None

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device or "cuda")
        return self.buf


_default_ws = {}


def paged_attention_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                           v_cache: torch.Tensor, block_tables: torch.Tensor,
                           seq_lens: torch.Tensor, scale: float, kv_scale: float = 1.0,
                           max_seq_len: Optional[int] = None, partition_tokens: int = 0,
                           workspace: Optional[DecodeWorkspace] = None, stream=None,
                           window: int = 0, sinks: int = 0) -> torch.Tensor:
    """One decode step: ``out[s, qh] = softmax(scale * q[s, qh] . K_s^T) . V_s``.

    ``max_seq_len`` is a host upper bound of ``seq_lens`` (the decode never
    synchronises to read it); by default the table capacity is used.
    ``window > 0``: each sequence attends only its last ``window`` tokens and
    its first ``sinks`` tokens (blocks outside them are never read)."""
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    _same_layout(out, q, k_cache, v_cache)
    B, Hq, d = q.shape
    desc = _desc(k_cache, None)
    mbps = int(block_tables.shape[1])
    if max_seq_len is None:
        max_seq_len = mbps * desc.block_size
    nbytes = decode_workspace_bytes(B, Hq, desc.num_kv_heads, d, max_seq_len, partition_tokens)
    if workspace is None:
        dev = q.device.index if q.device.index is not None else torch.cuda.current_device()
        workspace = _default_ws.setdefault(dev, DecodeWorkspace(q.device))
    ws = workspace.get(nbytes)
    qdt = F32 if q.dtype == torch.float32 else BF16
    if window:
        _check(library().pkv_paged_attention_decode_window(
            _ptr(out), _ptr(q), qdt, B, Hq, _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc),
            _ptr(block_tables), mbps, _ptr(seq_lens), int(max_seq_len), float(scale), float(kv_scale),
            int(window), int(sinks), int(partition_tokens), _ptr(ws), ws.numel(), _stream(stream)),
            "paged_attention_decode_window")
        return out
    _check(library().pkv_paged_attention_decode(
        _ptr(out), _ptr(q), qdt, B, Hq, _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc),
        _ptr(block_tables), mbps, _ptr(seq_lens), int(max_seq_len), float(scale), float(kv_scale),
        int(partition_tokens), _ptr(ws), ws.numel(), _stream(stream)), "paged_attention_decode")
    return out


def cascade_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                            max_seq_len: int) -> int:
    return int(library().pkv_cascade_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                     max_seq_len))


def cascade_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                   block_tables: torch.Tensor, seq_lens: torch.Tensor, prefix_blocks: int, scale: float,
                   kv_scale: float = 1.0, max_seq_len: Optional[int] = None,
                   workspace: Optional[DecodeWorkspace] = None, stream=None) -> torch.Tensor:
    """paged_attention_decode for a batch whose tables all begin with the same
    ``prefix_blocks`` blocks: the shared prefix is attended once for every
    query row of the batch, then each sequence's own blocks, and the two
    partial results are merged (bf16 and fp8 caches)."""
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    _same_layout(out, q, k_cache, v_cache)
    B, Hq, d = q.shape
    desc = _desc(k_cache, None)
    mbps = int(block_tables.shape[1])
    if max_seq_len is None:
        max_seq_len = mbps * desc.block_size
    nbytes = cascade_workspace_bytes(B, Hq, desc.num_kv_heads, d, max_seq_len)
    if workspace is None:
        dev = q.device.index if q.device.index is not None else torch.cuda.current_device()
        workspace = _default_ws.setdefault(dev, DecodeWorkspace(q.device))
    ws = workspace.get(nbytes)
    qdt = F32 if q.dtype == torch.float32 else BF16
    _check(library().pkv_cascade_decode(
        _ptr(out), _ptr(q), qdt, B, Hq, _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc),
        _ptr(block_tables), mbps, _ptr(seq_lens), int(max_seq_len), int(prefix_blocks), float(scale),
        float(kv_scale), _ptr(ws), ws.numel(), _stream(stream)), "cascade_decode")
    return out


def multi_workspace_bytes(num_seqs: int, total_q: int, max_q: int, num_q_heads: int, num_kv_heads: int,
                          head_dim: int) -> int:
    return int(library().pkv_multi_workspace_bytes(num_seqs, total_q, max_q, num_q_heads, num_kv_heads,
                                                   head_dim))


MULTI_KERNELS = {0: None, 1: "tcgen05", 2: "multi_query_decode", 3: "mma_sync"}


def multi_kernel_for(num_seqs: int, max_q: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                     block_size: int, cache_dtype: str, num_blocks: int = 1) -> str | None:
    """The kernel :func:`paged_attention_multi` runs for a call of this shape
    under the current :func:`set_tcgen05` setting: "tcgen05" (128-row
    tcgen05 tiles), "multi_query_decode" (the balanced decode kernel, 16
    (token, head) rows per unit), "mma_sync" (16-row mma.sync tiles), or None
    for a shape no kernel serves.  Host only."""
    dt = {"f32": F32, "bf16": BF16, "fp8_e4m3": FP8_E4M3}[cache_dtype]
    desc = CacheDesc(num_blocks, block_size, num_kv_heads, head_dim, dt)
    return MULTI_KERNELS[library().pkv_multi_kernel_for(num_seqs, max_q, num_q_heads, ctypes.byref(desc))]


def paged_attention_multi(out: torch.Tensor, q: torch.Tensor, q_start: torch.Tensor, k_cache: torch.Tensor,
                          v_cache: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                          scale: float, kv_scale: float = 1.0, max_q: Optional[int] = None,
                          max_seq_len: Optional[int] = None, workspace: Optional[DecodeWorkspace] = None,
                          stream=None) -> torch.Tensor:
    """Attention of several query tokens per sequence (a prefill chunk, a
    speculative step's tokens): sequence s owns rows ``q_start[s] ..
    q_start[s+1]-1`` of ``q [total, Hq, d]``, its last positions, each
    attending every position up to its own.  ``max_q`` is a host bound of the
    rows per sequence (read from ``q_start`` with a synchronisation when
    omitted)."""
    if q_start.dtype != torch.int32 or block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("q_start, block_tables and seq_lens must be int32")
    _same_layout(out, q, k_cache, v_cache)
    total, Hq, d = q.shape
    B = int(seq_lens.shape[0])
    if q_start.shape[0] != B + 1:
        raise ValueError("q_start must have num_seqs + 1 entries")
    desc = _desc(k_cache, None)
    mbps = int(block_tables.shape[1])
    if max_seq_len is None:
        max_seq_len = mbps * desc.block_size
    if max_q is None:
        max_q = int((q_start[1:] - q_start[:-1]).max().item()) if B else 0
    nbytes = multi_workspace_bytes(B, total, max_q, Hq, desc.num_kv_heads, d)
    if workspace is None:
        dev = q.device.index if q.device.index is not None else torch.cuda.current_device()
        workspace = _default_ws.setdefault(dev, DecodeWorkspace(q.device))
    ws = workspace.get(nbytes)
    qdt = F32 if q.dtype == torch.float32 else BF16
    _check(library().pkv_paged_attention_multi(
        _ptr(out), _ptr(q), qdt, _ptr(q_start), B, total, int(max_q), Hq, _ptr(k_cache), _ptr(v_cache),
        ctypes.byref(desc), _ptr(block_tables), mbps, _ptr(seq_lens), int(max_seq_len), float(scale),
        float(kv_scale), _ptr(ws), ws.numel(), _stream(stream)), "paged_attention_multi")
    return out


def decode_step(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, out: torch.Tensor,
                q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                kv_scale: float = 1.0, max_seq_len: Optional[int] = None,
                partition_tokens: int = 0, workspace: Optional[DecodeWorkspace] = None,
                stream=None) -> torch.Tensor:
    """One decode step: write the new tokens ``k, v [T, Hkv, d]`` into their
    slots, then attend (the decode overlaps its prologue with the write)."""
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    if k.dtype not in (torch.float32, torch.bfloat16) or v.dtype != k.dtype:
        raise TypeError("k and v must both be float32 or bfloat16")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    _same_layout(out, q, k_cache, v_cache)
    B, Hq, d = q.shape
    desc = _desc(k_cache, None)
    mbps = int(block_tables.shape[1])
    if max_seq_len is None:
        max_seq_len = mbps * desc.block_size
    nbytes = decode_workspace_bytes(B, Hq, desc.num_kv_heads, d, max_seq_len, partition_tokens)
    if workspace is None:
        dev = q.device.index if q.device.index is not None else torch.cuda.current_device()
        workspace = _default_ws.setdefault(dev, DecodeWorkspace(q.device))
    ws = workspace.get(nbytes)
    qdt = F32 if q.dtype == torch.float32 else BF16
    _check(library().pkv_decode_step(
        _ptr(k), _ptr(v), _dt(k), int(k.shape[0]), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
        ctypes.byref(desc), _ptr(out), _ptr(q), qdt, B, Hq, _ptr(block_tables), mbps, _ptr(seq_lens),
        int(max_seq_len), float(scale), float(kv_scale), int(partition_tokens), _ptr(ws), ws.numel(),
        _stream(stream)), "decode_step")
    return out


def split_kv_reduce(out: torch.Tensor, o_part: torch.Tensor, m_part: torch.Tensor,
                    l_part: torch.Tensor, seq_lens: torch.Tensor, partition_tokens: int,
                    stream=None) -> torch.Tensor:
    """Merge ``o_part [B, Hq, P, d]``, ``m_part / l_part [B, Hq, P]`` (fp32)."""
    B, Hq, P, d = o_part.shape
    odt = F32 if out.dtype == torch.float32 else BF16
    _check(library().pkv_split_kv_reduce(
        _ptr(out), odt, _ptr(o_part), _ptr(m_part), _ptr(l_part), _ptr(seq_lens), B, Hq, d,
        int(partition_tokens), P, _stream(stream)), "split_kv_reduce")
    return out


def gather_kv(k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
              seq_lens: torch.Tensor, max_seq_len: int, cu_seq_lens: Optional[torch.Tensor] = None,
              total_tokens: Optional[int] = None, stream=None):
    """Contiguous ``[sum(seq_lens), Hkv, d]`` copies of K and V."""
    desc = _desc(k_cache, None)
    if cu_seq_lens is None:
        cu_seq_lens = torch.zeros(seq_lens.numel() + 1, dtype=torch.int64, device=seq_lens.device)
        cu_seq_lens[1:] = torch.cumsum(seq_lens.to(torch.int64), 0)
    if total_tokens is None:
        total_tokens = int(cu_seq_lens[-1].item())
    k_out = torch.empty((total_tokens, desc.num_kv_heads, desc.head_dim), dtype=k_cache.dtype,
                        device=k_cache.device)
    v_out = torch.empty_like(k_out)
    _check(library().pkv_gather_kv(
        _ptr(k_out), _ptr(v_out), _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc),
        _ptr(block_tables), int(block_tables.shape[1]), _ptr(seq_lens), _ptr(cu_seq_lens),
        int(seq_lens.numel()), int(max_seq_len), _stream(stream)), "gather_kv")
    return k_out, v_out


def _addr(t: torch.Tensor):
    """Device address of a CUDA tensor or of a pinned host tensor (pinned
    host memory is mapped into the device's address space)."""
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("tensors must live on the CUDA device or in pinned host memory")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def copy_blocks(k_dst: torch.Tensor, v_dst: torch.Tensor, k_src: torch.Tensor, v_src: torch.Tensor,
                block_pairs: torch.Tensor, stream=None) -> None:
    """Copy blocks ``block_pairs[i] = (src, dst)`` (int64 ``[n, 2]``) of the
    pool ``k_src / v_src`` into the pool ``k_dst / v_dst`` (the same pool for
    copy-on-write; a pinned host pool for swap).  Every tensor may be a CUDA
    tensor or a pinned host tensor."""
    if block_pairs.dtype != torch.int64 or block_pairs.dim() != 2 or block_pairs.shape[1] != 2:
        raise ValueError("block_pairs must be int64 [n, 2]")
    dd, sd = _desc(k_dst, None), _desc(k_src, None)
    _check(library().pkv_copy_blocks(_addr(k_dst), _addr(v_dst), ctypes.byref(dd), _addr(k_src), _addr(v_src),
                                     ctypes.byref(sd), _addr(block_pairs), int(block_pairs.shape[0]),
                                     _stream(stream)), "copy_blocks")


def selftest_wait_timeout(stream=None) -> None:
    """Run the library's bounded-wait failure path once (an mbarrier armed for
    bytes no copy delivers): afterwards :func:`get_device_error` reports
    ``DEVERR_WAIT_TIMEOUT``.  Takes up to about a second of GPU time."""
    _check(library().pkv_selftest_wait_timeout(_stream(stream)), "selftest_wait_timeout")


def get_device_error(stream=None) -> int:
    """Synchronise the stream, then read and clear the device error word."""
    code = ctypes.c_uint32(0)
    _check(library().pkv_get_device_error(ctypes.byref(code), _stream(stream)), "get_device_error")
    return int(code.value)
