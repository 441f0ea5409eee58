"""Shared test helpers: marshalling between torch tensors and the oracle's
numpy arrays, and the oracle-side cache fill.  No attention arithmetic here."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads


def to_np(t: torch.Tensor) -> np.ndarray:
    """Raw oracle array for a tensor: float32 stays float32, bfloat16 becomes
    its uint16 bit pattern, uint8 (fp8 codes) stays uint8."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if t.dtype == torch.uint8:
        return t.numpy().copy()
    if t.dtype in (torch.int32, torch.int64):
        return t.numpy().copy()
    raise TypeError(t.dtype)


def from_np_bits(a: np.ndarray, like: torch.dtype) -> torch.Tensor:
    if like == torch.bfloat16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    return torch.from_numpy(a.copy())


def empty_cache_np(w: workloads.Workload) -> np.ndarray:
    dt = {"f32": np.float32, "bf16": np.uint16, "fp8_e4m3": np.uint8}[w.cache_dtype]
    shape = workloads.cache_shape(w)
    raw = np.full(int(np.prod(shape)) * np.dtype(dt).itemsize,
                  workloads.poison_bits(w.cache_dtype), dtype=np.uint8)
    return raw.view(dt).reshape(shape)


def oracle_caches(w: workloads.Workload, include_new: bool = True):
    """Oracle-side caches filled with the workload's history (and new) tokens."""
    kc, vc = empty_cache_np(w), empty_cache_np(w)
    if w.hist_slots.numel():
        oracle.reshape_and_cache(to_np(w.hist_k), to_np(w.hist_v), kc, vc,
                                 to_np(w.hist_slots), w.kv_scale)
    if include_new and w.new_slots.numel():
        oracle.reshape_and_cache(to_np(w.new_k), to_np(w.new_v), kc, vc,
                                 to_np(w.new_slots), w.kv_scale)
    return kc, vc


def oracle_decode(w: workloads.Workload, kc=None, vc=None, threads: int = 1) -> np.ndarray:
    if kc is None:
        kc, vc = oracle_caches(w)
    return oracle.paged_attention_decode(to_np(w.q), kc, vc, to_np(w.block_tables),
                                         to_np(w.seq_lens), w.scale, w.kv_scale, threads)
