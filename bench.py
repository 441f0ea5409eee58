"""Benchmark of one paged-decode step on GB300.

A step is the whole hot path for one decode iteration of one attention layer:
``kv_reshape_and_cache`` of the step's new K/V tokens (one per sequence), then
``paged_attention_decode`` over every sequence's paged cache.  The default
workload is the Llama-3-8B-shaped decode layer: 64 sequences with lengths
uniform in [128, 2048], 32 query / 8 kv heads, head_dim 128, bf16 cache,
block_size 16, a shuffled 16384-block pool.

Metric: effective HBM GB/s of the step -- algorithmic bytes (K/V of every
valid token, q, out, the block-table entries used, seq_lens, plus the cache
write's bytes) divided by the device time of the step -- with decode tokens/s
per layer beside it.  L2 is flushed between timed steps: a 256 MiB write, then a
256 MiB read of a second buffer, so the timed kernels start on a cold L2 that
holds no dirty line of the flush.

``--impl reference`` times the CPU oracle on the same workload instead (a
bounded sample of sequences per step) and prints the same JSON line.

Multi-GPU (torchrun): every rank runs its own replica of the workload with a
different seed (the sequences of a decode batch are independent; no
collective sits on the data path); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402
from paged_kv_cache_22_gb300 import metrics  # noqa: E402

METRIC = ("paged decode attention effective HBM GB/s (% of GB300 peak); decode tok/s/layer")
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20

# DRAM traffic of one decode launch on the default workload, from an ncu
# capture, valid only for the kernel sources it was taken on.
TRAFFIC = {"sources_sha256": "e2e92ca10a5eb5dedb6e155ad5f693c7c174ec151d02ce146ba8100d34690ea3",
           "bytes_per_launch": 319391744}  # mean of two launches: 316.93 MB read + 2.47 MB written

WORKLOAD_TEXT = {
    "llama3_8b": "Llama-3-8B-shaped decode layer: 64 seqs, L~U[128,2048], 32 q / 8 kv heads, "
                 "head_dim 128, bf16 KV, block 16, 16384-block shuffled pool",
    "llama70b_128": "Llama-70B-shaped decode layer: 128 seqs, L lognormal(median 800, sigma 1) "
                    "in [16,8192], 64 q / 8 kv heads, head_dim 128, bf16 KV, block 16",
    "long_split_kv": "long-context split-KV: 8 seqs x 32768 tokens, 32 q / 8 kv heads, head_dim "
                     "128, bf16 KV, block 16, 512-token partitions",
    "prefix_fp8": "prefix sharing + fp8 KV: 256 seqs = 2048 shared prefix + U[1,512] suffix, "
                  "32 q / 8 kv heads, head_dim 128, fp8-e4m3 KV, bf16 q/out",
    "tiny_mha": "tiny MHA: 4 seqs {1,17,33,100}, 4 heads, head_dim 64, fp32",
}


def kernel_sources_sha() -> str:
    """Hash of the files that define the tensor-core decode kernel's device
    code (host-side launch code does not change its DRAM traffic)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_22_gb300", "csrc")
    for f in ("pkv_device.cuh", "decode_common.cuh", "decode_tc.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor-core peak (TFLOP/s): the measured cuBLAS burst figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, device) -> float:
    """The largest `value` over all ranks (the identity without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world_size: int, bytes_per_rank_step: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank moves the same bytes per step (weak
    scaling); the step time is the slowest rank's."""
    return world_size * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def step_bytes(w: workloads.Workload, window: int = 0, sinks: int = 0):
    lens = w.seq_lens.tolist()
    dec = metrics.decode_bytes(lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.cache_dtype,
                               w.q_dtype, w.block_size, window, sinks)
    rc = metrics.reshape_bytes(int(w.new_slots.numel()), w.num_kv_heads, w.head_dim, w.src_dtype,
                               w.cache_dtype)
    return dec, rc


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed loop runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            target = f"GPU-{uuid}" if not uuid.startswith("GPU-") else uuid
        except Exception:
            target = str(device_index)
        self.target = target

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.target, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------ GPU arm
class L2Flush:
    """Cold L2 before a timed step, outside its events: write a buffer larger
    than L2 (evicts every line), then read a second one, so that the lines
    left behind are clean and the timed kernels do not pay the write-back of
    the flush's own data."""

    def __init__(self, dev):
        n = L2_FLUSH_BYTES // 4
        self.dirty = torch.empty(n, dtype=torch.float32, device=dev)
        self.clean = torch.ones(n, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self, i: int = 0):
        self.dirty.fill_(float(i))
        torch.sum(self.clean, dim=0, out=self.sink)


def run_gpu(args):
    import paged_kv_cache_22_gb300 as pkv

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pkv.library()
    pkv.set_decode_engine(args.engine)

    w = workloads.CONFIGS[args.config](seed=1234 + list(workloads.CONFIGS).index(args.config)
                                       + 1000 * rank)
    pt = args.partition_tokens
    shape = workloads.cache_shape(w)
    cdt = workloads.cache_torch_dtype(w.cache_dtype)
    kc = torch.zeros(shape, dtype=cdt, device=dev)
    vc = torch.zeros(shape, dtype=cdt, device=dev)
    # history tokens are state carried from earlier steps: written once, untimed
    if w.hist_slots.numel():
        pkv.kv_reshape_and_cache(w.hist_k.to(dev), w.hist_v.to(dev), kc, vc, w.hist_slots.to(dev),
                                 w.kv_scale)
    q = w.q.to(dev)
    new_k, new_v, new_slots = w.new_k.to(dev), w.new_v.to(dev), w.new_slots.to(dev)
    tables, lens = w.block_tables.to(dev), w.seq_lens.to(dev)
    out = torch.empty_like(q)
    max_len = w.max_seq_len
    workspace = pkv.DecodeWorkspace(dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    win, sinks = args.window, args.sinks
    pblocks = w.shared_prefix_blocks if args.cascade else 0
    if args.cascade and not pblocks:
        raise SystemExit("--cascade needs a workload whose tables share a prefix (prefix_fp8)")

    def step():
        if pblocks:  # cache write, then the cascade's prefix pass and decode (three launches)
            pkv.kv_reshape_and_cache(new_k, new_v, kc, vc, new_slots, w.kv_scale)
            pkv.cascade_decode(out, q, kc, vc, tables, lens, pblocks, w.scale, w.kv_scale,
                               max_seq_len=max_len, workspace=workspace)
            return
        if win:  # the windowed decode after the cache write (two launches)
            pkv.kv_reshape_and_cache(new_k, new_v, kc, vc, new_slots, w.kv_scale)
            pkv.paged_attention_decode(out, q, kc, vc, tables, lens, w.scale, w.kv_scale,
                                       max_seq_len=max_len, partition_tokens=pt, workspace=workspace,
                                       window=win, sinks=sinks)
            return
        pkv.decode_step(new_k, new_v, new_slots, out, q, kc, vc, tables, lens, w.scale, w.kv_scale,
                        max_seq_len=max_len, partition_tokens=pt, workspace=workspace)

    def decode_only():
        if pblocks:
            pkv.cascade_decode(out, q, kc, vc, tables, lens, pblocks, w.scale, w.kv_scale,
                               max_seq_len=max_len, workspace=workspace)
            return
        pkv.paged_attention_decode(out, q, kc, vc, tables, lens, w.scale, w.kv_scale,
                                   max_seq_len=max_len, partition_tokens=pt, workspace=workspace,
                                   window=win, sinks=sinks)

    for _ in range(args.warmup):
        flush(1)
        step()
    torch.cuda.synchronize()
    if pkv.get_device_error():
        raise RuntimeError("device error during warm-up")

    K = args.steps
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)  # let the sampler come up before the timed region
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # timed region: K steps (cache write + decode), L2 flushed before each
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush(i)  # untimed: evicts the previous step's lines from L2
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    # the dominant kernel alone, same inputs and flushing, for its roofline
    evd = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush(i)
        evd[i][0].record(stream)
        decode_only()
        evd[i][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    dec_ms = [e[0].elapsed_time(e[1]) for e in evd]
    tot_ms = max_over_ranks(sum(step_ms), dev)
    if pkv.get_device_error():
        raise RuntimeError("device error during the timed steps")

    dec_b, rc_b = step_bytes(w, win, sinks)
    ms_per_step = tot_ms / K
    value = job_throughput(ws, dec_b + rc_b, ms_per_step)
    dec_avg_ms = sum(dec_ms) / K
    # roofline bytes: what the timed call must move (a shared prefix once)
    roof_b = (metrics.cascade_bytes(w.seq_lens.tolist(), pblocks * w.block_size, w.num_q_heads,
                                    w.num_kv_heads, w.head_dim, w.cache_dtype, w.q_dtype, w.block_size)
              if pblocks else dec_b)
    achieved = roof_b / (dec_avg_ms * 1e-3) / 1e9
    peak, peak_src = measured_peak()

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(pkv, w, kc, vc, dev, pt, max(10, min(K, 200)), flush, win, sinks, pblocks)
    e2e["ms_per_step"] = max_over_ranks(e2e["ms_per_step"], dev)
    e2e["host_ms_per_step"] = max_over_ranks(e2e["host_ms_per_step"], dev)
    e2e_value = job_throughput(ws, dec_b + rc_b, e2e["ms_per_step"])

    traffic = None
    if (TRAFFIC["sources_sha256"] == kernel_sources_sha() and args.config == "llama3_8b" and pt == 0
            and args.engine == "tensor_cores" and not win and not pblocks):
        traffic = TRAFFIC["bytes_per_launch"]

    tc_decode = w.cache_dtype != "f32" and args.engine == "tensor_cores"
    # the kernel of the cascade's prefix pass (tcgen05 once a kv head has 128 rows)
    prefix_kernel = ("attn_tc05_kernel (tcgen05.mma, S and O in TMEM)"
                     if pblocks and pkv.get_tcgen05() and w.head_dim == 128
                     and w.num_seqs * (w.num_q_heads // w.num_kv_heads) >= 128
                     else "prefix_attention_kernel")
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.cache_dtype == "bf16" else w.cache_dtype,
        "data": "synthetic (seeded N(0,1) q/k/v, shuffled block pool)",
        "config": {
            "workload": WORKLOAD_TEXT.get(args.config, args.config),
            "name": args.config,
            "num_seqs": w.num_seqs, "sum_seq_len": int(w.seq_lens.sum()),
            "max_seq_len": max_len, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "cache_dtype": w.cache_dtype,
            "split": "balanced (1 launch)" if pt == 0 else f"fixed {pt}-token partitions + reduce",
            **({"window": win, "sinks": sinks,
                "step_launches": "kv_reshape_and_cache, then the windowed decode"} if win else {}),
            **({"cascade": {"prefix_blocks": pblocks,
                            "step_launches": f"kv_reshape_and_cache, {prefix_kernel}, decode_tc_kernel",
                            "metric_bytes": "logical: every sequence's prefix counted (as plain decode reads it)",
                            "roofline_bytes": "unique: the shared prefix once"}} if pblocks else {}),
            "engine": ("cuda_cores" if w.cache_dtype == "f32" else args.engine)
                      + " (q.K and P.V; softmax and accumulation in fp32)",
            "l2": "flushed between timed steps, outside the timed events: 256 MiB write, then "
                  "256 MiB read of a second buffer (cold L2 holding no dirty line)",
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
        },
        "decode_tok_s_per_layer": round(ws * w.num_seqs / (ms_per_step * 1e-3), 1),
        "step": ("kv_reshape_and_cache + cascade_decode (prefix pass, then suffix decode)" if pblocks else
                 "kv_reshape_and_cache + paged_attention_decode (windowed)" if win else
                 "kv_reshape_and_cache + paged_attention_decode (pkv_decode_step: the decode "
                 "is the cache write's programmatic dependent)"),
        "decode_only": {"ms": round(dec_avg_ms, 6), "gbs": round(dec_b / (dec_avg_ms * 1e-3) / 1e9, 1),
                        "frac_of_8TBs": round(dec_b / (dec_avg_ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
                        "bytes": dec_b, **({"unique_bytes": roof_b} if pblocks else {})},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": (f"{prefix_kernel} + decode_tc_kernel + merge_cut_kernel (cascade, all launches)"
                                if pblocks else
                                ("decode_tc_kernel" if tc_decode else "decode_kernel")
                                + ((" + merge_cut_kernel (balanced split)" if tc_decode else " (balanced split)")
                                   if pt == 0 else " + split_kv_reduce_kernel (partitions)"))},
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e["ms_per_step"], 6),
                "host_wall": {"ms_per_step": round(e2e["host_ms_per_step"], 6),
                              "value": round(job_throughput(ws, dec_b + rc_b, e2e["host_ms_per_step"]), 1),
                              "what": "host clock from the first call of a step until its output "
                                      "is on the host (binding, C ABI, launches, copies, GPU time)"}},
        # cache write, decode, then the merge grid (balanced split on the tensor cores) or the reduce
        # (partitions); a cascade adds its prefix pass
        "gpu_launches": K * (2 + (1 if (pt or tc_decode) else 0) + (1 if pblocks else 0)),
        "clocks": clocks,
    }
    if (ws == 1 and args.config == "llama3_8b" and pt == 0 and not win and not pblocks
            and args.engine == "tensor_cores" and not args.no_per_config):
        line["per_config"] = per_config(pkv, dev, flush, min(K, 50), dec_avg_ms)
        if pkv.get_device_error():
            raise RuntimeError("device error in the per-config measurements")
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, win, sinks)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def time_calls(fn, flush, stream, K: int, warmup: int = 3) -> float:
    """Mean device time (ms) of `fn` over K calls, each after an L2 flush,
    with CUDA events on the launching stream."""
    for i in range(warmup):
        flush(i)
        fn()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush(i)
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return sum(e[0].elapsed_time(e[1]) for e in ev) / K


MULTI_KERNEL_LABELS = {
    "tcgen05": "attn_tc05_kernel (tcgen05.mma, S and O in TMEM)",
    "multi_query_decode": "decode_tc_kernel (multi-query: 16 (token, head) rows per unit, balanced split, "
                          "mma.sync m16n8k16) + merge_cut_kernel (segments cut between warps)",
    "mma_sync": "prefix_attention_kernel (MULTI, mma.sync m16n8k16)",
}


def multi_kernel_label(pkv, w, max_q: int) -> str:
    """The kernel pkv_paged_attention_multi launches for this workload, as the
    library decides it under the current tcgen05 setting."""
    k = pkv.multi_kernel_for(w.num_seqs, max_q, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                             w.cache_dtype, w.num_blocks)
    return MULTI_KERNEL_LABELS.get(k, "none")


def per_config(pkv, dev, flush, K: int, main_decode_ms: float):
    """Decode-only figures of the other workloads, measured in this process
    with the same flush and events: each entry gives the time per call, the
    algorithmic GB/s (TFLOP/s for prefill chunks) and its fraction of the
    measured and nominal peaks.  Also the paged-vs-contiguous control
    (identity block tables) and block sizes 8 and 32 on the Llama-3-8B-shaped
    batch, and the multi-token workloads on both of their kernels."""
    stream = torch.cuda.current_stream()
    hbm_peak, _ = measured_peak()
    tc_peak = tensor_peak()[0]
    res = {}

    def caches(w):
        shape = workloads.cache_shape(w)
        cdt = workloads.cache_torch_dtype(w.cache_dtype)
        kc = torch.zeros(shape, dtype=cdt, device=dev)
        vc = torch.zeros(shape, dtype=cdt, device=dev)
        k, v, sl = w.all_tokens()
        pkv.kv_reshape_and_cache(k.to(dev), v.to(dev), kc, vc, sl.to(dev), w.kv_scale)
        return kc, vc

    def hbm_entry(ms, nbytes, kernel, extra=None):
        gbs = nbytes / (ms * 1e-3) / 1e9
        e = {"ms": round(ms, 6), "bytes": nbytes, "gbs": round(gbs, 1),
             "frac_of_measured": round(gbs / hbm_peak, 4), "frac_of_8TBs": round(gbs / NOMINAL_HBM_GBS, 4),
             "kernel": kernel}
        e.update(extra or {})
        return e

    def decode_entries(name, w, variants):
        kc, vc = caches(w)
        q = w.q.to(dev)
        out = torch.empty_like(q)
        tables, lens = w.block_tables.to(dev), w.seq_lens.to(dev)
        wsp = pkv.DecodeWorkspace(dev)
        lens_l = w.seq_lens.tolist()
        for tag, pt, win, sinks, pblocks in variants:
            def call():
                if pblocks:
                    pkv.cascade_decode(out, q, kc, vc, tables, lens, pblocks, w.scale, w.kv_scale,
                                       max_seq_len=w.max_seq_len, workspace=wsp)
                else:
                    pkv.paged_attention_decode(out, q, kc, vc, tables, lens, w.scale, w.kv_scale,
                                               max_seq_len=w.max_seq_len, partition_tokens=pt,
                                               workspace=wsp, window=win, sinks=sinks)
            ms = time_calls(call, flush, stream, K)
            nbytes = metrics.decode_bytes(lens_l, w.num_q_heads, w.num_kv_heads, w.head_dim, w.cache_dtype,
                                          w.q_dtype, w.block_size, win, sinks)
            extra = {"tok_s_per_layer": round(w.num_seqs / (ms * 1e-3), 1)}
            if pblocks:
                ub = metrics.cascade_bytes(lens_l, pblocks * w.block_size, w.num_q_heads, w.num_kv_heads,
                                           w.head_dim, w.cache_dtype, w.q_dtype, w.block_size)
                ugbs = ub / (ms * 1e-3) / 1e9
                e = {"ms": round(ms, 6), "bytes": nbytes, "logical_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                     "unique_bytes": ub, "unique_gbs": round(ugbs, 1),
                     "unique_frac_of_measured": round(ugbs / hbm_peak, 4),
                     "kernel": "prefix pass (attn_tc05_kernel once a kv head has >= 128 rows, else "
                               "prefix_attention_kernel) + decode_tc_kernel + merge_cut_kernel", **extra}
            else:
                kern = "decode_kernel (CUDA cores)" if w.cache_dtype == "f32" else "decode_tc_kernel"
                kern += (" + split_kv_reduce_kernel (fixed partitions)" if pt else
                         " (balanced split)" if w.cache_dtype == "f32" else " + merge_cut_kernel (balanced split)")
                e = hbm_entry(ms, nbytes, kern, extra)
            if win:
                e["window"], e["sinks"] = win, sinks
            res[name + tag] = e
        del kc, vc
        torch.cuda.empty_cache()

    decode_entries("llama70b_128", workloads.llama70b_128(seed=1236), [("", 0, 0, 0, 0)])
    decode_entries("long_split_kv", workloads.long_split_kv(seed=1237),
                   [("", 0, 0, 0, 0), ("_partitions512", 512, 0, 0, 0), ("_window4096_sinks4", 0, 4096, 4, 0)])
    pf = workloads.prefix_fp8(seed=1238)
    decode_entries("prefix_fp8", pf, [("", 0, 0, 0, 0), ("_cascade", 0, 0, 0, pf.shared_prefix_blocks)])
    decode_entries("tiny_mha", workloads.tiny_mha(seed=1234), [("", 0, 0, 0, 0)])
    decode_entries("llama3_8b_identity_tables", workloads.llama3_8b(seed=1235, identity_tables=True),
                   [("", 0, 0, 0, 0)])
    for bsz in (8, 32):
        decode_entries(f"llama3_8b_block{bsz}", workloads.llama3_8b(seed=1235, block_size=bsz), [("", 0, 0, 0, 0)])
    ident = res["llama3_8b_identity_tables"]["ms"]
    res["paged_vs_contiguous"] = {
        "shuffled_ms": round(main_decode_ms, 6), "identity_ms": ident,
        "ratio": round(main_decode_ms / ident, 4),
        "what": "the llama3_8b decode over a shuffled pool vs the same batch with block tables dealt in order"}

    for mname in ("verify4_llama3_8b", "prefill_chunk512"):
        w, q_cpu, qs_cpu = workloads.MULTI_CONFIGS[mname](seed=1301 + list(workloads.MULTI_CONFIGS).index(mname))
        kc, vc = caches(w)
        q, qs = q_cpu.to(dev), qs_cpu.to(dev)
        out = torch.empty_like(q)
        tables, lens = w.block_tables.to(dev), w.seq_lens.to(dev)
        q_lens = (qs_cpu[1:] - qs_cpu[:-1]).tolist()
        max_q = max(q_lens)
        wsp = pkv.DecodeWorkspace(dev)
        lens_l = w.seq_lens.tolist()
        nbytes = metrics.multi_bytes(lens_l, q_lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.cache_dtype,
                                     w.q_dtype, w.block_size)
        flops = metrics.multi_flops(lens_l, q_lens, w.num_q_heads, w.head_dim)
        rows = max_q * (w.num_q_heads // w.num_kv_heads)

        def call():
            pkv.paged_attention_multi(out, q, qs, kc, vc, tables, lens, w.scale, w.kv_scale, max_q=max_q,
                                      max_seq_len=w.max_seq_len, workspace=wsp)
        # both kernels where the tcgen05 one applies (a (sequence, kv head) of >= 128 rows)
        for tag, tc in (("", True), ("_mma_sync", False)) if rows >= 128 else (("", False),):
            with pkv.tcgen05(tc):
                ms = time_calls(call, flush, stream, K)
                kern = multi_kernel_label(pkv, w, max_q)
            if mname == "prefill_chunk512":
                tf = flops / (ms * 1e-3) / 1e12
                res[mname + tag] = {"ms": round(ms, 6), "flop": flops, "tflops": round(tf, 2),
                                    "frac_of_bf16_peak": round(tf / tc_peak, 4), "kernel": kern}
            else:
                res[mname + tag] = hbm_entry(ms, nbytes, kern)
        del kc, vc
        torch.cuda.empty_cache()
    return res


class StagedInputs:
    """A step's host inputs packed into one pinned buffer (256-byte aligned
    fields) and its device twin, so that a step uploads them with one copy;
    `dev[name]` are the device views the calls take."""

    def __init__(self, tensors: dict, device):
        offs, total = {}, 0
        for name, t in tensors.items():
            total = (total + 255) // 256 * 256
            n = t.numel() * t.element_size()
            offs[name] = (total, n, t)
            total += n
        self.host = torch.empty(max(total, 1), dtype=torch.uint8).pin_memory()
        self.device_buf = torch.empty_like(self.host, device=device)
        self.dev = {}
        for name, (o, n, t) in offs.items():
            self.host[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
            self.dev[name] = self.device_buf[o:o + n].view(t.dtype).view(t.shape)
        self.nbytes = total

    def upload(self):
        self.device_buf.copy_(self.host, non_blocking=True)


def run_e2e(pkv, w, kc, vc, dev, pt, steps, flush, window=0, sinks=0, prefix_blocks=0):
    """Per step: the host->device copy of the step's inputs from pinned
    memory (packed into one buffer), the calls, and a device->host read of
    the output, all timed."""
    staged = StagedInputs({"q": w.q, "k": w.new_k, "v": w.new_v, "slots": w.new_slots,
                           "tables": w.block_tables, "lens": w.seq_lens}, dev)
    dbuf = staged.dev
    out = torch.empty_like(dbuf["q"])
    out_host = torch.empty_like(w.q).pin_memory()
    workspace = pkv.DecodeWorkspace(dev)
    stream = torch.cuda.current_stream()
    h2d = staged.nbytes
    d2h = out_host.numel() * out_host.element_size()

    def one():
        staged.upload()
        if prefix_blocks:
            pkv.kv_reshape_and_cache(dbuf["k"], dbuf["v"], kc, vc, dbuf["slots"], w.kv_scale)
            pkv.cascade_decode(out, dbuf["q"], kc, vc, dbuf["tables"], dbuf["lens"], prefix_blocks, w.scale,
                               w.kv_scale, max_seq_len=w.max_seq_len, workspace=workspace)
        elif window:
            pkv.kv_reshape_and_cache(dbuf["k"], dbuf["v"], kc, vc, dbuf["slots"], w.kv_scale)
            pkv.paged_attention_decode(out, dbuf["q"], kc, vc, dbuf["tables"], dbuf["lens"], w.scale,
                                       w.kv_scale, max_seq_len=w.max_seq_len, partition_tokens=pt,
                                       workspace=workspace, window=window, sinks=sinks)
        else:
            pkv.decode_step(dbuf["k"], dbuf["v"], dbuf["slots"], out, dbuf["q"], kc, vc, dbuf["tables"],
                            dbuf["lens"], w.scale, w.kv_scale, max_seq_len=w.max_seq_len,
                            partition_tokens=pt, workspace=workspace)
        out_host.copy_(out, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    tot, host = 0.0, 0.0
    for i in range(steps):
        flush(i)
        torch.cuda.synchronize()  # the flush is not part of the host-side time either
        t0 = time.perf_counter()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        one()
        b.record(stream)
        b.synchronize()
        host += time.perf_counter() - t0
        tot += a.elapsed_time(b)
    return {"ms_per_step": tot / steps, "host_ms_per_step": host * 1e3 / steps, "h2d": h2d, "d2h": d2h}


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(w, max_seqs=None):
    """(q, caches, tables, lens) numpy inputs for the oracle over the first
    sequences of the workload, caches filled by the oracle's own cache write."""
    import oracle

    def np_of(t):
        t = t.contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16).copy()
        return t.numpy().copy()

    B = w.num_seqs if max_seqs is None else min(max_seqs, w.num_seqs)
    shape = workloads.cache_shape(w)
    dt = {"f32": np.float32, "bf16": np.uint16, "fp8_e4m3": np.uint8}[w.cache_dtype]
    kc = np.zeros(shape, dtype=dt)
    vc = np.zeros(shape, dtype=dt)
    k, v, slots = w.all_tokens()
    oracle.reshape_and_cache(np_of(k), np_of(v), kc, vc, slots.numpy().copy(), w.kv_scale)
    return (np_of(w.q[:B]), kc, vc, w.block_tables[:B].numpy().copy(),
            w.seq_lens[:B].numpy().copy(), np_of(w.new_k), np_of(w.new_v),
            w.new_slots.numpy().copy(), B)


def cpu_baseline(w, seconds: float, window: int = 0, sinks: int = 0):
    """The oracle, as it stands, timed on this host's cores: repeated full
    decode steps (cache write of the new tokens + attention) for ~`seconds`
    on every core, then for ~`seconds` / 2 on one thread."""
    import oracle
    q, kc, vc, tables, lens, nk, nv, ns, B = oracle_sample(w)
    dec_b, rc_b = step_bytes(w, window, sinks)

    def timed(threads, budget):
        reps, t0 = 0, time.perf_counter()
        while True:
            oracle.reshape_and_cache(nk, nv, kc, vc, ns, w.kv_scale)
            oracle.paged_attention_decode(q, kc, vc, tables, lens, w.scale, w.kv_scale, threads,
                                          window=window, sinks=sinks)
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget or reps >= 1000:
                return reps, el

    threads = os.cpu_count() or 1
    reps, el = timed(threads, seconds)
    reps1, el1 = timed(1, seconds / 2)
    return {"value": round(reps * (dec_b + rc_b) / el / 1e9, 3), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{reps} full decode steps of the same workload ({B} seqs), fp64 C loops, "
                      f"{el:.1f} s wall",
            "single_thread": {"value": round(reps1 * (dec_b + rc_b) / el1 / 1e9, 3), "unit": "GB/s", "cores": 1,
                              "sample": f"{reps1} full decode steps on one thread, {el1:.1f} s wall"}}


def run_reference(args):
    """The CPU oracle as the reference arm: each step is a bounded sample
    (the first few sequences of the workload), scaled to GB/s."""
    ws, rank, _ = dist_env()
    if ws > 1 and rank != 0:
        return
    import oracle
    w = workloads.CONFIGS[args.config](seed=1234 + list(workloads.CONFIGS).index(args.config))
    sample = max(1, min(w.num_seqs, args.ref_seqs))
    q, kc, vc, tables, lens, nk, nv, ns, B = oracle_sample(w, sample)
    threads = os.cpu_count() or 1
    lens_l = lens.tolist()
    dec_b = metrics.decode_bytes(lens_l, w.num_q_heads, w.num_kv_heads, w.head_dim, w.cache_dtype,
                                 w.q_dtype, w.block_size, args.window, args.sinks)
    rc_b = metrics.reshape_bytes(B, w.num_kv_heads, w.head_dim, w.src_dtype, w.cache_dtype)
    nk, nv, ns = nk[:B], nv[:B], ns[:B]

    def step():
        oracle.reshape_and_cache(nk, nv, kc, vc, ns, w.kv_scale)
        oracle.paged_attention_decode(q, kc, vc, tables, lens, w.scale, w.kv_scale, threads,
                                      window=args.window, sinks=args.sinks)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    ms = el * 1e3 / args.steps
    value = (dec_b + rc_b) / (ms * 1e-3) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q/k/v, shuffled block pool)",
        "config": {"workload": WORKLOAD_TEXT.get(args.config, args.config), "name": args.config,
                   "sample_seqs": B},
        "decode_tok_s_per_layer": round(B / (ms * 1e-3), 2),
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"first {B} of {w.num_seqs} sequences per step, fp64 C loops"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_copy(args):
    """Block copies on the Llama-3-8B-shaped pool (16,384 blocks of 8 kv heads
    x 16 tokens x 128 dims, bf16): copy-on-write of random block pairs inside
    the device pool, or swap of blocks to a pinned host pool and back.  One
    JSON line; GB/s counts every byte read and written."""
    import paged_kv_cache_22_gb300 as pkv
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pkv.library()
    nb, hkv, bs, d = 16384, 8, 16, 128
    block_bytes = hkv * bs * d * 2
    g = torch.Generator().manual_seed(77 + rank)
    kc = torch.randn((nb, hkv, bs, d), generator=g).to(torch.bfloat16).to(dev)
    vc = torch.randn((nb, hkv, bs, d), generator=g).to(torch.bfloat16).to(dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    if args.op == "copy_blocks":
        n = 4096  # 2 x 4096 x 32 KiB read + written per call
        perm = torch.randperm(nb, generator=g)
        pairs = torch.stack([perm[:n], perm[n:2 * n]], 1).to(torch.int64).to(dev)
        calls = [lambda: pkv.copy_blocks(kc, vc, kc, vc, pairs)]
        moved = n * 2 * block_bytes * 2
        what = "copy-on-write of 4096 random block pairs inside one device pool"
    else:
        n = 2048
        hk = torch.empty((n, hkv, bs, d), dtype=torch.bfloat16).pin_memory()
        hv = torch.empty_like(hk).pin_memory()
        perm = torch.randperm(nb, generator=g)
        out_pairs = torch.stack([perm[:n], torch.arange(n)], 1).to(torch.int64).to(dev)
        in_pairs = torch.stack([torch.arange(n), perm[n:2 * n]], 1).to(torch.int64).to(dev)
        calls = [lambda: pkv.copy_blocks(hk, hv, kc, vc, out_pairs),
                 lambda: pkv.copy_blocks(kc, vc, hk, hv, in_pairs)]
        moved = 2 * n * 2 * block_bytes * 2
        what = "swap of 2048 blocks device -> pinned host, then 2048 host -> device"
    for _ in range(args.warmup):
        flush(1)
        for c in calls:
            c()
    torch.cuda.synchronize()
    if pkv.get_device_error():
        raise RuntimeError("device error during warm-up")
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    K = min(args.steps, 200)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush(i)
        ev[i][0].record(stream)
        for c in calls:
            c()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if pkv.get_device_error():
        raise RuntimeError("device error during the timed steps")
    ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    gbs = moved / (ms * 1e-3) / 1e9
    peak, peak_src = measured_peak()
    line = {
        "metric": f"{args.op} effective GB/s (bytes read + written)", "value": round(gbs, 1),
        "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic (seeded N(0,1) pool)",
        "config": {"workload": what, "block_bytes_per_cache": block_bytes, "pool_blocks": nb,
                   "l2": "flushed between timed steps, outside the timed events"},
        "roofline": ({"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "peak_source": peak_src,
                      "unit": "GB/s", "frac": round(gbs / peak, 4)} if args.op == "copy_blocks" else
                     {"bound": "host link", "achieved": round(gbs, 1), "peak": None, "unit": "GB/s",
                      "frac": None}),
        "gpu_launches": K * len(calls), "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_multi(args):
    """Paged attention for several query tokens per sequence
    (pkv_paged_attention_multi) on a multi-token workload: speculative
    verification of 4 tokens on the Llama-3-8B-shaped batch (HBM-bound:
    GB/s), or 512-token prefill chunks (a contraction: TFLOP/s).  The step is
    the attention call; the chunk's K/V are in the cache before timing (their
    write is the decode step's cache-write kernel)."""
    import paged_kv_cache_22_gb300 as pkv
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pkv.library()
    w, q_cpu, qs_cpu = workloads.MULTI_CONFIGS[args.multi_config](seed=1301 + 1000 * rank
                                                                  + list(workloads.MULTI_CONFIGS).index(
                                                                      args.multi_config))
    shape = workloads.cache_shape(w)
    cdt = workloads.cache_torch_dtype(w.cache_dtype)
    kc = torch.zeros(shape, dtype=cdt, device=dev)
    vc = torch.zeros(shape, dtype=cdt, device=dev)
    k, v, sl = w.all_tokens()
    pkv.kv_reshape_and_cache(k.to(dev), v.to(dev), kc, vc, sl.to(dev), w.kv_scale)
    q, q_start = q_cpu.to(dev), qs_cpu.to(dev)
    tables, lens = w.block_tables.to(dev), w.seq_lens.to(dev)
    q_lens = (qs_cpu[1:] - qs_cpu[:-1]).tolist()
    max_q = max(q_lens)
    # the kernel pkv_paged_attention_multi runs on this workload (the library's own choice)
    multi_kernel = multi_kernel_label(pkv, w, max_q)
    out = torch.empty_like(q)
    workspace = pkv.DecodeWorkspace(dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def call(o=out, qq=q, qs=q_start, tb=tables, ln=lens):
        pkv.paged_attention_multi(o, qq, qs, kc, vc, tb, ln, w.scale, w.kv_scale, max_q=max_q,
                                  max_seq_len=w.max_seq_len, workspace=workspace)

    for _ in range(args.warmup):
        flush(1)
        call()
    torch.cuda.synchronize()
    if pkv.get_device_error():
        raise RuntimeError("device error during warm-up")
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    K = args.steps
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush(i)
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if pkv.get_device_error():
        raise RuntimeError("device error during the timed steps")
    ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in ev) / K, dev)
    lens_l = w.seq_lens.tolist()
    nbytes = metrics.multi_bytes(lens_l, q_lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.cache_dtype,
                                 w.q_dtype, w.block_size)
    flops = metrics.multi_flops(lens_l, q_lens, w.num_q_heads, w.head_dim)
    gbs = ws * nbytes / (ms * 1e-3) / 1e9
    tflops = ws * flops / (ms * 1e-3) / 1e12
    compute = args.multi_config == "prefill_chunk512"

    # end to end: q, offsets, tables and lengths from pinned host memory, out read back
    staged = StagedInputs({"q": q_cpu, "qs": qs_cpu, "tb": w.block_tables, "ln": w.seq_lens}, dev)
    dbuf = staged.dev
    out_host = torch.empty_like(q_cpu).pin_memory()
    h2d = staged.nbytes
    d2h = out_host.numel() * out_host.element_size()
    tot, n_e2e = 0.0, max(10, min(K, 200))
    for i in range(n_e2e + 3):
        flush(i)
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        staged.upload()
        call(out, dbuf["q"], dbuf["qs"], dbuf["tb"], dbuf["ln"])
        out_host.copy_(out, non_blocking=True)
        b_.record(stream)
        b_.synchronize()
        if i >= 3:
            tot += a_.elapsed_time(b_)
    e2e_ms = max_over_ranks(tot / n_e2e, dev)

    hbm_peak, hbm_src = measured_peak()
    tc_peak, tc_src = tensor_peak()
    unit = "TFLOP/s" if compute else "GB/s"
    value = tflops if compute else gbs
    e2e_value = (ws * flops / (e2e_ms * 1e-3) / 1e12) if compute else (ws * nbytes / (e2e_ms * 1e-3) / 1e9)
    line = {
        "metric": ("multi-token paged attention (prefill chunks) TFLOP/s" if compute else
                   "multi-token paged attention (speculative verify) effective HBM GB/s"),
        "value": round(value, 2 if compute else 1), "unit": unit, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) q/k/v, shuffled block pool)",
        "config": {"workload": args.multi_config, "num_seqs": w.num_seqs, "query_rows": int(qs_cpu[-1]),
                   "query_tokens_per_seq": max_q, "sum_seq_len": int(sum(lens_l)),
                   "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "block_size": w.block_size, "cache_dtype": w.cache_dtype,
                   "step": "pkv_paged_attention_multi (the chunk's K/V already in the cache)",
                   "l2": "flushed between timed steps, outside the timed events",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "bytes_per_step": nbytes, "flop_per_step": flops,
        "gbs": round(gbs, 1), "tflops": round(tflops, 3),
        "roofline": ({"bound": "tensor", "achieved": round(tflops, 2), "peak": tc_peak, "peak_source": tc_src,
                      "unit": "TFLOP/s", "frac": round(tflops / tc_peak, 4), "traffic": None,
                      "kernel": multi_kernel} if compute else
                     {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "peak_source": hbm_src,
                      "unit": "GB/s", "frac": round(gbs / hbm_peak, 4), "traffic": None,
                      "kernel": multi_kernel}),
        "e2e": {"value": round(e2e_value, 2 if compute else 1), "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 6)},
        "gpu_launches": K * (2 if "merge_cut_kernel" in multi_kernel else 1), "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_multi(w, q_cpu, qs_cpu, args.cpu_seconds, compute)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def cpu_baseline_multi(w, q_cpu, qs_cpu, seconds: float, compute: bool):
    """The oracle's multi-token attention, as it stands, on this host's cores:
    the first sequences of the workload (enough for ~`seconds`), repeated."""
    import oracle
    _, kc, vc, tables, lens, _, _, _, _ = oracle_sample(w)
    threads = os.cpu_count() or 1
    q_lens = (qs_cpu[1:] - qs_cpu[:-1]).tolist()
    n = 2 if compute else 8  # sequences in the sample
    qs = qs_cpu[:n + 1].numpy().copy()
    qrows = q_cpu[:int(qs[-1])].contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    nbytes = metrics.multi_bytes(lens[:n], q_lens[:n], w.num_q_heads, w.num_kv_heads, w.head_dim,
                                 w.cache_dtype, w.q_dtype, w.block_size)
    flops = metrics.multi_flops(lens[:n], q_lens[:n], w.num_q_heads, w.head_dim)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.paged_attention_multi(qrows, qs, kc, vc, tables[:n], lens[:n], w.scale, w.kv_scale, threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 1000:
            break
    value = reps * flops / el / 1e12 if compute else reps * nbytes / el / 1e9
    return {"value": round(value, 5 if compute else 3), "unit": "TFLOP/s" if compute else "GB/s",
            "cores": threads, "kind": "oracle",
            "sample": f"{reps} passes over the first {n} sequences of the workload, fp64 C loops, {el:.1f} s wall"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=list(workloads.CONFIGS), default="llama3_8b")
    ap.add_argument("--partition-tokens", type=int, default=0,
                    help="0 = balanced split (default); >0 = fixed partitions + reduce")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seqs", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other workloads' decode-only figures of the default run")
    ap.add_argument("--engine", choices=["tensor_cores", "cuda_cores"], default="tensor_cores",
                    help="units that run q.K and P.V for bf16 / fp8 caches")
    ap.add_argument("--window", type=int, default=0,
                    help="> 0: sliding-window decode over the last WINDOW tokens (plus --sinks)")
    ap.add_argument("--sinks", type=int, default=0, help="attention-sink tokens kept with --window")
    ap.add_argument("--cascade", action="store_true",
                    help="decode a shared-prefix workload as prefix pass + suffix decode (prefix_fp8)")
    ap.add_argument("--op", choices=["decode", "copy_blocks", "swap", "multi"], default="decode",
                    help="decode step (default), the block-copy kernels alone, or multi-token attention")
    ap.add_argument("--multi-config", choices=list(workloads.MULTI_CONFIGS), default="verify4_llama3_8b",
                    help="workload of --op multi")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "multi":
        run_multi(args)
    elif args.op != "decode":
        run_copy(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
