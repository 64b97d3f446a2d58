"""Benchmark of the paged decode hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl native|reference]

One step = one decode layer-step of the whole hot path on one batch: the
cache write of the step's new K/V (one appended token per sequence) and
paged attention over every cached token, in one pa_decode_append launch,
then its split-K merge launch.  The FP8 and NVFP4 figures write the new rows
with their own launch (pa_cache_write_fp8 / _nvfp4) and then decode: for
them that measured faster than the fused calls.  The K timed steps are
launched back to back on one stream, CUDA events before the first and after
the last.
The host block manager has already placed the appended tokens (its cost is
reported separately).  Inputs are seeded synthetic tensors shaped like the
workload, resident in HBM; consecutive steps rotate over several
independent layer pools so that each step streams its KV from DRAM rather
than from the 129 MB L2.

The JSON line reports algorithmic KV-read GB/s (sum over sequences of
n * Hkv * d * 2 * bytes, the per-token footprint formula with L = 1) per
step, sequences/s, the decode kernel's roofline against the measured HBM
copy bandwidth, an end-to-end figure through the public API with host
buffers, and the fp64 CPU oracle timed on a bounded sample.

N > 1 (torchrun): every rank runs an independent replica on its own GPU
(the path needs no collective); value = bytes of all ranks / slowest rank.
``--impl reference`` times the fp64 CPU oracle on the same workload instead.
"""
from __future__ import annotations

import os

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import math
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-decode KV-read HBM GB/s (% of GB300 peak) and seqs/s per layer-step"
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------- setup ---
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_value(step_s, nbytes, ws, device):
    """Whole-job figure of N independent replicas: the slowest rank's step
    time (max over ranks) and the bytes of all ranks per that time, GB/s."""
    if ws > 1:
        t = torch.tensor([step_s], device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        step_s = float(t.item())
    return step_s, nbytes * ws / step_s / 1e9


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash():
    """Hash of every kernel and launch source (csrc/*, include/*.h): a DRAM
    traffic figure counts only while it was captured on these sources."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_228_gb300", "csrc")
    inc = os.path.join(ROOT, "include")
    for d in (csrc, inc):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cu", ".cuh", ".cpp", ".h")):
                h.update(f.encode())
                h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """Per-launch DRAM bytes of the decode kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "decode_dram_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(workload)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed loop runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- workloads ---
def make_pools(w, n_pools, device):
    from paged_kv_cache_228_gb300 import workloads as W
    shape = (w.pool_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    pools = []
    for i in range(n_pools):
        k = W.normal_bf16(shape, w.seed * 100 + 2 * i, device, w.outlier_prob, w.outlier_scale)
        v = W.normal_bf16(shape, w.seed * 100 + 2 * i + 1, device, w.outlier_prob,
                          w.outlier_scale)
        pools.append((k, v))
    return pools


def step_inputs(w, device):
    """Block manager (native) places the pre-step tokens and the appended
    ones; returns tables, lens, slots and the host-manager time per append."""
    from paged_kv_cache_228_gb300 import pa
    from paged_kv_cache_228_gb300 import workloads as W
    maxb = w.max_blocks_per_seq
    alloc, tables, lens = pa.replay_script(W.build_script(w), w.num_seqs, w.block_size, maxb,
                                           w.pool_blocks)
    # the step's appends: one native call for the batch (timed)
    ba = pa.BatchAppender(alloc, tables, maxb)
    ones = [1] * w.num_seqs
    st, slots, _, done = ba.append(lens, ones, w.block_size)
    host_us = ba.last_call_us  # the native call (one per step) with its FFI entry
    assert st == pa.PA_OK and done == w.num_seqs
    tab = torch.from_numpy(ba.tables.copy())
    tables = [list(r[r >= 0]) for r in ba.tables]
    return (tables, tab.to(device), torch.tensor(w.seq_lens, dtype=torch.int32, device=device),
            torch.from_numpy(slots.copy()).to(device), host_us)


def fragmentation_report(w, max_len):
    """Host block manager's usage after the step's appends (the pages'
    fragmentation claim): share of reserved slots holding no token, against
    a contiguous cache reserving ``max_len`` (and the batch's own maximum)
    per sequence."""
    from paged_kv_cache_228_gb300 import pa
    from paged_kv_cache_228_gb300 import workloads as W
    alloc, tables, lens = pa.replay_script(W.build_script(w), w.num_seqs, w.block_size,
                                           w.max_blocks_per_seq, w.pool_blocks)
    ba = pa.BatchAppender(alloc, tables, w.max_blocks_per_seq)
    st, _, _, _ = ba.append(lens, [1] * w.num_seqs, w.block_size)
    assert st == pa.PA_OK
    u = pa.allocator_usage(alloc, ba.tables, w.seq_lens, w.block_size)
    return {
        **u,
        "paged_waste": 1.0 - u["tokens_stored"] / u["slots_reserved"],
        "contiguous_waste_at_max_len": 1.0 - u["tokens_logical"] / (w.num_seqs * max_len),
        "contiguous_waste_at_batch_max": 1.0 - u["tokens_logical"] /
                                         (w.num_seqs * max(w.seq_lens)),
        "max_len": max_len,
        "sharing": u["tokens_logical"] / u["tokens_stored"],
    }


def offload_figure(w, device, reps=5):
    """Swap the batch's blocks out to pinned host memory and back in
    (pa_swap_out / pa_swap_in, zero-copy over the host link): GB/s each way."""
    from paged_kv_cache_228_gb300 import pa
    from paged_kv_cache_228_gb300 import workloads as W
    tables, _, _, _, _ = step_inputs(w, "cpu")
    used = sorted({b for t in tables for b in t})
    ids = torch.tensor(used, dtype=torch.int32, device=device)
    shape = (w.pool_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    k = W.normal_bf16(shape, w.seed * 10 + 1, device)
    v = W.normal_bf16(shape, w.seed * 10 + 2, device)
    hk = torch.empty((len(used),) + shape[1:], dtype=torch.bfloat16, pin_memory=True)
    hv = torch.empty_like(hk, pin_memory=True)
    nbytes = 2 * hk.numel() * hk.element_size()
    out = {"blocks": len(used), "bytes": nbytes}
    for name, fn in (("out", lambda: pa.pa_swap_out(k, v, ids, hk, hv)),
                     ("in", lambda: pa.pa_swap_in(hk, hv, ids, k, v))):
        fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        out[name + "_GB_per_s"] = nbytes * reps / (a.elapsed_time(b) / 1e3) / 1e9
    if pa.pa_get_device_error():
        raise RuntimeError("device error during the swap figure")
    return out


def kv_bytes_nvfp4(w):
    """Algorithmic bytes of one NVFP4 layer-step: half a byte per value plus
    one E4M3 block scale per 16 values, K and V, every cached token."""
    return sum(w.seq_lens) * 2 * w.num_kv_heads * (w.head_dim // 2 + w.head_dim // 16)


def kv_bytes(w, bytes_per_scalar=2, scale_bytes=0):
    """Algorithmic KV bytes of one layer-step: per-token footprint
    2 * H_kv * d_h * s (one layer) for every cached token, plus, for FP8,
    the K and V scales of every (block, KV head) a sequence touches."""
    total = 0
    for n in w.seq_lens:
        total += n * 2 * w.num_kv_heads * w.head_dim * bytes_per_scalar
        if scale_bytes:
            total += 2 * (-(-n // w.block_size)) * w.num_kv_heads * scale_bytes
    return total


def block_size_sweep(args, device, peak):
    """The shared-prefix batch (256 forks of a 2048-token prompt, private
    suffixes of 1..512 tokens) at block sizes 8, 16 and 32, each through the
    plain paged decode and the cascade: time per step and per decode call,
    logical KV bytes (the prefix counted once per sequence) and unique KV
    bytes (every stored token once: the least DRAM traffic a step can
    have), and the paging waste of the host block manager's layout."""
    from paged_kv_cache_228_gb300 import workloads as W
    out = {}
    for bs in (8, 16, 32):
        wl = W.shared_prefix(bs)
        frag = fragmentation_report(wl, 2048 + 512)
        unique = frag["tokens_stored"] * 2 * wl.num_kv_heads * wl.head_dim * 2
        nb = kv_bytes(wl)
        for casc in (False, True):
            r = run_native(wl, max(50, args.steps // 20), max(3, args.warmup // 10), device,
                           profile_only=True, cascade=casc)
            dec_s = r["decode_ms_mean"] / 1e3
            out[wl.name + ("_cascade" if casc else "")] = {
                "block_size": bs,
                "kv_bytes_per_step": nb,
                "unique_kv_bytes_per_step": unique,
                "us_per_step": r["ms_per_step"] * 1e3,
                "decode_us": dec_s * 1e6,
                "decode_GB_per_s": nb / dec_s / 1e9,
                "unique_GB_per_s": unique / dec_s / 1e9,
                "unique_frac_of_measured_hbm": unique / dec_s / 1e9 / peak,
                "paged_waste": frag["paged_waste"],
                "dram_bytes_per_step": ncu_traffic(wl.name + ("_cascade" if casc else "")),
                "call": "pa_decode_cascade (the prefix's attention once for all sequences, "
                        "suffixes paged), after pa_cache_write" if casc else "pa_decode_append "
                        "(every sequence walks the shared prefix blocks through its own "
                        "table)",
            }
    return out


# ----------------------------------------------------------- native arm ---
def run_native(w, steps, warmup, device, fp8=False, n_pools=None, sample_clocks=None,
               profile_only=False, cascade=False, nvfp4=False):
    from paged_kv_cache_228_gb300 import pa
    from paged_kv_cache_228_gb300 import workloads as W
    per_pool = w.pool_blocks * w.num_kv_heads * w.block_size * w.head_dim * 2 * 2
    if nvfp4:
        per_pool = per_pool * 9 // 32  # 4.5 bits per value
    if n_pools is None:
        n_pools = max(1, min(8, math.ceil(4 * L2_BYTES / per_pool)))
    pools = make_pools(w, n_pools, device)
    tables, tab, lens, slots, host_us = step_inputs(w, device)
    q = W.normal_bf16((w.num_seqs, w.num_q_heads, w.head_dim), w.seed * 100 + 50, device)
    kn = W.normal_bf16((w.num_seqs, w.num_kv_heads, w.head_dim), w.seed * 100 + 51, device)
    vn = W.normal_bf16((w.num_seqs, w.num_kv_heads, w.head_dim), w.seed * 100 + 52, device)
    out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.bfloat16,
                      device=device)
    if cascade:
        ws_n = pa.pa_decode_cascade_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                                   w.head_dim, w.block_size, w.shared_prefix)
    else:
        ws_n = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                           w.head_dim)
    ws = torch.empty(max(16, ws_n), dtype=torch.uint8, device=device)
    scales = [(None, None)] * n_pools
    if fp8:
        qpools, scales = [], []
        ids = torch.arange(w.pool_blocks, dtype=torch.int32, device=device)
        valid = torch.full((w.pool_blocks,), w.block_size, dtype=torch.int32, device=device)
        for k, v in pools:
            kq = torch.empty(k.shape, dtype=torch.uint8, device=device)
            vq = torch.empty_like(kq)
            ks = torch.empty((w.pool_blocks, w.num_kv_heads), device=device)
            vs = torch.empty_like(ks)
            pa.pa_quantize_fp8(k, v, ids, valid, kq, vq, ks, vs)
            qpools.append((kq, vq))
            scales.append((ks, vs))
        del pools
        pools = qpools
    if nvfp4:
        # every slot of each pool quantised; tensor scales amax / (6 * 448)
        qpools, scales = [], []
        nb, bs, h, d = w.pool_blocks, w.block_size, w.num_kv_heads, w.head_dim
        all_slots = torch.arange(nb * bs, dtype=torch.int64, device=device)
        for k, v in pools:
            gs = (float(k.abs().amax()) / 2688.0, float(v.abs().amax()) / 2688.0)
            c = pa.nvfp4_empty_cache(nb, h, bs, d, device)
            pa.pa_cache_write_nvfp4(k.permute(0, 2, 1, 3).reshape(nb * bs, h, d).contiguous(),
                                    v.permute(0, 2, 1, 3).reshape(nb * bs, h, d).contiguous(),
                                    all_slots, c, *gs)
            qpools.append(c)
            scales.append(gs)
        del pools
        pools = qpools
        torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    pa.pa_get_device_error()

    def step(i, ev=None):
        if nvfp4:
            # NVFP4 cache: the step's tokens written by their own launch, then
            # the decode (measured faster than pa_decode_append_nvfp4 here)
            c, (kg, vg) = pools[i % n_pools], scales[i % n_pools]
            pa.pa_cache_write_nvfp4(kn, vn, slots, c, kg, vg, stream=stream)
            if ev is not None:
                ev[0].record(stream)
            pa.pa_decode_nvfp4(q, c, kg, vg, tab, lens, w.scale, out, ws, stream=stream)
            if ev is not None:
                ev[1].record(stream)
            return
        k, v = pools[i % n_pools]
        ks, vs = scales[i % n_pools]
        if cascade:
            pa.pa_cache_write(kn, vn, slots, k, v, stream=stream)
        elif fp8:
            pa.pa_cache_write_fp8(kn, vn, slots, k, v, ks, vs, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        if cascade:
            # the shared prefix read once for all sequences
            pa.pa_decode_cascade(q, k, v, tab, lens, w.shared_prefix, w.scale, out, ws,
                                 stream=stream)
        elif fp8:
            # FP8 cache: the decode after its own write launch (measured faster
            # than pa_decode_append_fp8 here)
            pa.pa_decode(q, k, v, tab, lens, w.scale, out, ws, k_scale=ks, v_scale=vs,
                         stream=stream)
        else:
            # this step's cache write and decode in one launch
            pa.pa_decode_append(q, kn, vn, slots, k, v, tab, lens, w.scale, out, ws,
                                stream=stream)
        if ev is not None:
            ev[1].record(stream)

    # nvidia-smi samples clocks from before the warm-up to after the timed
    # region, so that no idle gap precedes the timed steps
    sampler = sample_clocks() if sample_clocks else None
    if sampler:
        time.sleep(0.3)  # let nvidia-smi start sampling
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if torch.distributed.is_initialized():
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(steps):
        step(i, evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    if torch.distributed.is_initialized():
        torch.distributed.barrier()
    total_ms = t_start.elapsed_time(t_end)
    dec_ms = [a.elapsed_time(b) for a, b in evs]
    err = pa.pa_get_device_error()
    if err:
        raise RuntimeError(f"device error word 0x{err:x} during the benchmark")
    if profile_only:
        if sampler:
            sampler.stop()
        return {"ms_per_step": total_ms / steps, "decode_ms_mean": statistics.mean(dec_ms)}

    # The headline timed region: exactly `steps` steps launched back to back
    # on one stream with no event between them, so that each step's
    # programmatic dependent launches overlap its start with the previous
    # step's tail, as consecutive calls do in use.  It follows the loop
    # above directly (the GPU does not idle in between).
    if torch.distributed.is_initialized():
        torch.distributed.barrier()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        step(i)
    b.record(stream)
    torch.cuda.synchronize()
    clocks = None
    if sampler:
        sampler.stop()
        clocks = sampler.summary()
    if torch.distributed.is_initialized():
        torch.distributed.barrier()
    stream_ms = a.elapsed_time(b) / steps
    err = pa.pa_get_device_error()
    if err:
        raise RuntimeError(f"device error word 0x{err:x} during the benchmark")

    # The same steps replayed from CUDA graphs (one graph per layer pool;
    # reported, not the headline: a graph boundary ends the overlap).
    graphs = []
    try:
        s2 = torch.cuda.Stream()
        s2.wait_stream(stream)
        with torch.cuda.stream(s2):
            for i in range(n_pools):
                g = torch.cuda.CUDAGraph()
                if nvfp4:
                    c, (kg, vg) = pools[i], scales[i]
                    with torch.cuda.graph(g, stream=s2):
                        pa.pa_cache_write_nvfp4(kn, vn, slots, c, kg, vg, stream=s2)
                        pa.pa_decode_nvfp4(q, c, kg, vg, tab, lens, w.scale, out, ws,
                                           stream=s2)
                    graphs.append(g)
                    continue
                k, v = pools[i]
                ks, vs = scales[i]
                with torch.cuda.graph(g, stream=s2):
                    if fp8:
                        pa.pa_cache_write_fp8(kn, vn, slots, k, v, ks, vs, stream=s2)
                        pa.pa_decode(q, k, v, tab, lens, w.scale, out, ws, k_scale=ks,
                                     v_scale=vs, stream=s2)
                    else:
                        pa.pa_decode_append(q, kn, vn, slots, k, v, tab, lens, w.scale, out,
                                            ws, stream=s2)
                graphs.append(g)
        stream.wait_stream(s2)
        for i in range(max(3, warmup)):
            graphs[i % n_pools].replay()
        torch.cuda.synchronize()
    except Exception as e:  # no graph: the eager loop above is the figure
        graphs = f"unavailable: {type(e).__name__}: {e}"
    graph_ms = None
    if isinstance(graphs, list):
        if torch.distributed.is_initialized():
            torch.distributed.barrier()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            graphs[i % n_pools].replay()
        b.record(stream)
        torch.cuda.synchronize()
        if torch.distributed.is_initialized():
            torch.distributed.barrier()
        graph_ms = a.elapsed_time(b) / steps
        err = pa.pa_get_device_error()
        if err:
            raise RuntimeError(f"device error word 0x{err:x} during the graph replays")

    # end to end through the public API with host buffers
    e2e = run_e2e(w, pools[0], scales[0], tab, lens, slots, q, kn, vn, ws, fp8, stream,
                  max(20, min(steps, 2000)), nvfp4=nvfp4)
    return {
        "ms_per_step": stream_ms,
        "eager_ms_per_step": total_ms / steps,
        "timed": "stream",
        "decode_ms_mean": statistics.mean(dec_ms),
        "decode_ms_median": statistics.median(dec_ms),
        "graph_ms_per_step": graph_ms if graph_ms is not None else graphs,
        "host_append_us": host_us,
        "n_pools": n_pools,
        "pool_bytes": per_pool // (2 if fp8 else 1),
        "clocks": clocks,
        "e2e": e2e,
        # bf16: decode (with the fused cache write) + merge; FP8, NVFP4: + the
        # cache write
        "launches_per_step": 3 if (nvfp4 or fp8) else 2,
    }


def run_e2e(w, pool, scale, tab, lens, slots, q, kn, vn, ws, fp8, stream, steps, nvfp4=False):
    """Per step: one pinned host -> device copy of the step's inputs (q, new
    K/V, slots, block tables, lengths, packed in one staging buffer); cache
    write + decode; device -> host copy of out.  Two buffer sets and a copy
    stream pipeline the steps: step i+1's inputs go up and step i-1's output
    comes down while step i computes."""
    from paged_kv_cache_228_gb300 import pa
    src = dict(q=q, kn=kn, vn=vn, slots=slots, tab=tab, lens=lens)
    offs, total = {}, 0
    for n, t in src.items():
        nb = t.numel() * t.element_size()
        offs[n] = (total, nb)
        total += -(-nb // 256) * 256
    hbuf = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    for n, t in src.items():
        o, nb = offs[n]
        hbuf[o:o + nb].copy_(t.contiguous().reshape(-1).view(torch.uint8).cpu())
    shape = (w.num_seqs, w.num_q_heads, w.head_dim)
    bufs = []
    for _ in range(2):
        dbuf = torch.empty(total, dtype=torch.uint8, device=q.device)
        d = {n: dbuf[o:o + nb].view(src[n].dtype).view(src[n].shape)
             for n, (o, nb) in offs.items()}
        bufs.append((dbuf, d, torch.empty(shape, dtype=torch.bfloat16, device=q.device),
                     torch.empty(shape, dtype=torch.bfloat16, pin_memory=True)))
    h2d_bytes = total
    d2h_bytes = bufs[0][3].numel() * bufs[0][3].element_size()
    xs = torch.cuda.Stream(device=q.device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def h2d(i, first):
        dbuf = bufs[i % 2][0]
        with torch.cuda.stream(xs):
            if not first:
                xs.wait_event(ev_comp[i % 2])  # step i-2 has read this buffer
            dbuf.copy_(hbuf, non_blocking=True)
            ev_in[i % 2].record(xs)

    def compute(i, first):
        _, d, out_d, _ = bufs[i % 2]
        stream.wait_event(ev_in[i % 2])
        if not first:
            stream.wait_event(ev_out[i % 2])  # step i-2's output is down
        if nvfp4:
            pa.pa_cache_write_nvfp4(d["kn"], d["vn"], d["slots"], pool, *scale, stream=stream)
            pa.pa_decode_nvfp4(d["q"], pool, *scale, d["tab"], d["lens"], w.scale, out_d, ws,
                               stream=stream)
        elif fp8:
            k, v = pool
            ks, vs = scale
            pa.pa_cache_write_fp8(d["kn"], d["vn"], d["slots"], k, v, ks, vs, stream=stream)
            pa.pa_decode(d["q"], k, v, d["tab"], d["lens"], w.scale, out_d, ws, k_scale=ks,
                         v_scale=vs, stream=stream)
        else:
            k, v = pool
            pa.pa_decode_append(d["q"], d["kn"], d["vn"], d["slots"], k, v, d["tab"],
                                d["lens"], w.scale, out_d, ws, stream=stream)
        ev_comp[i % 2].record(stream)

    def d2h(i):
        _, _, out_d, out_h = bufs[i % 2]
        with torch.cuda.stream(xs):
            xs.wait_event(ev_comp[i % 2])
            out_h.copy_(out_d, non_blocking=True)
            ev_out[i % 2].record(xs)

    def run(n):
        h2d(0, True)
        for i in range(n):
            compute(i, i < 2)
            if i + 1 < n:
                h2d(i + 1, i + 1 < 2)
            d2h(i)

    run(5)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(steps)
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / steps
    return {"ms_per_step": ms, "h2d_bytes_per_step": h2d_bytes,
            "d2h_bytes_per_step": d2h_bytes,
            "pipeline": "two buffer sets; uploads and downloads on a copy stream overlap "
                        "the neighbouring steps' kernels"}


# ------------------------------------------------------------ oracle arm ---
_ORACLE_INPUTS = {}


def _oracle_inputs(w, b, device):
    """Sequence b's blocks and queries for the oracle, as float arrays: the
    ceil(n_b / block_size) blocks it owns, generated from b's own seeds (the
    oracle gathers through its local ids 0, 1, 2, ...).  Generated once per
    process and kept, so the timed samples spend their time in the oracle."""
    key = (w.name, b)
    if key not in _ORACLE_INPUTS:
        from paged_kv_cache_228_gb300 import workloads as W
        nblk = -(-w.seq_lens[b] // w.block_size)
        shape = (nblk, w.num_kv_heads, w.block_size, w.head_dim)
        kk = W.normal_bf16(shape, w.seed * 1000 + b, device).float().cpu().numpy()
        vv = W.normal_bf16(shape, w.seed * 1000 + b + 500, device).float().cpu().numpy()
        qq = W.normal_bf16((w.num_q_heads, w.head_dim), w.seed * 1000 + b + 900,
                           device).double().cpu().numpy()
        _ORACLE_INPUTS[key] = (kk, vv, qq, np.arange(nblk))
    return _ORACLE_INPUTS[key]


def oracle_sample(w, device, budget_s, part=(0, 1)):
    """Time the fp64 oracle (as it stands) on whole (sequence, KV head)
    segments of this workload -- the sequences b with b % part[1] ==
    part[0], repeated -- until about ``budget_s`` seconds of oracle time;
    returns (GB/s, segments, seconds).  Runs on the host alone: the inputs
    come from the seeded generators, the lengths from the workload."""
    from oracle import paged_attention as OPA
    done_bytes, done, t_used = 0, 0, 0.0
    G = w.group
    mine = [b for b in range(w.num_seqs) if b % part[1] == part[0]]
    while mine:
        for b in mine:
            kk, vv, qq, local = _oracle_inputs(w, b, device)
            for gk in range(w.num_kv_heads):
                t0 = time.perf_counter()
                kc = OPA.gather_sequence(kk[:, gk:gk + 1], local, w.seq_lens[b],
                                         w.block_size)[:, 0]
                vc = OPA.gather_sequence(vv[:, gk:gk + 1], local, w.seq_lens[b],
                                         w.block_size)[:, 0]
                for h in range(gk * G, (gk + 1) * G):
                    OPA.attend(qq[h], kc, vc, w.scale)
                t_used += time.perf_counter() - t0
                done += 1
                done_bytes += w.seq_lens[b] * w.head_dim * 2 * 2
                if t_used >= budget_s:
                    return done_bytes / t_used / 1e9, done, t_used
    return done_bytes / max(t_used, 1e-9) / 1e9, done, t_used


def _oracle_part(args):
    """Worker of oracle_sample_all_cores (a spawned process)."""
    name, rank, n, budget = args
    from paged_kv_cache_228_gb300 import workloads as W
    gbs, segs, secs = oracle_sample(W.WORKLOADS[name](), "cpu", budget, (rank, n))
    return gbs * secs * 1e9, segs, secs


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the
    cpu_baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_sample_all_cores(name, budget_s):
    """The oracle on every host core: one spawned process per core, each on
    its share of the sequences (single-threaded BLAS in each); returns
    (GB/s = all bytes / the slowest process's oracle time, segments, cores)."""
    import multiprocessing as mp
    n = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(n) as pool:
        res = pool.map(_oracle_part, [(name, r, n, budget_s) for r in range(n)])
    total = sum(r[0] for r in res)
    return total / max(r[2] for r in res) / 1e9, sum(r[1] for r in res), n


def workload_config(w, world_size=1):
    """The workload's identity, the same dict in both arms' JSON lines (how
    each arm ran goes in its own keys)."""
    return {"workload": w.name, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "kv_bytes_per_step": kv_bytes(w),
            "mean_seq_len": sum(w.seq_lens) / w.num_seqs,
            "parallelism": f"{world_size} independent replicas" if world_size > 1 else "none"}


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    # about 10x the cpu_baseline budget over the whole run (120 s by default)
    budget = 10.0 * args.cpu_budget / max(1, args.steps + args.warmup)
    vals, secs = [], []
    segs = 0
    for i in range(args.warmup + args.steps):
        v, n, t = oracle_sample(w, "cpu", budget)
        if i >= args.warmup:
            vals.append(v)
            secs.append(t)
            segs = n
    value = statistics.mean(vals)
    cpu = {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
           "cpu_model": cpu_model(),
           "sample": f"{segs} whole (sequence, KV head) segments of {w.name} per step, "
                     f"fp64 numpy, single-threaded BLAS"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            # each step is a bounded sample of the workload (above), not the
            # whole batch: its oracle time
            "ms_per_step": 1e3 * statistics.mean(secs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "setup": {"arm": "the fp64 CPU oracle on host cores",
                      "step": f"a bounded sample of {budget:.2f} s of oracle time"},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ------------------------------------------------------------------ main ---
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="llama3.1-8b")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle time for cpu_baseline; the reference "
                         "arm spends 10x this over its warm-up and timed steps")
    ap.add_argument("--fp8", action="store_true",
                    help="with --profile: run the FP8 cache path of the workload")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="with --profile: a smaller batch of the 128K workload "
                         "(ncu captures that must stay a few GB)")
    ap.add_argument("--nvfp4", action="store_true",
                    help="with --profile: run the NVFP4 cache path of the workload")
    ap.add_argument("--cascade", action="store_true",
                    help="with --profile on a shared_prefix workload: pa_decode_cascade")
    ap.add_argument("--profile", action="store_true",
                    help="only the warm-up and timed steps of the main workload "
                         "(for ncu captures); prints the step time")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    from paged_kv_cache_228_gb300 import workloads as W
    if args.num_seqs is not None:
        if not args.profile or args.workload != "llama3.1-70b-128k":
            ap.error("--num-seqs only goes with --profile --workload llama3.1-70b-128k")
        w = W.llama31_70b_128k(num_seqs=args.num_seqs)
    else:
        w = W.WORKLOADS[args.workload]()
    if args.impl == "reference":
        run_reference(args, w)
        return

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    device = f"cuda:{local}" if ws > 1 else "cuda"
    from paged_kv_cache_228_gb300 import build as B
    if rank == 0:
        B.build()
    if ws > 1:
        torch.distributed.barrier()
    from paged_kv_cache_228_gb300 import pa
    pa.lib()

    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_index = int(vis.split(",")[local])
        except ValueError:
            pass
    if args.profile:
        if args.cascade and not w.shared_prefix:
            ap.error("--cascade needs a shared_prefix workload")
        r = run_native(w, args.steps, args.warmup, device, fp8=args.fp8,
                       n_pools=1 if w.num_seqs * max(w.seq_lens) > 10 ** 6 else None,
                       profile_only=True, cascade=args.cascade, nvfp4=args.nvfp4)
        print(json.dumps({"workload": w.name, "ms_per_step": r["ms_per_step"],
                          "decode_ms_mean": r["decode_ms_mean"]}))
        return
    res = run_native(w, args.steps, args.warmup, device,
                     sample_clocks=(lambda: ClockSampler(gpu_index)) if rank == 0 else None)
    nbytes = kv_bytes(w)
    step_s = res["ms_per_step"] / 1e3
    step_s, value = replica_value(step_s, nbytes, ws, device)
    peak, peak_kind = peaks()
    # roofline: the decode + merge launch pair over the timed region (the K
    # steps back to back, each a programmatic dependent of the one before);
    # the same pair timed with CUDA events around every call is reported
    # beside it (events between calls end that overlap)
    achieved = nbytes / (res["ms_per_step"] / 1e3) / 1e9
    dec_s = res["decode_ms_mean"] / 1e3
    achieved_eager = nbytes / dec_s / 1e9
    secondary = {}
    if rank == 0 and not args.no_secondary and args.workload == "llama3.1-8b":
        # paging tax: the same batch with contiguous physical blocks; the
        # other report-only shapes (decode kernel pair only, logical bytes)
        for wl, casc in ((W.contiguous(w), False), (W.llama32_1b(), False)):
            r = run_native(wl, max(50, args.steps // 20), max(3, args.warmup // 10), device,
                           profile_only=True, cascade=casc)
            nb = kv_bytes(wl)
            secondary[wl.name + ("_cascade" if casc else "")] = {
                "kv_bytes_per_step": nb,
                "decode_us": r["decode_ms_mean"] * 1e3,
                "decode_GB_per_s": nb / (r["decode_ms_mean"] / 1e3) / 1e9,
                "us_per_step": r["ms_per_step"] * 1e3,
            }
        secondary.update(block_size_sweep(args, device, peak))
        r = run_native(w, max(50, args.steps // 20), max(3, args.warmup // 10), device,
                       fp8=True)
        nb = kv_bytes(w, 1, 4)
        secondary[w.name + "_fp8"] = {
            "kv_bytes_per_step": nb,
            "decode_us": r["decode_ms_mean"] * 1e3,
            "decode_GB_per_s": nb / (r["decode_ms_mean"] / 1e3) / 1e9,
            "hbm_frac_of_measured": nb / (r["decode_ms_mean"] / 1e3) / 1e9 / peak,
            "us_per_step": r["ms_per_step"] * 1e3,
            "kernel": "paged_decode_tc_fp8_kernel<128> + merge",
            "note": "pa_cache_write_fp8 of the step's tokens + pa_decode (+ merge) on an E4M3 "
                    "cache; bytes: codes and per-(block, head) scales",
        }
        r = run_native(w, max(50, args.steps // 20), max(3, args.warmup // 10), device,
                       nvfp4=True)
        nb = kv_bytes_nvfp4(w)
        secondary[w.name + "_nvfp4"] = {
            "kv_bytes_per_step": nb,
            "decode_us": r["decode_ms_mean"] * 1e3,
            "decode_GB_per_s": nb / (r["decode_ms_mean"] / 1e3) / 1e9,
            "hbm_frac_of_measured": nb / (r["decode_ms_mean"] / 1e3) / 1e9 / peak,
            "us_per_step": r["ms_per_step"] * 1e3,
            "e2e_us_per_step": r["e2e"]["ms_per_step"] * 1e3,
            "note": "pa_cache_write_nvfp4 of the step's tokens + pa_decode_nvfp4 (+ merge); "
                    "bytes: 4-bit values and E4M3 block scales",
        }
        secondary["offload"] = offload_figure(w, device)
        secondary["offload"]["note"] = (
            "pa_swap_out / pa_swap_in of every block the 8B batch uses, between HBM and "
            "pinned host memory read and written in place by the kernel")
        secondary["fragmentation"] = {w.name: fragmentation_report(w, 4096)}
        for bs in (8, 16, 32):
            secondary["fragmentation"][W.shared_prefix(bs).name] = fragmentation_report(
                W.shared_prefix(bs), 2048 + 512)
        c = secondary[W.contiguous(w).name]["decode_GB_per_s"]
        # both sides timed the same way (CUDA events around every call)
        secondary["paging_tax"] = {
            "scattered_decode_GB_per_s": achieved_eager, "contiguous_decode_GB_per_s": c,
            "tax": 1.0 - achieved_eager / c}
    if rank == 0 and not args.no_secondary and args.workload != "llama3.1-70b-128k":
        wl = W.llama31_70b_128k()
        for fmt in ("bf16", "fp8", "nvfp4"):
            fp8, fp4 = fmt == "fp8", fmt == "nvfp4"
            r = run_native(wl, max(20, args.steps // 50), max(3, args.warmup // 10), device,
                           fp8=fp8, n_pools=1, nvfp4=fp4)
            nb = kv_bytes_nvfp4(wl) if fp4 else kv_bytes(wl, 1 if fp8 else 2, 4 if fp8 else 0)
            dec_gbs = nb / (r["decode_ms_mean"] / 1e3) / 1e9
            secondary["llama3.1-70b-128k_" + fmt] = {
                "roofline": {
                    "bound": "hbm", "achieved": dec_gbs, "peak": peak, "unit": "GB/s",
                    "frac": dec_gbs / peak,
                    "traffic": ncu_traffic(wl.name if fmt == "bf16" else f"{wl.name}_{fmt}"),
                    "kernel": {"bf16": "paged_decode_ws_kernel<128,bf16>",
                               "fp8": "paged_decode_tc_fp8_kernel<128>",
                               "nvfp4": "paged_decode_nvfp4_kernel<128>"}[fmt] + " + merge "
                              "(per launch pair, CUDA events around each call)",
                    "peak_source": peak_kind},
                "kv_bytes_per_step": nb,
                "us_per_step": r["ms_per_step"] * 1e3,
                "GB_per_s": nb / (r["ms_per_step"] / 1e3) / 1e9,
                "decode_us": r["decode_ms_mean"] * 1e3,
                "decode_GB_per_s": nb / (r["decode_ms_mean"] / 1e3) / 1e9,
                "hbm_frac_of_measured": nb / (r["decode_ms_mean"] / 1e3) / 1e9 / peak,
                "seqs_per_s": wl.num_seqs / (r["ms_per_step"] / 1e3),
                "graph_us_per_step": (r["graph_ms_per_step"] * 1e3
                                      if isinstance(r["graph_ms_per_step"], float) else
                                      r["graph_ms_per_step"]),
            }
    cpu = None
    if rank == 0:
        v, segs, secs = oracle_sample(w, "cpu", args.cpu_budget)
        cpu = {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "cpu_model": cpu_model(),
               "sample": f"{segs} whole (sequence, KV head) segments of {w.name}, "
                         f"the batch repeated ({secs:.1f} s of oracle time), fp64 numpy, "
                         f"single-threaded BLAS"}
        if not args.no_secondary and args.workload in W.WORKLOADS:
            va, sega, cores = oracle_sample_all_cores(args.workload, args.cpu_budget / 3)
            cpu["all_cores"] = {"value": va, "unit": "GB/s", "cores": cores,
                                "sample": f"{sega} segments, one process per core"}
    e2e = res["e2e"]
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 K/V, Q; scattered blocks)",
            "config": workload_config(w, ws),
            "setup": {
                "l2": f"inputs larger than L2: {res['n_pools']} rotating layer pools of "
                      f"{res['pool_bytes'] / 1e9:.2f} GB",
                "step": "pa_decode_append: cache write fused into the decode launch, "
                        "+ merge launch",
                "timing": "the timed steps launched back to back on one stream (no event "
                          "between steps); CUDA events before the first and after the last",
            },
            "seqs_per_s": w.num_seqs * ws / step_s,
            "us_per_step": step_s * 1e6,
            "hbm_frac": value / ws / peak,
            "eager_us_per_step": res["eager_ms_per_step"] * 1e3,
            "eager_value": nbytes / res["eager_ms_per_step"] * 1e3 / 1e9 * ws,
            "graph_us_per_step": (res["graph_ms_per_step"] * 1e3
                                  if isinstance(res["graph_ms_per_step"], float)
                                  else res["graph_ms_per_step"]),
            "host_block_manager_us_per_step": res["host_append_us"],
            "host_block_manager_us_per_append": res["host_append_us"] / w.num_seqs,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": ncu_traffic(w.name),
                         "kernel": "paged_decode_ws_kernel<128,bf16> (fused append) + "
                                   "paged_decode_merge_kernel: the launch pair of each step, "
                                   "CUDA events around the timed region of back-to-back steps",
                         "peak_source": peak_kind,
                         "pair_eager": {"achieved": achieved_eager,
                                        "frac": achieved_eager / peak,
                                        "us": dec_s * 1e6,
                                        "timing": "CUDA events around every call of a separate "
                                                  "loop of the same steps"}},
            "cpu_baseline": cpu,
            "e2e": {"value": nbytes / (e2e["ms_per_step"] / 1e3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                    "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
                    "ms_per_step": e2e["ms_per_step"], "pipeline": e2e["pipeline"]},
            "gpu_launches": res["launches_per_step"] * args.steps,
            "clocks": res["clocks"],
            "secondary": secondary,
        }
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
