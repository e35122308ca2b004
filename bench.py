#!/usr/bin/env python
"""Benchmark: sink+window attention over the 30-layer rolling KV cache stack.

Workload (default ``stream30``): Wan2.1-1.3B-shaped self-attention -- 30 layers,
12 heads of dimension 128, 1560 tokens per latent frame, chunks of 3 frames,
a 3-frame sink and a 9-frame window, bf16.  One step = one whole stream from an
empty cache: 20 chunks (60 latent frames), each chunk attended and committed in
all 30 layers (600 ll_attend_chunk calls with commit; independent seeded q/k/v
per layer and chunk, all resident in HBM before timing starts: 25.9 GB, well
above the 126 MB L2, so no flush is needed between steps).  The warm-up chunks
attend to 3, 6, 9 and 12 frames, the rest to 15 (23400 keys); the first FIFO
eviction happens at the commit of chunk 4.

Printed (rank 0, one JSON line): latent frames/s of the stack (all ranks),
TFLOPS, the attend kernel's roofline against the measured bf16 peak, the
append kernel's HBM bandwidth, an end-to-end number with host<->device copies,
the float64 oracle's CPU throughput on a bounded sample, and sampled clocks.

``--impl reference`` times the float64 CPU oracle instead (the only
reference implementation there is), on bounded samples of the same workload.
Multi-GPU (torchrun): every rank runs its own independent stream (weak
scaling, no collective on the data path); timing is max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import llsynth  # noqa: E402

METRIC = "sink+window attention TFLOPS & latent frames/s (30-layer stack); % bf16 peak"
UNIT = "latent_frames/s"
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ----------------------------------------------------------------------------
# workload arithmetic (what counts as algorithmic work)
# ----------------------------------------------------------------------------

def resident_count(S, W, n):
    return min(S, n) + min(W, max(0, n - S))


def stream_plan(shape: llsynth.Shape, chunks: int):
    """Per chunk: (t0, keys attended).  Work counts only the keys the method attends."""
    T, C = shape.tokens_per_frame, shape.chunk_frames
    plan = []
    for c in range(chunks):
        t0 = c * C
        plan.append((t0, (resident_count(shape.sink_frames, shape.window_frames, t0) + C) * T))
    return plan


def attend_flops(Lq, Lkv, H, d):
    return 4.0 * Lq * Lkv * H * d


def masked_pairs(Lq, La, Lb, block):
    """Query-key pairs an attention visits: every row sees La cached keys plus, of the Lb
    fresh keys, all of them (block None) or the blocks up to its own (block-causal)."""
    if block is None:
        return Lq * (La + Lb)
    total = Lq * La
    for g0 in range(0, Lq, block):
        total += min(block, Lq - g0) * min(Lb, g0 + block)
    return total


def chunk_pairs(shape, t0, chunk_mask):
    """Pairs of one chunk attend at frame t0 (frame mask: the chunk's keys in frame blocks)."""
    T, C = shape.tokens_per_frame, shape.chunk_frames
    L = C * T
    La = resident_count(shape.sink_frames, shape.window_frames, t0) * T
    return masked_pairs(L, La, L, T if (chunk_mask == "frame" and C > 1) else None)


def prefill_pairs(shape, n, chunk_mask, recache_scope):
    """Pairs of one recache prefill after n committed frames."""
    T, C, S, W = shape.tokens_per_frame, shape.chunk_frames, shape.sink_frames, shape.window_frames
    block = (1 if chunk_mask == "frame" else C) * T
    sink = min(S, n)
    win = min(W, max(0, n - S))
    if recache_scope == "window":
        return masked_pairs(win * T, sink * T, win * T, block)
    R = (sink + win) * T
    return masked_pairs(R, 0, R, block)


def pair_flops(pairs, H, d):
    return 4.0 * pairs * H * d


def set_options(ll, cache, args):
    ll.ll_set_chunk_mask(cache, args.chunk_mask)
    ll.ll_set_recache_scope(cache, args.recache_scope)
    if args.pair:
        ll.ll_debug_pair_kernel(cache, True)


def append_bytes(shape: llsynth.Shape, frames_written: int, kv_elem_bytes: int = 4):
    """K and V: read from the chunk tensors (or the e4m3 staging) and written to the cache,
    per committed frame.  kv_elem_bytes: bytes of one K element plus one V element in the
    cache (4 in bf16, 3 with e4m3 keys, 2 with e4m3 keys and values)."""
    return 2 * frames_written * shape.tokens_per_frame * shape.heads * shape.head_dim * kv_elem_bytes


def kv_elem_bytes(args):
    return 2 if args.kv_fp8 else 3 if args.key_fp8 else 4


def frames_written(shape: llsynth.Shape, t0: int):
    S, W, C = shape.sink_frames, shape.window_frames, shape.chunk_frames
    lo = max(S, t0 + C - W)
    return sum(1 for f in range(t0, t0 + C) if f < S or f >= lo)


# ----------------------------------------------------------------------------
# environment: distributed, peaks, clocks
# ----------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while work runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


def code_hash(texts):
    """Hash of C++/CUDA source texts with // comments, trailing blanks and blank lines removed,
    so that an edit to comments alone leaves it unchanged (the sources hold no // inside a
    string literal and no block comments)."""
    h = hashlib.sha256()
    for text in texts:
        for line in text.splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
        h.update(b"\0")
    return h.hexdigest()[:16]


def kernel_source_hash():
    """Code hash of the attention kernel's sources (ll_attend_tc.cu + ll_tc_common.cuh + ll_internal.h)."""
    texts = []
    for f in ("ll_attend_tc.cu", "ll_tc_common.cuh", "ll_internal.h"):
        with open(os.path.join(ROOT, "windowed_sink_attention_ll_b300", "csrc", f)) as fh:
            texts.append(fh.read())
    return code_hash(texts)


def attend_bytes(shape: llsynth.Shape, resident_frames: int):
    """Algorithmic DRAM bytes of one attend launch: q, the resident cache rows, the chunk's
    k and v, and out (bf16)."""
    row = shape.heads * shape.head_dim * 2
    L = shape.chunk_tokens
    return (3 * L + 2 * resident_frames * shape.tokens_per_frame + L) * row


def traffic_record():
    """DRAM bytes per attend launch from the committed ncu summary, if it matches this source."""
    p = os.path.join(ROOT, "profiles", "attend_tc_traffic.txt")
    if not os.path.exists(p):
        return None
    rec = {}
    with open(p) as f:
        for line in f:
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                rec[k.strip()] = v.strip()
    if rec.get("source_hash") != kernel_source_hash():
        return None
    return rec


def traffic_per_launch(alg_bytes_per_launch: float):
    """Measured DRAM bytes per launch, scaled from the captured launch to this workload's
    average launch by algorithmic bytes (the traffic grows with the keys read)."""
    rec = traffic_record()
    if rec is None:
        return None, None
    measured = float(rec["dram_bytes_per_launch"])
    captured_alg = float(rec["algorithmic_bytes_per_launch"])
    return measured * alg_bytes_per_launch / captured_alg, rec.get("workload")


# ----------------------------------------------------------------------------
# CPU baseline: the float64 oracle on a bounded sample
# ----------------------------------------------------------------------------

def oracle_rate(shape: llsynth.Shape, budget_s: float = 12.0):
    """Attention flop/s of the float64 oracle on one steady-state attend (sampled rows)."""
    import numpy as np

    import oracle

    try:
        from threadpoolctl import threadpool_info

        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        threads = os.cpu_count()
    H, d, T, S, W, C = (shape.heads, shape.head_dim, shape.tokens_per_frame, shape.sink_frames,
                        shape.window_frames, shape.chunk_frames)
    orc = oracle.OracleCache(1, H, d, T, S, W, C)
    rng = np.random.default_rng(0)
    L = C * T
    z = rng.standard_normal((L, H, d))
    steady = S + W
    while orc.state(0)[0] < steady:
        orc.commit(0, z, z)
    q = rng.standard_normal((L, H, d))
    Lkv = (resident_count(S, W, orc.state(0)[0]) + C) * T
    rows, done_rows, spent = 16, 0, 0.0
    while True:
        sel = np.arange(rows) * (L // rows)
        t = time.perf_counter()
        orc.attend(0, q, z, z, commit=False, rows=sel)
        dt = time.perf_counter() - t
        spent += dt
        done_rows += rows
        left = budget_s - spent
        if left < 0.6 * dt:
            break
        # size the next call to fit what is left of the budget
        rows = int(max(16, min(L, rows * left / dt * 0.8)))
    rate = attend_flops(done_rows, Lkv, H, d) / spent
    sample = ("float64 oracle attend of %d sampled query rows (all %d heads, %d keys) of a steady-state "
              "chunk, %.1f s; rate scaled by the step's attention flops" % (done_rows, H, Lkv, spent))
    return rate, threads, sample


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def timed_region(args, world, local, caches, step, profile_every=1):
    """W warm-up steps, then exactly K timed steps between barriers and synchronisations.

    The library brackets one launch in every `profile_every` of each kind with CUDA events
    inside the timed region (fewer event records perturb the step less).
    Returns (ms, clocks, launches, per-kind (bracketed launches, ms) summed over ``caches``)."""
    import windowed_sink_attention_ll_b300 as ll

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    kinds = (ll.LL_KERNEL_ATTEND, ll.LL_KERNEL_PREFILL, ll.LL_KERNEL_COPY)
    for cache in caches:
        for kind in kinds:
            ll.ll_profile_read(cache, kind)
        ll.ll_profile_enable(cache, True, profile_every)
    launches0 = ll.ll_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    launches = ll.ll_launch_count() - launches0
    prof = {}
    for cache in caches:
        ll.ll_profile_enable(cache, False)
        for kind in kinds:
            n, ms_k = ll.ll_profile_read(cache, kind)
            a, b = prof.get(kind, (0, 0.0))
            prof[kind] = (a + n, b + ms_k)
    return ev0.elapsed_time(ev1), clk.summary(), launches, prof


def attend_kernel_name(args):
    if args.kv_fp8:
        return "attend_tc_kernel<128, e4m3 keys and values>"
    if args.key_fp8:
        return "attend_tc_kernel<128, e4m3 keys>"
    return "attend_pair_kernel (CTA pair)" if args.pair else "attend_tc_kernel<128>"


def cache_dtype(ll, args):
    if args.kv_fp8:
        return ll.LL_FP8
    return ll.LL_BF16_K8 if args.key_fp8 else ll.LL_BF16


def peak_scale(args):
    """Tensor peak of the attention relative to the bf16 peak.  With e4m3 keys Q K^T (half
    the flops) runs at the FP8 rate, twice the bf16 rate (the nominal ratio, 4.5 / 2.25
    PFLOP/s), and P V at the bf16 rate: 1 / (0.5 / 2 + 0.5 / 1) = 4 / 3.  With e4m3 values
    as well P V runs on fp16 operands, at the same rate as bf16: 4 / 3 again."""
    return 4.0 / 3.0 if args.key_fp8 else 1.0


def tensor_roofline(kernel, flops, n, ms, pk, pk_src, sustained=True, scale=1.0):
    """Tensor-bound roofline object of one kernel: flops over its summed CUDA-event time.
    scale: the kernel's peak relative to the bf16 peak (4/3 with e4m3 keys, see peak_scale)."""
    achieved = flops / (ms / 1e3) / 1e12 if ms > 0 else 0.0
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    peak = pk.get(key, FALLBACK[key]) * scale
    src = "%s %s (%s)" % (pk_src, key, "kernel timed inside a long step" if sustained else "kernel timed in isolation")
    if scale != 1.0:
        src += " x %.4g: Q K^T at the FP8 rate (2x bf16, nominal ratio), P V at the bf16 rate" % scale
    return {"kernel": kernel, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak,
            "peak_source": src,
            "frac_of_burst_peak": achieved / (pk.get("bf16_tflops", FALLBACK["bf16_tflops"]) * scale),
            "frac_of_nominal_2250": achieved / (2250.0 * scale),
            "launches": n, "ms_per_launch": ms / max(n, 1), "flops_per_launch": flops / max(n, 1)}


def hbm_roofline(kernel, nbytes, n, ms, pk):
    achieved = nbytes / (ms / 1e3) / 1e9 if ms > 0 else 0.0
    peak = pk.get("hbm_gbs", FALLBACK["hbm_gbs"])
    return {"kernel": kernel, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "frac_of_nominal_8000": achieved / 8000.0, "launches": n,
            "us_per_launch": 1e3 * ms / max(n, 1), "bytes_per_launch": nbytes / max(n, 1)}


def base_result(args, world, value, ms_max, config):
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 (keys and values e4m3)" if args.kv_fp8 else "bf16 (keys e4m3)" if args.key_fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v per layer and chunk, Wan2.1-1.3B shapes; no weights)",
        "config": config,
    }


def shape_config(shape, extra):
    cfg = {"layers": shape.layers, "heads": shape.heads, "head_dim": shape.head_dim,
           "tokens_per_frame": shape.tokens_per_frame, "sink_frames": shape.sink_frames,
           "window_frames": shape.window_frames, "chunk_frames": shape.chunk_frames}
    cfg.update(extra)
    return cfg


def run_ours(args, world, rank, local):
    import windowed_sink_attention_ll_b300 as ll

    shape = llsynth.STREAM30
    chunks = llsynth.STREAM30_CHUNKS
    H, d, T, S, W, C = (shape.heads, shape.head_dim, shape.tokens_per_frame, shape.sink_frames,
                        shape.window_frames, shape.chunk_frames)
    L = C * T
    plan = stream_plan(shape, chunks)
    step_frames = chunks * C
    P = args.passes  # query passes per chunk through all layers; the last one commits
    step_flops = sum(pair_flops(chunk_pairs(shape, t0, args.chunk_mask), H, d) for t0, _ in plan) * shape.layers * P

    # inputs: independent seeded q/k/v per (rank, layer, chunk), resident before timing; with
    # several passes, the earlier (non-committing) passes get their own q/k/v too
    inputs = [[tuple(llsynth.seeded_normal(("bench", rank, l, c, t), (L, H, d), device="cuda") for t in "qkv")
               for c in range(chunks)] for l in range(shape.layers)]
    early = [[[tuple(llsynth.seeded_normal(("bench-pass", rank, l, c, p, t), (L, H, d), device="cuda") for t in "qkv")
               for p in range(P - 1)] for c in range(chunks)] for l in range(shape.layers)]
    outs = [torch.empty((L, H, d), dtype=torch.bfloat16, device="cuda") for _ in range(shape.layers)]
    cache = ll.ll_cache_create(shape.layers, H, d, T, S, W, C, cache_dtype(ll, args))
    set_options(ll, cache, args)
    stream = torch.cuda.current_stream()

    def step():
        ll.ll_reset(cache)
        st = torch.cuda.current_stream()  # the capture stream while a CUDA graph is recorded
        for c in range(chunks):
            # as a denoising loop runs the stack: every pass through all layers, the last commits
            for p in range(P - 1):
                for l in range(shape.layers):
                    q, k, v = early[l][c][p]
                    ll.ll_attend_chunk(cache, l, q, k, v, outs[l], False, st)
            for l in range(shape.layers):
                q, k, v = inputs[l][c]
                ll.ll_attend_chunk(cache, l, q, k, v, outs[l], True, st)

    if args.graph:
        return run_graph(args, world, local, ll, cache, step, step_frames, step_flops, shape, L, chunks)
    ms, clocks, launches, prof = timed_region(args, world, local, [cache], step, profile_every=10)
    ms_max = max_over_ranks(ms, world)
    n_att, ms_att = prof[ll.LL_KERNEL_ATTEND]
    n_cp, ms_cp = prof[ll.LL_KERNEL_COPY]
    # the bracketed launches are one in ten of each kind: layers 0, 10, 20 of every pass of every chunk
    att_sampled = sum(pair_flops(chunk_pairs(shape, t0, args.chunk_mask), H, d) * 3 * P
                      for t0, _ in plan) * args.steps
    cp_sampled = sum(append_bytes(shape, frames_written(shape, t0), kv_elem_bytes(args)) * 3
                     for t0, _ in plan) * args.steps
    pk, pk_src = peaks()
    config = {"workload": "stream30: 30 layers x 20 chunks (60 latent frames), H=12, d=128, "
                          "T=1560, C=3, S=3, W=9, %s" % (
                              "1 committed pass per chunk" if P == 1 else
                              "%d passes per chunk through all layers (the last commits)" % P)}
    config.update(shape_config(shape, {
        "chunks": chunks, "passes": P,
        "l2": "inputs larger than L2 (%.1f GB q/k/v + %.2f GB cache per rank)" % (
            3 * L * H * d * 2 * chunks * shape.layers * P / 1e9, 2 * shape.layers * (S + W) * T * H * d * 2 / 1e9),
        "chunk_mask": args.chunk_mask, "recache_scope": args.recache_scope,
        "parallelism": "replicas x%d (independent streams, no collective)" % world}))
    result = base_result(args, world, step_frames * args.steps * world / (ms_max / 1e3), ms_max, config)
    roof = tensor_roofline(attend_kernel_name(args), att_sampled, n_att, ms_att, pk, pk_src, scale=peak_scale(args))
    roof["sampling"] = "one launch in ten of each kind bracketed with CUDA events in the timed region"
    alg = sum(attend_bytes(shape, resident_count(S, W, t0)) for t0, _ in plan) / len(plan)
    roof["algorithmic_bytes_per_launch"] = alg
    roof["traffic"], src = traffic_per_launch(alg) if not (args.pair or args.key_fp8) else (None, None)
    if src:
        roof["traffic_source"] = "ncu capture of %s, scaled by algorithmic bytes" % src
    in_stream = hbm_roofline("copy_frames_kernel", cp_sampled, n_cp, ms_cp, pk)
    in_stream["how"] = "one commit copy in ten bracketed singly with CUDA events inside the timed stream"
    result.update({
        "tflops": step_flops * args.steps * world / (ms_max / 1e3) / 1e12,
        "roofline": roof,
        "append": append_batch(ll, cache, shape, inputs, pk) if not args.key_fp8 else None,
        "append_in_stream_brackets": in_stream,
        "gpu_launches": launches,
        "clocks": clocks,
    })
    if not args.no_e2e and P == 1:
        result["e2e"] = run_e2e(ll, cache, shape, chunks, step_frames, world, rank, args)
    cache.close()
    del inputs, early
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, threads, sample = oracle_rate(shape)
        result["cpu_baseline"] = {"value": step_frames / (step_flops / rate), "unit": UNIT, "cores": threads,
                                  "kind": "oracle", "sample": sample}
    return result


def append_batch(ll, cache, shape, inputs, pk, reps=5):
    """HBM roofline of the commit copy, batch-timed.

    Every layer of the 30-layer cache holds one committed chunk (the 3 sink frames), and
    ll_recache then rewrites those 3 frames in every layer: the same copy kernel moving the
    same bytes as a commit (3 frames x 12 heads x 1560 tokens x 128, K and V, read + write).
    The 30 launches, on distinct layers and distinct source buffers (1.7 GB in all, well
    above the 126 MB L2), are recorded once as a CUDA graph, so that host-side call overhead
    does not starve the GPU, and each replay is timed between one pair of CUDA events: the
    figure includes the DRAM write-back of each launch and the gaps between launches, but no
    per-launch event overhead."""
    layers = shape.layers
    ll.ll_reset(cache)
    for l in range(layers):
        q, k, v = inputs[l][0]
        ll.ll_attend_chunk(cache, l, q, k, v, torch.empty_like(q), True)
    assert all(ll.ll_recache_tokens(cache, l) == shape.chunk_tokens for l in range(layers))
    srcs = [inputs[l][1 + l % (len(inputs[l]) - 1)][1:] for l in range(layers)]

    def batch():
        st = torch.cuda.current_stream()
        for l in range(layers):
            ll.ll_recache(cache, l, *srcs[l], st)

    batch()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    n0 = ll.ll_launch_count()
    with torch.cuda.graph(g):
        batch()
    assert ll.ll_launch_count() - n0 == layers
    stream = torch.cuda.current_stream()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    nbytes = append_bytes(shape, shape.chunk_frames) * layers
    roof = hbm_roofline("copy_frames_kernel", nbytes * reps, layers * reps, ms * reps, pk)
    roof["how"] = ("30 commit-sized copies (one per layer, distinct buffers) recorded as one CUDA graph; each "
                   "replay timed between one pair of CUDA events, median of %d replays" % reps)
    return roof


def run_graph(args, world, local, ll, cache, step, step_frames, step_flops, shape, L, chunks):
    """The whole stream step (600 attention calls from an empty cache) recorded once as one
    CUDA graph after an eager warm-up step; every timed step replays it.  The library keeps its
    frame bookkeeping on the host, so the graph replays exactly the calls it recorded."""
    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    n0 = ll.ll_launch_count()
    with torch.cuda.graph(g):
        step()
    per_step = ll.ll_launch_count() - n0
    ms, clocks, _, _ = timed_region(args, world, local, [cache], g.replay)
    ms_max = max_over_ranks(ms, world)
    H, d = shape.heads, shape.head_dim
    P = args.passes
    config = {"workload": "stream30 as one CUDA graph: 30 layers x 20 chunks (60 latent frames), H=12, d=128, "
                          "T=1560, C=3, S=3, W=9, %s" % (
                              "1 committed pass per chunk" if P == 1 else
                              "%d passes per chunk through all layers (the last commits)" % P)}
    config.update(shape_config(shape, {"chunks": chunks, "passes": P, "chunk_mask": args.chunk_mask,
                                       "l2": "inputs larger than L2 (%.1f GB q/k/v)" % (
                                           3 * L * H * d * 2 * chunks * shape.layers * P / 1e9),
                                       "parallelism": "replicas x%d (independent streams, no collective)" % world}))
    result = base_result(args, world, step_frames * args.steps * world / (ms_max / 1e3), ms_max, config)
    result.update({
        "tflops": step_flops * args.steps * world / (ms_max / 1e3) / 1e12,
        "roofline": None,
        "roofline_note": "per-kernel event brackets are not recorded in graph mode; see the eager run",
        "gpu_launches": per_step * args.steps,
        "clocks": clocks,
    })
    cache.close()
    return result


def run_single(args, world, rank, local):
    """Single Wan-shaped layer at steady state (23400 keys): one step = 4 query passes of a
    chunk, the last one committing (per-head input scales 0.5-2.0)."""
    import windowed_sink_attention_ll_b300 as ll

    shape = llsynth.SINGLE_LAYER
    H, d, T, S, W, C = (shape.heads, shape.head_dim, shape.tokens_per_frame, shape.sink_frames,
                        shape.window_frames, shape.chunk_frames)
    L = C * T
    passes = llsynth.SINGLE_LAYER_PASSES
    cache = ll.ll_cache_create(1, H, d, T, S, W, C, cache_dtype(ll, args))
    set_options(ll, cache, args)
    for c in range((S + W) // C):
        q, k, v = (llsynth.seeded_normal(("bench-single-fill", rank, c, t), (L, H, d), device="cuda",
                                         per_head_scale=True) for t in "qkv")
        ll.ll_attend_chunk(cache, 0, q, k, v, torch.empty_like(q), True)
    pool = 8  # distinct chunks cycled (8 x 4 passes x 43 MB of q/k/v: far beyond L2)
    inputs = [[tuple(llsynth.seeded_normal(("bench-single", rank, i, p, t), (L, H, d), device="cuda",
                                           per_head_scale=True) for t in "qkv") for p in range(passes)]
              for i in range(pool)]
    out = torch.empty((L, H, d), dtype=torch.bfloat16, device="cuda")
    pass_flops = pair_flops(chunk_pairs(shape, S + W, args.chunk_mask), H, d)
    it = [0]

    def step():
        chunk = inputs[it[0] % pool]
        it[0] += 1
        for p in range(passes):
            ll.ll_attend_chunk(cache, 0, *chunk[p], out, p == passes - 1)

    ms, clocks, launches, prof = timed_region(args, world, local, [cache], step)
    ms_max = max_over_ranks(ms, world)
    n_att, ms_att = prof[ll.LL_KERNEL_ATTEND]
    n_cp, ms_cp = prof[ll.LL_KERNEL_COPY]
    pk, pk_src = peaks()
    config = {"workload": "single: 1 Wan-shaped layer at steady state, H=12, d=128, T=1560, C=3, S=3, W=9, "
                          "Lkv=23400, 4 passes per chunk (commit on the last), per-head scales 0.5-2.0"}
    config.update(shape_config(shape, {"passes": passes, "l2": "8 distinct chunks cycled (1.4 GB of q/k/v)",
                                       "chunk_mask": args.chunk_mask}))
    result = base_result(args, world, C * args.steps * world / (ms_max / 1e3), ms_max, config)
    roof = tensor_roofline(attend_kernel_name(args), pass_flops * passes * args.steps, n_att, ms_att, pk, pk_src,
                           sustained=False, scale=peak_scale(args))
    alg = attend_bytes(shape, S + W)
    roof["algorithmic_bytes_per_launch"] = alg
    roof["traffic"], src = traffic_per_launch(alg) if not (args.pair or args.key_fp8) else (None, None)
    if src:
        roof["traffic_source"] = "ncu capture of %s" % src
    result.update({
        "tflops": pass_flops * passes * args.steps * world / (ms_max / 1e3) / 1e12,
        "roofline": roof,
        "append": hbm_roofline("copy_frames_kernel", append_bytes(shape, C, kv_elem_bytes(args)) * args.steps,
                               n_cp, ms_cp, pk),
        "gpu_launches": launches, "clocks": clocks,
    })
    cache.close()
    return result


def run_recache30(args, world, rank, local):
    """30 layers x 40 chunks with a recache prefill of the 12 resident frames in every layer
    before chunks 10, 20 and 30 (prompt switches)."""
    import windowed_sink_attention_ll_b300 as ll

    shape = llsynth.RECACHE30
    chunks = llsynth.RECACHE30_CHUNKS
    H, d, T, S, W, C = (shape.heads, shape.head_dim, shape.tokens_per_frame, shape.sink_frames,
                        shape.window_frames, shape.chunk_frames)
    L = C * T
    R = W if args.recache_scope == "window" else S + W  # frames a recache rewrites at a switch
    pool = 20  # chunk inputs cycled per layer (26 GB in total: far beyond L2)
    inputs = [[tuple(llsynth.seeded_normal(("bench-rc", rank, l, c, t), (L, H, d), device="cuda") for t in "qkv")
               for c in range(pool)] for l in range(shape.layers)]
    rc_inputs = [[tuple(llsynth.seeded_normal(("bench-rc-win", rank, l, sw, t), (R * T, H, d), device="cuda")
                        for t in "qkv") for sw in range(len(llsynth.RECACHE30_SWITCHES))]
                 for l in range(shape.layers)]
    outs = [torch.empty((L, H, d), dtype=torch.bfloat16, device="cuda") for _ in range(shape.layers)]
    out_rc = torch.empty((R * T, H, d), dtype=torch.bfloat16, device="cuda")
    cache = ll.ll_cache_create(shape.layers, H, d, T, S, W, C, cache_dtype(ll, args))
    set_options(ll, cache, args)
    stream = torch.cuda.current_stream()
    plan = stream_plan(shape, chunks)
    att_flops = sum(pair_flops(chunk_pairs(shape, t0, args.chunk_mask), H, d) for t0, _ in plan) * shape.layers
    # block-causal prefill (blocks of C frames, or of one frame with the frame mask); the
    # switches come after at least S + W frames, so the prefill shape is the same at each
    pre_flops = pair_flops(prefill_pairs(shape, S + W, args.chunk_mask, args.recache_scope), H, d)
    switches = len(llsynth.RECACHE30_SWITCHES)
    step_pre_flops = pre_flops * shape.layers * switches

    def step():
        ll.ll_reset(cache)
        for c in range(chunks):
            if c in llsynth.RECACHE30_SWITCHES:
                sw = llsynth.RECACHE30_SWITCHES.index(c)
                for l in range(shape.layers):
                    ll.ll_recache_attend(cache, l, *rc_inputs[l][sw], out_rc, stream)
            for l in range(shape.layers):
                ll.ll_attend_chunk(cache, l, *inputs[l][c % pool], outs[l], True, stream)

    ms, clocks, launches, prof = timed_region(args, world, local, [cache], step)
    ms_max = max_over_ranks(ms, world)
    pk, pk_src = peaks()
    n_att, ms_att = prof[ll.LL_KERNEL_ATTEND]
    n_pre, ms_pre = prof[ll.LL_KERNEL_PREFILL]
    config = {"workload": "recache30: 30 layers x 40 chunks (120 latent frames), recache prefill of 12 frames "
                          "(18720 tokens, block-causal in 3-frame blocks) in every layer before chunks 10, 20, 30"}
    config.update(shape_config(shape, {"chunks": chunks, "switches": list(llsynth.RECACHE30_SWITCHES),
                                       "l2": "inputs larger than L2 (41 GB per rank)",
                                       "chunk_mask": args.chunk_mask, "recache_scope": args.recache_scope}))
    result = base_result(args, world, chunks * C * args.steps * world / (ms_max / 1e3), ms_max, config)
    result.update({
        "tflops": (att_flops + step_pre_flops) * args.steps * world / (ms_max / 1e3) / 1e12,
        "roofline": tensor_roofline(attend_kernel_name(args), att_flops * args.steps, n_att, ms_att, pk, pk_src,
                                    scale=peak_scale(args)),
        "prefill": dict(tensor_roofline(attend_kernel_name(args) + " (prefill mode)", step_pre_flops * args.steps, n_pre,
                                        ms_pre, pk, pk_src, scale=peak_scale(args)),
                        ms_per_switch_30_layers=ms_pre / max(1, args.steps * switches)),
        "gpu_launches": launches, "clocks": clocks,
    })
    cache.close()
    return result


def run_sweep(args, world, rank, local):
    """Window/sink sweep: steady-state chunk attend TFLOPS for W in {3,6,9,12,18} x S in {0,3}."""
    import windowed_sink_attention_ll_b300 as ll

    base = llsynth.WAN
    H, d, T, C = base["heads"], base["head_dim"], base["tokens_per_frame"], base["chunk_frames"]
    L = C * T
    pool = 8
    inputs = [tuple(llsynth.seeded_normal(("bench-sweep", rank, i, t), (L, H, d), device="cuda") for t in "qkv")
              for i in range(pool)]
    out = torch.empty((L, H, d), dtype=torch.bfloat16, device="cuda")
    pk, pk_src = peaks()
    rows, total_ms, total_frames = [], 0.0, 0
    for W in llsynth.SWEEP_W:
        for S in llsynth.SWEEP_S:
            cache = ll.ll_cache_create(1, H, d, T, S, W, C, cache_dtype(ll, args))
            set_options(ll, cache, args)
            while ll.ll_cache_state(cache, 0)[0] < S + W + C:  # steady state: sink and window full
                ll.ll_attend_chunk(cache, 0, *inputs[0], out, True)
            lkv = (S + W + C) * T
            it = [0]

            def step():
                for _ in range(10):
                    ll.ll_attend_chunk(cache, 0, *inputs[it[0] % pool], out, True)
                    it[0] += 1

            ms, clocks, launches, prof = timed_region(args, world, local, [cache], step)
            n_att, ms_att = prof[ll.LL_KERNEL_ATTEND]
            flops = pair_flops(chunk_pairs(llsynth.Shape(1, H, d, T, S, W, C), S + W, args.chunk_mask), H, d) \
                * 10 * args.steps
            rows.append({"W": W, "S": S, "Lkv": lkv, "ms_per_chunk": ms / (10 * args.steps),
                         "attend_tflops": flops / (ms_att / 1e3) / 1e12,
                         "attend_frac_of_burst": flops / (ms_att / 1e3) / 1e12 / pk.get("bf16_tflops", 1800.0)})
            total_ms += ms
            total_frames += 10 * C * args.steps
            cache.close()
    ms_max = max_over_ranks(total_ms, world)
    config = {"workload": "sweep: 1 Wan-shaped layer, W in {3,6,9,12,18} x S in {0,3}, steady state, "
                          "10 committed chunks per step and setting"}
    result = base_result(args, world, total_frames * world / (ms_max / 1e3), ms_max, config)
    result.update({"sweep": rows, "clocks": clocks})
    return result


def run_e2e(ll, cache, shape, chunks, step_frames, world, rank, args):
    """Same stream through the public API with q/k/v copied in from pinned host memory and every
    output copied back.  q, k and v go up on separate copy streams (several copy engines work
    at once); `out` comes back on another; NB device buffer sets rotate so copies overlap the
    attention of the previous layers."""
    H, d, T, C = shape.heads, shape.head_dim, shape.tokens_per_frame, shape.chunk_frames
    L = C * T
    pool = 4  # distinct pinned host input sets, cycled
    NB = 3    # device buffer sets in flight
    host_in = [tuple(llsynth.seeded_normal(("bench-e2e", rank, i, t), (L, H, d)).pin_memory() for t in "qkv")
               for i in range(pool)]
    host_out = [torch.empty((L, H, d), dtype=torch.bfloat16).pin_memory() for _ in range(NB)]
    dev_in = [tuple(torch.empty((L, H, d), dtype=torch.bfloat16, device="cuda") for _ in range(3)) for _ in range(NB)]
    dev_out = [torch.empty((L, H, d), dtype=torch.bfloat16, device="cuda") for _ in range(NB)]
    comp = torch.cuda.current_stream()
    n_in = max(1, args.e2e_streams)
    s_in = [torch.cuda.Stream() for _ in range(n_in)]
    s_out = torch.cuda.Stream()
    done = [torch.cuda.Event() for _ in range(NB)]     # attention of buffer set b finished
    drained = [torch.cuda.Event() for _ in range(NB)]  # out of buffer set b copied back
    for e in done + drained:
        e.record(comp)
    bytes_in = bytes_out = 0

    def step():
        nonlocal bytes_in, bytes_out
        ll.ll_reset(cache)
        i = 0
        for c in range(chunks):
            for l in range(shape.layers):
                b = i % NB
                src = host_in[i % pool]
                ready = []
                for ti, (dst, h) in enumerate(zip(dev_in[b], src)):
                    st = s_in[ti % n_in]
                    st.wait_event(done[b])
                    with torch.cuda.stream(st):
                        dst.copy_(h, non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(st)
                    ready.append(ev)
                for ev in ready:
                    comp.wait_event(ev)
                comp.wait_event(drained[b])
                ll.ll_attend_chunk(cache, l, *dev_in[b], dev_out[b], True, comp)
                done[b].record(comp)
                s_out.wait_event(done[b])
                with torch.cuda.stream(s_out):
                    host_out[b].copy_(dev_out[b], non_blocking=True)
                drained[b].record(s_out)
                bytes_in += 3 * L * H * d * 2
                bytes_out += L * H * d * 2
                i += 1

    step()
    torch.cuda.synchronize()
    bytes_in = bytes_out = 0
    steps = max(1, min(args.steps, 2))
    barrier(world)
    torch.cuda.synchronize()
    t = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    el = max_over_ranks(time.perf_counter() - t, world)
    barrier(world)
    return {"value": step_frames * steps * world / el, "unit": UNIT, "steps": steps,
            "h2d_bytes_per_step": bytes_in // steps, "d2h_bytes_per_step": bytes_out // steps,
            "h2d_GBps": bytes_in / el / 1e9, "d2h_GBps": bytes_out / el / 1e9,
            "how": "pinned host q/k/v -> device (%d copy stream%s) -> ll_attend_chunk -> out -> pinned host "
                   "(copy stream), %d buffer sets in flight; wall clock" % (n_in, "s" if n_in > 1 else "", NB)}


# ----------------------------------------------------------------------------
# reference arm: the float64 oracle, on bounded samples of the same workload
# ----------------------------------------------------------------------------

def run_reference(args, world, rank):
    shape = llsynth.STREAM30
    chunks = llsynth.STREAM30_CHUNKS
    H, d, T, C = shape.heads, shape.head_dim, shape.tokens_per_frame, shape.chunk_frames
    L = C * T
    plan = stream_plan(shape, chunks)
    step_frames = chunks * C
    step_flops = sum(attend_flops(L, lkv, H, d) for _, lkv in plan) * shape.layers * args.passes
    budget = max(2.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    if args.ref_budget_s is not None:
        budget = args.ref_budget_s
    for _ in range(args.warmup):
        oracle_rate(shape, budget_s=min(budget, 3.0))
    times, rates, threads, sample = [], [], 1, ""
    for _ in range(args.steps):
        rate, threads, sample = oracle_rate(shape, budget_s=budget)
        rates.append(rate)
        times.append(step_flops / rate)
    ms_step = 1e3 * statistics.mean(times)
    value = step_frames / (ms_step / 1e3)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "stream30: 30 layers x 20 chunks (60 latent frames), H=12, d=128, T=1560, "
                               "C=3, S=3, W=9, %s (float64 CPU oracle, sampled rows; step time scaled by "
                               "flops)" % ("1 committed pass per chunk" if args.passes == 1 else
                                           "%d passes per chunk (the last commits)" % args.passes)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["stream30", "single", "recache30", "sweep"], default="stream30",
                    help="stream30 (default: the 30-layer stack the metric names); the others time the "
                         "single-layer, prompt-switch recache and window/sink sweep workloads")
    ap.add_argument("--graph", action="store_true",
                    help="stream30: record the whole step as one CUDA graph and time its replays")
    ap.add_argument("--chunk-mask", choices=["chunk", "frame"], default="chunk",
                    help="chunk (default): a chunk sees all its frames; frame: the frame-causal reading")
    ap.add_argument("--recache-scope", choices=["resident", "window"], default="resident",
                    help="resident (default): recache rewrites sink and window; window: the sink keeps its K/V")
    ap.add_argument("--key-fp8", action="store_true",
                    help="an FP8-key cache (LL_BF16_K8): keys stored in e4m3, Q K^T at the FP8 tensor rate")
    ap.add_argument("--passes", type=int, default=1,
                    help="stream30: query passes per chunk through all layers, the last one committing "
                         "(default 1; e2e is measured at 1 only)")
    ap.add_argument("--kv-fp8", action="store_true",
                    help="an FP8 cache (LL_FP8): keys and values stored in e4m3, Q K^T at the FP8 tensor rate, "
                         "P V on fp16 operands")
    ap.add_argument("--pair", action="store_true",
                    help="run head_dim 128 on the CTA-pair tensor-core kernel instead of the default one-CTA kernel")
    ap.add_argument("--ref-budget-s", type=float, default=None,
                    help="seconds of oracle work per step of the reference arm (default: sized so the run takes "
                         "about two minutes)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-streams", type=int, default=3, help="host-to-device copy streams of the e2e measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.key_fp8 = args.key_fp8 or args.kv_fp8  # an FP8 cache stores its keys in e4m3 too
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        # CPU-only arm: rank 0 alone times the oracle; other ranks exit without work
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if rank == 0:
            print(json.dumps(run_reference(args, world, rank)), flush=True)
        return
    world, rank, local = dist_setup()
    run = {"stream30": run_ours, "single": run_single, "recache30": run_recache30, "sweep": run_sweep}
    res = run[args.workload](args, world, rank, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
