"""Decode-step benchmark: KV append + paged decode attention over every layer
of a Llama-3-8B-shaped decode batch (batch 64, context 1024, block_size 16,
32 layers), through the C ABI on one GB300 per rank.

One JSON line (rank 0):
  value       decode tokens/s per layer, whole job (all ranks), inputs resident
  e2e         the same metric with per-step inputs copied from pinned host
              memory and the outputs read back inside the timed region
  roofline    achieved HBM bandwidth of the paged attention call (its
              kernels: one for the tensor-core path) from CUDA events in the
              timed region, against the measured copy bandwidth of this GPU model
  cpu_baseline  the CPU fp64 oracle on a bounded sample of the same workload
  legs        contiguous-layout attention on the same logical KV, the append
              kernel alone, and a Yi-34B-shaped copy-on-write block copy

--impl reference times the CPU oracle instead (the only reference there is).
Multi-GPU (torchrun): every rank runs its own replica of the batch (weak
scaling, no collective on the data path); the barrier and the max over ranks
of the timed region use torch.distributed.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "decode-attn achieved HBM TB/s (% of GB300 8 TB/s); decode tokens/s/layer"
UNIT = "tokens/s/layer"
WORKLOADS = {
    # name: (shape, batch, context, block_size, seed)
    "llama3_8b_b64": (W.LLAMA3_8B, 64, 1024, 16, W.SEED_LLAMA),
    "yi6b_b64": (W.YI_6B, 64, 1024, 16, W.SEED_YI6B),
}
for _b in W.LLAMA_SWEEP_BATCHES:
    WORKLOADS["llama3_8b_b%d" % _b] = (W.LLAMA3_8B, _b, 1024, 16, W.SEED_LLAMA)
# ragged serving batch (context = prompt + generated so far, max 8192)
for _bs in W.RAGGED_BLOCK_SIZES:
    WORKLOADS["llama3_8b_ragged_bs%d" % _bs] = (W.LLAMA3_8B, 256, "ragged", _bs, W.SEED_RAGGED)
# parallel sampling over shared prompts: the first decode step after copy on write
WORKLOADS["yi34b_sharing"] = (W.YI_34B, 128, "sharing", 16, W.SEED_YI34B)
DEFAULT_WORKLOAD = "llama3_8b_b64"


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _describe(name):
    shape, B, ctx, bs, _ = WORKLOADS[name]
    ctx_text = {"ragged": "ragged contexts (prompt ~ Exp(1024) + generated ~ U{0..Exp(256)}, "
                          "max 8192)",
                "sharing": "32 prompts ~ U[1024, 8192] x 4 sampled branches sharing prompt "
                           "blocks, first step after copy on write"}.get(ctx, "context %s" % ctx)
    return ("%s-shaped decode: batch %d, %s, block_size %d, %d layers, "
            "%d query / %d KV heads, head_dim %d"
            % (shape.name, B, ctx_text, bs, shape.num_layers, shape.num_q_heads,
               shape.num_kv_heads, shape.head_dim))


def rank_workload(name, rank):
    """(batch, copy-on-write pairs [n, 2] or None) that a rank decodes: every
    rank gets the workload's full shape (weak scaling) with its own seed, so
    ranks hold different sequences.  The sharing workload's step is the first
    decode step after forking, so it starts with the copies on write."""
    shape, B, ctx, bs, seed = WORKLOADS[name]
    seed = seed + 1000 * rank
    if ctx == "ragged":
        return W.make_paged_batch(shape, W.ragged_lengths(B, seed=seed), bs, seed), None
    if ctx == "sharing":
        sc = W.sharing_scenario(seed=seed, decode_steps=1)
        return sc.steps[0], (sc.cow_pairs if len(sc.cow_pairs) else None)
    return W.uniform_batch(shape, B, ctx, bs, seed=seed), None


def rank_batch(name, rank):
    return rank_workload(name, rank)[0]


def algorithmic_bytes(batch):
    """Bytes one paged attention call must move: K and V of every attended
    position, Q and O, the block-table entries read and the context lengths."""
    s = batch.shape
    ctx = batch.ctx.astype(np.int64)
    kv = int(ctx.sum()) * s.num_kv_heads * s.head_dim * 2 * 2
    qo = 2 * batch.B * s.num_q_heads * s.head_dim * 2
    tables = int(((ctx + batch.block_size - 1) // batch.block_size).sum()) * 4
    return kv + qo + tables + 4 * batch.B


def unique_kv_bytes(batch):
    """K and V bytes of the distinct cache rows the call reads: sequences
    that share prompt blocks read those rows once each, so this is below the
    algorithmic count exactly when blocks are shared."""
    s = batch.shape
    bs = batch.block_size
    rows = []
    for i in range(batch.B):
        c = int(batch.ctx[i])
        if c <= 0:
            continue
        pos = np.arange(c, dtype=np.int64)
        rows.append(batch.block_tables[i, pos // bs].astype(np.int64) * bs + pos % bs)
    n = len(np.unique(np.concatenate(rows))) if rows else 0
    return n * s.num_kv_heads * s.head_dim * 2 * 2


def attention_flops(batch):
    """q.K and p.V: 4 flops per (position, query head, dimension)."""
    s = batch.shape
    return 4 * int(batch.ctx.astype(np.int64).sum()) * s.num_q_heads * s.head_dim


class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.device_index = device_index
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# The sources the attention call's kernel (decode_tc_kernel, which merges
# the pieces of cut pairs itself) is built from; the DRAM counters of a
# profile summary stand for the kernel only while these are unchanged.
DECODE_SOURCES = ("decode_tc.cu", "decode_tc.cuh", "decode_tc_launch.h", "pkv_device.cuh")


def _source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_245_gb300", "csrc")
    for f in DECODE_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def _profiled_traffic(name):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "paged_decode_%s.md" % name)
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256_16") != _source_hash():
        return None
    try:
        return int(float(vals["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------------ GPU arm

class DeviceWorkload:
    def __init__(self, name, dev, rank):
        import paged_kv_cache_245_gb300 as pkv
        self.pkv = pkv
        shape, B, ctx, bs, seed = WORKLOADS[name]
        self.name = name
        self.shape = shape
        self.batch, pairs = rank_workload(name, rank)
        self.dev = dev
        b = self.batch
        self.layers = []
        for l in range(shape.num_layers):
            li = W.layer_inputs(b, l, device=dev, fast_cache=True)
            self.layers.append(li)
        self.cow = None if pairs is None else torch.as_tensor(pairs, device=dev)
        # sequences forked from one prompt: attend their shared blocks once
        # per group (the sharing workload: groups of `n` consecutive branches)
        self.groups = None
        if ctx == "sharing":
            n = W.sharing_scenario(decode_steps=1).n
            starts = np.arange(0, b.B + 1, n, dtype=np.int32)
            shared = W.shared_prefix_blocks(b.block_tables, b.ctx, bs, starts)
            own = int((b.ctx - np.repeat(shared, n) * bs).max())  # own positions per sequence
            self.groups = (torch.as_tensor(starts, device=dev), torch.as_tensor(shared, device=dev),
                           n, own)
        self.k_caches = [li.k_cache for li in self.layers]
        self.v_caches = [li.v_cache for li in self.layers]
        self.tables = torch.as_tensor(b.block_tables, device=dev)
        self.ctx = torch.as_tensor(b.ctx, device=dev)
        self.slots = torch.as_tensor(b.slot_mapping, device=dev)
        self.scale = W.default_scale(shape)
        self.out = [torch.empty_like(li.q) for li in self.layers]
        nbytes = pkv.decode_workspace_size(b.B, shape.num_q_heads, shape.num_kv_heads,
                                           b.max_context)
        if self.groups is not None:
            nbytes = max(nbytes, pkv.lib().pkv_shared_decode_workspace_size(
                b.B, len(self.groups[1]), self.groups[2], b.block_tables.shape[1],
                pkv.binding.heads(shape.num_q_heads, shape.num_kv_heads, shape.head_dim)))
        self.workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
        self.nsplit = pkv.decode_num_splits(b.B, shape.num_q_heads, shape.num_kv_heads,
                                            b.max_context)

    @property
    def uses_tc(self):
        # the library's own choice for this batch (variant, block size, tiles per SM)
        return self.pkv.decode_uses_tensor_cores(self.batch.B, self.shape.num_q_heads,
                                                 self.shape.num_kv_heads, self.batch.max_context,
                                                 self.batch.block_size, self.shape.head_dim)

    def shared_kernels(self):
        """The kernels of one shared-prefix call, by the library's launch count."""
        n = (self.launches_per_step() - (0 if self.cow is None else 1)) // self.shape.num_layers - 1
        return {1: "prefix_kernel alone: own positions as masked key tiles, output written there",
                2: "prefix_kernel, then cascade_merge_kernel",
                }.get(n, "cascade_prep_kernel, prefix_kernel, decode_tc_kernel over the own "
                         "positions, cascade_merge_kernel")

    def launches_per_step(self):
        # per layer: the decode step's kernels (the tensor-core kernel alone,
        # which does the append and merges its split pairs itself; else the
        # append, the split kernel and its combine), or the append and the
        # shared-prefix call's kernels as the library reports them; plus one
        # block copy launch (all layers) when the step copies on write
        cow = 0 if self.cow is None else 1
        if self.groups is not None:
            gs, sb, n, own = self.groups
            b = self.batch
            attn = self.pkv.shared_decode_launches(
                b.B, int(gs.numel()) - 1, n, b.block_tables.shape[1], b.max_context,
                b.block_size, own, self.shape.num_q_heads, self.shape.num_kv_heads)
            return self.shape.num_layers * (1 + attn) + cow
        if self.uses_tc:
            return self.shape.num_layers + cow
        return self.shape.num_layers * (2 + (1 if self.nsplit > 1 else 0)) + cow

    def copy_on_write(self, pairs=None):
        pairs = self.cow if pairs is None else pairs
        if pairs is not None:
            self.pkv.block_copy(pairs, self.k_caches, self.v_caches)

    def attend(self, l):
        li = self.layers[l]
        if self.groups is not None:
            gs, sb, n, own = self.groups
            self.pkv.paged_decode_attention_shared(li.q, li.k_cache, li.v_cache, self.tables,
                                                   self.ctx, self.batch.max_context, self.scale,
                                                   gs, sb, n, max_own_tokens=own,
                                                   out=self.out[l], workspace=self.workspace)
        else:
            self.pkv.paged_decode_attention(li.q, li.k_cache, li.v_cache, self.tables, self.ctx,
                                            self.batch.max_context, self.scale, out=self.out[l],
                                            workspace=self.workspace)

    def layer(self, l):
        """One layer's decode step: append + attention in one C-ABI call (the
        sharing workload: append, then attention with its shared blocks read
        once per group)."""
        li = self.layers[l]
        if self.groups is not None:
            self.pkv.kv_append(self.slots, li.k_new, li.v_new, li.k_cache, li.v_cache)
            self.attend(l)
            return
        self.pkv.paged_decode_step(self.slots, li.k_new, li.v_new, li.q, li.k_cache, li.v_cache,
                                   self.tables, self.ctx, self.batch.max_context, self.scale,
                                   out=self.out[l], workspace=self.workspace)

    def step(self):
        self.copy_on_write()
        for l in range(self.shape.num_layers):
            self.layer(l)

    def attention_only(self):
        for l in range(self.shape.num_layers):
            self.attend(l)


def _barrier(world):
    if world > 1:
        torch.distributed.barrier()


def _max_over_ranks(x, world, dev):
    """Max of a per-rank value over all ranks (the slowest rank's time)."""
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def run_gpu(args, world, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from __graft_entry__ import build
    if rank == 0 or world == 1:
        build()
    _barrier(world)
    wl = DeviceWorkload(args.workload, dev, rank)
    nl = wl.shape.num_layers
    stream = torch.cuda.current_stream(dev)

    # Direct launches first (sets kernel attributes, warms caches), then the
    # step and the attention calls alone are captured as CUDA graphs: a decode
    # loop replays the same launches every step, so the host's per-call
    # overhead stays out of the device-time measurement.
    for _ in range(3):
        wl.step()
    torch.cuda.synchronize(dev)
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph):
        wl.step()
    attn_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(attn_graph):
        wl.attention_only()
    torch.cuda.synchronize(dev)
    for _ in range(max(args.warmup, 3)):
        step_graph.replay()
    torch.cuda.synchronize(dev)

    # ---- timed region: K decode steps (graph replays) between two events
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    _barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    t0.record()
    for k in range(args.steps):
        step_graph.replay()
    t1.record()
    torch.cuda.synchronize(dev)
    _barrier(world)
    # ---- the attention calls alone (same calls, same data), for the roofline
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # at least 50 replays (1,600 calls at 32 layers): the number that decides
    # the roofline fraction is averaged over tens of milliseconds
    attn_reps = max(args.steps // 2, 50)
    a0.record()
    for k in range(attn_reps):
        attn_graph.replay()
    a1.record()
    torch.cuda.synchronize(dev)
    clock_info = clocks.stop()
    elapsed_ms = _max_over_ranks(t0.elapsed_time(t1), world, dev)
    attn_avg_ms = _max_over_ranks(a0.elapsed_time(a1) / (attn_reps * nl), world, dev)

    B = wl.batch.B
    ms_per_step = elapsed_ms / args.steps
    value = world * B / (ms_per_step / 1e3 / nl)
    alg = algorithmic_bytes(wl.batch)
    peak, peak_kind = _peaks()
    achieved_gbs = alg / (attn_avg_ms / 1e3) / 1e9

    legs = {}
    e2e = None
    cpu = None
    if rank == 0 and not args.skip_legs:
        legs = measure_legs(wl, dev, args)
    if not args.skip_e2e:
        e2e = measure_e2e(wl, dev, args, world)
    if rank == 0 and world == 1 and not args.skip_cpu:
        cpu = cpu_baseline(wl, args)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": _describe(args.workload), "global_batch": B * world,
                   "seq_len": int(wl.batch.ctx.max()), "mean_context": round(float(wl.batch.ctx.mean()), 1),
                   "layers": nl,
                   "block_size": wl.batch.block_size, "num_splits": wl.nsplit,
                   "parallelism": "replicas (one batch per GPU, no collective)" if world > 1
                   else "single GPU",
                   "l2": "inputs larger than L2: %.1f GB of distinct K/V per step, "
                         "%.0f MB per layer" % (nl * alg / 1e9, alg / 1e6),
                   "step": ("block_copy of %d copy-on-write pairs (all layers), then "
                            % len(wl.cow) if wl.cow is not None else "")
                           + ("per layer: kv_append + paged_decode_attention_shared (each "
                              "group's shared prompt blocks read once for all its branches)"
                              if wl.groups is not None
                              else "per layer: paged_decode_step (kv_append + "
                              "paged_decode_attention; with the tensor-core kernel one launch "
                              "that also appends)")},
        "hbm_tbs": round(achieved_gbs / 1e3, 4),
        "hbm_pct_of_8tbs": round(100 * achieved_gbs / 8000.0, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved_gbs / peak, 4),
                     "traffic": _profiled_traffic(args.workload),
                     "kernel": "paged_decode_attention_shared call (%s)" % wl.shared_kernels()
                               if wl.groups is not None else
                               "paged_decode_attention call (decode_tc_kernel, merging the "
                               "pairs its CTA ranges cut)" if wl.uses_tc else
                               "paged_decode_attention call (decode_attention_kernel + "
                               "decode_combine_kernel)",
                     "algorithmic_bytes_per_launch": alg,
                     "unique_kv_bytes_per_launch": unique_kv_bytes(wl.batch),
                     "flops_per_launch": attention_flops(wl.batch),
                     "avg_launch_us": round(attn_avg_ms * 1e3, 3),
                     "timed_over": "%d replays of the step's %d attention calls" % (attn_reps, nl),
                     "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind},
        "gpu_launches": wl.launches_per_step() * args.steps,
        "timing": "CUDA-graph replay of the step; roofline from a replay of the %d "
                  "attention calls alone" % nl,
        "clocks": clock_info,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if legs:
        line["legs"] = legs
    if rank == 0:
        print(json.dumps(line), flush=True)


def _time_graph(fn, reps, dev, calls=1):
    """Device time of one call of fn: `calls` calls captured in a CUDA graph,
    replayed `reps` times between CUDA events (after a warm replay)."""
    fn()
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(calls):
            fn()
    g.replay()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b) / (reps * calls)


def measure_legs(wl, dev, args):
    """Per-kernel figures beside the step: contiguous-layout attention over the
    same logical K/V, the append alone, and a copy-on-write block copy."""
    pkv = wl.pkv
    b = wl.batch
    alg = algorithmic_bytes(b)
    # the contiguous layout's per-request capacity S: the ragged batch's
    # maximum length (8192), else the longest context of the batch
    S = 8192 if WORKLOADS[wl.name][2] == "ragged" else int(b.ctx.max())
    # distinct layers cycled (far above L2), within about 24 GB of buffers
    buf_bytes = 2 * b.B * wl.shape.num_kv_heads * S * wl.shape.head_dim * 2
    nl = max(1, min(8, wl.shape.num_layers, int(24e9 // buf_bytes)))
    bufs = []
    for l in range(nl):
        li = wl.layers[l]
        bufs.append((W.paged_to_contig(li.k_cache, b, S), W.paged_to_contig(li.v_cache, b, S)))
    req = torch.arange(b.B, dtype=torch.int32, device=dev)
    it = {"i": 0}

    def contig():
        l = it["i"] % nl
        it["i"] += 1
        pkv.contig_decode_attention(wl.layers[l].q, bufs[l][0], bufs[l][1], req, wl.ctx,
                                    b.max_context, wl.scale, out=wl.out[l],
                                    workspace=wl.workspace)

    def paged():
        l = it["i"] % nl
        it["i"] += 1
        li = wl.layers[l]
        pkv.paged_decode_attention(li.q, li.k_cache, li.v_cache, wl.tables, wl.ctx,
                                   b.max_context, wl.scale, out=wl.out[l],
                                   workspace=wl.workspace)

    reps = max(10, args.steps // 20)
    t_contig = _time_graph(contig, reps, dev, calls=nl)
    t_paged = _time_graph(paged, reps, dev, calls=nl)
    vmm = measure_vmm(wl, dev, bufs[0], S, req, reps)
    del bufs
    # the split (CUDA-core) kernel on the same calls, for comparison
    pkv.set_decode_variant(pkv.VARIANT_SPLIT)
    try:
        t_split = _time_graph(paged, reps, dev, calls=nl)
    finally:
        pkv.set_decode_variant(pkv.VARIANT_AUTO)

    def append():
        l = it["i"] % wl.shape.num_layers
        it["i"] += 1
        li = wl.layers[l]
        pkv.kv_append(wl.slots, li.k_new, li.v_new, li.k_cache, li.v_cache)

    t_append = _time_graph(append, reps, dev, calls=wl.shape.num_layers)
    append_bytes = 2 * 2 * b.B * wl.shape.num_kv_heads * wl.shape.head_dim * 2 + 8 * b.B

    # Yi-34B-shaped copy on write: 96 block pairs x 60 layers of 32 KiB blocks
    L, nb = 60, 192
    g = torch.Generator(device=dev)
    g.manual_seed(W.SEED_YI34B)
    ks = [torch.empty((nb, 8, 16, 128), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    vs = [torch.empty((nb, 8, 16, 128), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    pairs = torch.stack([torch.arange(0, 96), torch.arange(96, 192)], 1).to(dev)
    t_copy = _time_graph(lambda: pkv.block_copy(pairs, ks, vs), 20, dev)
    copy_bytes = 2 * 96 * L * 2 * 8 * 16 * 128 * 2
    del ks, vs
    return {
        "paged_attention_us": round(t_paged * 1e3, 3),
        "contig_attention_us": round(t_contig * 1e3, 3),
        "paged_over_contig_time": round(t_paged / t_contig, 4),
        "contig_S": S, "contig_layers": nl,
        "split_kernel_attention_us": round(t_split * 1e3, 3),
        "split_kernel_hbm_gbs": round(alg / (t_split / 1e3) / 1e9, 1),
        "contig_hbm_gbs": round(alg / (t_contig / 1e3) / 1e9, 1),
        "kv_append_us": round(t_append * 1e3, 3),
        "kv_append_gbs": round(append_bytes / (t_append / 1e3) / 1e9, 1),
        "block_copy_us": round(t_copy * 1e3, 3),
        "block_copy_gbs": round(copy_bytes / (t_copy / 1e3) / 1e9, 1),
        "block_copy_shape": "96 pairs x 60 layers x (K,V) of 32 KiB blocks (read + write)",
        "on_demand_contig": vmm,
        "prefill": measure_prefill(wl, dev, reps),
        "swap": measure_swap(pkv, dev),
    }


def measure_swap(pkv, dev, reps=8):
    """Pre-emption by swapping, Llama-3-8B-shaped: four sequences of 1024
    tokens (256 blocks scattered over the pool) x 32 layers x (K, V) of
    32 KiB blocks, out to a page-locked host pool and back, one block_swap
    launch each way.  Beside it, one contiguous copy of the same bytes by
    the copy engine (cudaMemcpyAsync), the link's plain transfer rate."""
    L, nb, n = 32, 512, 256
    shape = (nb, 8, 16, 128)
    dk = [torch.zeros(shape, dtype=torch.bfloat16, device=dev) for _ in range(L)]
    dv = [torch.zeros(shape, dtype=torch.bfloat16, device=dev) for _ in range(L)]
    hk = [torch.zeros((n,) + shape[1:], dtype=torch.bfloat16, pin_memory=True) for _ in range(L)]
    hv = [torch.zeros((n,) + shape[1:], dtype=torch.bfloat16, pin_memory=True) for _ in range(L)]
    g = torch.Generator().manual_seed(W.SEED_LLAMA)
    blocks = torch.randperm(nb, generator=g)[:n]
    out = torch.stack([blocks, torch.arange(n)], 1).to(dev)
    back = torch.stack([torch.arange(n), blocks], 1).to(dev)
    moved = 2 * L * n * 8 * 16 * 128 * 2

    def timed(fn):
        fn()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / reps / 1e3

    try:
        t_out = timed(lambda: pkv.block_swap(out, dk, dv, hk, hv))
        t_in = timed(lambda: pkv.block_swap(back, hk, hv, dk, dv))
        flat_d = torch.empty(moved // 2, dtype=torch.bfloat16, device=dev)
        flat_h = torch.empty(moved // 2, dtype=torch.bfloat16, pin_memory=True)
        t_d2h = timed(lambda: flat_h.copy_(flat_d, non_blocking=True))
        t_h2d = timed(lambda: flat_d.copy_(flat_h, non_blocking=True))
    finally:
        torch.cuda.synchronize(dev)
    gbs = lambda t: round(moved / t / 1e9, 1)
    return {"bytes": moved, "swap_out_us": round(t_out * 1e6, 1), "swap_out_gbs": gbs(t_out),
            "swap_in_us": round(t_in * 1e6, 1), "swap_in_gbs": gbs(t_in),
            "copy_engine_d2h_gbs": gbs(t_d2h), "copy_engine_h2d_gbs": gbs(t_h2d),
            "shape": "256 scattered blocks x 32 layers x (K,V) of 32 KiB, device <-> "
                     "page-locked host, one launch each way"}


def _bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops)"
    return 1900.0, "fallback"


def measure_prefill(wl, dev, reps):
    """Causal prefill over a paged cache with the workload's head shape:
    8 fresh prompts of 2048 tokens, and 8 chunks of 512 tokens after 1536
    cached positions (random blocks, block_size 16).  Flops: 4 * D per
    (query token, head, attended position)."""
    pkv = wl.pkv
    shape = wl.shape
    peak, peak_src = _bf16_peak()
    res = {}
    for name, cached, lq in (("fresh_8x2048", 0, 2048), ("chunk_8x512_after_1536", 1536, 512)):
        ctx = np.full(8, cached + lq, np.int32)
        b = W.make_paged_batch(shape, ctx, 16, 250)
        li = W.layer_inputs(b, 0, device=dev, fast_cache=True)
        cu = torch.as_tensor(np.arange(0, 8 * lq + 1, lq, dtype=np.int32), device=dev)
        g = torch.Generator(device=dev)
        g.manual_seed(251)
        q = torch.randn((8 * lq, shape.num_q_heads, shape.head_dim), generator=g,
                        device=dev).to(torch.bfloat16)
        out = torch.empty_like(q)
        tables = torch.as_tensor(b.block_tables, device=dev)
        ctx_d = torch.as_tensor(b.ctx, device=dev)

        def call():
            pkv.paged_prefill_attention(q, cu, li.k_cache, li.v_cache, tables, ctx_d, lq,
                                        W.default_scale(shape), out=out)

        t = _time_graph(call, max(5, reps // 4), dev, calls=2)
        attended = 8 * sum(cached + j + 1 for j in range(lq))  # per head
        flops = 4.0 * shape.head_dim * shape.num_q_heads * attended
        res[name] = {"us": round(t * 1e3, 2), "tflops": round(flops / (t / 1e3) / 1e12, 1),
                     "frac_of_bf16_peak": round(flops / (t / 1e3) / 1e12 / peak, 3)}
        del li
    res["peak_tflops"] = peak
    res["peak_source"] = peak_src
    res["kernel"] = ("prefill_kernel (tcgen05.mma 128x128x16 bf16, S and O in tensor memory; "
                     "persistent, one CTA per SM over items of 256 query rows)")
    return res


def measure_vmm(wl, dev, buf, S, req, reps):
    """The contiguous layout on memory mapped on demand: back every request's
    rows (timed on the host: the mapping rate), copy layer 0's rows in, and
    time the same attention call there and on regular device memory."""
    pkv = wl.pkv
    b = wl.batch
    vm = pkv.VmmBuffer(b.B, wl.shape.num_kv_heads, (S + 15) // 16 * 16)
    try:
        t0 = time.perf_counter()
        for r in range(b.B):
            vm.ensure(r, int(b.ctx[r]))
        t_map = time.perf_counter() - t0
        st = vm.stats()
        for r in range(b.B):   # kernels below touch only backed rows
            assert vm.backed_tokens(r) >= int(b.ctx[r])
        for r in range(b.B):
            c = int(b.ctx[r])
            vm.k[r, :, :c].copy_(buf[0][r, :, :c])
            vm.v[r, :, :c].copy_(buf[1][r, :, :c])
        li = wl.layers[0]
        out = torch.empty_like(li.q)

        def on_vmm():
            pkv.contig_decode_attention(li.q, vm.k, vm.v, req, wl.ctx, b.max_context, wl.scale,
                                        out=out, workspace=wl.workspace)

        def on_regular():
            pkv.contig_decode_attention(li.q, buf[0], buf[1], req, wl.ctx, b.max_context,
                                        wl.scale, out=out, workspace=wl.workspace)

        t_vmm = _time_graph(on_vmm, reps, dev, calls=4)
        t_reg = _time_graph(on_regular, reps, dev, calls=4)
        mapped = 2 * st["mapped_pages"] * st["page_bytes"]
        return {"page_bytes": st["page_bytes"], "mapped_bytes": mapped,
                "map_ms": round(t_map * 1e3, 3),
                "map_gbs": round(mapped / t_map / 1e9, 2),
                "attention_us": round(t_vmm * 1e3, 3),
                "regular_memory_attention_us": round(t_reg * 1e3, 3),
                "how": "one layer's rows; the same call repeated 4x per graph on either memory"}
    finally:
        torch.cuda.synchronize(dev)
        vm.close()


def measure_e2e(wl, dev, args, world, chunks=8):
    """Each step copies its inputs -- every layer's q and new k/v rows plus the
    batch's slots, block tables and context lengths -- from pinned host
    memory to the device, runs the step through the C ABI (append + attention
    per layer), and reads every layer's output back to pinned host memory.
    The copies are pipelined as a serving loop would, in `chunks` groups of
    layers: a group's inputs go up on one copy stream and its outputs come
    back on another while other groups compute (8 groups measured best on
    GB300: 1.616 ms per Llama-3-8B b64 step against 1.631 with 4 groups,
    1.627 with 16 and 1.664 with 32).  The whole step -- copies
    and C-ABI calls -- is captured once as a CUDA graph and replayed every
    step, as a serving loop would; every replay moves the step's inputs and
    outputs across the host link, inside the timed region."""
    nl = wl.shape.num_layers
    b = wl.batch
    shared = [torch.as_tensor(b.slot_mapping), torch.as_tensor(b.block_tables),
              torch.as_tensor(b.ctx)]
    if wl.cow is not None:
        shared.append(wl.cow)
    bounds = [round(c * nl / chunks) for c in range(chunks + 1)]
    groups = [(bounds[c], bounds[c + 1]) for c in range(chunks) if bounds[c + 1] > bounds[c]]

    def packed(parts):
        sizes = [t.numel() * t.element_size() for t in parts]
        offs = [0]
        for n in sizes:
            offs.append(offs[-1] + (n + 255) // 256 * 256)
        host = torch.empty(offs[-1], dtype=torch.uint8, pin_memory=True)
        for t, o, n in zip(parts, offs, sizes):
            host[o:o + n].copy_(t.detach().to("cpu").contiguous().view(-1).view(torch.uint8))
        bufs = [torch.empty(offs[-1], dtype=torch.uint8, device=dev) for _ in range(2)]
        views = [[d[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(parts, offs, sizes)]
                 for d in bufs]
        return host, bufs, views, sum(sizes)

    sh = packed(shared)
    grp_in = [packed([x for l in range(l0, l1)
                      for x in (wl.layers[l].q, wl.layers[l].k_new, wl.layers[l].v_new)])
              for l0, l1 in groups]
    out_dev = [torch.empty((nl,) + tuple(wl.layers[0].q.shape), dtype=torch.bfloat16, device=dev)
               for _ in range(2)]
    host_out = torch.empty(out_dev[0].shape, dtype=torch.bfloat16, pin_memory=True)
    h2d = sh[3] + sum(x[3] for x in grp_in)
    d2h = out_dev[0].numel() * out_dev[0].element_size()
    pkv = wl.pkv
    comp = torch.cuda.current_stream(dev)
    up = torch.cuda.Stream(dev)
    down = torch.cuda.Stream(dev)
    ev = torch.cuda.Event
    in_ready = [[ev() for _ in range(len(groups) + 1)] for _ in range(2)]
    grp_done = [[ev() for _ in groups] for _ in range(2)]
    step_done = [ev() for _ in range(2)]
    out_read = [ev() for _ in range(2)]
    used = [False, False]

    def step(bi=0):
        with torch.cuda.stream(up):
            up.wait_stream(comp)  # fork from the capturing stream
            if used[bi]:
                up.wait_event(step_done[bi])  # kernels of two steps ago done with the buffers
            sh[1][bi].copy_(sh[0], non_blocking=True)
            in_ready[bi][0].record(up)
            for g in range(len(groups)):
                grp_in[g][1][bi].copy_(grp_in[g][0], non_blocking=True)
                in_ready[bi][g + 1].record(up)
        if used[bi]:
            comp.wait_event(out_read[bi])  # outputs of two steps ago read back
        used[bi] = True
        comp.wait_event(in_ready[bi][0])
        slots, tables, ctx = sh[2][bi][:3]
        cow = sh[2][bi][3] if wl.cow is not None else None
        wl.copy_on_write(cow)
        out_all = out_dev[bi]
        for g, (l0, l1) in enumerate(groups):
            comp.wait_event(in_ready[bi][g + 1])
            views = grp_in[g][2][bi]
            for l in range(l0, l1):
                q, kn, vn = views[3 * (l - l0):3 * (l - l0) + 3]
                li = wl.layers[l]
                if wl.groups is not None:
                    gs, sb, n, own = wl.groups
                    pkv.kv_append(slots, kn, vn, li.k_cache, li.v_cache)
                    pkv.paged_decode_attention_shared(q, li.k_cache, li.v_cache, tables, ctx,
                                                      b.max_context, wl.scale, gs, sb, n,
                                                      max_own_tokens=own, out=out_all[l],
                                                      workspace=wl.workspace)
                else:
                    pkv.paged_decode_step(slots, kn, vn, q, li.k_cache, li.v_cache, tables, ctx,
                                          b.max_context, wl.scale, out=out_all[l],
                                          workspace=wl.workspace)
            grp_done[bi][g].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(grp_done[bi][g])
                host_out[l0:l1].copy_(out_all[l0:l1], non_blocking=True)
        step_done[bi].record(comp)
        out_read[bi].record(down)
        comp.wait_event(out_read[bi])  # join: the step ends when its outputs are on the host

    # Graph of one step (buffers 0); replays run in stream order, one whole
    # step after another.
    for _ in range(2):
        step()
    torch.cuda.synchronize(dev)
    used[0] = used[1] = False  # the graph waits on no event from outside it
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        comp = torch.cuda.current_stream(dev)
        step()
    iters = max(20, args.steps // 10)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize(dev)
    _barrier(world)
    comp = torch.cuda.current_stream(dev)
    a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    for _ in range(iters):
        graph.replay()
    c.record(comp)
    torch.cuda.synchronize(dev)
    _barrier(world)
    ms = _max_over_ranks(a.elapsed_time(c) / iters, world, dev)
    return {"value": round(world * b.B / (ms / 1e3 / nl), 1), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms, 4), "steps": iters,
            "how": "the step's C-ABI calls and its pinned H2D inputs / D2H outputs (in %d "
                   "groups of layers on two copy streams, pipelined with the kernels) "
                   "captured as one CUDA graph and replayed every step; every copy inside "
                   "the timed region" % len(groups)}


# ------------------------------------------------------------------ CPU oracle

def _oracle_layer_host(name, layer=0, rank=0):
    b, pairs = rank_workload(name, rank)
    li = W.layer_inputs(b, layer, device="cpu")
    return b, {"q": W.to_u16(li.q), "k_new": W.to_u16(li.k_new), "v_new": W.to_u16(li.v_new),
               "k": W.to_u16(li.k_cache).copy(), "v": W.to_u16(li.v_cache).copy(),
               "cow": pairs}


def _oracle_step_text(h):
    return ("copy on write + " if h["cow"] is not None else "") + "append + attention"


def _oracle_step(oracle, b, h, scale, nthreads):
    if h["cow"] is not None:
        oracle.block_copy(h["cow"], [h["k"]], [h["v"]])
    oracle.kv_append(b.slot_mapping, h["k_new"], h["v_new"], h["k"], h["v"])
    oracle.paged_decode(h["q"], h["k"], h["v"], b.block_tables, b.ctx, scale, nthreads)


def cpu_baseline(wl, args, budget_s=15.0):
    """The oracle as it stands, on all host cores, on layers of the same
    workload until about budget_s seconds of work."""
    import oracle
    cores = os.cpu_count() or 1
    b, h = _oracle_layer_host(args.workload)
    scale = W.default_scale(b.shape)
    _oracle_step(oracle, b, h, scale, cores)       # warm
    done, t_total = 0, 0.0
    while t_total < budget_s and done < 64:
        t = time.perf_counter()
        _oracle_step(oracle, b, h, scale, cores)
        t_total += time.perf_counter() - t
        done += 1
    # the same on one core, over a shorter sample
    one, t_one = 0, 0.0
    while t_one < budget_s / 3 and one < 16:
        t = time.perf_counter()
        _oracle_step(oracle, b, h, scale, 1)
        t_one += time.perf_counter() - t
        one += 1
    return {"value": round(b.B * done / t_total, 2), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": "%d repetitions of one layer (%s, all %d sequences) of "
                      "the same workload, fp64 C oracle, %d threads"
                      % (done, _oracle_step_text(h), b.B, cores),
            "single_core": {"value": round(b.B * one / t_one, 2), "unit": UNIT, "cores": 1,
                            "sample": "%d repetitions of the same layer, 1 thread" % one}}


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    from oracle.build_oracle import build as build_oracle
    build_oracle()
    cores = os.cpu_count() or 1
    b, h = _oracle_layer_host(args.workload)
    scale = W.default_scale(b.shape)
    for _ in range(max(args.warmup, 0)):
        _oracle_step(oracle, b, h, scale, cores)
    steps = args.steps
    t = time.perf_counter()
    for _ in range(steps):
        _oracle_step(oracle, b, h, scale, cores)
    el = time.perf_counter() - t
    value = b.B * steps / el
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
            "n_gpus": world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * el / steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": _describe(args.workload), "global_batch": b.B,
                       "seq_len": int(b.ctx.max()), "layers_per_step": 1,
                       "step": "one layer of the workload (%s, all sequences)"
                               % _oracle_step_text(h)},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores,
                             "kind": "oracle",
                             "sample": "one layer per step, all %d sequences" % b.B},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def profile_case(args):
    """A small case for ncu: a few layers of the workload (about 1 GB at the
    Llama shape; 2 layers of the ragged and sharing workloads;
    --profile-layers overrides), a few attention calls through the C ABI --
    the shared-prefix call on the sharing workload.  --profile-contig S lays
    the workload's first --profile-requests requests out contiguously (offset
    reqId x S) and runs the contiguous call instead."""
    import paged_kv_cache_245_gb300 as pkv
    from __graft_entry__ import build
    build()
    dev = torch.device("cuda", 0)
    b = rank_batch(args.workload, 0)
    shape, _, kind, bs, _ = WORKLOADS[args.workload]
    nl = 2 if kind in ("sharing", "ragged") else 4
    if args.profile_layers > 0:
        nl = args.profile_layers
    if args.profile_contig > 0:
        n = min(args.profile_requests or b.B, b.B)
        S = args.profile_contig
        sub = W.PagedBatch(shape=b.shape, seed=b.seed, block_size=b.block_size,
                           num_blocks=b.num_blocks, ctx_pre=b.ctx_pre[:n], ctx=b.ctx[:n],
                           block_tables=b.block_tables[:n], slot_mapping=b.slot_mapping[:n],
                           req_ids=np.arange(n, dtype=np.int32), max_reqs=n)
        bufs = []
        for l in range(nl):
            li = W.layer_inputs(b, l, device=dev, fast_cache=True)
            bufs.append((li.q[:n].contiguous(), W.paged_to_contig(li.k_cache, sub, S),
                         W.paged_to_contig(li.v_cache, sub, S)))
            del li
        req = torch.as_tensor(sub.req_ids, device=dev)
        ctx = torch.as_tensor(sub.ctx, device=dev)
        for i in range(args.profile_calls):
            q, kb, vb = bufs[i % nl]
            pkv.contig_decode_attention(q, kb, vb, req, ctx, int(sub.max_context),
                                        W.default_scale(b.shape))
        torch.cuda.synchronize(dev)
        return
    layers = [W.layer_inputs(b, l, device=dev, fast_cache=True) for l in range(nl)]
    tables = torch.as_tensor(b.block_tables, device=dev)
    ctx = torch.as_tensor(b.ctx, device=dev)
    scale = W.default_scale(b.shape)
    if kind == "sharing":
        n = W.sharing_scenario(decode_steps=1).n
        starts = np.arange(0, b.B + 1, n, dtype=np.int32)
        shared = W.shared_prefix_blocks(b.block_tables, b.ctx, bs, starts)
        own = int((b.ctx - np.repeat(shared, n) * bs).max())
        gs = torch.as_tensor(starts, device=dev)
        sb = torch.as_tensor(shared, device=dev)
    for i in range(args.profile_calls):
        li = layers[i % nl]
        if kind == "sharing":
            pkv.paged_decode_attention_shared(li.q, li.k_cache, li.v_cache, tables, ctx,
                                              b.max_context, scale, gs, sb, n,
                                              max_own_tokens=own)
        else:
            pkv.paged_decode_attention(li.q, li.k_cache, li.v_cache, tables, ctx, b.max_context,
                                       scale)
    torch.cuda.synchronize(dev)


def profile_prefill_case(args):
    """A small case for ncu: a few prefill calls over 8 fresh 2048-token
    prompts with the workload's head shape (block_size 16)."""
    import paged_kv_cache_245_gb300 as pkv
    from __graft_entry__ import build
    build()
    dev = torch.device("cuda", 0)
    shape = rank_batch(args.workload, 0).shape
    ctx = np.full(8, 2048, np.int32)
    b = W.make_paged_batch(shape, ctx, 16, 250)
    li = W.layer_inputs(b, 0, device=dev, fast_cache=True)
    cu = torch.as_tensor(np.arange(0, 8 * 2048 + 1, 2048, dtype=np.int32), device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(251)
    q = torch.randn((8 * 2048, shape.num_q_heads, shape.head_dim), generator=g,
                    device=dev).to(torch.bfloat16)
    out = torch.empty_like(q)
    for _ in range(args.profile_prefill_calls):
        pkv.paged_prefill_attention(q, cu, li.k_cache, li.v_cache,
                                    torch.as_tensor(b.block_tables, device=dev),
                                    torch.as_tensor(b.ctx, device=dev), 2048,
                                    W.default_scale(shape), out=out)
    torch.cuda.synchronize(dev)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--skip-legs", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--profile-calls", type=int, default=0,
                    help="profiling case: run this many paged attention calls over 4 layers "
                         "of the workload and exit (no timing, no JSON)")
    ap.add_argument("--profile-layers", type=int, default=0,
                    help="profiling case: layers to cycle over (default 4; 2 for the ragged "
                         "and sharing workloads)")
    ap.add_argument("--profile-contig", type=int, default=0,
                    help="profiling case: contiguous layout with this S (tokens per request)")
    ap.add_argument("--profile-requests", type=int, default=0,
                    help="profiling case, contiguous layout: the first this many requests")
    ap.add_argument("--profile-prefill-calls", type=int, default=0,
                    help="profiling case: run this many prefill calls over 8 fresh 2048-token "
                         "prompts and exit (no timing, no JSON)")
    args = ap.parse_args()
    world, rank, local = _dist()
    if args.profile_calls > 0:
        profile_case(args)
        return
    if args.profile_prefill_calls > 0:
        profile_prefill_case(args)
        return
    if args.impl == "reference":
        # CPU-only arm: rank 0 runs it; other ranks exit without work.
        run_reference(args, world, rank)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        run_gpu(args, world, rank, local)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
