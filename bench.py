"""Benchmark of the paged decode hot path on one GB300 (or N independent replicas).

One step = the whole hot path over one batch of the workload: the KV append
of the step's new tokens (slot scatter kernel) and single-query paged decode
attention (decode kernel + split-context merge kernel).  Inputs are seeded
and synthetic; the caches are built through the library before timing.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--partition P]
                    [--window W] [--block-size 8|16|32] [--no-cpu-baseline] [--no-workloads]
    python bench.py --impl reference ...     # the oracle on the host cores

NAME is longctx_fp8 (the default: the 70B-shaped 4 x 131072-token FP8
cache, in 512-token partitions), gqa_bf16, mha_f16, prefix_bf16 or tiny.

Prints one JSON line.  ``value`` is decode tokens/s (batch x steps / time)
with every input resident in HBM; ``e2e`` is the same metric through the
public API from pinned host buffers, copies included.  Between timed steps
the caches rotate over replicas whose total size exceeds L2, so each step
streams its KV from HBM.  Unless a partition, window or block size is
forced, the line also carries ``workloads``: the device figures of every
other workload, each on its own set-up and timed the same way.
"""

import argparse
import json
import platform
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode-attn tokens/s and KV HBM GB/s (fraction of GB300 peak), 1 GPU"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0   # HBM3e nominal bandwidth of one GB300 (about 8 TB/s)
L2_BYTES = 129 * 2**20


# tokens per KV block of the workload (None: its own)
BLOCK_SIZE = None


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default="longctx_fp8")
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--partition", type=int, default=None, help="tokens per partition (default: the workload's)")
    p.add_argument("--window", type=int, default=0,
                   help="attend only each sequence's last W tokens (a slid window; 0: the whole context)")
    p.add_argument("--block-size", type=int, default=None, choices=[8, 16, 32],
                   help="re-block gqa_bf16 / mha_f16 / longctx_fp8 (default: their 16-token blocks)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the device records of the other workloads (the line's \"workloads\" key)")
    p.add_argument("--cpu-seconds", type=float, default=16.0,
                   help="budget of the oracle baseline (half on one core, half on every core)")
    p.add_argument("--clock-probe-s", type=float, default=2.0,
                   help="seconds of untimed load before the timed steps, for the clock sampler")
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------ clock sampler

class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------- workload set-up

class GpuWorkload:
    """A workload's caches, block tables and step inputs on the device."""

    def __init__(self, name, device, replicas, partition=None, window=0):
        import torch

        import paged_kv_cache_257_gb300 as pa
        from synth import workloads as wl
        self.pa, self.torch = pa, torch
        self.w = w = wl.make(name, BLOCK_SIZE)
        self.device = device
        self.partition = w.partition_size if partition is None else partition
        bs = w.block_size
        self.alloc_tables(wl)
        ctx = self.ctx_decode
        # 0 = the library plans it from the batch's context lengths, which a
        # serving host knows when it builds the block tables
        self.plan = self.partition == 0
        # a slid window: positions [ctx - W, ctx) of each row are attended
        self.window = window
        self.starts_host = np.maximum(ctx - window, 0).astype(np.int32) if window > 0 else None
        # source values of every cached token (in the cache's source type)
        k_scale = v_scale = 1.0
        seqs_k, seqs_v = [], []
        for s in range(w.batch):
            n = int(w.context_lens[s]) + (1 if w.prefix_len else 0)
            seqs_k.append(wl.kv_tokens_f32(w, "k", s, 0, n))
            seqs_v.append(wl.kv_tokens_f32(w, "v", s, 0, n))
        if w.kv_dtype == "fp8_e4m3":
            k_scale = float(max(wl.fp8_scale_of(x) for x in seqs_k))
            v_scale = float(max(wl.fp8_scale_of(x) for x in seqs_v))
        self.desc = pa.CacheDesc(w.num_blocks, bs, w.n_kv_heads, w.head_dim, w.kv_dtype, k_scale, v_scale)
        src = w.src_dtype
        torch_src = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[src]

        def dev(arr_f32):
            t = torch.from_numpy(np.ascontiguousarray(arr_f32))
            return t.to(torch_src).to(device) if src != "f32" else t.to(device)

        # fill the caches through the library: slot mapping then append, in chunks
        seq_ids = np.concatenate([np.full(len(x), s, np.int32) for s, x in enumerate(seqs_k)])
        pos = np.concatenate([np.arange(len(x), dtype=np.int32) for x in seqs_k])
        slots = pa.compute_slot_mapping(self.tables_np, seq_ids, pos, bs)
        self.pools = []
        for r in range(replicas):
            kc, vc = self.desc.new_pools(device, fill=0)
            self.pools.append((kc, vc))
        chunk = 1 << 16
        allk = np.concatenate(seqs_k)
        allv = np.concatenate(seqs_v)
        for lo in range(0, len(slots), chunk):
            k = dev(allk[lo:lo + chunk])
            v = dev(allv[lo:lo + chunk])
            sl = torch.from_numpy(slots[lo:lo + chunk]).to(device)
            for kc, vc in self.pools:
                pa.kv_append(self.desc, k, v, sl, kc, vc)
        del allk, allv
        torch.cuda.synchronize()
        self.kv_tokens = int(np.sum(ctx - (self.starts_host if window > 0 else 0)))
        self.kv_bytes = self.kv_tokens * 2 * w.n_kv_heads * w.head_dim * w.kv_elem_bytes
        self.unique_kv_bytes = self.kv_bytes
        if w.prefix_len and window <= 0:
            uniq = w.prefix_len + int(np.sum(ctx - w.prefix_len))
            self.unique_kv_bytes = uniq * 2 * w.n_kv_heads * w.head_dim * w.kv_elem_bytes
        # step inputs
        q = wl.cast(wl.queries_f32(w), w.q_dtype)
        if w.q_dtype == "bf16":
            self.q = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(device)
        else:
            self.q = torch.from_numpy(q).to(device)
        self.block_tables = torch.from_numpy(self.tables_np).to(device)
        self.context_lens = torch.from_numpy(ctx.astype(np.int32)).to(device)
        self.ctx_host = ctx.astype(np.int32)
        self.context_starts = None
        if window > 0:
            self.context_starts = torch.from_numpy(self.starts_host).to(device)
        if self.plan:
            self.partition = self.plan_partition()
        self.new_k, self.new_v, self.new_slots = self.step_append_inputs(wl, dev)
        self.workspace = None
        need = pa.decode_workspace_size(self.desc, w.batch, w.n_q_heads, self.tables_np.shape[1], self.partition)
        if need:
            self.workspace = pa.new_workspace(need, device)
        self.out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float32, device=device)
        self.resolved_partition = pa.partition_size(self.desc, w.batch, w.n_q_heads, self.tables_np.shape[1],
                                                    self.partition)
        # the merge kernel runs when a sequence may hold more than 16 partitions
        cap = self.tables_np.shape[1] * bs
        self.merge_launches = 1 if -(-cap // self.resolved_partition) > 16 else 0

    def alloc_tables(self, wl):
        w = self.w
        if w.block_tables is not None:
            self.tables_np = w.block_tables
            self.ctx_decode = w.context_lens.astype(np.int64)
            self.append_positions = None
            return
        # prefix sharing: blocks handed out by the library's allocator; the
        # prefix blocks are shared by every sequence (reference count = batch)
        self.allocator = self.pa.BlockAllocator(w.num_blocks, w.alloc_seed)
        self.tables_np, self.ctx_decode, self.append_slots = wl.build_prefix_tables(w, self.allocator)
        self.append_positions = w.context_lens.copy()

    def plan_partition(self):
        w = self.w
        lens = self.ctx_host
        if self.starts_host is not None:        # a window's partitions start at its start rounded down to 16
            lens = self.ctx_host - (self.starts_host & ~15)
        return self.pa.plan_partition(self.desc, w.batch, w.n_q_heads, self.tables_np.shape[1], lens)

    def step_append_inputs(self, wl, dev):
        torch = self.torch
        w = self.w
        if w.name == "gqa_bf16":
            slots = wl.append_slots(w)
            k, v = wl.append_tokens_f32(w, "k"), wl.append_tokens_f32(w, "v")
        elif w.prefix_len:
            slots = np.array(self.append_slots, dtype=np.int64)
            k = np.stack([wl.kv_tokens_f32(w, "k", s, int(c), int(c) + 1)[0] for s, c in enumerate(w.context_lens)])
            v = np.stack([wl.kv_tokens_f32(w, "v", s, int(c), int(c) + 1)[0] for s, c in enumerate(w.context_lens)])
        else:
            return None, None, None
        return dev(k), dev(v), torch.from_numpy(np.asarray(slots, dtype=np.int64)).to(self.device)

    def step(self, r, ev=None, decode_only=False):
        """One step on cache replica r; ``ev``: None or four events (append
        start, end, decode start, end); ``decode_only`` leaves the append
        out.  Returns the kernels it launched."""
        pa = self.pa
        kc, vc = self.pools[r % len(self.pools)]
        n = 0
        if self.new_k is not None and not decode_only:
            if ev is not None:
                ev[0].record()
            pa.kv_append(self.desc, self.new_k, self.new_v, self.new_slots, kc, vc)
            if ev is not None:
                ev[1].record()
            n += 1
        if ev is not None:
            ev[2].record()
        pa.decode_attention(self.desc, self.q, kc, vc, self.block_tables, self.context_lens, self.w.scale,
                            partition=self.partition, workspace=self.workspace, out=self.out,
                            context_starts=self.context_starts)
        if ev is not None:
            ev[3].record()
        return n + 1 + self.merge_launches


# Counters of one launch of each workload's decode kernel (the warp-per-item
# kernel for longctx_fp8, the CTA-per-item kernel for the others), from the
# ncu captures summarised in profiles/: DRAM bytes read + written, and L2
# read sectors / requests from the SMs' load unit (four 32-byte sectors per
# request = whole 128-byte lines).  They hold for the kernel code they were
# taken on (the fingerprint of the files below, see _code_fingerprint);
# after any change to that code they are reported as null until a new
# capture is recorded here.
TRAFFIC_SOURCES = ("paged_kv_cache_257_gb300/csrc/decode_mma.cu", "paged_kv_cache_257_gb300/csrc/decode_warp.cu",
                   "paged_kv_cache_257_gb300/csrc/mma_chunk.cuh", "paged_kv_cache_257_gb300/csrc/common.cuh",
                   "paged_kv_cache_257_gb300/csrc/decode.h", "paged_kv_cache_257_gb300/csrc/decode_epilogue.cuh",
                   "paged_kv_cache_257_gb300/csrc/window.cuh")
NCU_TRAFFIC = {"4cdd1064cf872625": {"longctx_fp8": 1_074_022_912 + 7_592_448,
                                    "gqa_bf16": 283_151_360 + 3_324_672,
                                    "mha_f16": 671_249_152 + 2_931_200,
                                    "prefix_bf16": 72_591_104 + 977_920}}
NCU_L2_SECTORS = {"4cdd1064cf872625": {"longctx_fp8": (42_150_239, 10_572_906),
                                       "gqa_bf16": (11_124_599, 2_794_323),
                                       "mha_f16": (26_238_115, 6_562_870),
                                       "prefix_bf16": (14_301_736, 3_591_418)}}
DECODE_KERNEL_OF = {"longctx_fp8": "decode_warp_kernel", "gqa_bf16": "decode_mma_kernel",
                    "mha_f16": "decode_mma_kernel", "prefix_bf16": "decode_mma_kernel"}


def _code_fingerprint(paths):
    """First 16 hex digits of the sha256 of the files' code with comments
    and runs of white space removed, so that edits to comments alone keep
    the recorded counters valid and any change to the code voids them."""
    import hashlib
    import re
    root = os.path.dirname(os.path.abspath(__file__))
    h = hashlib.sha256()
    for f in paths:
        with open(os.path.join(root, f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def captured_traffic(workload):
    return NCU_TRAFFIC.get(_code_fingerprint(TRAFFIC_SOURCES), {}).get(workload)


def captured_sectors_per_request(workload):
    sr = NCU_L2_SECTORS.get(_code_fingerprint(TRAFFIC_SOURCES), {}).get(workload)
    return None if sr is None else sr[0] / sr[1]


def copy_blocks_timing(pa, torch, w, device, pairs=4096):
    """Copy-on-write's device half (pa_copy_blocks) on this workload's block
    geometry: `pairs` shuffled block pairs of a scratch pool, K and V, timed
    with CUDA events on the launching stream after a warm-up call."""
    import synth
    desc = pa.CacheDesc(2 * pairs, w.block_size, w.n_kv_heads, w.head_dim, w.kv_dtype, 1.0, 1.0)
    kc, vc = desc.new_pools(device, fill=0)
    perm = synth.permutation(92, 0, 2 * pairs).astype(np.int32)
    src = torch.from_numpy(perm[:pairs].copy()).to(device)
    dst = torch.from_numpy(perm[pairs:].copy()).to(device)
    pa.copy_blocks(desc, kc, vc, src, dst)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    reps = 10
    ev[0].record()
    for _ in range(reps):
        pa.copy_blocks(desc, kc, vc, src, dst)
    ev[1].record()
    torch.cuda.synchronize()
    us = ev[0].elapsed_time(ev[1]) * 1e3 / reps
    block_bytes = w.n_kv_heads * w.block_size * w.head_dim * w.kv_elem_bytes
    moved = 2 * pairs * block_bytes * 2          # K and V, read + write
    del kc, vc
    return {"pairs": pairs, "block_bytes": block_bytes, "us": us, "gbs": moved / us / 1e3,
            "frac_of_peak": moved / us / 1e3 / measured_peak()[0],
            "note": "pa_copy_blocks on a scratch pool (2 x pairs blocks), read + write bytes, after warm-up"}


def prefix_cache_host_timing(pa, w):
    """Host cost of the prefix cache on this workload's shape: one request
    computes and caches the shared prefix; each of the others maps it
    (pa_prefix_match) and caches its own full blocks (pa_prefix_insert).
    Token ids are seeded synthetic values."""
    import synth
    bs = w.block_size
    alloc = pa.BlockAllocator(w.num_blocks, 1)
    cache = pa.PrefixCache(alloc, bs)
    prefix = [int(x) for x in synth.uniform_int(90, 0, w.prefix_len, 0, 1 << 17)]
    cap = -(-int(max(w.context_lens) + 1) // bs)
    rows, match_s, insert_s, matched = [], 0.0, 0.0, 0
    for s in range(w.batch):
        n_tok = int(w.context_lens[s]) + 1
        toks = prefix + [int(x) for x in synth.uniform_int(91, s, n_tok - w.prefix_len, 0, 1 << 17)]
        row = [-1] * cap
        t0 = time.perf_counter()
        m = cache.match(toks, row)
        match_s += time.perf_counter() - t0
        matched += m
        n = m
        for t in range(m * bs, n_tok):
            _, n, _ = alloc.append_slot(row, n, t, bs)
        t0 = time.perf_counter()
        cache.insert(toks, row, n)
        insert_s += time.perf_counter() - t0
        rows.append((row, n))
    blocks_private = sum(-(-(int(c) + 1) // bs) for c in w.context_lens)
    out = {"requests": w.batch, "prefix_tokens": w.prefix_len,
           "match_us_per_request": match_s / w.batch * 1e6, "insert_us_per_request": insert_s / w.batch * 1e6,
           "blocks_matched": matched, "blocks_held": w.num_blocks - alloc.free_count,
           "blocks_without_sharing": blocks_private,
           "note": "host-side, through the Python binding (ctypes); not in the timed GPU region"}
    cache.destroy()
    return out


def capture(wk, fn):
    """A CUDA graph of the library calls ``fn`` makes (captured on a side
    stream; replayed on the current one).  Returns (graph, fn's result)."""
    torch = wk.torch
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side):
        res = fn()
    torch.cuda.current_stream().wait_stream(side)
    return g, res


def replay_ms(wk, g):
    """Device time of one replay of ``g`` (CUDA events on the current stream,
    synchronised on both sides)."""
    torch = wk.torch
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    start.record()
    g.replay()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def time_device(wk, steps, warmup, probe_s=0.0):
    """The device-side timings of a workload.

    W eager warm-up steps, then the K timed steps launched as one CUDA graph
    (so that the host's launch rate never paces the GPU), bracketed by a
    barrier and synchronisation; then a graph of K decode launches alone,
    whose replay time / K is the decode's average launch duration; then the
    same K steps again, launched eagerly with events around each append and
    decode (per-launch spread; the events and the host's launches add gaps).

    Returns (total ms of the timed steps, decode ms per launch in the
    decode-only region, evented decode ms per step, evented append ms per
    step or [], kernels launched in the timed region).

    ``probe_s`` seconds of extra untimed replays run first so that the clock
    sampler (nvidia-smi, 200 ms period) sees the GPU under this load."""
    torch = wk.torch
    for i in range(warmup):
        wk.step(i)
    torch.cuda.synchronize()
    g_steps, launches = capture(wk, lambda: sum(wk.step(warmup + i) for i in range(steps)))
    g_dec, _ = capture(wk, lambda: [wk.step(warmup + i, decode_only=True) for i in range(steps)])
    g_steps.replay()
    g_dec.replay()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < probe_s:
        g_steps.replay()
        torch.cuda.synchronize()
    total_ms = replay_ms(wk, g_steps)
    dec_launch_ms = replay_ms(wk, g_dec) / steps
    del g_steps, g_dec
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for i in range(steps):
        wk.step(warmup + i, ev[i])
    torch.cuda.synchronize()
    dec_ms = [e[2].elapsed_time(e[3]) for e in ev]
    app_ms = [e[0].elapsed_time(e[1]) for e in ev] if wk.new_k is not None else []
    return total_ms, dec_launch_ms, dec_ms, app_ms, launches


def time_decode_no_flush(wk, steps):
    """Decode average launch duration with one cache replica reused launch
    after launch (its KV stays in L2 as far as it fits): a graph of K decode
    launches on replica 0, after a warm-up replay."""
    g, _ = capture(wk, lambda: [wk.step(0, decode_only=True) for _ in range(steps)])
    g.replay()
    wk.torch.cuda.synchronize()
    return replay_ms(wk, g) / steps


DECODE_US_NOTE = ("launch_avg: K decode launches replayed from one CUDA graph, region time / K (the roofline's "
                  "duration); mean/median/min: the same launches made eagerly with CUDA events around each "
                  "(they include the events' and the host's launch gaps)")


def _stats_us(ms):
    return {"mean": statistics.mean(ms) * 1e3, "median": statistics.median(ms) * 1e3, "min": min(ms) * 1e3}


class E2EBuffers:
    """Pinned host and device buffers of the end-to-end loop.  Every input
    of a step sits in one pinned staging buffer (256-byte aligned pieces), so
    a step uploads with one copy; typed views name the pieces on the device."""

    def __init__(self, wk):
        torch = wk.torch
        host = {"q": wk.q.cpu().pin_memory(), "bt": wk.block_tables.cpu().pin_memory(),
                "ctx": wk.context_lens.cpu().pin_memory()}
        if wk.context_starts is not None:
            host["starts"] = wk.context_starts.cpu().pin_memory()
        if wk.new_k is not None:
            host.update(k=wk.new_k.cpu().pin_memory(), v=wk.new_v.cpu().pin_memory(),
                        slots=wk.new_slots.cpu().pin_memory())
        self.out_host = [torch.empty(wk.out.shape, dtype=wk.out.dtype).pin_memory() for _ in range(2)]
        self.outs = [torch.empty_like(wk.out) for _ in range(2)]
        offs, size = {}, 0
        for k, v in host.items():
            offs[k] = size
            size += (v.numel() * v.element_size() + 255) // 256 * 256
        self.stage = torch.empty(size, dtype=torch.uint8).pin_memory()
        for k, v in host.items():
            n = v.numel() * v.element_size()
            self.stage[offs[k]:offs[k] + n].copy_(v.contiguous().view(-1).view(torch.uint8))
        self.bufs = [torch.empty(size, dtype=torch.uint8, device=wk.device) for _ in range(2)]
        self.dev = [{k: buf[offs[k]:offs[k] + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
                     for k, v in host.items()} for buf in self.bufs]
        self.h2d = sum(v.numel() * v.element_size() for v in host.values())
        self.d2h = self.out_host[0].numel() * self.out_host[0].element_size()


def e2e_compute(wk, d, out, r, part):
    """One step's device work through the public API on the current stream."""
    kc, vc = wk.pools[r % len(wk.pools)]
    if "k" in d:
        wk.pa.kv_append(wk.desc, d["k"], d["v"], d["slots"], kc, vc)
    wk.pa.decode_attention(wk.desc, d["q"], kc, vc, d["bt"], d["ctx"], wk.w.scale, partition=part,
                           workspace=wk.workspace, out=out, context_starts=d.get("starts"))


def time_e2e(wk, steps, warmup):
    """The public API from pinned host buffers, as a serving loop drives it:
    every step uploads its inputs and downloads its output.  The uploads and
    downloads run on their own streams into two sets of buffers, so the next
    step's inputs and the previous step's output move while this step
    computes; a buffer is reused only after the step two back has finished
    with it.  The timed region ends when the last output is in host memory."""
    torch = wk.torch
    eb = E2EBuffers(wk)
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    computed = [torch.cuda.Event() for _ in range(2)]     # step done with dev[b], outs[b] written
    uploaded = [torch.cuda.Event() for _ in range(2)]
    downloaded = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):
        computed[b].record(comp)
        downloaded[b].record(comp)

    def one(r):
        b = r % 2
        with torch.cuda.stream(up):
            up.wait_event(computed[b])
            eb.bufs[b].copy_(eb.stage, non_blocking=True)
            uploaded[b].record(up)
        comp.wait_event(uploaded[b])
        comp.wait_event(downloaded[b])
        part = wk.plan_partition() if wk.plan else wk.partition   # host work of a serving step
        e2e_compute(wk, eb.dev[b], eb.outs[b], r, part)
        computed[b].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(computed[b])
            eb.out_host[b].copy_(eb.outs[b], non_blocking=True)
            downloaded[b].record(down)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    start.record(comp)
    up.wait_event(start)
    for i in range(steps):
        one(warmup + i)
    comp.wait_event(downloaded[(warmup + steps - 1) % 2])
    end.record(comp)
    torch.cuda.synchronize()
    return start.elapsed_time(end), eb.h2d, eb.d2h


def time_e2e_graph(wk, steps, warmup):
    """The same serving loop with each step replayed from a CUDA graph, the
    way decode steps of a fixed batch shape are usually launched.

    Graph i (buffer set b = i % 2, cache replica i % R) computes on dev[b]
    (uploaded by the graph before it), uploads the next step's inputs into
    dev[1 - b] and downloads the previous step's output from outs[1 - b]; the
    copies are branches of the graph that run beside the kernels.  Graphs
    replay in stream order, so each buffer's writer has finished before its
    reader starts.  The partition size is planned once on the host: the
    batch's lengths do not change between these steps (a serving loop keeps
    one graph per batch shape and partition size).  Returns (ms, h2d, d2h) of
    the timed steps, including the first upload and the last download."""
    torch = wk.torch
    eb = E2EBuffers(wk)
    part = wk.plan_partition() if wk.plan else wk.partition
    n_graphs = 2 * len(wk.pools) // math.gcd(2, len(wk.pools))
    side = torch.cuda.Stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    for buf in eb.bufs:                                 # valid inputs in both sets before any compute
        buf.copy_(eb.stage)
    with torch.cuda.stream(side):                       # warm-up before capture
        for i in range(n_graphs):
            e2e_compute(wk, eb.dev[i % 2], eb.outs[i % 2], i, part)
    torch.cuda.synchronize()
    graphs = []
    for i in range(n_graphs):
        b = i % 2
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            cs = torch.cuda.current_stream()
            up.wait_stream(cs)
            down.wait_stream(cs)
            with torch.cuda.stream(up):
                eb.bufs[1 - b].copy_(eb.stage, non_blocking=True)
            with torch.cuda.stream(down):
                eb.out_host[1 - b].copy_(eb.outs[1 - b], non_blocking=True)
            e2e_compute(wk, eb.dev[b], eb.outs[b], i, part)
            cs.wait_stream(up)
            cs.wait_stream(down)
        graphs.append(g)
    comp = torch.cuda.current_stream()

    def run(n):
        eb.bufs[0].copy_(eb.stage, non_blocking=True)
        for i in range(n):
            graphs[i % n_graphs].replay()
        eb.out_host[(n - 1) % 2].copy_(eb.outs[(n - 1) % 2], non_blocking=True)

    run(max(warmup, n_graphs))
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    start.record(comp)
    run(steps)
    end.record(comp)
    torch.cuda.synchronize()
    return start.elapsed_time(end), eb.h2d, eb.d2h


# -------------------------------------------------------------- oracle arm
#
# The oracle timed on the host cores: bench's cpu_baseline leg and the
# reference arm (--impl reference).  Workers are separate processes started
# with `spawn` (never forked from a process that has touched the GPU), each
# with one BLAS thread, each timing the oracle's paged decode over its own
# share of the workload.  Long contexts are sampled: a worker attends the
# first ORACLE_TOKEN_CAP tokens of its sequence and counts that call as the
# matching fraction of a sequence-step.

ORACLE_TOKEN_CAP = 8192
_ONE_THREAD_ENV = {k: "1" for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS",
                                     "NUMEXPR_NUM_THREADS", "VECLIB_MAXIMUM_THREADS")}


def oracle_share(w_name, worker, n_workers, window=0):
    """(sequence ids, token cap or None) of one worker's sample."""
    from synth import workloads as wl
    w = wl.make(w_name, BLOCK_SIZE)
    cap = ORACLE_TOKEN_CAP if int(np.max(w.context_lens)) > 4 * ORACLE_TOKEN_CAP and window <= 0 else None
    if cap is None and n_workers <= w.batch:
        return list(range(worker, w.batch, n_workers)), None
    return [worker % w.batch], cap


def oracle_sample(w_name, seqs, cap, window=0):
    """The oracle's own paged cache for sequences ``seqs`` of the workload (at
    most their first ``cap`` tokens when ``cap`` is set).  The pool holds
    only those sequences' blocks, in the workload's physical order and
    sharing (ids renumbered), so the sample reads scattered blocks as the
    full workload does.  Returns the inputs of decode_attention_paged and
    the sequence-steps one call stands for."""
    from oracle import allocator as oalloc
    from oracle import cache as ocache
    from synth import workloads as wl
    w = wl.make(w_name, BLOCK_SIZE)
    if w.block_tables is None:
        tables, ctx, _ = wl.build_prefix_tables(w, oalloc.BlockAllocator(w.num_blocks, w.alloc_seed))
    else:
        tables, ctx = w.block_tables, w.context_lens.astype(np.int64)
    bs = w.block_size
    full = np.asarray([int(ctx[s]) for s in seqs], dtype=np.int64)
    lens = np.minimum(full, cap) if cap else full
    nblk = [-(-int(n) // bs) for n in lens]
    used = sorted({int(tables[s, j]) for s, n in zip(seqs, nblk) for j in range(n)})
    renum = {b: i for i, b in enumerate(used)}
    t2 = np.zeros((len(seqs), max(1, max(nblk))), dtype=np.int32)
    for i, (s, n) in enumerate(zip(seqs, nblk)):
        t2[i, :n] = [renum[int(b)] for b in tables[s, :n]]
    kp = ocache.new_pool(max(1, len(used)), w.n_kv_heads, bs, w.head_dim, w.kv_dtype)
    vp = ocache.new_pool(max(1, len(used)), w.n_kv_heads, bs, w.head_dim, w.kv_dtype)
    vals = [(wl.kv_tokens_f32(w, "k", s, 0, int(n)), wl.kv_tokens_f32(w, "v", s, 0, int(n)))
            for s, n in zip(seqs, lens)]
    scales = (1.0, 1.0)
    if w.kv_dtype == "fp8_e4m3":
        scales = (float(wl.fp8_scale_of(np.concatenate([k.ravel() for k, _ in vals]))),
                  float(wl.fp8_scale_of(np.concatenate([v.ravel() for _, v in vals]))))
    for i, ((k, v), n) in enumerate(zip(vals, lens)):
        slots = ocache.slot_mapping(t2, [i] * int(n), range(int(n)), bs)
        ocache.kv_append(kp, vp, wl.cast(k, w.src_dtype), wl.cast(v, w.src_dtype), slots, w.src_dtype,
                         w.kv_dtype, *scales)
    q = wl.cast(wl.queries_f32(w), w.q_dtype)[list(seqs)]
    starts = np.maximum(lens - window, 0) if window > 0 else None
    units = float(np.sum(lens / full))
    return dict(w=w, q=q, kp=kp, vp=vp, tables=t2, ctx=lens, scales=scales, starts=starts, units=units)


def _oracle_call(s):
    from oracle import attention as oatt  # test infrastructure: the oracle legs of this file only
    w = s["w"]
    oatt.decode_attention_paged(s["q"], s["kp"], s["vp"], s["tables"], s["ctx"], w.scale, w.kv_dtype,
                                *s["scales"], q_dtype=w.q_dtype, context_starts=s["starts"])


def _oracle_worker(w_name, worker, n_workers, window, block_size, calls, warmup, budget_s, barrier_, queue):
    """One spawned worker: set up its share, wait for the others, then time
    ``calls`` oracle calls (or as many as fit in ``budget_s``)."""
    global BLOCK_SIZE
    BLOCK_SIZE = block_size
    try:
        seqs, cap = oracle_share(w_name, worker, n_workers, window)
        s = oracle_sample(w_name, seqs, cap, window)
        for _ in range(warmup):
            _oracle_call(s)
        barrier_.wait(timeout=900)
        t0 = time.perf_counter()
        done = 0
        while (calls is not None and done < calls) or (calls is None and (done == 0 or
                                                                            time.perf_counter() - t0 < budget_s)):
            _oracle_call(s)
            done += 1
        queue.put((worker, done * s["units"], time.perf_counter() - t0, done, seqs, cap))
    except BaseException as e:  # reported to the parent, which raises
        queue.put((worker, None, repr(e), 0, [], None))


def run_oracle(w_name, n_workers, calls=None, warmup=0, budget_s=None, window=0):
    """The oracle's throughput on ``n_workers`` host cores: each worker a
    spawned single-threaded process over its own share of the workload,
    all timed together.  Returns (sequence-steps per second, seconds,
    sequence-steps, sample text)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    saved = {k: os.environ.get(k) for k in _ONE_THREAD_ENV}
    os.environ.update(_ONE_THREAD_ENV)              # children start with one BLAS thread
    try:
        queue, barrier_ = ctx.Queue(), ctx.Barrier(n_workers)
        procs = [ctx.Process(target=_oracle_worker, args=(w_name, i, n_workers, window, BLOCK_SIZE, calls, warmup,
                                                          budget_s, barrier_, queue)) for i in range(n_workers)]
        for p in procs:
            p.start()
        res = []
        t0 = time.perf_counter()
        while len(res) < len(procs):
            try:
                res.append(queue.get(timeout=2.0))
            except Exception:   # queue.Empty: a worker that died without a result ends the wait
                dead = [p.exitcode for p in procs if p.exitcode not in (None, 0)]
                if dead or time.perf_counter() - t0 > 1800:
                    for p in procs:
                        if p.is_alive():
                            p.terminate()
                    raise RuntimeError(f"oracle workers ended without results (exit codes {dead})")
        for p in procs:
            p.join(timeout=60)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    bad = [r for r in res if r[1] is None]
    if bad:
        raise RuntimeError(f"oracle worker failed: {bad[0][2]}")
    secs = max(r[2] for r in res)
    units = sum(r[1] for r in res)
    calls_done = sum(r[3] for r in res)
    cap = res[0][5]
    sample = (f"oracle decode_attention_paged (numpy, float64) in {n_workers} spawned single-threaded "
              f"process(es), each over its share of {w_name}'s sequences (their block tables, context lengths"
              + (f" capped at the first {cap} tokens, counted as {cap}/{int(max(wl_ctx(w_name)))} of a "
                 f"sequence-step" if cap else "") + (f", last {window} tokens" if window > 0 else "")
              + f"): {calls_done} calls, {units:.3f} sequence-steps in {secs:.1f} s")
    return units / secs, secs, units, sample


def wl_ctx(w_name):
    from synth import workloads as wl
    return wl.make(w_name, BLOCK_SIZE).context_lens


def cpu_baseline(w_name, budget_s, window=0):
    """The oracle on one core and on every core of the host, same sample."""
    n = os.cpu_count() or 1
    v1, s1, u1, sample1 = run_oracle(w_name, 1, budget_s=budget_s / 2, window=window)
    vn, sn, un, samplen = run_oracle(w_name, n, budget_s=budget_s / 2, window=window)
    return {"value": vn, "unit": "tokens/s", "cores": n, "kind": "oracle", "sample": samplen,
            "value_all_cores": vn, "value_1thread": v1, "sample_1thread": sample1, **host_cpu()}


def host_cpu():
    """The host's CPU model and logical core count."""
    model = None
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.split(":")[0].strip().lower() == "model name":
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    key = line.split(":")[0].strip().lower()
                    if key in ("model name", "cpu model"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"cpu_model": f"{model or platform.machine()} ({platform.machine()})", "nproc": os.cpu_count()}

# ----------------------------------------------------------- distributed

_dist = None


def barrier():
    if _dist is not None:
        _dist.barrier()


def max_over_ranks(x):
    if _dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    _dist.all_reduce(t, op=_dist.ReduceOp.MAX)
    return float(t.item())


def init_distributed(world):
    """One process per GPU: a gloo group for the barrier and the max over
    ranks (the replicas exchange no data)."""
    global _dist
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        _dist = dist


def job_rate(units_per_step, steps, world, local_ms):
    """Whole-job rate: every rank's units over the slowest rank's time.
    Returns (units per second, that time in ms)."""
    t = max_over_ranks(local_ms)
    return units_per_step * steps * world / (t / 1e3), t


def replicas_for(w):
    """Cache replicas whose total exceeds L2 several times (one when a single
    copy already does), so that every step streams its KV from HBM."""
    per = w.num_blocks * w.n_kv_heads * w.block_size * w.head_dim * w.kv_elem_bytes * 2
    return max(1, min(4, math.ceil(3 * L2_BYTES / per))), per


OTHER_WORKLOADS = ("gqa_bf16", "mha_f16", "prefix_bf16", "tiny", "longctx_fp8")


def workload_record(name, device, steps, warmup):
    """Device-side figures of one more workload (its own set-up, the same
    timing as the headline's, no end-to-end loop and no clock probe)."""
    import torch
    from synth import workloads as wl
    w = wl.make(name, BLOCK_SIZE)
    replicas, per = replicas_for(w)
    wk = GpuWorkload(name, device, replicas)
    total_ms, dec_launch_ms, dec_ms, app_ms, launches = time_device(wk, steps, warmup)
    peak = measured_peak()[0]
    step_s = total_ms / 1e3 / steps
    dec_s = dec_launch_ms / 1e3
    rec = {"batch": w.batch, "kv_dtype": w.kv_dtype, "kv_tokens": wk.kv_tokens, "kv_bytes": wk.kv_bytes,
           "partition_size": wk.resolved_partition, "tokens_per_s": w.batch / step_s, "ms_per_step": step_s * 1e3,
           "decode_us": dict(_stats_us(dec_ms), launch_avg=dec_launch_ms * 1e3, note=DECODE_US_NOTE),
           "kv_gbs": wk.kv_bytes / dec_s / 1e9,
           "frac": wk.kv_bytes / dec_s / 1e9 / peak, "traffic": captured_traffic(name),
           "l2_sectors_per_request": captured_sectors_per_request(name),
           "kv_gbs_step": wk.kv_bytes / step_s / 1e9, "gpu_launches": launches,
           "l2": (f"{replicas} cache replicas rotated per step ({replicas * per / 2**20:.0f} MiB > L2)"
                  if replicas * per > L2_BYTES else f"KV ({per / 2**10:.0f} KiB) fits in L2: launch-bound")}
    if wk.unique_kv_bytes != wk.kv_bytes:
        rec["unique_kv_gbs"] = wk.unique_kv_bytes / dec_s / 1e9
        rec["unique_frac"] = rec["unique_kv_gbs"] / peak
    if app_ms:
        rec["append_us"] = dict(_stats_us(app_ms), tokens=w.append_tokens)
    del wk
    torch.cuda.empty_cache()
    return rec


def main():
    global BLOCK_SIZE
    args = parse()
    BLOCK_SIZE = args.block_size
    rank, world, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args)
    init_distributed(world)
    import torch
    from paged_kv_cache_257_gb300 import build
    if rank == 0:          # one build for all ranks: they share the source tree
        build.build()
    barrier()
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    from synth import workloads as wl
    w = wl.make(args.workload, BLOCK_SIZE)
    replicas, per = replicas_for(w)
    wk = GpuWorkload(args.workload, device, replicas, args.partition, args.window)
    with ClockSampler(local) as clk:
        total_ms, dec_launch_ms, dec_ms, app_ms, launches = time_device(wk, args.steps, args.warmup,
                                                                       args.clock_probe_s)
    no_flush_ms = time_decode_no_flush(wk, args.steps)
    eager_ms, h2d, d2h = time_e2e(wk, args.steps, args.warmup)
    try:
        e2e_ms, h2d, d2h = time_e2e_graph(wk, args.steps, args.warmup)
        e2e_mode = "graph"
    except RuntimeError as e:                            # capture refused: the eager loop's number stands
        e2e_ms, e2e_mode = eager_ms, f"eager (graph capture failed: {str(e).splitlines()[0][:120]})"
    value, total_ms = job_rate(w.batch, args.steps, world, total_ms)
    e2e_value, e2e_ms = job_rate(w.batch, args.steps, world, e2e_ms)
    eager_value, eager_ms = job_rate(w.batch, args.steps, world, eager_ms)
    dec_avg_s = dec_launch_ms / 1e3
    peak, peak_src = measured_peak()
    achieved = wk.kv_bytes / dec_avg_s / 1e9
    step_s = total_ms / 1e3 / args.steps
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.kv_dtype, "data": "synthetic",
        "config": {"workload": args.workload, "batch": w.batch, "n_q_heads": w.n_q_heads,
                   "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
                   "kv_dtype": w.kv_dtype, "q_dtype": w.q_dtype, "kv_tokens": wk.kv_tokens,
                   "partition_size": wk.resolved_partition, "append_tokens": w.append_tokens,
                   "l2": f"{replicas} cache replicas rotated per step ({replicas * per / 2**20:.0f} MiB > L2)",
                   "parallelism": f"replicas x{world}",
                   "decode_schedule": "deterministic" if wk.pa.decode_deterministic() else
                   "balanced tail (the library's default; reproducible to bf16 rounding)",
                   **({"window": args.window} if args.window > 0 else {})},
        "kv_tokens_per_s": wk.kv_tokens * world / step_s,
        "kv_gbs": wk.kv_bytes * world / step_s / 1e9,
        "decode_kernel_us": dec_avg_s * 1e6,
        "decode_us": dict(_stats_us(dec_ms), launch_avg=dec_launch_ms * 1e3, note=DECODE_US_NOTE,
                          no_flush_launch_avg=no_flush_ms * 1e3,
                          no_flush_note="one replica reused: its KV stays in L2 as far as it fits"),
        "roofline": {"bound": "hbm", "kernel": "paged decode (decode + split merge)", "achieved": achieved,
                     "duration": "decode_us.launch_avg: a CUDA-graph region of K decode launches / K",
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": captured_traffic(args.workload),
                     "traffic_of": f"one {DECODE_KERNEL_OF.get(args.workload, 'decode')} launch (ncu)",
                     "l2_sectors_per_request": captured_sectors_per_request(args.workload),
                     "peak_source": f"{peak_src} hbm_gbs", "bytes_per_launch": wk.kv_bytes,
                     "nominal_peak_gbs": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "launch": e2e_mode, "eager_value": eager_value,
                "eager_note": "the same loop launching each call from Python, planning the partition every step"},
        "gpu_launches": launches,
        "clocks": dict(clk.summary(), window=f"{args.clock_probe_s:.1f} s of the same steps + the timed steps"),
    }
    if wk.unique_kv_bytes != wk.kv_bytes:
        line["unique_kv_gbs"] = wk.unique_kv_bytes * world / step_s / 1e9
    if app_ms:
        line["append_us"] = dict(_stats_us(app_ms), tokens=w.append_tokens)
    if w.prefix_len and rank == 0:
        line["prefix_cache"] = prefix_cache_host_timing(wk.pa, w)
    line["copy_blocks"] = copy_blocks_timing(wk.pa, torch, w, device)
    del wk
    torch.cuda.empty_cache()
    # the other workloads, each measured the same way on its own set-up
    plain = args.partition is None and args.window <= 0 and args.block_size is None
    if plain and not args.no_workloads:
        recs = {}
        for name in OTHER_WORKLOADS:
            if name != args.workload:
                recs[name] = workload_record(name, device, args.steps, args.warmup)
        line["workloads"] = recs
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds, args.window)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if _dist is not None:
        _dist.destroy_process_group()
    return 0


def run_reference(args):
    """The oracle as the reference arm on every host core: W untimed calls,
    then K timed calls per worker, each call a bounded sample of the
    workload (the worker's share of the sequences)."""
    from synth import workloads as wl
    w = wl.make(args.workload, BLOCK_SIZE)
    n = os.cpu_count() or 1
    value, secs, units, sample = run_oracle(args.workload, n, calls=args.steps, warmup=args.warmup,
                                            window=args.window)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": secs * 1e3 / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": args.workload, "batch": w.batch, "n_q_heads": w.n_q_heads,
                       "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
                       "kv_dtype": w.kv_dtype, "q_dtype": w.q_dtype, "partition_size": w.partition_size or None,
                       "parallelism": f"{n} host processes",
                       **({"window": args.window} if args.window > 0 else {})},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": n, "kind": "oracle",
                             "sample": sample, **host_cpu()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
