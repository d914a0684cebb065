"""Benchmark: paged decode attention KV GB/s (and decode tokens/s) on GB300.

One step = the whole hot path over one decode batch: the host block manager
reserves one slot per sequence (copy-on-write pairs included), then on the
device the copy-on-write block copy, the slot write of the new token's K/V
in every layer, and per layer the split-K decode pass and its merge.

* ``value``: unique K/V bytes the step's attention must read from HBM per
  second of device time (inputs resident in HBM; host reservations for all
  steps made before timing, per-step metadata uploaded beforehand; each
  step replayed as a CUDA graph; L2 flushed between steps outside the timed
  windows by a 256 MiB write followed by a 256 MiB read).
* ``e2e``: the same metric through the C-ABI call ``kv_decode_step_host``
  with pinned host buffers: host reservation, H2D of q / new K,V / slots /
  pairs / tables / lengths, kernels, D2H of the float32 outputs, synchronise.
* ``roofline``: the split pass (dominant kernel), its algorithmic bytes per
  launch over its CUDA-event duration, against MEASURED_PEAKS.json.
* ``cpu_baseline``: the CPU oracle (fp64, one thread) on a bounded sample of
  the same workload, in a subprocess.

``--impl reference`` times the CPU oracle itself as the reference arm.
Multi-GPU (torchrun): replicas only -- each rank runs its own pool and batch
(weak scaling); the value is the sum over ranks over the max time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "paged decode-attn KV GB/s (% of GB300 HBM peak) and decode tokens/s"
DEFAULT_WORKLOAD = "pool36"

# Per-launch DRAM traffic of the dominant kernel from an ncu capture, keyed by
# (workload, block size, kernel): ncu dram__bytes_read.sum + dram__bytes_write.sum of one
# launch (profiles/), valid only while the sources of that kernel family hash
# to "sha" (kernel_sha(family)).
TRAFFIC = {
    ("qwen_2k", 16, "decode_mma_kernel"): {"bytes": 331453952 + 3647232, "sha": "bbd095098e8316bd"},
    ("shared_8k", 16, "decode_mma_kernel"): {"bytes": 170885888 + 3263744, "sha": "bbd095098e8316bd"},
    ("gqa70b_32k", 16, "decode_tc_kernel"): {"bytes": 1615905024 + 6258432, "sha": "bbd095098e8316bd"},
    ("qwen_2k_fp8", 16, "decode_mma_kernel"): {"bytes": 169168128 + 3468032, "sha": "bbd095098e8316bd"},
    ("qwen_2k_q8", 16, "decode_mma_kernel"): {"bytes": 179549184 + 3918848, "sha": "bbd095098e8316bd"},
    ("gqa70b_32k_fp8", 16, "decode_tc_kernel"): {"bytes": 809733376 + 6476032,
                                                  "sha": "bbd095098e8316bd"},
    # one layer's launch of the 36-layer pool, captured on a one-layer pool of the same recipe
    ("pool36", 16, "decode_mma_kernel"): {"bytes": 3464012544 + 5924864, "sha": "bbd095098e8316bd"},
    ("prefill_4k", 16, "prefill_tc_kernel"): {"bytes": 164881920 + 33188864, "sha": "2d5b25821dda64ad"},
    # the attention launch over the bfloat16 copy of the FP8 pool's blocks
    ("prefill_4k_fp8", 16, "prefill_tc_kernel"): {"bytes": 166232832 + 34139136,
                                                  "sha": "2d5b25821dda64ad"},
}


# KV_OPT_DECODE_PATH values
KERNELS = {"auto": 0, "cuda": 1, "mma": 2, "tc": 3}

KERNEL_SOURCES = {
    "decode": ("decode.cuh", "decode_mma.cuh", "decode_tc.cuh", "tc.cuh", "ptx.cuh", "plan.h",
               "plan.cpp"),
    "prefill": ("prefill_tc.cuh", "prefill.h", "decode.cuh", "tc.cuh", "ptx.cuh"),
}


def kernel_sha(family: str = "decode") -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, "paged_kv_cache_65_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples every 50 ms with arrival times; the
    summary keeps the samples inside the timed window (widened by 0.3 s on
    each side so that a short window still has a sample next to it)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.perf_counter()
            while not self.lines and time.perf_counter() - t0 < 5.0:
                time.sleep(0.02)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def summary(self, t_begin: float, t_end: float):
        """Samples that arrived inside [t_begin - 0.3 s, t_end + 0.3 s]."""
        if self.proc is None:
            return None
        time.sleep(0.35)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in list(self.lines):
            if not (t_begin - 0.3 <= t <= t_end + 0.3):
                continue
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}

    def close(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.proc = None

    def stop(self, t_begin: float, t_end: float):
        out = self.summary(t_begin, t_end)
        self.close()
        return out


# ------------------------------------------------------------ distributed
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist

        backend = "nccl" if os.environ.get("BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend)
    return rank, local, ws


def aggregate(local_bytes: float, local_seconds: float, world: int, device=None):
    """Whole-job bytes and max-over-ranks seconds (barrier included)."""
    if world <= 1:
        return local_bytes, local_seconds
    import torch
    import torch.distributed as dist

    t = torch.tensor([local_bytes, local_seconds], dtype=torch.float64, device=device)
    b = t[:1].clone()
    s = t[1:].clone()
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    dist.all_reduce(s, op=dist.ReduceOp.MAX)
    return float(b.item()), float(s.item())


# -------------------------------------------------------------- workload
def setup(name: str, block_size: int = 16, device="cuda", fill: str = "device",
          placement_seed=None, n_layers=None):
    """Build the workload's pool on the device.  ``fill="device"`` fills the
    whole pool with seeded N(0,1) values generated on the GPU by torch and
    skips history writes (the history values are whatever the pool holds);
    ``fill="host"`` writes the recipe's CPU-generated values slot by slot."""
    import torch

    from paged_kv_cache_65_gb300 import PagedKVCache
    from paged_kv_cache_65_gb300.driver import DeviceRun

    wl = recipe(name, block_size, n_layers)
    if placement_seed is not None:
        import dataclasses

        wl = dataclasses.replace(wl, free_order=synth.permutation((placement_seed, 99),
                                                                   wl.n_blocks))
    cache = PagedKVCache(wl.n_layers, wl.n_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim,
                         wl.dtype, free_order=wl.free_order, device=device)
    fp8 = wl.dtype == "fp8_e4m3"
    if fp8:
        cache.kv_pool_set_fp8_scales(wl.k_scale, wl.v_scale)
    if fill == "device":
        g = torch.Generator(device=device)
        g.manual_seed(synth.torch_seed((wl.seed, 5)))
        for t in (cache.k, cache.v):
            flat = t.view(-1)
            step = 1 << 28
            for i in range(0, flat.numel(), step):
                seg = flat[i:i + step]
                x = torch.randn(seg.numel(), generator=g, device=device, dtype=torch.float32)
                if wl.dtype == "q8_0":  # codes of N(0,1) values at scale 1/32
                    seg.copy_(torch.clamp(torch.round(x * 32), -127, 127).to(torch.int8)
                              .view(torch.uint8))
                    continue
                # FP8 pools: the values' E4M3 codes (torch's conversion; synthetic fill only)
                seg.copy_(x.to(torch.float8_e4m3fn).view(torch.uint8) if fp8 else x)
        if wl.dtype == "q8_0":
            cache.k_sc.fill_(1.0 / 32)
            cache.v_sc.fill_(1.0 / 32)
    run = DeviceRun(cache, wl.n_q_heads)
    values = None if fill == "device" else wl.append_values
    for op in wl.build_ops:
        if op[0] == "append" and values is None:
            slots, pairs = cache.seq_append_tokens(op[1], op[2])
            if len(pairs):
                d = torch.from_numpy(np.ascontiguousarray(pairs)).to(device)
                cache.cow_copy(d, len(pairs))
            run.lengths[op[1]] = run.lengths.get(op[1], 0) + op[2]
        else:
            run.apply(op, values)
    torch.cuda.synchronize()
    return wl, cache, run


def unique_kv_bytes(cache, seq_ids, lengths, esize):
    """Distinct (block, valid rows) the step's attention reads, all layers."""
    B = cache.B
    table, lens = cache.seq_block_table(seq_ids, max(1, max(-(-lengths[s] // B) for s in seq_ids)))
    rows = {}
    for i in range(len(seq_ids)):
        n = int(lens[i])
        for j in range(-(-n // B)):
            r = min(B, n - j * B)
            p = int(table[i, j])
            rows[p] = max(rows.get(p, 0), r)
    per_row = 2 * cache.H * cache.D * esize * cache.L
    return sum(rows.values()) * per_row, int(lens.sum()) * per_row


# ----------------------------------------------------------------- ours
def workload_config(wl, world: int, placement_seed=None) -> dict:
    """The workload a line measures, from its recipe alone (both arms print
    the same dict): shapes, pool, the mean context after the first decode
    step, how L2 is handled and the replica count."""
    lens = synth.recipe_lengths(wl)
    ctx = [lens.get(s, 0) + 1 for s in wl.decode_seqs]
    return {"workload": wl.name, "n_layers": wl.n_layers, "n_seq": len(wl.decode_seqs),
            "block_size": wl.block_size, "H_q": wl.n_q_heads, "H_kv": wl.n_kv_heads,
            "D_h": wl.head_dim, "kv_dtype": wl.dtype, "mean_context": round(float(np.mean(ctx)), 1),
            "n_blocks": wl.n_blocks, "l2": "flushed between steps (256 MiB write + 256 MiB read)",
            "placement_seed": placement_seed, "parallelism": f"replicas x{world}"}


def recipe(name: str, block_size: int = 16, n_layers=None):
    wl = synth.workload(name, **({"block_size": block_size} if name == "pool36" else {}))
    if n_layers is not None and n_layers != wl.n_layers:
        import dataclasses

        wl = dataclasses.replace(wl, n_layers=int(n_layers))
    return wl


def agree_max(x: int, world: int, device=None) -> int:
    """The largest of the ranks' values (every rank times the same count)."""
    if world <= 1:
        return int(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([int(x)], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return int(t.item())


def read_stream_gbs(dev) -> float | None:
    """Read-only HBM stream rate on this GPU: a float32 sum over 4 GiB (a
    reduction reads every byte once and writes nothing), best of 5, CUDA
    events; a roofline denominator beside the copy peak."""
    import torch

    try:
        x = torch.ones(1 << 30, dtype=torch.float32, device=dev)
    except Exception:
        return None
    best = None
    for _ in range(6):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        x.sum()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None else min(best, ms)
    del x
    torch.cuda.empty_cache()
    return round(4.0 * (1 << 30) / (best / 1e3) / 1e9, 1)


def measure_decode(args, name, block_size, steps, dev, world, clocks, min_timed_s=0.0,
                   n_layers=None):
    """One decode workload on this rank's GPU: the step timing (``steps``
    graph replays, or more when ``min_timed_s`` asks for a longer timed
    region), the split pass's roofline, the host-buffer step (e2e) and the
    clock record of the timed window.  Returns the measurement as a dict."""
    import torch

    from paged_kv_cache_65_gb300 import _lib

    wl, cache, run = setup(name, block_size, dev, placement_seed=args.placement_seed,
                           n_layers=n_layers)
    if args.cuda_cores:
        args.kernel = "cuda"
    cache.kv_pool_set_option(_lib.KV_OPT_DECODE_PATH, KERNELS[args.kernel])
    cache.kv_pool_set_option(_lib.KV_OPT_PDL, 0 if args.no_pdl else 1)
    esize = wl.elem_bytes
    seqs = wl.decode_seqs
    n = len(seqs)
    L = wl.n_layers
    stream = torch.cuda.current_stream()
    # host part of the steps first (reservations + tables), then upload; the
    # timed loop cycles over n_plans distinct steps so that contexts grow by
    # at most n_plans tokens however many steps are timed
    n_plans = args.plans if min_timed_s > 0 else min(args.warmup + steps, args.plans)

    use_plan = not (args.plain or args.kernel == "cuda") and \
        wl.dtype in ("bf16", "fp8_e4m3", "q8_0") and \
        wl.block_size % 8 == 0
    plans, host_plans = [], []
    max_blocks = 1
    for i in range(n_plans):
        slots, pairs = run.reserve(seqs)
        table, lens = cache.seq_block_table(seqs, run.max_blocks(seqs))
        ub, lb = unique_kv_bytes(cache, seqs, run.lengths, esize)
        plans.append((slots, pairs, table, lens, ub, lb))
        max_blocks = max(max_blocks, table.shape[1])
        if use_plan:  # the sharing-aware plan of exactly this step's tables
            host_plans.append(cache.paged_decode_plan(seqs, wl.n_q_heads, 1 << 24))
    dplans = []
    ws_bytes = cache.paged_decode_workspace_bytes(n, wl.n_q_heads)
    for i, (slots, pairs, table, lens, ub, lb) in enumerate(plans):
        tpad = np.full((n, max_blocks), -1, dtype=np.int32)
        tpad[:, :table.shape[1]] = table
        d = dict(
            slots=torch.from_numpy(slots).to(dev),
            pairs=torch.from_numpy(np.ascontiguousarray(pairs)).to(dev) if len(pairs) else None,
            npairs=len(pairs), table=torch.from_numpy(tpad).to(dev),
            lens=torch.from_numpy(lens).to(dev), ub=ub, lb=lb, ctx=int(lens.sum()))
        dplans.append(d)
    for d, hp in zip(dplans, host_plans):
        d["h_plan"], d["ws"] = hp
        d["d_plan"] = torch.from_numpy(hp[0]).to(dev)
        ws_bytes = max(ws_bytes, hp[1])
    g = torch.Generator(device=dev)
    g.manual_seed(synth.torch_seed((wl.seed, 6)))
    tdt = torch.float32 if wl.dtype == "f32" else torch.bfloat16  # FP8 pools take bf16
    q = torch.randn((L, n, wl.n_q_heads, wl.head_dim), generator=g, device=dev).to(tdt)
    kn = torch.randn((L, n, wl.n_kv_heads, wl.head_dim), generator=g, device=dev).to(tdt)
    vn = torch.randn((L, n, wl.n_kv_heads, wl.head_dim), generator=g, device=dev).to(tdt)
    out = torch.empty((L, n, wl.n_q_heads, wl.head_dim), dtype=torch.float32, device=dev)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(64 << 20, dtype=torch.float32, device=dev)

    def flush_l2(i):
        # write 256 MiB, then read another 256 MiB: L2 ends up holding only
        # clean lines of the flush buffers, so the timed step neither hits its
        # own data nor pays for write-back of dirty flush lines
        flush.fill_(i & 0xFF)
        flush_r.sum()

    # one CUDA graph per step plan: cow copy, slot write, per layer split + merge
    # (with --fused-write the planned pass writes each layer's new tokens
    # itself); event-record nodes around each split pass time the dominant kernel
    fused = use_plan and args.fused_write

    def enqueue(p, ext=None, split=True, merge=True):
        cnt = 0
        if p["npairs"]:
            cache.cow_copy(p["pairs"], p["npairs"])
            cnt += 1
        if not fused:
            cache.reshape_and_cache(-1, kn, vn, p["slots"], n)
            cnt += 1
        for layer in range(L):
            if ext is not None:
                ext[layer][0].record()
            if fused and split:
                cache.paged_decode_partials_planned_write(layer, q[layer], wl.n_q_heads,
                                                          kn[layer], vn[layer], p["table"],
                                                          max_blocks, p["d_plan"], p["h_plan"],
                                                          ws)
            elif use_plan and split:
                cache.paged_decode_partials_planned(layer, q[layer], wl.n_q_heads, p["table"],
                                                    max_blocks, p["d_plan"], p["h_plan"], ws)
            elif split:
                cache.paged_decode_partials(layer, q[layer], wl.n_q_heads, p["table"], max_blocks,
                                            p["lens"], n, ws, 0.0)
            if ext is not None:
                ext[layer][1].record()
            if use_plan and merge:
                cache.paged_decode_merge_planned(wl.n_q_heads, p["d_plan"], p["h_plan"],
                                                 out[layer], ws)
            elif merge:
                cache.paged_decode_merge(wl.n_q_heads, p["lens"], n, out[layer], ws)
            cnt += int(split) + int(merge)
        return cnt

    for i in range(args.warmup):  # eager: first launches size grids, set attributes
        enqueue(dplans[i % n_plans])
    torch.cuda.synchronize()
    try:
        ext_events = [[[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
                       for _ in range(L)] for _ in range(n_plans)]
    except TypeError:
        ext_events = None
    graphs, instr_graphs, split_graphs, nosplit_graphs, noattn_graphs = [], [], [], [], []
    nomerge_graphs = []
    launches_of = []
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        for pi in range(n_plans):
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_, stream=cap):
                launches_of.append(enqueue(dplans[pi]))
            graphs.append(g_)
            gn = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gn, stream=cap):
                enqueue(dplans[pi], split=False)
            nosplit_graphs.append(gn)
            ga = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ga, stream=cap):
                enqueue(dplans[pi], split=False, merge=False)
            noattn_graphs.append(ga)
            gs = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gs, stream=cap):
                enqueue(dplans[pi], merge=False)
            nomerge_graphs.append(gs)
            gi = torch.cuda.CUDAGraph()
            if ext_events is not None:
                with torch.cuda.graph(gi, stream=cap):
                    enqueue(dplans[pi], ext_events[pi])
                instr_graphs.append(gi)
            else:
                gs = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gs, stream=cap):
                    for layer in range(L):
                        if use_plan:
                            cache.paged_decode_partials_planned(
                                layer, q[layer], wl.n_q_heads, dplans[pi]["table"], max_blocks,
                                dplans[pi]["d_plan"], dplans[pi]["h_plan"], ws)
                        else:
                            cache.paged_decode_partials(layer, q[layer], wl.n_q_heads,
                                                        dplans[pi]["table"], max_blocks,
                                                        dplans[pi]["lens"], n, ws, 0.0)
                split_graphs.append(gs)
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    t_w0 = time.perf_counter()
    for i in range(args.warmup):
        flush_l2(i)
        graphs[i % n_plans].replay()
    torch.cuda.synchronize()
    per_iter_s = (time.perf_counter() - t_w0) / max(1, args.warmup)
    if min_timed_s > 0:  # a timed region of at least min_timed_s of replays
        steps = max(steps, int(np.ceil(min_timed_s / max(per_iter_s, 1e-6))))
    steps = agree_max(steps, world, dev)
    n_steps = args.warmup + steps

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_steps)]
    split_ms = []
    launches = 0
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for i in range(args.warmup, n_steps):
        pi = i % n_plans
        flush_l2(i)  # evict L2 outside the timed windows
        ev[i][0].record(stream)
        graphs[pi].replay()
        ev[i][1].record(stream)
        launches += launches_of[pi]
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    t_wall = t_wall1 - t_wall0
    clk = clocks.summary(t_wall0, t_wall1) if clocks is not None else None
    step_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.warmup, n_steps)]
    # the split pass alone: the same steps replayed from graphs that hold
    # event-record nodes around each split launch (a second timed loop, so
    # that the step timing above keeps the kernels' programmatic edges)
    n_split = min(steps, 200)
    if ext_events is not None:
        split_src = "event-record nodes around each split launch in the step graphs"
        for j in range(n_split):
            pi = j % n_plans
            flush_l2(j)
            instr_graphs[pi].replay()
            torch.cuda.synchronize()
            split_ms.extend(ext_events[pi][l][0].elapsed_time(ext_events[pi][l][1])
                            for l in range(L))
    else:
        split_src = "events around graphs holding only the split launches"
        e0s = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_split)]
        for j in range(n_split):
            flush_l2(j)
            e0s[j][0].record(stream)
            split_graphs[j % n_plans].replay()
            e0s[j][1].record(stream)
        torch.cuda.synchronize()
        split_ms = [a.elapsed_time(b) / L for a, b in e0s]
    # the split passes' device time: the step graphs without the merge
    # launches (each ending with its layer's split pass) against the same
    # graphs with neither, replayed the same way (L2 flushed before each,
    # events around the replay); per launch = the difference of the medians
    # / L.  The merge is left out of both, so its own speed, after the split
    # pass or alone, does not enter the split's figure.
    n_inc = min(steps, 200)
    with_ms, without_ms, noattn_ms, nomerge_ms = [], [], [], []
    for j in range(n_inc):
        for gr_, acc in ((graphs, with_ms), (nosplit_graphs, without_ms),
                         (noattn_graphs, noattn_ms), (nomerge_graphs, nomerge_ms)):
            flush_l2(j)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gr_[j % n_plans].replay()
            e1.record(stream)
            acc.append((e0, e1))
    torch.cuda.synchronize()
    with_ms = [a.elapsed_time(b) for a, b in with_ms]
    without_ms = [a.elapsed_time(b) for a, b in without_ms]
    noattn_ms = [a.elapsed_time(b) for a, b in noattn_ms]
    nomerge_ms = [a.elapsed_time(b) for a, b in nomerge_ms]
    # the step minus the step without the split launches (the merge kept)
    inc_s = (float(np.median(with_ms)) - float(np.median(without_ms))) / L / 1e3
    split_only_s = (float(np.median(nomerge_ms)) - float(np.median(noattn_ms))) / L / 1e3
    # split and merge launches together (the attention of the layer)
    attn_s = (float(np.median(with_ms)) - float(np.median(noattn_ms))) / L / 1e3
    # steps whose plan carries copy-on-write pairs (the first step after a
    # fork) apart from the rest
    cow_ms = [t for i, t in zip(range(args.warmup, n_steps), step_ms)
              if dplans[i % n_plans]["npairs"]]
    steady_ms = [t for i, t in zip(range(args.warmup, n_steps), step_ms)
                 if not dplans[i % n_plans]["npairs"]]
    dev_s = sum(step_ms) / 1e3
    ub = sum(dplans[i % n_plans]["ub"] for i in range(args.warmup, n_steps))
    lb = sum(dplans[i % n_plans]["lb"] for i in range(args.warmup, n_steps))
    tot_b, max_s = aggregate(float(ub), dev_s, world, dev)
    value = tot_b / max_s / 1e9
    ms_per_step = max_s / steps * 1e3
    toks = world * n * steps / max_s

    # roofline of the split pass: algorithmic bytes per launch (2 * H_kv * D_h
    # * b bytes per distinct context token row of the layer) / mean duration
    per_launch_alg = [dplans[j % n_plans]["ub"] / L for j in range(n_split)]
    alg = float(np.mean(per_launch_alg))
    split_ev_s = float(np.mean(split_ms)) / 1e3
    split_s = split_only_s
    peak, peak_kind = read_peaks()
    achieved = alg / split_s / 1e9
    # the split-pass kernel that ran: a plan records its own; otherwise the option
    tensor_shape = wl.dtype in ("bf16", "fp8_e4m3", "q8_0") and wl.block_size % 8 == 0
    if use_plan:
        from paged_kv_cache_65_gb300.cache import parse_plan

        kname = {2: "decode_mma_kernel", 3: "decode_tc_kernel"}[
            parse_plan(host_plans[0][0])["kernel"]]
    elif args.kernel == "cuda" or not tensor_shape:
        kname = "decode_split_kernel"
    elif args.kernel == "tc" and wl.head_dim == 128:
        kname = "decode_tc_kernel"
    else:
        kname = "decode_mma_kernel"
    traffic = TRAFFIC.get((name, wl.block_size, kname))
    traffic_v = traffic["bytes"] if traffic and traffic.get("sha") == kernel_sha() else None

    # e2e through the public C-ABI call with pinned host buffers
    e2e = bench_e2e(args, wl, cache, run, dev, world, min(steps, args.plans))
    res = {
        "config": workload_config(wl, world, args.placement_seed),
        "path": {"decode_path": "planned" if use_plan else "plain",
                 "kernel_option": args.kernel, "kernel": kname, "pdl": not args.no_pdl,
                 "slot_write": "fused into the split pass" if fused else "separate launch"},
        "dtype": wl.dtype,
        "value": round(value, 2), "unit": "GB/s", "steps": steps,
        "ms_per_step": round(ms_per_step, 4),
        "step_us_median_p10_p90": [round(1e3 * float(np.percentile(step_ms, p)), 2)
                                   for p in (50, 10, 90)],
        "pct_of_hbm_peak": round(100 * value / peak, 2),
        "pct_of_8tbs_nominal": round(100 * value / 8000.0, 2),
        "logical_kv_gbs": round(lb / dev_s / 1e9, 2),
        "decode_tokens_per_s": round(toks, 1),
        "decode_tokens_per_s_36_layers": round(toks * L / 36.0, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic_v,
                     "kernel": kname,
                     "peak_source": peak_kind,
                     "timing": ("device time of the split launches: median of the step "
                                "graphs without the merge launches minus median of the "
                                "same graphs without split or merge, per launch (CUDA "
                                "events around each replay, L2 flushed before each)"),
                     "alg_bytes_per_launch": int(alg),
                     "mean_launch_us": round(split_s * 1e6, 2),
                     "event_node_launch_us": round(split_ev_s * 1e6, 2),
                     "step_minus_nosplit_us": round(inc_s * 1e6, 2),
                     "split_and_merge_us": round(attn_s * 1e6, 2),
                     "split_and_merge_frac": round(alg / attn_s / 1e9 / peak, 4),
                     "event_node_timing": split_src},
        "gpu_launches": launches,
        "graphs": "one CUDA graph per step plan, replayed",
        "cow_steps": ({"n": len(cow_ms), "step_ms": round(float(np.mean(cow_ms)), 4),
                       "steady_step_ms": round(float(np.mean(steady_ms)), 4)}
                      if cow_ms and steady_ms else None),
        "e2e": e2e,
        "clocks": clk,
        "wall_s_timed": round(t_wall, 4),
    }
    del graphs, instr_graphs, split_graphs, nosplit_graphs, noattn_graphs, nomerge_graphs
    cache.close()
    return res


# the target configs and config 1, then the same steps over FP8 pools (the
# warp-level pass on qwen_2k_fp8, the tcgen05 pass on gqa70b_32k_fp8)
PER_CONFIG = ("shared_8k", "gqa70b_32k", "qwen_2k", "qwen_2k_fp8", "gqa70b_32k_fp8")


def free_device():
    import gc

    import torch

    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def bench_ours(args):
    import torch

    rank, local, world = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    clocks = ClockSampler(torch.cuda.current_device() if world == 1 else local)
    clocks.start()
    stream_gbs = read_stream_gbs(dev)
    head = measure_decode(args, args.workload, args.block_size, args.steps, dev, world, clocks,
                          n_layers=args.layers)
    per = {}
    if args.per_config:
        for w in PER_CONFIG:
            if w == args.workload:
                continue
            free_device()
            per[w] = measure_decode(args, w, 16, args.steps, dev, world, clocks,
                                    min_timed_s=args.min_timed_s)
    clocks.close()
    free_device()
    cpu = cpu_par = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, args.cpu_seconds)
        cpu_par = cpu_baseline_parallel(args.workload, args.cpu_seconds)
        for w in per:
            per[w]["cpu_baseline"] = cpu_baseline(w, args.per_config_cpu_seconds)

    if rank == 0:
        peak, peak_kind = read_peaks()
        line = {
            "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": head["dtype"], "data": "synthetic (seeded N(0,1) K/V/q; torch device generator)",
            "config": head["config"],
        }
        line.update({k: v for k, v in head.items() if k not in line and k != "steps"})
        line["peaks"] = {"measured_copy_gbs": peak, "measured_copy_source": peak_kind,
                         "read_stream_gbs": stream_gbs,
                         "read_stream_how": "float32 sum over 4 GiB on this GPU, best of 5",
                         "nominal_gbs": 8000.0}
        for res in [line] + list(per.values()):
            rf = res["roofline"]
            rf["frac_of_nominal"] = round(rf["achieved"] / 8000.0, 4)
            if stream_gbs:
                rf["frac_of_read_stream"] = round(rf["achieved"] / stream_gbs, 4)
        if cpu is not None:
            line["cpu_baseline"] = cpu
            line["cpu_baseline_parallel"] = cpu_par
        if per:
            line["per_config"] = per
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()


def bench_e2e(args, wl, cache, run, dev, world, steps):
    import torch

    seqs = wl.decode_seqs
    n = len(seqs)
    L = wl.n_layers
    # each e2e step advances the host state by one token per sequence
    steps = max(1, steps)
    max_blocks = run.max_blocks(seqs) + (steps + args.warmup) // wl.block_size + 2
    staging = torch.empty(cache.kv_decode_step_staging_bytes(n, wl.n_q_heads, max_blocks),
                          dtype=torch.uint8, device=dev)
    tdt = torch.float32 if wl.dtype == "f32" else torch.bfloat16  # FP8 pools take bf16
    g = torch.Generator()
    g.manual_seed(synth.torch_seed((wl.seed, 7)))
    hq = torch.randn((L, n, wl.n_q_heads, wl.head_dim), generator=g).to(tdt).pin_memory()
    hk = torch.randn((L, n, wl.n_kv_heads, wl.head_dim), generator=g).to(tdt).pin_memory()
    hv = torch.randn((L, n, wl.n_kv_heads, wl.head_dim), generator=g).to(tdt).pin_memory()
    ho = torch.empty((L, n, wl.n_q_heads, wl.head_dim), dtype=torch.float32).pin_memory()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(64 << 20, dtype=torch.float32, device=dev)
    esize = wl.elem_bytes
    seq_arr = np.asarray(seqs, dtype=np.int32)  # the caller's id array, built once
    total_s, total_b = 0.0, 0
    h2d = d2h = 0
    for i in range(args.warmup + steps):
        flush.fill_(i & 0xFF)
        flush_r.sum()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        cache.kv_decode_step_host(seq_arr, wl.n_q_heads, max_blocks, hq, hk, hv, ho, staging)
        dt = time.perf_counter() - t0
        for s in seqs:
            run.lengths[s] += 1
        if i >= args.warmup:
            total_s += dt
            ub, _ = unique_kv_bytes(cache, seqs, run.lengths, esize)
            total_b += ub
    # q and the new rows as the caller holds them (bf16 for code pools)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv)) + n * 8 + n * 8 + \
        n * max_blocks * 4 + n * 4
    d2h = ho.numel() * 4
    tot_b, max_s = aggregate(float(total_b), total_s, world, dev)
    return {"value": round(tot_b / max_s / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(max_s / steps * 1e3, 4), "api": "kv_decode_step_host"}


# ------------------------------------------------------ chunked prefill
PREFILL_METRIC = ("chunked-prefill attention TFLOP/s (% of GB300 bf16 tensor peak) and "
                  "prefill tokens/s")


def read_tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s) for a kernel timed alone."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def prefill_flops(wl) -> float:
    """Algorithmic flops of a round: per admitted (query, key) pair and query
    head, 2 D for the score and 2 D for the weighted value; a chunk of c
    tokens after h admits c h + c (c + 1) / 2 pairs ("第 8 章 推理优化"
    §8.2.3)."""
    pairs = 0
    for seq, c in wl.chunks:
        h = wl.history[seq]
        pairs += c * h + c * (c + 1) // 2
    return 4.0 * wl.head_dim * wl.n_q_heads * pairs


def bench_prefill(args):
    """Time chunked-prefill rounds: each step rewrites the chunks' K/V into
    their slots (reserved once, before timing) and runs the prefill
    attention of every chunk over its paged context, replayed as one CUDA
    graph with L2 flushed between steps."""
    import torch

    rank, local, world = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl, cache, run = setup(args.workload, device=dev, placement_seed=args.placement_seed)
    cache.kv_pool_set_option(_lib_mod().KV_OPT_PDL, 0 if args.no_pdl else 1)
    wl.history = {s: run.lengths.get(s, 0) for s, _ in wl.chunks}
    seqs = [s for s, _ in wl.chunks]
    slot_list = []
    for seq, c in wl.chunks:
        slots, pairs = cache.seq_append_tokens(seq, c)
        assert len(pairs) == 0
        run.lengths[seq] = run.lengths.get(seq, 0) + c
        slot_list.append(slots)
    n_tok = sum(c for _, c in wl.chunks)
    d_slots = torch.from_numpy(np.concatenate(slot_list)).to(dev)
    d_table, d_lens, mb = run.tables(seqs)
    starts = np.zeros(len(seqs) + 1, dtype=np.int32)
    starts[1:] = np.cumsum([c for _, c in wl.chunks])
    d_starts = torch.from_numpy(starts).to(dev)
    max_chunk = max(c for _, c in wl.chunks)
    # heaviest-first work order from the host's copy of the chunk geometry
    sched = cache.paged_prefill_schedule(starts, d_lens.cpu().numpy(), wl.n_q_heads)
    d_sched = torch.from_numpy(sched).to(dev)
    natural = args.prefill_order == "natural"
    g = torch.Generator(device=dev)
    g.manual_seed(synth.torch_seed((wl.seed, 8)))
    q = torch.randn((n_tok, wl.n_q_heads, wl.head_dim), generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn((wl.n_layers, n_tok, wl.n_kv_heads, wl.head_dim), generator=g,
                    device=dev).to(torch.bfloat16)
    v = torch.randn_like(k)
    out = torch.empty((n_tok, wl.n_q_heads, wl.head_dim), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    # an FP8 pool goes through a bfloat16 copy of the blocks read (the staged
    # call: a conversion launch before each layer's attention)
    fp8 = wl.dtype == "fp8_e4m3"
    ws = (torch.empty(cache.paged_prefill_staging_bytes(len(seqs), mb), dtype=torch.uint8,
                      device=dev) if fp8 else None)

    def attend(s):
        for layer in range(wl.n_layers):
            if fp8:
                cache.paged_prefill_attention_staged(
                    layer, q, wl.n_q_heads, d_table, mb, d_starts, d_lens, len(seqs), out, ws,
                    max_chunk=max_chunk if natural else 0, d_sched=None if natural else d_sched,
                    n_items=0 if natural else len(sched), stream=s.cuda_stream)
            elif natural:
                cache.paged_prefill_attention(layer, q, wl.n_q_heads, d_table, mb, d_starts,
                                              d_lens, len(seqs), max_chunk, out, 0.0,
                                              s.cuda_stream)
            else:
                cache.paged_prefill_attention_scheduled(layer, q, wl.n_q_heads, d_table, mb,
                                                        d_starts, d_lens, len(seqs), d_sched,
                                                        len(sched), out, 0.0, s.cuda_stream)

    def step(s):
        cache.reshape_and_cache(-1, k, v, d_slots, n_tok, s.cuda_stream)
        attend(s)

    graphs = {}
    for name, fn in (("step", step), ("attn", attend)):
        with torch.cuda.stream(stream):
            fn(stream)  # warm (module load, attributes)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            fn(stream)
        graphs[name] = gr
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(64 << 20, dtype=torch.float32, device=dev)
    clk = ClockSampler(local)
    clk.start()

    def timed(gr, n):
        evs = []
        with torch.cuda.stream(stream):
            for i in range(n):
                flush.fill_(i & 0xFF)
                flush_r.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                gr.replay()
                e1.record(stream)
                evs.append((e0, e1))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    timed(graphs["step"], args.warmup)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    step_ms = timed(graphs["step"], args.steps)
    t1 = time.perf_counter()
    attn_ms = timed(graphs["attn"], min(args.steps, 200))
    clocks = clk.stop(t0, t1)
    assert cache.kv_pool_device_status() == 0
    flops = prefill_flops(wl) * wl.n_layers
    ms = float(np.mean(step_ms))
    tot_f, max_s = aggregate(flops * args.steps, ms * args.steps / 1e3, world, dev)
    value = tot_f / max_s / 1e12
    attn_s = float(np.mean(attn_ms)) / 1e3
    peak, peak_kind = read_tensor_peak()
    achieved = flops / attn_s / 1e12
    traffic = TRAFFIC.get((args.workload, wl.block_size, "prefill_tc_kernel"))
    traffic_v = traffic["bytes"] if traffic and traffic.get("sha") == kernel_sha("prefill") else None
    e2e = bench_prefill_e2e(args, wl, cache, dev, q, k, v, d_slots, d_table, d_lens, mb, d_starts,
                            starts, max_chunk, n_tok, flops, world, ws)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, args.cpu_seconds)
        cpu_par = cpu_baseline_parallel(args.workload, args.cpu_seconds)
    if rank == 0:
        line = {
            "metric": PREFILL_METRIC, "value": round(value, 2), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic (seeded N(0,1) pool, q and chunk K/V; torch device generator)",
            "config": {"workload": args.workload, "n_layers": wl.n_layers,
                       "chunks": [c for _, c in wl.chunks],
                       "histories": [wl.history[s] for s in seqs], "kernel": "prefill_tc_kernel",
                       "kv_dtype": wl.dtype,
                       "staging": ("prefill_stage_fp8_kernel: the blocks read, as exact "
                                   "bfloat16, before each layer's attention" if fp8 else None),
                       "pdl": not args.no_pdl, "block_size": wl.block_size,
                       "work_order": ("natural grid" if natural else
                                      "heaviest first (host schedule, paged_prefill_schedule)"),
                       "H_q": wl.n_q_heads, "H_kv": wl.n_kv_heads, "D_h": wl.head_dim,
                       "l2": "flushed between steps (256 MiB write + 256 MiB read)",
                       "placement_seed": args.placement_seed,
                       "parallelism": f"replicas x{world}"},
            "pct_of_tensor_peak": round(100 * value / peak, 2),
            "prefill_tokens_per_s": round(n_tok * world / (ms / 1e3), 1),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                         "traffic": traffic_v, "kernel": "prefill_tc_kernel",
                         "peak_source": peak_kind,
                         "timing": ("CUDA events around a graph holding the attention launches"
                                    + (" (each layer's conversion launch included)"
                                       if fp8 else "")),
                         "alg_flops_per_launch": int(flops / wl.n_layers),
                         "mean_launch_us": round(attn_s * 1e6 / wl.n_layers, 2),
                         "note": "the weights go through the tensor core twice (bf16 high part "
                                 "and remainder), so the P.V half of the flops runs twice"},
            "gpu_launches": 1 + wl.n_layers * (2 if fp8 else 1),
            "graphs": "one CUDA graph per step, replayed",
            "e2e": e2e, "clocks": clocks,
            "wall_s_timed": round(t1 - t0, 4),
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
            line["cpu_baseline_parallel"] = cpu_par
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def bench_prefill_e2e(args, wl, cache, dev, q, k, v, d_slots, d_table, d_lens, mb, d_starts,
                      starts, max_chunk, n_tok, flops, world, ws=None):
    """The same round through the public calls with page-locked host buffers:
    host -> device copies of q and the chunks' K/V, the host work order and
    its copy (unless the natural grid is asked for), the slot write and the
    attention, the device -> host copy of the outputs, and a synchronise."""
    import torch

    natural = args.prefill_order == "natural"
    h_lens = d_lens.cpu().numpy()
    d_sched = torch.empty((cache.paged_prefill_schedule_bytes_for(starts, wl.n_q_heads) // 16, 4),
                          dtype=torch.int32, device=dev)
    h_sched = torch.empty(d_sched.shape, dtype=torch.int32).pin_memory()

    hq, hk, hv = q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()
    ho = torch.empty((n_tok, wl.n_q_heads, wl.head_dim), dtype=torch.float32).pin_memory()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dout = torch.empty((n_tok, wl.n_q_heads, wl.head_dim), dtype=torch.float32, device=dev)
    n = max(1, min(args.steps, 50))
    total = 0.0
    for i in range(args.warmup + n):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        if not natural:
            sc = cache.paged_prefill_schedule(starts, h_lens, wl.n_q_heads)
            h_sched[: len(sc)].numpy()[:] = sc
            d_sched[: len(sc)].copy_(h_sched[: len(sc)], non_blocking=True)
        cache.reshape_and_cache(-1, dk, dv, d_slots, n_tok)
        for layer in range(wl.n_layers):
            if ws is not None:
                cache.paged_prefill_attention_staged(
                    layer, dq, wl.n_q_heads, d_table, mb, d_starts, d_lens, len(wl.chunks), dout,
                    ws, max_chunk=max_chunk if natural else 0,
                    d_sched=None if natural else d_sched, n_items=0 if natural else len(sc))
            elif natural:
                cache.paged_prefill_attention(layer, dq, wl.n_q_heads, d_table, mb, d_starts,
                                              d_lens, len(wl.chunks), max_chunk, dout)
            else:
                cache.paged_prefill_attention_scheduled(layer, dq, wl.n_q_heads, d_table, mb,
                                                        d_starts, d_lens, len(wl.chunks), d_sched,
                                                        len(sc), dout)
        ho.copy_(dout, non_blocking=True)
        torch.cuda.synchronize()
        if i >= args.warmup:
            total += time.perf_counter() - t0
    tot_f, max_s = aggregate(flops * n, total, world, dev)
    h2d = (hq.numel() + hk.numel() + hv.numel()) * 2 + (0 if natural else len(sc) * 16)
    return {"value": round(tot_f / max_s / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(ho.numel() * 4),
            "ms_per_step": round(max_s / n * 1e3, 4),
            "api": ("reshape_and_cache + paged_prefill_attention"
                    + ("_staged" if ws is not None else "") if natural else
                    "paged_prefill_schedule + reshape_and_cache + "
                    + ("paged_prefill_attention_staged" if ws is not None
                       else "paged_prefill_attention_scheduled"))}


def _lib_mod():
    from paged_kv_cache_65_gb300 import _lib

    return _lib


# ------------------------------------------------------------- CPU oracle
# Workloads whose whole oracle pool is too large (36 layers of 167 GB) or too
# slow to build for a CPU leg of seconds: the leg runs on some of their
# sequences (with the prefixes they share) and, for pool36, on one layer.
CPU_SAMPLE = {"pool36": (list(range(0, 128, 16)), 1), "gqa70b_32k": (list(range(8)), None)}


def cpu_recipe(workload: str):
    wl = synth.workload(workload)
    if workload in CPU_SAMPLE:
        seqs, n_layers = CPU_SAMPLE[workload]
        wl = synth.restrict(wl, seqs, n_layers)
    return wl


def cpu_subset_note(workload: str) -> str:
    if workload not in CPU_SAMPLE:
        return ""
    full = synth.workload(workload)
    seqs, n_layers = CPU_SAMPLE[workload]
    return (f" (sequences {seqs} of the batch's {len(full.decode_seqs)}, with the prefixes "
            f"they share{', one layer' if n_layers else ''})")


def oracle_sample(workload: str):
    """Build the oracle's pool for the workload and make one decode step's
    host reservation and writes (setup, untimed)."""
    from oracle.runner import OracleRun

    wl = cpu_recipe(workload)
    orc = OracleRun(wl)
    slots, cows = orc.reserve_step()
    q = orc.write_step(0, slots, cows)
    return wl, orc, q


def oracle_attend(wl, orc, q, seconds: float, max_seqs: int | None = None, start: int = 0):
    """The oracle as it stands: layer-0 attention sequence by sequence until
    ``seconds`` have passed.  Returns (bytes of K/V read, seconds, count)."""
    per_tok = 2 * wl.n_kv_heads * wl.head_dim * wl.elem_bytes
    done, nbytes = 0, 0
    n = len(wl.decode_seqs)
    t0 = time.perf_counter()
    while True:
        i = (start + done) % n
        orc.attend(0, q, seq_index=[i])
        done += 1
        nbytes += orc.bm.lengths[wl.decode_seqs[i]] * per_tok
        if time.perf_counter() - t0 > seconds or (max_seqs and done >= max_seqs):
            break
    return nbytes, time.perf_counter() - t0, done


def prefill_oracle_leg(workload: str, seconds: float, start: int = 0):
    """The oracle's chunked-prefill attention as it stands on whole chunks of
    the round, one after the other (from chunk ``start``), until ``seconds``
    have passed."""
    from oracle.runner import OracleRun

    wl = synth.workload(workload)
    orc = OracleRun(wl)
    hist = {s: orc.bm.lengths.get(s, 0) for s, _ in wl.chunks}
    _, _, q = orc.prefill_step(0)
    flops, done = 0.0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds or done == 0:
        i = (start + done) % len(wl.chunks)
        orc.prefill_attend(0, q, [i])
        seq, c = wl.chunks[i]
        flops += 4.0 * wl.head_dim * wl.n_q_heads * (c * hist[seq] + c * (c + 1) // 2)
        done += 1
    dt = time.perf_counter() - t0
    return flops, dt, done


def cpu_leg(workload: str, seconds: float, start: int = 0):
    if isinstance(synth.workload(workload), synth.PrefillWorkload):
        flops, dt, done = prefill_oracle_leg(workload, seconds, start)
        return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
                "kind": "oracle", "seconds": round(dt, 3), "chunks": done, "flops": flops,
                "sample": f"{workload}: {done} whole chunks of the round, cycling over its "
                          f"{len(synth.workload(workload).chunks)} chunks (fp64 masked "
                          f"softmax over the paged context, one thread), {dt:.1f} s"}
    wl, orc, q = oracle_sample(workload)
    nbytes, dt, done = oracle_attend(wl, orc, q, seconds, start=start)
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{workload}: {done} single-sequence layer-0 decode attentions, cycling "
                      f"over {len(wl.decode_seqs)} sequences{cpu_subset_note(workload)} (paged "
                      f"gather + fp64 softmax, one thread), {dt:.1f} s",
            "seconds": round(dt, 3), "sequences": done, "bytes": int(nbytes)}


def cpu_baseline(workload: str, seconds: float):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-leg", workload,
                        "--cpu-seconds", str(seconds)], capture_output=True, text=True, env=env,
                       timeout=600)
    for ln in r.stdout.splitlines()[::-1]:
        if ln.startswith("{"):
            return json.loads(ln)
    return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "failed: " + r.stderr[-200:]}


def cpu_baseline_parallel(workload: str, seconds: float):
    """The same oracle leg in one single-threaded process per host core, all
    at once, each starting at a different sequence (or chunk) of the batch:
    the work they finish together over the longest one's time."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    wl = cpu_recipe(workload)
    n = len(wl.chunks) if isinstance(wl, synth.PrefillWorkload) else len(wl.decode_seqs)
    P = max(1, os.cpu_count() or 1)
    procs = [subprocess.Popen([sys.executable, os.path.abspath(__file__), "--cpu-leg", workload,
                               "--cpu-seconds", str(seconds), "--cpu-start", str(k * n // P)],
                              stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True,
                              env=env) for k in range(P)]
    legs = []
    for pr in procs:
        out, _ = pr.communicate(timeout=900)
        for ln in out.splitlines()[::-1]:
            if ln.startswith("{"):
                legs.append(json.loads(ln))
                break
    if len(legs) != P:
        return {"value": None, "kind": "oracle", "cores": P, "sample": "failed"}
    dt = max(x["seconds"] for x in legs)
    if "flops" in legs[0]:
        value, unit = round(sum(x["flops"] for x in legs) / dt / 1e12, 6), "TFLOP/s"
        done = sum(x["chunks"] for x in legs)
        what = f"{done} whole chunks"
    else:
        value, unit = round(sum(x["bytes"] for x in legs) / dt / 1e9, 4), "GB/s"
        done = sum(x["sequences"] for x in legs)
        what = f"{done} single-sequence layer-0 decode attentions"
    return {"value": value, "unit": unit, "cores": P, "kind": "oracle",
            "sample": f"{workload}{cpu_subset_note(workload)}: {P} single-threaded oracle "
                      f"processes at once, {what} in all, {dt:.1f} s", "seconds": round(dt, 3)}


def bench_reference(args):
    """The reference arm: the CPU oracle as it stands, each step a bounded
    sample (two sequences' layer-0 attention) of the same workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(k, "1")
    wl, orc, q = oracle_sample(args.workload)
    secs, nbytes = [], []
    for i in range(args.warmup + args.steps):
        b, dt, _ = oracle_attend(wl, orc, q, 1e9, max_seqs=2, start=2 * i)
        if i >= args.warmup:
            secs.append(dt)
            nbytes.append(b)
    value = round(sum(nbytes) / sum(secs) / 1e9, 4)
    sample = (f"{args.workload}: per step, layer-0 decode attention of 2 of "
              f"{len(wl.decode_seqs)} sequences{cpu_subset_note(args.workload)} (paged gather "
              f"+ fp64 softmax, one thread)")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    config = workload_config(recipe(args.workload, args.block_size, args.layers), world,
                             args.placement_seed)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * float(np.mean(secs)), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": config,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def bench_prefill_reference(args):
    """Reference arm of a prefill round: the CPU oracle as it stands, each
    step one whole chunk of the round."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(k, "1")
    flops_all, secs = 0.0, 0.0
    for i in range(args.warmup + args.steps):
        f, dt, _ = prefill_oracle_leg(args.workload, 0.0)
        if i >= args.warmup:
            flops_all += f
            secs += dt
    value = round(flops_all / secs / 1e12, 6)
    sample = f"{args.workload}: per step, one whole chunk of the round (fp64, one thread)"
    print(json.dumps({
        "impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": {"workload": args.workload},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


# ------------------------------------------------------- prefix cache (host)
def bench_prefix(args):
    """Host path of the prefix cache through the C ABI: a 4096-token system
    prompt (256 blocks of 16) is cached, then each request matches it, appends
    32 new tokens and releases ("KV 缓存管理", radix-tree section: the host
    resolves the block table of a hit in well under 50 us)."""
    from paged_kv_cache_65_gb300 import PagedKVCache

    B, S, NEW, N = 16, 4096, 32, 4096
    rng = np.random.default_rng(synth.torch_seed((11, 1)) & 0xFFFFFFFF)
    sysp = [int(x) for x in rng.integers(0, 151936, S)]
    c = PagedKVCache(1, N, B, 8, 128, "bf16", allocate=False)
    c.kv_prefix_cache_enable(0x5A17)
    c.seq_match_prefix(0, sysp)
    c.seq_append_tokens(0, S, sysp)
    c.seq_release(0)  # the prompt's 256 blocks stay cached, dormant
    n = args.warmup + min(args.steps, 2000)
    t_match, t_req = [], []
    # the requests' token arrays are built before timing
    reqs = [np.ascontiguousarray(np.concatenate([np.asarray(sysp, dtype=np.int32),
                                                 rng.integers(0, 151936, NEW).astype(np.int32)]))
            for _ in range(n)]
    for i in range(n):
        toks = reqs[i]
        sid = 1 + i
        t0 = time.perf_counter()
        m = c.seq_match_prefix(sid, toks)
        t1 = time.perf_counter()
        c.seq_append_tokens(sid, len(toks) - m, toks[m:])
        c.seq_release(sid)
        t2 = time.perf_counter()
        assert m == S
        if i >= args.warmup:
            t_match.append(t1 - t0)
            t_req.append(t2 - t0)
    us_match = float(np.mean(t_match)) * 1e6
    us_req = float(np.mean(t_req)) * 1e6
    # the oracle's match on the same prompt, timed on the same host core
    cpu = None
    if not args.no_cpu_baseline:
        from oracle.prefix_cache import PrefixCachingBlockManager

        o = PrefixCachingBlockManager(N, B, salt=0x5A17)
        o.match_prefix(0, sysp)
        o.append_tokens(0, S, sysp)
        o.release(0)
        ts = []
        for i in range(50):
            toks = sysp + [1 + i] * NEW
            t0 = time.perf_counter()
            o.match_prefix(1 + i, toks)
            ts.append(time.perf_counter() - t0)
            o.release(1 + i)
        cpu = {"value": round(1.0 / float(np.mean(ts)), 1), "unit": "match/s", "cores": 1,
               "kind": "oracle", "sample": "50 matches of the same 4096-token prompt"}
    line = {
        "metric": "prefix-cache hit of a 4096-token prompt on the host (match/s, us per match)",
        "value": round(1e6 / us_match, 1), "unit": "match/s", "n_gpus": 0,
        "steps": len(t_match), "warmup": args.warmup, "ms_per_step": round(us_req / 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic token ids (seeded)",
        "config": {"workload": "prefix_4k", "block_size": B, "prompt_tokens": S,
                   "new_tokens": NEW, "blocks": N, "path": "C ABI through ctypes"},
        "us_per_match": round(us_match, 2), "us_per_request": round(us_req, 2),
        "roofline": None, "cpu_baseline": cpu,
        "e2e": {"value": round(1e6 / us_req, 1), "unit": "request/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--plans", type=int, default=32,
                    help="distinct decode steps the timed loop cycles over")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--block-size", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", default="auto", choices=sorted(KERNELS),
                    help="split-pass kernel: automatic, CUDA cores, warp-level MMA, tcgen05")
    ap.add_argument("--cuda-cores", action="store_true",
                    help="decode on CUDA cores even where the tensor-core pass applies")
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch without programmatic dependencies between kernels")
    ap.add_argument("--plain", action="store_true",
                    help="no sharing-aware plan: one segment per (sequence, K/V head)")
    ap.add_argument("--fused-write", action="store_true",
                    help="planned steps: the slot write inside each layer's split pass "
                         "(paged_decode_partials_planned_write) instead of its own launch")
    ap.add_argument("--prefill-order", default="heaviest", choices=["heaviest", "natural"],
                    help="chunked prefill: launch the work items heaviest first (host "
                         "schedule) or in the natural grid order")
    ap.add_argument("--prefix-cache", action="store_true",
                    help="host prefix-cache hit of a 4096-token prompt instead of a GPU step")
    ap.add_argument("--layers", type=int, default=None,
                    help="override the workload's layer count (pool36: a one-layer pool for "
                         "ncu captures of the same per-layer launch)")
    ap.add_argument("--per-config", dest="per_config", action="store_true", default=None,
                    help="also measure " + ", ".join(PER_CONFIG) + " (default with the "
                         "default workload)")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false")
    ap.add_argument("--min-timed-s", type=float, default=0.5,
                    help="per-config workloads: replay at least this long in the timed loop")
    ap.add_argument("--per-config-cpu-seconds", type=float, default=8.0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-leg", default=None)
    ap.add_argument("--cpu-start", type=int, default=0)
    ap.add_argument("--placement-seed", type=int, default=None,
                    help="re-randomise the physical placement of the pool's blocks (the "
                         "free-list order) with this seed; contents and lengths unchanged")
    args = ap.parse_args()
    if args.cpu_leg:
        print(json.dumps(cpu_leg(args.cpu_leg, args.cpu_seconds, args.cpu_start)), flush=True)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.per_config is None:
        args.per_config = args.workload == DEFAULT_WORKLOAD and args.layers is None
    if args.prefix_cache:
        bench_prefix(args)
        return
    prefill = isinstance(synth.workload(args.workload), synth.PrefillWorkload)
    if args.impl == "reference":
        (bench_prefill_reference if prefill else bench_reference)(args)
    elif prefill:
        bench_prefill(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
