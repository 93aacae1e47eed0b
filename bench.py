"""Throughput of the paged KV-cache hot path on GB300.

One step = one pass of the whole path over one synthetic batch already resident
in HBM: copy-on-write block copies (when the workload forks), the K/V append
scatter, paged-attention decode (partitions + log-sum-exp reduce) and, for the
mixed workload, the chunked-prefill attention.  The default workload is the
Llama-3-8B-shaped decode layer (64 sequences, 32 q / 8 kv heads, d 128,
context U[512, 4096], bf16).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference]

N > 1 runs one rank per GPU under torch.distributed.run (started by this
script itself when no launcher did): each rank serves its own independent
batch of the same shape (sequences shard with no exchange), the timed region
is bracketed by barriers and the slowest rank's time is used.  Rank 0 prints
one JSON line.  ``--impl reference`` times the fp64 host oracle
on the same workload instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_297_gb300 import accounting  # noqa: E402
from paged_kv_cache_297_gb300 import workloads as W  # noqa: E402

METRIC = ("paged decode KV-read GB/s & fraction of HBM peak; sequence-steps/sec at 1 GB300")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------------------
# distributed plumbing
# ----------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device: str = "cpu") -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# measurement helpers
# ----------------------------------------------------------------------------

def kernel_source_hash(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_cache_297_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, files):
    """DRAM bytes per call from the committed ncu summary, only while the
    kernel's sources still hash to what was profiled (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel, {}).get(workload)
    if not rec or rec.get("source_sha") != kernel_source_hash(files):
        return None
    return rec.get("dram_bytes_per_call")


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[4], parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        mhz = sorted(r[0] for r in rows)
        loaded = [r for r in rows if r[0] >= 0.5 * max(mhz)] or rows
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in loaded:
            for name, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        lm = sorted(r[0] for r in loaded)
        return {"sm_mhz": lm[len(lm) // 2], "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

class Step:
    """Device-resident inputs and the calls of one step of the hot path."""

    def __init__(self, batch: W.Batch, dev: str, partition: int = 0, unfused: bool = False,
                 no_cascade: bool = False):
        import paged_kv_cache_297_gb300 as pkv
        self.pkv = pkv
        self.b = batch
        self.dev = dev
        t = {}
        for name in ("k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "q", "block_tables",
                     "context_lens", "copy_pairs", "prefill_q", "prefill_cu_q_lens",
                     "prefill_block_tables", "prefill_context_lens"):
            x = getattr(batch, name)
            t[name] = None if x is None else x.to(dev)
        self.t = t
        S, Hq, d = batch.q.shape
        self.out = torch.empty((S, Hq, d), dtype=batch.dtype, device=dev)
        self.max_ctx = max(1, batch.max_context_len)
        self.partition = partition
        # the partition the library uses (decides whether the reduce launches)
        self.part_used = pkv.decode_partition_size(S, batch.spec.num_kv_heads, self.max_ctx, partition)
        if batch.k_scale is not None:  # the fp8 kernel's own adaptive choice
            self.part_used = pkv.decode_partition_size_fp8(S, Hq, batch.spec.num_kv_heads, self.max_ctx, partition)
        ws = pkv.decode_workspace_bytes(S, Hq, d, self.max_ctx, partition)
        self.ws = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
        self.pout = None
        if batch.prefill_q is not None:
            self.pout = torch.empty(batch.prefill_q.shape, dtype=batch.dtype, device=dev)
            cu = batch.prefill_cu_q_lens
            self.max_q = int((cu[1:] - cu[:-1]).max())
            self.max_pctx = int(batch.prefill_context_lens.max())
        self.has_copy = batch.copy_pairs is not None and batch.copy_pairs.numel() > 0
        # decode-only steps whose new tokens are exactly one per sequence at
        # position L-1 take the fused append + decode call
        self.fused = (not unfused) and batch.prefill_q is None and self._one_token_per_seq()
        # a batch over one shared prefix takes the cascade: the prefix once for
        # all queries on the tensor cores, then each sequence's own tokens
        self.prefix_len = 16 * int(batch.meta.get("prefix_blocks", 0))
        # fp8 E4M3 caches: the quantising append, then the fp8 decode
        self.fp8 = batch.k_scale is not None
        if self.fp8:
            t["k_scale"], t["v_scale"] = batch.k_scale.to(dev), batch.v_scale.to(dev)
        self.cascade = (self.fused and not self.fp8 and not no_cascade and self.prefix_len > 0
                        and batch.dtype == torch.bfloat16 and d == 128)
        if self.cascade:
            ws = pkv.decode_shared_prefix_workspace_bytes(S, Hq, d, self.max_ctx, self.prefix_len, partition)
            self.ws = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)

    def _one_token_per_seq(self) -> bool:
        b = self.b
        L = b.context_lens.long()
        if b.slot_mapping.numel() != L.numel() or bool((L <= 0).any()):
            return False
        pos = L - 1
        blk = b.block_tables.long().gather(1, (pos // 16).unsqueeze(1)).squeeze(1)
        return bool(torch.equal(blk * 16 + pos % 16, b.slot_mapping.long()))

    def launches_per_step(self) -> int:
        n = 1 if self.fused else 2  # (append +) decode partitions
        if self.cascade:
            n += 2  # shared-prefix kernel, log-sum-exp merge
        elif self.max_ctx > self.part_used:
            n += 1  # log-sum-exp reduce
        if self.has_copy:
            n += 1
        if self.pout is not None:
            n += 1
        return n

    def calls(self):
        """(name, thunk) for every call of one step, in order."""
        t, b, pkv = self.t, self.b, self.pkv
        out = []
        if self.has_copy:
            out.append(("copy_blocks", lambda: pkv.copy_blocks(t["copy_pairs"], t["k_cache"],
                                                               t["v_cache"])))
        if self.fp8 and self.fused:
            out.append(("decode", lambda: pkv.decode_step_fp8(
                t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["k_scale"], t["v_scale"],
                t["block_tables"], t["context_lens"], b.scale, self.out, max_context_len=self.max_ctx,
                partition_size=self.partition, workspace=self.ws)))
            return out
        if self.fp8:
            out.append(("kv_append", lambda: pkv.kv_append_fp8(t["k_new"], t["v_new"], t["slot_mapping"],
                                                               t["k_cache"], t["v_cache"], t["k_scale"],
                                                               t["v_scale"])))
            out.append(("decode", lambda: pkv.paged_attention_decode_fp8(
                t["q"], t["k_cache"], t["v_cache"], t["k_scale"], t["v_scale"], t["block_tables"],
                t["context_lens"], b.scale, self.out, max_context_len=self.max_ctx,
                partition_size=self.partition, workspace=self.ws)))
            return out
        if self.cascade:
            out.append(("decode", lambda: pkv.decode_shared_prefix(
                t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"], b.scale,
                self.out, self.prefix_len, k_new=t["k_new"], v_new=t["v_new"],
                max_context_len=self.max_ctx, partition_size=self.partition, workspace=self.ws)))
            return out
        if self.fused:
            out.append(("decode", lambda: pkv.decode_step(
                t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["block_tables"],
                t["context_lens"], b.scale, self.out, max_context_len=self.max_ctx,
                partition_size=self.partition, workspace=self.ws)))
            return out
        out.append(("kv_append", lambda: pkv.kv_append(t["k_new"], t["v_new"], t["slot_mapping"],
                                                       t["k_cache"], t["v_cache"])))
        out.append(("decode", lambda: pkv.paged_attention_decode(
            t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"], b.scale,
            self.out, max_context_len=self.max_ctx, partition_size=self.partition, workspace=self.ws)))
        if self.pout is not None:
            out.append(("prefill_chunk", lambda: pkv.paged_attention_prefill_chunk(
                t["prefill_q"], t["prefill_cu_q_lens"], t["k_cache"], t["v_cache"],
                t["prefill_block_tables"], t["prefill_context_lens"], b.scale, self.pout,
                max_q_len=self.max_q, max_context_len=self.max_pctx)))
        return out


DECODE_SOURCES = ("common.cuh", "decode.cu")
# the shared-prefix call also runs the tcgen05 kernel on the prefix
CASCADE_SOURCES = DECODE_SOURCES + ("prefill_common.cuh", "prefill_tc.cu", "tcgen05.cuh")


def sleep_ahead(ms: float) -> None:
    """Keep the current stream busy for about `ms` milliseconds (a spin
    kernel of torch's; nothing of this library runs)."""
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is None or ms <= 0:
        return
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    mhz = getattr(props, "clock_rate", 0) / 1e3  # kHz -> MHz
    sleep(int(ms * 1e3 * (mhz if mhz > 0 else 2070.0)))


def capture_step(calls):
    """One step's calls captured in a CUDA graph (the library's launches,
    programmatic dependencies included), or None if capture is refused."""
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _, fn in calls:
                fn()
        g.replay()
        torch.cuda.synchronize()
        return g
    except Exception as e:  # noqa: BLE001 - fall back to eager dispatch
        print(f"bench: CUDA graph capture refused ({type(e).__name__}: {e}); timing eager dispatch",
              file=sys.stderr)
        torch.cuda.synchronize()
        return None


def time_device(step: Step, steps: int, warmup: int, world: int):
    """Timed passes of `steps` steps each.  Throughput: the calls dispatched
    eagerly through the API, then the same step captured once in a CUDA graph
    and replayed (as a serving loop dispatches a decode step); each pass
    records an event only before the first and after the last step, and the
    faster of the two is the step's time (both are kept in
    `step.dispatch_ms`).  Eager steps keep the programmatic-dependent overlap
    of consecutive launches, but a short step's calls can outrun the host's
    dispatch; a graph replay takes no host time per call but starts each
    step as a new graph launch.  The breakdown pass calls the API eagerly and
    brackets every call with events (per-call durations and the roofline),
    which serialises the calls."""
    calls = step.calls()
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for _, fn in calls:
            fn()
    torch.cuda.synchronize()

    def timed(run_step):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e0.record(stream)
        for _ in range(steps):
            run_step()
        e1.record(stream)
        torch.cuda.synchronize()
        wall_s = time.perf_counter() - t0
        barrier(world)
        return e0.elapsed_time(e1), wall_s

    def eager():
        for _, fn in calls:
            fn()

    span_ms, wall = timed(eager)
    step.dispatch, step.dispatch_ms = "eager", {"eager": round(span_ms / steps, 5)}
    graph = capture_step(calls)
    dev = f"cuda:{torch.cuda.current_device()}"
    # every rank takes the same path: graphs only if every rank captured one,
    # and used only if they are faster on every rank
    if max_over_ranks(0.0 if graph is not None else 1.0, world, dev) == 0.0:
        g_ms, g_wall = timed(graph.replay)
        step.dispatch_ms["cuda_graph"] = round(g_ms / steps, 5)
        if max_over_ranks(g_ms - span_ms, world, dev) < 0:
            span_ms, wall, step.dispatch = g_ms, g_wall, "cuda_graph"
    del graph

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
          for _ in range(steps)]
    torch.cuda.synchronize()
    # The host needs about as long to enqueue a short step with its events as
    # the GPU needs to run it; an idle gap between an event and the launch
    # after it would count as call time.  A device-side sleep ahead of the
    # loop (as long as the throughput pass, at most 200 ms) lets the host
    # queue steps while the GPU is busy, so the events time only the calls.
    sleep_ahead(min(200.0, span_ms))
    for i in range(steps):
        ev[i][0].record(stream)
        for j, (_, fn) in enumerate(calls):
            fn()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    per_call = {}
    for j, (name, _) in enumerate(calls):
        per_call[name] = sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)) / steps
    step_ms = sorted(ev[i][0].elapsed_time(ev[i][-1]) for i in range(steps))
    serial_ms = sum(step_ms) / steps
    # spread of the serialised step times (nearest-rank percentiles)
    pct = {f"p{q}": round(step_ms[min(steps - 1, (q * steps) // 100)], 5) for q in (10, 50, 90)}
    return span_ms, serial_ms, per_call, wall, pct


def _pack(tensors, device):
    """One uint8 buffer holding every tensor (each at a 256-byte aligned
    offset) and views of it with the tensors' dtypes and shapes."""
    offs, total = [], 0
    for x in tensors:
        offs.append(total)
        total += (x.numel() * x.element_size() + 255) // 256 * 256
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device=device,
                      pin_memory=(device == "cpu" and torch.cuda.is_available()))
    views = [buf[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape)
             for o, x in zip(offs, tensors)]
    return buf, views


def time_e2e(step: Step, steps: int, warmup: int, world: int):
    """Same step through the public API with host buffers: each step copies its
    inputs from pinned host memory and reads the outputs back.  The inputs sit
    in one pinned staging buffer (as a serving loop would assemble them) and
    cross in one copy; the outputs come back in one copy.  The copies run on
    a second stream into double-buffered device inputs and outputs, as a
    serving loop pipelines them: step i+1's inputs cross while step i
    computes, and step i's outputs cross after it finishes (every copy of
    every step is inside the timed region)."""
    b = step.b
    names = ["q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens"]
    if step.has_copy:
        names.append("copy_pairs")
    if step.pout is not None:
        names += ["prefill_q", "prefill_cu_q_lens", "prefill_block_tables", "prefill_context_lens"]
    src = [getattr(b, n).contiguous() for n in names]
    hin, hviews = _pack(src, "cpu")
    for v, x in zip(hviews, src):
        v.copy_(x)
    outs = [step.out] + ([] if step.pout is None else [step.pout])
    dins = [_pack(src, step.dev) for _ in range(2)]
    douts = [_pack(outs, step.dev) for _ in range(2)]
    houts = [torch.empty(douts[0][0].numel(), dtype=torch.uint8).pin_memory() for _ in range(2)]
    saved = ({n: step.t[n] for n in names}, step.out, step.pout)
    h2d = sum(x.numel() * x.element_size() for x in src)
    d2h = sum(x.numel() * x.element_size() for x in outs)
    calls = step.calls()
    main = torch.cuda.current_stream()
    cs = torch.cuda.Stream(device=step.dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]

    def bind(j):  # the calls read buffer set j
        for n, v in zip(names, dins[j][1]):
            step.t[n] = v
        step.out = douts[j][1][0]
        if step.pout is not None:
            step.pout = douts[j][1][1]

    def run(n):
        # inputs of step 0, then: compute i on the main stream while the copy
        # stream brings step i+1's inputs and takes step i-1's outputs
        with torch.cuda.stream(cs):
            cs.wait_stream(main)
            dins[0][0].copy_(hin, non_blocking=True)
            ev_in[0].record(cs)
        for i in range(n):
            j = i & 1
            main.wait_event(ev_in[j])
            bind(j)
            for _, fn in calls:
                fn()
            ev_done[j].record(main)
            with torch.cuda.stream(cs):
                if i + 1 < n:
                    if i >= 1:
                        cs.wait_event(ev_done[j ^ 1])  # step i-1 no longer reads buffer set j^1
                    dins[j ^ 1][0].copy_(hin, non_blocking=True)
                    ev_in[j ^ 1].record(cs)
                cs.wait_event(ev_done[j])
                houts[j].copy_(douts[j][0], non_blocking=True)
        main.wait_stream(cs)

    try:
        run(warmup)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        e0.record(main)
        run(steps)
        e1.record(main)
        torch.cuda.synchronize()
        barrier(world)
    finally:
        step.t.update(saved[0])
        step.out, step.pout = saved[1], saved[2]
    return e0.elapsed_time(e1), h2d, d2h


def cpu_baseline(batch: W.Batch, budget_s: float = 12.0):
    """The fp64 oracle as it stands, on this host's cores, on whole steps of
    the same batch repeated for about `budget_s` seconds."""
    import oracle
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    reps, seqs, rows = 0, 0, 0
    t0 = time.perf_counter()
    while True:
        if batch.copy_pairs is not None and batch.copy_pairs.numel():
            oracle.copy_blocks(kc, vc, batch.copy_pairs)
        if batch.k_scale is not None:
            oracle.kv_append_fp8(batch.k_new, batch.v_new, batch.slot_mapping, kc, vc, batch.k_scale,
                                 batch.v_scale)
        else:
            oracle.kv_append(batch.k_new, batch.v_new, batch.slot_mapping, kc, vc)
        oracle.decode(batch.q, kc, vc, batch.block_tables, batch.context_lens, batch.scale, batch.k_scale,
                      batch.v_scale)
        if batch.prefill_q is not None:
            oracle.prefill_chunk(batch.prefill_q, batch.prefill_cu_q_lens, kc, vc,
                                 batch.prefill_block_tables, batch.prefill_context_lens,
                                 batch.scale)
        reps += 1
        seqs += batch.num_seqs + (0 if batch.prefill_context_lens is None
                                  else int(batch.prefill_context_lens.numel()))
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    cores = oracle.threads()
    # one thread, on the first 8 decode sequences of the batch (about 1/8 of
    # the budget), for the single-core figure
    one = None
    if batch.prefill_q is None:
        sub = slice(0, min(8, batch.num_seqs))
        oracle.set_threads(1)
        try:
            r1, t1 = 0, time.perf_counter()
            while True:
                oracle.decode(batch.q[sub], kc, vc, batch.block_tables[sub], batch.context_lens[sub], batch.scale,
                              batch.k_scale, batch.v_scale)
                r1 += 1
                if time.perf_counter() - t1 >= budget_s / 8:
                    break
            one = {"value": r1 * (sub.stop - sub.start) / (time.perf_counter() - t1), "cores": 1,
                   "sample": f"{r1} decodes of the first {sub.stop - sub.start} sequences"}
        finally:
            oracle.set_threads(cores)
    return {"value": seqs / dt, "unit": "seq-steps/s", "cores": cores,
            "kind": "oracle", "cpu": cpu_model(),
            "sample": f"{reps} whole steps of the {batch.spec.name} batch "
                      f"({batch.num_seqs} decode seqs), fp64, {dt:.1f} s",
            "single_thread": one}


# Arm "CPU part" codes of the server cores this may run on
ARM_PARTS = {"0xd0c": "Neoverse N1", "0xd40": "Neoverse V1", "0xd49": "Neoverse N2", "0xd4f": "Neoverse V2",
             "0xd83": "Neoverse V3", "0xd84": "Neoverse V3AE", "0xd8e": "Neoverse N3"}


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    v = line.split(":", 1)[1].strip()
                    return f"Arm {ARM_PARTS[v]} ({v})" if v in ARM_PARTS else v
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def step_rooflines(step: Step, per_call: dict, peaks: dict, workload: str):
    """The decode call's HBM roofline (and the prefill chunk's tensor roofline,
    the copy and append figures when the step has them) from the per-call
    CUDA-event durations of one breakdown pass."""
    batch = step.b
    S, Hq, d = batch.q.shape
    Hkv = batch.spec.num_kv_heads
    elem = batch.q.element_size()
    kv_elem = batch.k_cache.element_size()  # 1 for fp8 caches
    # context lengths the decode call sees (after this step's append)
    db = accounting.decode_bytes(batch.context_lens, Hq, Hkv, d, kv_elem, elem, elem)
    dec_ms = per_call["decode"]
    # the fused call also writes the appended K and V rows (it reads them from
    # k_new/v_new instead of the cache, which the KV count already covers)
    dec_bytes = db["total"] + (2 * S * Hkv * d * kv_elem if step.fused else 0)
    if step.cascade:
        # the prefix's K/V are read once, not once per sequence: count them once
        dec_bytes -= step.prefix_len * (S - 1) * 2 * Hkv * d * elem
    achieved = dec_bytes / (dec_ms / 1e3) / 1e9
    kname = ("decode_shared_prefix" if step.cascade else "decode_step_fp8" if step.fp8 and step.fused
             else "decode_step" if step.fused else "paged_attention_decode_fp8" if step.fp8
             else "paged_attention_decode")
    traffic = recorded_traffic(kname, workload, CASCADE_SOURCES if step.cascade else DECODE_SOURCES)
    roofline = {"kernel": ("decode_shared_prefix (fused append; shared-prefix tile on the tensor cores, "
                           "partition kernel over each sequence's own tokens, log-sum-exp merge; bytes "
                           "count the prefix once)" if step.cascade else
                           "decode_step_fp8 (fused quantising append; fp8 E4M3 cache widened to fp16 in "
                           "registers, transposed fp16 tile products; one wave without a split when it "
                           "covers the batch, else partitions + log-sum-exp reduce)" if step.fp8 and step.fused else
                           "decode_step (fused append + partition kernel + log-sum-exp reduce)"
                           if step.fused else
                           "paged_attention_decode_fp8 (fp8 E4M3 cache widened to fp16 in registers, "
                           "transposed fp16 tile products; one wave without a split when it covers the "
                           "batch, else partitions + log-sum-exp reduce)" if step.fp8 else
                           "paged_attention_decode (partition kernel + log-sum-exp reduce)"),
                "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "peak_source": f"{peaks['source']} hbm_gbs (copy bandwidth)",
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": traffic, "traffic_unit": "bytes per call (ncu dram read+write)",
                "algorithmic_bytes": dec_bytes, "partition": step.part_used,
                "kv_bytes": db["kv"], "decode_us": round(dec_ms * 1e3, 2)}
    extra = {}
    if step.pout is not None:
        fl = accounting.prefill_flops(batch.prefill_cu_q_lens, batch.prefill_context_lens, Hq, d)
        tf = fl / (per_call["prefill_chunk"] / 1e3) / 1e12
        extra["prefill_roofline"] = {
            "kernel": "prefill_tc_kernel (tcgen05, chunked-prefill tile)", "bound": "tensor",
            "achieved": round(tf, 1), "peak": peaks["bf16_tflops"],
            "peak_source": f"{peaks['source']} bf16_tflops (cuBLAS burst)", "unit": "TFLOP/s",
            "frac": round(tf / peaks["bf16_tflops"], 4),
            "frac_of_sustained": round(tf / peaks["bf16_tflops_sustained"], 4),
            "flops": fl, "us": round(per_call["prefill_chunk"] * 1e3, 2)}
    if step.has_copy:
        cb = accounting.copy_blocks_bytes(int(batch.copy_pairs.shape[0]), Hkv, d, elem)
        extra["copy_blocks"] = {"pairs": int(batch.copy_pairs.shape[0]), "bytes": cb,
                                "us": round(per_call["copy_blocks"] * 1e3, 2)}
    if "kv_append" in per_call:
        ab = accounting.append_bytes(int(batch.slot_mapping.numel()), Hkv, d, elem)
        extra["append_gbs"] = round(ab / (per_call["kv_append"] / 1e3) / 1e9, 1)
    return roofline, extra, db


def seqs_per_step(batch: W.Batch) -> int:
    return batch.num_seqs + (0 if batch.prefill_context_lens is None else int(batch.prefill_context_lens.numel()))


# Workloads whose own targets ride on the headline run as sub-records: the
# long-context decode (HBM roofline) and the mixed step (its prefill chunk
# against the bf16 tensor roofline), plus the headline batch itself over a
# long timed region.
TARGET_WORKLOADS = ("llama3_8b_decode", "long_context", "mixed_step")
# Further records on the same line: the same decode batches over fp8 E4M3
# caches and the shared-prefix (cascade) step, each with its own roofline.
EXTRA_RECORDS = (("llama3_8b_decode_fp8", "llama3_8b_decode", "fp8"),
                 ("long_context_fp8", "long_context", "fp8"),
                 ("shared_prefix_cow", "shared_prefix_cow", "bf16"))


def target_record(name: str, dev: str, peaks: dict, args, world: int, min_ms: float = 250.0,
                  kv_dtype: str = "bf16") -> dict:
    """One workload's step timed over at least `min_ms` of GPU time (so the
    clock sampler sees it under load), with its rooflines."""
    batch = W.make_batch(name, poison=False)
    if kv_dtype == "fp8":
        batch = W.fp8_batch(batch)
    step = Step(batch, dev, args.partition, args.unfused, args.no_cascade)
    calls = step.calls()
    for _ in range(3):
        for _, fn in calls:
            fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        for _, fn in calls:
            fn()
    e1.record()
    torch.cuda.synchronize()
    n = max(10, int(math.ceil(min_ms / max(1e-3, e0.elapsed_time(e1) / 5))))
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    span_ms, serial_ms, per_call, _, pct = time_device(step, n, 3, world)
    clk = clocks.stop()
    roofline, extra, _ = step_rooflines(step, per_call, peaks, name)
    rec = {"kv_dtype": kv_dtype, "step_dispatch": getattr(step, "dispatch", "eager"),
           "dispatch_ms_per_step": getattr(step, "dispatch_ms", None), "steps": n, "timed_ms": round(span_ms, 1), "ms_per_step": round(span_ms / n, 5),
           "value": round(world * seqs_per_step(batch) * n / (span_ms / 1e3), 1), "unit": "seq-steps/s",
           "calls_us": {k: round(v * 1e3, 2) for k, v in per_call.items()},
           "serial_ms_per_step": round(serial_ms, 5), "roofline": roofline, "clocks": clk}
    rec.update(extra)
    del step
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    world, rank, local = dist_env()
    init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    batch = W.make_batch(args.workload, poison=False)
    if args.kv_dtype == "fp8":
        if batch.prefill_q is not None or batch.spec.head_dim != 128 or batch.dtype != torch.bfloat16:
            raise SystemExit("--kv-dtype fp8 needs a bf16, head_dim 128, decode-only workload")
        batch = W.fp8_batch(batch)
    step = Step(batch, dev, args.partition, args.unfused, args.no_cascade)
    peaks = read_peaks()

    clocks = ClockSampler(local)
    clocks.start()
    span_ms, serial_ms, per_call, wall, step_pct = time_device(step, args.steps, args.warmup, world)
    clk = clocks.stop()
    span_ms = max_over_ranks(span_ms, world, dev)
    e2e_ms, h2d, d2h = time_e2e(step, args.steps, args.warmup, world)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)

    sps = seqs_per_step(batch)
    ms_per_step = span_ms / args.steps
    value = world * sps * args.steps / (span_ms / 1e3)
    S, Hq, d = batch.q.shape
    roofline, extra, db = step_rooflines(step, per_call, peaks, args.workload)
    dec_ms = per_call["decode"]
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "seq-steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3" if step.fp8 else "bf16"
        if batch.dtype == torch.bfloat16 else "f32", "data": "synthetic",
        "config": {"workload": args.workload + ("_fp8" if step.fp8 else ""), "seqs": S, "q_heads": Hq,
                   "kv_heads": batch.spec.num_kv_heads, "head_dim": d, "block_size": 16,
                   "max_context_len": batch.max_context_len,
                   "mean_context_len": round(float(batch.context_lens.float().mean()), 1),
                   "kv_bytes_per_step": db["kv"],
                   "l2": "inputs larger than L2 (KV per step %.0f MB > 129 MB L2); no flush"
                         % (db["kv"] / 1e6) if db["kv"] > 129e6 else
                         "working set fits L2; numbers are L2-assisted",
                   "parallelism": f"replicas x{world} (sequences shard, no collective)",
                   "step_dispatch": getattr(step, "dispatch", "eager"),
                   "dispatch_ms_per_step": getattr(step, "dispatch_ms", None)},
        "kv_gbs": round(db["kv"] / (dec_ms / 1e3) / 1e9, 1),
        "calls_us": {k: round(v * 1e3, 2) for k, v in per_call.items()},
        "serial_ms_per_step": round(serial_ms, 5),
        "serial_step_ms_pct": step_pct,
        "roofline": roofline,
        "e2e": {"value": round(world * sps * args.steps / (e2e_ms / 1e3), 1),
                "unit": "seq-steps/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": step.launches_per_step() * args.steps,
        "clocks": clk,
        "wall_s": round(wall, 4),
    }
    line.update(extra)
    del step
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(batch)
    if (world == 1 and not args.no_targets and args.workload == W.HEADLINE and args.kv_dtype == "bf16"
            and args.partition == 0 and not args.unfused and not args.no_cascade):
        line["targets"] = {name: target_record(name, dev, peaks, args, world) for name in TARGET_WORKLOADS}
        for key, name, kvd in EXTRA_RECORDS:
            line["targets"][key] = target_record(name, dev, peaks, args, world, kv_dtype=kvd)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ----------------------------------------------------------------------------
# reference arm: the fp64 oracle on host cores
# ----------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    batch = W.make_batch(args.workload, poison=False)
    S = batch.num_seqs
    # size each step's sample so that warmup + steps stay within ~2 minutes
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    t0 = time.perf_counter()
    oracle.decode(batch.q[:1], kc, vc, batch.block_tables[:1], batch.context_lens[:1], batch.scale)
    per_seq = max(1e-4, time.perf_counter() - t0)
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = max(1, min(S, int(budget / per_seq)))
    sub = slice(0, n)

    def one():
        oracle.kv_append(batch.k_new[sub], batch.v_new[sub], batch.slot_mapping[sub], kc, vc)
        oracle.decode(batch.q[sub], kc, vc, batch.block_tables[sub], batch.context_lens[sub],
                      batch.scale)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "seq-steps/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "seqs": S, "sample_seqs": n},
            "cpu_baseline": {"value": round(value, 3), "unit": "seq-steps/s",
                             "cores": oracle.threads(), "kind": "oracle", "cpu": cpu_model(),
                             "sample": f"first {n} of {S} sequences per step (append + decode), fp64"},
            "e2e": {"value": round(value, 3), "unit": "seq-steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _free_port() -> int:
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_ranks(n: int, argv) -> int:
    """Run this script as `n` ranks, one process per GPU, under
    torch.distributed.run on this node; returns its exit status.  Rank 0
    prints the JSON line."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.abspath(__file__), *argv]
    return subprocess.run(cmd).returncode


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=W.HEADLINE, choices=sorted(W.SPECS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--partition", type=int, default=0,
                    help="decode split-K partition in tokens (0: the library's adaptive choice)")
    ap.add_argument("--unfused", action="store_true",
                    help="separate append and decode calls even where the fused step applies")
    ap.add_argument("--no-cascade", action="store_true",
                    help="plain decode even where the batch shares a prefix")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"],
                    help="fp8: the same step over fp8 E4M3 caches (decode-only workloads)")
    ap.add_argument("--no-targets", action="store_true",
                    help="skip the long-timed records of the target workloads (headline run only)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    world = os.environ.get("WORLD_SIZE")
    if world is None and args.gpus > 1:
        # not started by a launcher: start the ranks here
        sys.exit(launch_ranks(args.gpus, argv))
    if world is not None and int(world) != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}: the launcher and the flag disagree")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
