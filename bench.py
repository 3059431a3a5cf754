#!/usr/bin/env python
"""Benchmark of the paged-KV decode hot path on one GB300 (or N replicas).

One *step* is one pass of the whole decode path over one synthetic batch:
for the ragged serving batch (the default workload) that is

    prepare_decode_metadata (copy_page_indices + compute_num_kv_splits in one
    launch; --metadata separate launches the two) -> paged_attention_v2_partition
    (reading block ids through the flat page list) -> paged_attention_v2_reduce

all launched through the C ABI on one stream, captured once as a CUDA graph
and replayed (--no-graph: plain stream launches).  The KV cache is resident
device state (as in serving); inputs are larger than L2, so no flush is
needed between steps (the tiny workload, which fits in L2, is flushed).

Printed (rank 0, one JSON line): the KV-read GB/s of the step (``value``),
microseconds per step, the roofline of the dominant kernel (the attention
partition pass) against the measured HBM copy bandwidth, the end-to-end
figure through host buffers, SM clocks sampled during the timed region and a
CPU baseline: the float64 oracle timed on a bounded sample on the host cores.

``--impl reference`` times that oracle alone as the reference arm.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "paged decode µs/step and KV-read GB/s (% of GB300 HBM peak) at 1 GPU"
UNIT = "GB/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
DEFAULT_WORKLOAD = "ragged_v2_bf16"


# ----------------------------------------------------------------- helpers --

def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, dist, device) -> float:
    """Largest value of ``x`` over all ranks (rank timing: the slowest rank
    defines the step); identity without a process group."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_rank: int, world: int, seconds: float) -> float:
    """Whole-job throughput: every rank moves its own batch's bytes (weak
    scaling) within the slowest rank's time."""
    return world * bytes_per_rank / seconds / 1e9


def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


ATTENTION_SOURCES = ("attention_kernel.cuh", "attention_unit.inc", "pkv_ptx.cuh")
METADATA_SOURCES = ("decode_metadata.cu", "pkv_ptx.cuh", "pkv_launch.cuh")


def kernel_source_sha(files=ATTENTION_SOURCES) -> str:
    """Hash of a kernel's source files (the kernel a traffic figure describes)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_tables_gb300", "csrc")
    for name in files:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the workload's dominant kernel from the committed
    ncu record, only while that kernel's sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_sha") == kernel_source_sha(tuple(e["source_files"])):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(n)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------- the decode step --

def kv_bytes_of(inp) -> int:
    """K/V bytes one step reads: every token of every sequence, per kv head."""
    kc = inp["key_cache"]
    return sum(inp["seq_lens_list"]) * kc.shape[1] * 2 * inp["query"].shape[2] * kc.element_size()


def flushes_l2(inp) -> bool:
    """Workloads whose K/V is not far larger than L2 get L2 flushed between steps."""
    return kv_bytes_of(inp) < 4 * L2_BYTES


def workload_overrides(name: str, num_seqs=None, seq_len=None, partition_size=None) -> dict:
    """Spec fields that a cut or resized batch replaces (profiling and sweeps
    only): fewer sequences, every sequence `seq_len` tokens, another fixed
    partition size.  Both arms apply the same ones."""
    over = {} if num_seqs is None else {"num_seqs": num_seqs}
    if seq_len is not None:
        n = num_seqs if num_seqs is not None else workloads.WORKLOADS[name].num_seqs
        over.update(seq_len_recipe="fixed", seq_lens=[int(seq_len)] * n)
    if partition_size is not None:
        over["partition_size"] = int(partition_size)
    return over


def workload_config(inp, world: int = 1) -> dict:
    """The workload's identifying configuration: the same dict in both arms."""
    spec = inp["spec"]
    B, H, D = inp["query"].shape
    kc = inp["key_cache"]
    kvb = kv_bytes_of(inp)
    return {
        "workload": spec.name,
        "description": spec.description,
        "num_seqs": B, "num_heads": H, "num_kv_heads": kc.shape[1],
        "head_size": D, "block_size": kc.shape[3],
        "kv_cache_dtype": spec.kv_cache_dtype, "alibi": spec.alibi,
        "total_tokens": sum(inp["seq_lens_list"]), "kv_bytes_per_step": kvb,
        "l2": ("flushed between steps (512 MB write)" if flushes_l2(inp) else
               f"inputs larger than L2: {kvb / 1e9:.2f} GB of K/V per step"),
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }


class DecodeStep:
    """Device buffers of one workload and the launches of one step, issued
    straight through the C ABI with argument structs prepared once."""

    def __init__(self, name: str, seed: int, device, num_seqs=None, fused_metadata=True,
                 lpt=True, seq_len=None, partition_size=None):
        import ctypes

        import paged_kv_decode_tables_gb300 as pkv

        self.pkv = pkv
        self.lib = pkv.lib()
        self.name = name
        over = workload_overrides(name, num_seqs, seq_len, partition_size)
        inp = workloads.make_workload(name, seed=seed, device=device, **over)
        self.inp = inp
        spec = inp["spec"]
        self.spec = spec
        self._input_arena(inp)
        q, kc, vc = inp["query"], inp["key_cache"], inp["value_cache"]
        B, H, D = q.shape
        Hk, bs = kc.shape[1], kc.shape[3]
        self.B, self.H, self.D, self.Hk, self.bs = B, H, D, Hk, bs
        lens = inp["seq_lens_list"]
        self.lens = lens
        e = q.element_size()
        ekv = kc.element_size()  # 1 for an fp8 cache
        nblk = [len(r) for r in inp["block_rows"]]
        self.kv_bytes = sum(lens) * Hk * 2 * D * ekv
        self.q_bytes = B * H * D * e
        self.out_bytes = B * H * D * e
        self.table_bytes = 4 * sum(nblk)
        self.mode = spec.mode
        dev = q.device
        self.out = torch.empty_like(q)
        c_i64x3 = ctypes.c_int64 * 3
        self.out_stride = c_i64x3(*self.out.stride())
        stream = 0  # replaced per call by the current stream
        self._stream = stream

        if self.mode == "v2_splits":
            self.cu = inp["cu_num_blocks"]
            self.page_indices = torch.empty(int(self.cu[-1].item()), dtype=torch.int32, device=dev)
            self.splits = torch.empty(B, dtype=torch.int32, device=dev)
            self.maxP = spec.max_kv_splits
            bt_for_attn, indptr = self.page_indices, self.cu
        else:
            bt_for_attn, indptr = inp["block_tables"], None
            if self.mode == "v2_fixed":
                self.maxP = -(-inp["max_blocks_per_seq"] * bs // spec.partition_size)
            else:
                self.maxP = 1
        if self.mode != "v1":
            self.tmp = torch.empty(B, H, self.maxP, D, dtype=torch.float32, device=dev)
            self.es = torch.empty(B, H, self.maxP, dtype=torch.float32, device=dev)
            self.ml = torch.empty(B, H, self.maxP, dtype=torch.float32, device=dev)
            self.partial_bytes = 0
        self.args = pkv._decode_args(q, kc, vc, bt_for_attn, inp["seq_lens"], inp["scale"], indptr,
                                     None, None, spec.kv_cache_dtype, spec.k_scale, spec.v_scale,
                                     inp["alibi_slopes"])
        self.args_ref = ctypes.byref(self.args)
        self.fused_metadata = fused_metadata
        self.launches_per_step = {"v1": 1, "v2_fixed": 2,
                                  "v2_splits": 3 if fused_metadata else 4}[self.mode]
        # Single pass, longest sequence first: each step orders the batch on
        # the device (pkv_order_by_length) and the decode launches in that order.
        # Only a batch of several waves has a tail worth shortening: at least
        # 4 (sequence, kv head) units per SM.
        sms = torch.cuda.get_device_properties(dev).multi_processor_count if dev.type == "cuda" else 1
        units = B * Hk * -(-(H // Hk) // 8)
        self.lpt = lpt and self.mode == "v1" and units >= 4 * sms
        if self.lpt:
            self.order = torch.empty(B, dtype=torch.int32, device=dev)
            self.args.seq_order = self.order.data_ptr()
            self.launches_per_step += 1
        # Algorithmic bytes of one launch of the attention kernel: K+V of every
        # token, the queries, the block ids and lengths it reads, and (single
        # pass) its output.  The fp32 split-KV partials are counted apart.
        self.attn_alg_bytes = (self.kv_bytes + self.q_bytes + self.table_bytes + 4 * B +
                               (self.out_bytes if self.mode == "v1" else 0) +
                               (4 * B + 4 * (B + 1) if self.mode == "v2_splits" else 0) +
                               (4 * H if spec.alibi else 0))

    def _input_arena(self, inp):
        """Place the per-step inputs (query, lengths, indptr, the table or a
        packed copy of its strided view) in one device buffer, so that an
        end-to-end step brings them in with a single host-to-device copy (a
        pinned copy costs about 11 us before its first byte on this link).
        The step's tensors become views of that buffer; a strided table view
        is filled from its packed copy by a device copy."""
        parts = [("query", inp["query"]), ("seq_lens", inp["seq_lens"])]
        if "cu_num_blocks" in inp:
            parts.append(("cu_num_blocks", inp["cu_num_blocks"]))
        bt = inp["block_tables"]
        parts.append(("table", bt))
        layout, off = {}, 0
        for name, t in parts:
            off = -(-off // 256) * 256
            n = t.numel() * t.element_size()
            layout[name] = (off, n, t.dtype, tuple(t.shape))
            off += n
        arena = torch.empty(off, dtype=torch.uint8, device=bt.device)
        views = {name: arena[o:o + n].view(dt).view(shape)
                 for name, (o, n, dt, shape) in layout.items()}
        for name, t in parts:
            views[name].copy_(t)
        self.arena = arena
        # [0, query_end): the query; [rest_off, end): lengths, indptr, table
        self._query_end = layout["query"][0] + layout["query"][1]
        self._rest_off = layout["seq_lens"][0]
        for name in ("query", "seq_lens", "cu_num_blocks"):
            if name in views:
                inp[name] = views[name]
        if bt.is_contiguous():
            inp["block_tables"] = views["table"]
            self._table_stage = None
        else:
            self._table_stage = views["table"]

    def _check(self, st, what):
        if st != 0:
            raise RuntimeError(f"{what} failed with status {st}")

    def run(self, attn_events=None, kernel_events=None, before_attention=None):
        """Enqueue one step on the current stream.  ``attn_events`` (a pair)
        brackets the attention kernel; ``kernel_events`` (a dict of lists of
        event pairs keyed by kernel) brackets every launch;
        ``before_attention`` is called just before the attention launch is
        enqueued."""
        lib = self.lib
        s = torch.cuda.current_stream().cuda_stream

        def mark(name, i):
            if kernel_events is not None:
                kernel_events[name][-1][i].record()

        def begin(name):
            if kernel_events is not None:
                kernel_events.setdefault(name, []).append(
                    (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                mark(name, 0)

        if self.lpt:
            begin("pkv_order_by_length")
            self._check(lib.pkv_order_by_length(self.order.data_ptr(), self.inp["seq_lens"].data_ptr(),
                                                self.B, s), "order")
            mark("pkv_order_by_length", 1)
        if self.mode == "v2_splits" and self.fused_metadata:
            inp = self.inp
            bt = inp["block_tables"]
            sp = self.spec
            begin("prepare_decode_metadata")
            self._check(lib.prepare_decode_metadata(
                self.page_indices.data_ptr(), self.page_indices.numel(), bt.data_ptr(), bt.shape[1],
                bt.stride(0), bt.stride(1), self.cu.data_ptr(), self.B, self.splits.data_ptr(),
                inp["seq_lens"].data_ptr(), 1, self.H, self.Hk, sp.max_kv_splits,
                sp.device_core_count, None, s), "metadata")
            mark("prepare_decode_metadata", 1)
        elif self.mode == "v2_splits":
            inp = self.inp
            bt = inp["block_tables"]
            begin("copy_page_indices")
            self._check(lib.copy_page_indices(self.page_indices.data_ptr(), self.page_indices.numel(),
                                              bt.data_ptr(), bt.shape[1], bt.stride(0), bt.stride(1),
                                              self.cu.data_ptr(), self.B, None, s), "copy")
            mark("copy_page_indices", 1)
            sp = self.spec
            begin("compute_num_kv_splits")
            self._check(lib.compute_num_kv_splits(self.splits.data_ptr(), inp["seq_lens"].data_ptr(),
                                                  self.B, 1, self.H, self.Hk, sp.max_kv_splits,
                                                  sp.device_core_count, s), "splits")
            mark("compute_num_kv_splits", 1)
        if before_attention is not None:
            before_attention()
        if attn_events is not None:
            attn_events[0].record()
        if self.mode == "v1":
            begin("paged_attention_decode")
            self._check(lib.paged_attention_decode(self.out.data_ptr(), self.out_stride,
                                                   self.args_ref, s), "decode")
            mark("paged_attention_decode", 1)
        else:
            splits = self.splits.data_ptr() if self.mode == "v2_splits" else None
            P = 0 if self.mode == "v2_splits" else self.spec.partition_size
            begin("paged_attention_v2_partition")
            self._check(lib.paged_attention_v2_partition(self.tmp.data_ptr(), self.es.data_ptr(),
                                                         self.ml.data_ptr(), self.maxP, P, splits,
                                                         self.args_ref, s), "partition")
            mark("paged_attention_v2_partition", 1)
        if attn_events is not None:
            attn_events[1].record()
        if self.mode != "v1":
            splits = self.splits.data_ptr() if self.mode == "v2_splits" else None
            begin("paged_attention_v2_reduce")
            self._check(lib.paged_attention_v2_reduce(
                self.out.data_ptr(), self.out_stride, self.tmp.data_ptr(), self.es.data_ptr(),
                self.ml.data_ptr(), self.inp["seq_lens"].data_ptr(), splits, self.B, self.H,
                self.D, self.bs, self.maxP, self.spec.partition_size, self.args.dtype, None, s),
                "reduce")
            mark("paged_attention_v2_reduce", 1)

    def config(self, world: int = 1) -> dict:
        return workload_config(self.inp, world)

    def host_inputs(self):
        """A pinned host copy of the input buffer (query, lengths, indptr, the
        table's live view packed row by row) and a pinned host buffer for the
        result.  Only the table's view is sent, not its backing storage (a
        stride-2 view covers half of it)."""
        hin = {"arena": self.arena.cpu().pin_memory()}
        hout = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self._copy_stream = torch.cuda.Stream()
        return hin, hout

    def e2e_enqueue(self, hin, hout):
        """H2D of the step's inputs, the step, D2H of its output (enqueued
        only).  The lengths, indptr and table go first; the query follows on
        a second stream while the table's packed copy fills its strided view
        and the metadata (or order) launch runs, and only the attention
        launch waits for it."""
        cur = torch.cuda.current_stream()
        r = self._rest_off
        self.arena[r:].copy_(hin["arena"][r:], non_blocking=True)
        side = self._copy_stream
        side.wait_stream(cur)  # one copy at a time on the link
        with torch.cuda.stream(side):
            q = self._query_end
            self.arena[:q].copy_(hin["arena"][:q], non_blocking=True)
        if self._table_stage is not None:
            self.inp["block_tables"].copy_(self._table_stage)
        self.run(before_attention=lambda: cur.wait_stream(side))
        hout.copy_(self.out, non_blocking=True)

    def e2e_step(self, hin, hout, graph=None):
        """One end-to-end step; the host waits for the output.  With ``graph``
        (a capture of ``e2e_enqueue``) the same copies and launches replay as
        one graph launch."""
        if graph is not None:
            graph.replay()
        else:
            self.e2e_enqueue(hin, hout)
        torch.cuda.current_stream().synchronize()

    def e2e_bytes(self, hin, hout):
        h2d = sum(t.numel() * t.element_size() for t in hin.values())
        return h2d, hout.numel() * hout.element_size()


# ------------------------------------------------------------ CPU oracle --

def oracle_sample_inputs(step_or_inp, seq_ids):
    """CPU copies of the pages of ``seq_ids`` (renumbered 0..n-1: the oracle's
    result does not depend on physical block ids)."""
    inp = step_or_inp
    rows = [inp["block_rows"][s] for s in seq_ids]
    blocks = [b for r in rows for b in r]
    idx = torch.tensor(blocks, dtype=torch.long, device=inp["key_cache"].device)
    kc = inp["key_cache"].index_select(0, idx).cpu() if blocks else inp["key_cache"][:0].cpu()
    vc = inp["value_cache"].index_select(0, idx).cpu() if blocks else inp["value_cache"][:0].cpu()
    width = max([1] + [len(r) for r in rows])
    bt = torch.full((len(seq_ids), width), -1, dtype=torch.int32)
    off = 0
    for i, r in enumerate(rows):
        bt[i, :len(r)] = torch.arange(off, off + len(r), dtype=torch.int32)
        off += len(r)
    q = inp["query"][torch.tensor(seq_ids, device=inp["query"].device)].cpu()
    lens = [inp["seq_lens_list"][s] for s in seq_ids]
    return q, kc, vc, bt, lens


def oracle_step(inp, spec, seq_ids, all_splits):
    """The oracle's pass over the sampled sequences (the same steps as the
    GPU step: metadata, then split-KV partition + reduce or single pass).
    Returns (K/V bytes covered, wall seconds spent in the oracle itself, process
    CPU seconds over the same span, all threads); copying the sampled pages out
    of device memory is not counted."""
    import oracle

    q, kc, vc, bt, lens = oracle_sample_inputs(inp, seq_ids)
    kw = oracle_variant_kwargs(inp)
    c0 = time.process_time()
    t0 = time.perf_counter()
    if spec.mode == "v1":
        oracle.decode_v1(q, kc, vc, bt, lens, inp["scale"], **kw)
    elif spec.mode == "v2_fixed":
        maxP = -(-max(lens) // spec.partition_size)
        tmp, es, ml = oracle.v2_partition(q, kc, vc, bt, lens, inp["scale"], maxP,
                                          partition_size=spec.partition_size, **kw)
        oracle.v2_reduce(tmp, es, ml, lens, spec.block_size, partition_size=spec.partition_size)
    else:
        splits = [all_splits[s] for s in seq_ids]
        tmp, es, ml = oracle.v2_partition(q, kc, vc, bt, lens, inp["scale"], spec.max_kv_splits,
                                          num_kv_splits=splits, **kw)
        oracle.v2_reduce(tmp, es, ml, lens, spec.block_size, num_kv_splits=splits)
    dt = time.perf_counter() - t0
    dc = time.process_time() - c0
    e = inp["key_cache"].element_size()
    return sum(lens) * spec.num_kv_heads * 2 * spec.head_size * e, dt, dc


def oracle_variant_kwargs(inp):
    """Cache format and ALiBi slopes of a workload, as the oracle takes them."""
    sl = inp.get("alibi_slopes")
    return dict(kv_cache_dtype=inp.get("kv_cache_dtype", "auto"), k_scale=inp.get("k_scale", 1.0),
                v_scale=inp.get("v_scale", 1.0),
                alibi_slopes=None if sl is None else [float(v) for v in sl.cpu()])


def cpu_threads(n=None):
    """Use ``n`` intra-op threads (default: every core this process may run on)."""
    if n is None:
        try:
            n = len(os.sched_getaffinity(0))
        except Exception:
            n = os.cpu_count() or 1
    torch.set_num_threads(n)
    return torch.get_num_threads()


def oracle_metadata(inp, spec):
    import oracle

    splits = None
    if spec.mode == "v2_splits":
        bt = inp["block_tables"].cpu()
        cu = inp["cu_num_blocks"].cpu().tolist()
        oracle.copy_page_indices(bt, cu, cu[-1])
        splits = oracle.num_kv_splits(inp["seq_lens_list"], 1, spec.num_heads, spec.num_kv_heads,
                                      spec.max_kv_splits, spec.device_core_count)
    return splits


def cpu_baseline(inp, spec, budget_s=10.0, threads=None):
    """The oracle on a bounded sample: sequences in a seeded order (cycling
    through the batch when it is smaller than the budget) until the oracle has
    spent the time budget, after one untimed warm-up sequence; returns KV-read
    GB/s over the sample, the threads it was given and the process CPU time
    over its wall time (how many cores it kept busy)."""
    prev = torch.get_num_threads()
    cores = cpu_threads(threads)
    try:
        order = torch.randperm(len(inp["seq_lens_list"]),
                               generator=torch.Generator().manual_seed(0)).tolist()
        c0 = time.process_time()
        t0 = time.perf_counter()
        splits = oracle_metadata(inp, spec)
        spent = time.perf_counter() - t0
        cpu = time.process_time() - c0
        oracle_step(inp, spec, [order[-1]], splits)  # warm-up, not counted
        steps, nbytes, distinct = 0, 0, set()
        while True:
            s = order[steps % len(order)]
            nb, dt, dc = oracle_step(inp, spec, [s], splits)
            nbytes += nb
            spent += dt
            cpu += dc
            steps += 1
            distinct.add(s)
            if spent >= budget_s:
                break
    finally:
        torch.set_num_threads(prev)
    n = len(inp["seq_lens_list"])
    what = (f"{steps} of {n} sequences" if steps <= n else
            f"{steps} sequence decodes cycling through all {n} sequences")
    return {"value": nbytes / spent / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
            "wall_s": round(spent, 6), "cpu_time_s": round(cpu, 6),
            "cpu_time_over_wall": round(cpu / spent, 2),
            "sample": (f"{what} ({nbytes / 1e9:.3f} GB of K/V) of {spec.name} plus the whole "
                       f"batch's metadata, float64, {spent:.1f} s of oracle time on {cores} "
                       f"thread(s)")}


# ------------------------------------------------------------------ arms --

def run_reference(args):
    rank, world, _ = env_rank()
    if rank != 0:
        return 0
    device = "cuda" if torch.cuda.is_available() else "cpu"
    over = workload_overrides(args.workload, args.num_seqs, args.seq_len, args.partition_size)
    inp = workloads.make_workload(args.workload, seed=0, device=device, **over)
    spec = inp["spec"]
    cores = cpu_threads()
    # the whole --steps K --warmup W run stays within the budget: each step
    # processes sequences (at least one) for its share of it
    total_budget = args.reference_budget
    per_step = total_budget / max(1, args.steps + args.warmup)
    order = torch.randperm(len(inp["seq_lens_list"]), generator=torch.Generator().manual_seed(0))
    order = order.tolist()
    pos = 0
    splits = oracle_metadata(inp, spec)

    def one_step():
        nonlocal pos
        nb, n, spent, cpu = 0, 0, 0.0, 0.0
        while True:
            b, dt, dc = oracle_step(inp, spec, [order[pos % len(order)]], splits)
            nb += b
            spent += dt
            cpu += dc
            pos += 1
            n += 1
            if spent >= per_step:
                break
        return nb, spent, cpu, n

    for _ in range(args.warmup):
        one_step()
    tot_b, tot_t, tot_c, tot_n = 0, 0.0, 0.0, 0
    for _ in range(args.steps):
        b, t, c, n = one_step()
        tot_b += b
        tot_t += t
        tot_c += c
        tot_n += n
    value = tot_b / tot_t / 1e9
    cfg = workload_config(inp, world)
    # one whole decode step of the workload at the sampled rate
    ms_whole_step = cfg["kv_bytes_per_step"] / (value * 1e9) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_whole_step, 3),
        "ms_per_step_note": ("one whole step of the workload extrapolated from the sampled "
                             "rate: kv_bytes_per_step / value"),
        "sample_ms_per_step": round(1e3 * tot_t / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "wall_s": round(tot_t, 3),
                         "cpu_time_s": round(tot_c, 3),
                         "cpu_time_over_wall": round(tot_c / tot_t, 2),
                         "sample": (f"each step: sequences of {args.workload} in a seeded order "
                                    f"for ~{per_step:.1f} s ({tot_n} sequences over "
                                    f"{args.steps} steps), float64")},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# Workloads timed beside the headline in the same run, each with the same
# steps and warm-up: the other decode configurations (single-pass MHA and GQA,
# long-context split-KV, the tiny worked example) and the fp8-cache and ALiBi
# variants of the hot path.
COMPANION_WORKLOADS = ("mha_v1_fp16", "gqa_v1_bf16", "long_v2_bf16", "ragged_v2_fp8",
                       "long_v2_fp8", "mha_v1_alibi_fp16", "tiny_mha_fp32", "gqa_v1_fp32")
# Workloads whose oracle is also timed on one core (the small and mid-size
# configurations); the headline's oracle runs on every core.
ONE_CORE_WORKLOADS = ("tiny_mha_fp32", "mha_v1_fp16", "gqa_v1_bf16")

ATTENTION_KERNEL = {"v1": "paged_attention_decode", "v2_fixed": "paged_attention_v2_partition",
                    "v2_splits": "paged_attention_v2_partition"}


def percentile(sorted_vals, q):
    """Nearest-rank percentile of an ascending list (q in [0, 1])."""
    i = min(len(sorted_vals) - 1, max(0, int(round(q * (len(sorted_vals) - 1)))))
    return sorted_vals[i]


def capture_step_graph(step):
    """One step captured as a CUDA graph (after warm-up launches on a side stream)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            step.run()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.run()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    return graph


def time_steps(step, K, warmup, use_graph, dist=None, clocks=None):
    """Device time of K steps on the launching stream.  Inputs larger than L2:
    the K steps run back to back between two CUDA events (the timed span),
    then a second run of K steps, each bracketed by its own pair of events,
    gives the per-step distribution.  Smaller inputs: L2 is flushed before
    every step (outside its pair of events) and the span is the sum of the
    per-step times.  Returns the per-step times (ms), the span (ms), whether a
    graph was replayed and the clocks sampled during the timed span."""
    flush = flushes_l2(step.inp)
    flush_buf = (torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
                 if flush else None)
    for _ in range(max(3, warmup)):
        step.run()
    torch.cuda.synchronize()
    graph = capture_step_graph(step) if use_graph else None

    def one():
        if graph is not None:
            graph.replay()
        else:
            step.run()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    if flush:
        for i in range(K):
            flush_buf.fill_(float(i))
            ev[i][0].record()
            one()
            ev[i][1].record()
    else:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(K):
            one()
        t1.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    if flush:
        per_step = [a.elapsed_time(b) for a, b in ev]
        span = sum(per_step)
    else:
        span = t0.elapsed_time(t1)
        for i in range(K):
            ev[i][0].record()
            one()
            ev[i][1].record()
        torch.cuda.synchronize()
        per_step = [a.elapsed_time(b) for a, b in ev]
    del flush_buf
    return per_step, span, graph is not None, clk


def kernel_breakdown(step, nsteps):
    """Average device time of every launch of a step (events around each
    launch, plain stream launches) and the attention kernel's launch times."""
    kev = {}
    for _ in range(nsteps):
        step.run(kernel_events=kev)
    torch.cuda.synchronize()
    kernel_us = {k: round(sum(a.elapsed_time(b) for a, b in v) / len(v) * 1e3, 2)
                 for k, v in kev.items()}
    attn_ms = [a.elapsed_time(b) for a, b in kev[ATTENTION_KERNEL[step.mode]]]
    return kernel_us, attn_ms


def roofline_record(step, attn_ms, peak, peak_kind, workload):
    attn_sorted = sorted(attn_ms)
    avg_ms = sum(attn_ms) / len(attn_ms)
    achieved = step.attn_alg_bytes / (avg_ms * 1e-3) / 1e9
    return {
        "kernel": ATTENTION_KERNEL[step.mode],
        "bound": "hbm",
        "achieved": round(achieved, 1),
        "peak": peak,
        "peak_kind": f"{peak_kind} HBM copy bandwidth",
        "unit": "GB/s",
        "frac": round(achieved / peak, 4),
        "traffic": recorded_traffic(workload),
        "alg_bytes_per_launch": step.attn_alg_bytes,
        "avg_launch_us": round(avg_ms * 1e3, 2),
        "p10_p90_launch_us": [round(percentile(attn_sorted, 0.1) * 1e3, 2),
                              round(percentile(attn_sorted, 0.9) * 1e3, 2)],
    }


def step_stats(per_step_ms):
    v = sorted(per_step_ms)
    return {"median": round(percentile(v, 0.5) * 1e3, 2), "p10": round(percentile(v, 0.1) * 1e3, 2),
            "p90": round(percentile(v, 0.9) * 1e3, 2)}


def dtype_label(spec):
    return spec.dtype if spec.kv_cache_dtype == "auto" else f"{spec.dtype}+{spec.kv_cache_dtype}"


def companion_record(name, args, peak, peak_kind, want_one_core):
    """Time one companion workload (same steps and warm-up as the headline)
    and, for the small and mid-size configurations, its oracle on one core."""
    step = DecodeStep(name, seed=0, device="cuda",
                      lpt=args.launch_order == "longest-first")
    K = args.steps
    clocks = ClockSampler(torch.cuda.current_device()) if not args.no_clocks else None
    per_step, span, graphed, clk = time_steps(step, K, args.warmup, args.graph, clocks=clocks)
    kernel_us, attn_ms = kernel_breakdown(step, min(K, 200))
    ms = span / K
    rec = {
        "us_per_step": round(ms * 1e3, 2),
        "step_us": step_stats(per_step),
        "value": round(step.kv_bytes / (ms * 1e-3) / 1e9, 2),
        "unit": UNIT,
        "dtype": dtype_label(step.spec),
        "config": step.config(),
        "roofline": roofline_record(step, attn_ms, peak, peak_kind, name),
        "kernel_us": kernel_us,
        "gpu_launches": K * step.launches_per_step,
        "launch": "CUDA graph replay of the step" if graphed else "stream launches",
        "launch_order": ("longest first (pkv_order_by_length in the step)" if step.lpt
                         else "sequence order"),
        "clocks": clk,
    }
    if want_one_core:
        rec["cpu_baseline_1core"] = cpu_baseline(step.inp, step.spec, budget_s=args.one_core_budget,
                                                 threads=1)
    del step
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    rank, world, local_rank = env_rank()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU for the library arm")
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist_mod.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        dist = dist_mod

    from paged_kv_decode_tables_gb300 import _build

    if rank == 0 or dist is None:
        _build.build()
    if dist is not None:
        dist.barrier()
    step = DecodeStep(args.workload, seed=rank, device="cuda", num_seqs=args.num_seqs,
                      fused_metadata=args.metadata == "fused",
                      lpt=args.launch_order == "longest-first",
                      seq_len=args.seq_len, partition_size=args.partition_size)
    if args.warps:
        step.pkv.set_attention_warps(args.warps)
    if args.fp8_kernel == "tensor-memory":
        step.pkv.set_fp8_kernel(1)
    spec = step.spec
    K = args.steps
    clocks = ClockSampler(torch.cuda.current_device()) if (rank == 0 and not args.no_clocks) else None
    per_step, span_ms, graphed, clk = time_steps(step, K, args.warmup, args.graph, dist, clocks)
    elapsed_ms = max_over_ranks(span_ms, dist, "cuda")

    # per-kernel breakdown over a separate run of steps (events around every launch)
    kernel_us, attn_ms = kernel_breakdown(step, min(K, 200))

    # end to end through host buffers (per step: H2D of the inputs, the step,
    # D2H of the output, host waits for it)
    hin, hout = step.host_inputs()
    Ke = max(3, min(K, 200))
    e2e_graph = None
    if args.graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step.e2e_enqueue(hin, hout)
        torch.cuda.current_stream().wait_stream(side)
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph):
            step.e2e_enqueue(hin, hout)
    for _ in range(3):
        step.e2e_step(hin, hout, e2e_graph)
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(Ke):
        step.e2e_step(hin, hout, e2e_graph)
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, dist, "cuda")
    h2d, d2h = step.e2e_bytes(hin, hout)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    ms_step = elapsed_ms / K
    value = aggregate_gbs(step.kv_bytes, world, ms_step * 1e-3)
    peak, peak_kind = load_peak()
    # the committed DRAM record is for the full batch, not a cut or resized one
    full = (args.num_seqs, args.seq_len, args.partition_size) == (None, None, None)
    roofline = roofline_record(step, attn_ms, peak, peak_kind, args.workload if full else None)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(step.inp, spec, budget_s=args.cpu_budget)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": max(3, args.warmup),
        "ms_per_step": round(ms_step, 5),
        "us_per_step": round(ms_step * 1e3, 2),
        "step_us": step_stats(per_step),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_label(spec),
        "accumulate": "f32",
        "data": "synthetic (seeded; see workloads.py)",
        "config": step.config(world),
        "launch": ("CUDA graph replay of the step" if graphed else
                   "stream launches, programmatic dependent launch"),
        "fp8_kernel": args.fp8_kernel if spec.kv_cache_dtype != "auto" else None,
        "metadata": (("one launch (prepare_decode_metadata)" if step.fused_metadata else
                      "copy_page_indices + compute_num_kv_splits")
                     if step.mode == "v2_splits" else None),
        "launch_order": "longest first (pkv_order_by_length in the step)" if step.lpt else "sequence order",
        "roofline": roofline,
        "step_share": {"attention_kernel": round(roofline["avg_launch_us"] / 1e3 / ms_step, 4)},
        "kernel_us": kernel_us,
        "e2e": {"value": round(aggregate_gbs(step.kv_bytes, world, e2e_s / Ke), 2), "unit": UNIT,
                "us_per_step": round(e2e_s / Ke * 1e6, 2), "steps": Ke,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": ("K/V cache resident on the device; per step: H2D of the inputs from "
                         "one pinned host buffer (lengths, indptr and the table as its packed "
                         "live view first; the query behind them on a second stream, under the "
                         "metadata launch), the step, D2H of the output, host waits"
                         + ("; replayed as one CUDA graph" if e2e_graph is not None else "")),
                "graph": e2e_graph is not None},
        "gpu_launches": K * step.launches_per_step,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    resized = (args.num_seqs, args.seq_len, args.partition_size) != (None, None, None)
    if world == 1 and not args.no_companions and not resized:
        # the other configurations, one after another with the same steps and
        # warm-up; the headline's buffers are released first
        del step, hin, hout, e2e_graph
        torch.cuda.empty_cache()
        comp = {}
        for name in COMPANION_WORKLOADS:
            if name == args.workload:
                continue
            comp[name] = companion_record(name, args, peak, peak_kind,
                                          (not args.no_cpu_baseline) and name in ONE_CORE_WORKLOADS)
        line["workloads"] = comp
        line["gpu_launches"] += sum(r["gpu_launches"] for r in comp.values())
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_metadata(args):
    """The fused decode metadata kernel alone (normal_decode_set_metadata), one
    launch per step, L2 flushed between launches (its inputs are about L2-sized)."""
    import ctypes

    import paged_kv_decode_tables_gb300 as pkv
    from paged_kv_decode_tables_gb300 import _build

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU for the library arm")
    _build.build()
    inp = workloads.make_decode_metadata_inputs(args.workload, seed=0, device="cuda")
    B = inp["seq_lens"].shape[0]
    msp, ps = inp["max_seq_pages"], inp["page_size"]
    swa = inp["full_to_swa_mapping"] is not None
    cache = torch.empty(B, dtype=torch.int32, device="cuda")
    cu = torch.empty(B + 1, dtype=torch.int32, device="cuda")
    pt = torch.empty(B, msp, dtype=torch.int32, device="cuda")
    swa_t = torch.empty(B, msp, dtype=torch.int32, device="cuda") if swa else None
    a = pkv.decode_metadata_args(cache, cu, pt, inp["req_to_token"], inp["req_pool_indices"],
                                 inp["seq_lens"], seq_len_delta=inp["seq_len_delta"], page_size=ps,
                                 max_seq_pages=msp, swa_page_table=swa_t,
                                 full_to_swa_mapping=inp["full_to_swa_mapping"])
    ref = ctypes.byref(a)
    lib = pkv.lib()

    def launch():
        st = lib.normal_decode_set_metadata(ref, torch.cuda.current_stream().cuda_stream)
        if st != 0:
            raise RuntimeError(f"normal_decode_set_metadata failed with status {st}")

    flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    for _ in range(max(3, args.warmup)):
        launch()
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    clocks = ClockSampler(torch.cuda.current_device()) if not args.no_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    for i in range(K):
        flush_buf.fill_(float(i))
        ev[i][0].record()
        launch()
        ev[i][1].record()
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    ms = [x.elapsed_time(y) for x, y in ev]
    avg_ms = sum(ms) / K
    entries = B * msp
    alg = (entries * 4 * 2 + (entries * (8 + 4) if swa else 0) + B * 8 * 2 + B * 4 + (B + 1) * 4)
    peak, peak_kind = load_peak()
    achieved = alg / (avg_ms * 1e-3) / 1e9

    # end to end: lengths and request rows from pinned host memory, outputs back
    h_lens = inp["seq_lens"].cpu().pin_memory()
    h_pool = inp["req_pool_indices"].cpu().pin_memory()
    h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (cache, cu, pt)]
    Ke = max(3, min(K, 100))
    for it in range(Ke + 3):
        if it == 3:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
        inp["seq_lens"].copy_(h_lens, non_blocking=True)
        inp["req_pool_indices"].copy_(h_pool, non_blocking=True)
        launch()
        for h, d in zip(h_out, (cache, cu, pt)):
            h.copy_(d, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    e2e_s = (time.perf_counter() - t0) / Ke
    h2d = h_lens.numel() * 8 + h_pool.numel() * 8
    d2h = sum(h.numel() * h.element_size() for h in h_out)

    cpu = None
    if not args.no_cpu_baseline:
        import oracle

        cores = cpu_threads()
        rt = inp["req_to_token"].cpu()
        mapping = inp["full_to_swa_mapping"].cpu() if swa else None
        lens = inp["seq_lens"].cpu().tolist()
        pool = inp["req_pool_indices"].cpu().tolist()
        t0 = time.perf_counter()
        rows = 0
        while rows < B and time.perf_counter() - t0 < args.cpu_budget:
            n = min(8, B - rows)
            oracle.decode_set_metadata(lens[rows:rows + n], rt, pool[rows:rows + n], msp,
                                       inp["seq_len_delta"], ps, full_to_swa_mapping=mapping)
            rows += n
        dt = time.perf_counter() - t0
        per_row = alg / B
        cpu = {"value": round(per_row * rows / dt / 1e9, 5), "unit": UNIT, "cores": 1,
               "kind": "oracle",
               "sample": f"{rows} of {B} request rows, pure Python, {dt:.1f} s"}
        del cores

    line = {
        "metric": "fused decode metadata µs/launch and GB/s moved at 1 GPU",
        "value": round(achieved, 2), "unit": UNIT, "n_gpus": 1, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": round(avg_ms, 5),
        "us_per_step": round(avg_ms * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32", "data": "synthetic (seeded; see workloads.py)",
        "config": {"workload": args.workload, "description": inp["description"],
                   "batch": B, "page_size": ps, "max_seq_pages": msp, "swa": swa,
                   "l2": "flushed between launches (512 MB write)"},
        "roofline": {"kernel": "normal_decode_set_metadata", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} HBM copy bandwidth", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": recorded_traffic(args.workload),
                     "alg_bytes_per_launch": alg, "avg_launch_us": round(avg_ms * 1e3, 2)},
        "e2e": {"value": round(alg / e2e_s / 1e9, 2), "unit": UNIT,
                "us_per_step": round(e2e_s * 1e6, 2), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": K, "clocks": clk, "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_swa_spec(args):
    """The SWA speculative page-table kernel alone, L2 flushed between launches."""
    import paged_kv_decode_tables_gb300 as pkv
    from paged_kv_decode_tables_gb300 import _build

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU for the library arm")
    _build.build()
    inp = workloads.make_swa_spec_inputs(args.workload, seed=0, device="cuda")
    A, Bt = inp["page_table_a"], inp["page_table_b"]
    la, lb, R = inp["seq_len_a"], inp["seq_len_b"], inp["num_draft_tokens"]
    rows, width = Bt.shape[0], A.shape[1] + Bt.shape[1]
    dst = torch.zeros(rows, width, dtype=torch.int32, device="cuda")

    def launch():
        pkv.prepare_swa_spec_page_table(dst, A, Bt, la, lb, R)

    flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    for _ in range(max(3, args.warmup)):
        launch()
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for i in range(K):
        flush_buf.fill_(float(i))
        ev[i][0].record()
        launch()
        ev[i][1].record()
    torch.cuda.synchronize()
    avg_ms = sum(x.elapsed_time(y) for x, y in ev) / K
    la_rows = la.repeat_interleave(R).to(torch.int64)
    written = int(torch.clamp(la_rows + lb.to(torch.int64), max=width).sum())
    alg = written * 4 * 2 + la.numel() * 4 + lb.numel() * 4  # read + write each element
    peak, peak_kind = load_peak()
    achieved = alg / (avg_ms * 1e-3) / 1e9
    line = {
        "metric": "SWA speculative page table µs/launch and GB/s moved at 1 GPU",
        "value": round(achieved, 2), "unit": UNIT, "n_gpus": 1, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": round(avg_ms, 5),
        "us_per_step": round(avg_ms * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32", "data": "synthetic (seeded; see workloads.py)",
        "config": {"workload": args.workload, "description": inp["description"],
                   "l2": "flushed between launches (512 MB write)"},
        "roofline": {"kernel": "prepare_swa_spec_page_table", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} HBM copy bandwidth", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "alg_bytes_per_launch": alg, "avg_launch_us": round(avg_ms * 1e3, 2)},
        "gpu_launches": K, "cpu_baseline": None, "e2e": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(workloads.WORKLOADS) + sorted(workloads.METADATA_WORKLOADS)
                    + sorted(workloads.SWA_SPEC_WORKLOADS))
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="smaller batch of the same workload (profiling captures only)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="every sequence this many tokens (launch-size sweeps only)")
    ap.add_argument("--partition-size", type=int, default=None,
                    help="tokens per partition of a fixed-partition workload (sweeps only)")
    ap.add_argument("--warps", type=int, default=0, choices=[0, 1, 2, 4],
                    help="force warps per attention CTA (0: library default)")
    ap.add_argument("--fp8-kernel", choices=["mma", "tensor-memory"], default="mma",
                    help="kernel for fp8 caches of head size 128 / block size 16")
    ap.add_argument("--metadata", choices=["fused", "separate"], default="fused",
                    help="ragged step: metadata in one launch or the two separate kernels")
    ap.add_argument("--launch-order", choices=["longest-first", "sequence"],
                    default="longest-first",
                    help="single pass: order the batch longest first on the device each step "
                         "(pkv_order_by_length, one launch in the step) or keep sequence order")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="time stream launches instead of CUDA-graph replays of the step")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the CPU baseline sample")
    ap.add_argument("--reference-budget", type=float, default=120.0,
                    help="total seconds of oracle work for --impl reference (all steps)")
    ap.add_argument("--one-core-budget", type=float, default=3.0,
                    help="seconds of single-thread oracle work per small/mid-size workload")
    ap.add_argument("--no-companions", action="store_true",
                    help="time only the selected workload (no per-configuration records)")
    args = ap.parse_args(argv)
    if args.workload in workloads.SWA_SPEC_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm covers the "
                              "decode workloads; this workload is a library addition"}))
            return 0
        return run_swa_spec(args)
    if args.workload in workloads.METADATA_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm covers the "
                              "decode workloads; this workload is a library addition"}))
            return 0
        return run_metadata(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
