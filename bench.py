"""Benchmark of the paged decode hot path on GB300.

A step is one pass of the whole path over one batch: copy-on-write block copies (when
the workload has shared blocks), the new tokens' cache write, and paged decode
attention for every sequence.  Inputs are synthetic and seeded
(paged_kv_cache_90_gb300.workloads); the default workload is the Llama-3-8B-shaped
decode layer (64 sequences, contexts uniform in [128, 2048] plus the new token,
32/8 heads, head_dim 128, bf16, block size 16).

Metric: effective GB/s = algorithmic bytes of a step / step time, where the bytes are
those the step must move: every context token's K and V (for its KV head), the
queries, the outputs, the block-table entries and lengths, the new tokens read and
written, and the copied blocks.  Timing: CUDA events on the launching stream.  A step
that reads more than twice the L2 (the Llama-3-8B, long-context and continuous-batching
workloads) runs back to back with the others between two events: its K/V are streamed
with an evict-first policy, so no step finds the previous one's data in L2 (a
device-side spin queued before the first event lets the host queue the steps, so the
GPU never waits for a launch inside the timed region).  Smaller
steps, and steps whose sequences share blocks, are timed one by one with the L2 flushed
between them outside the events (a 256 MiB write, then a 256 MiB read so that the
write's dirty lines are written back before the step starts); the flushed per-step
figures of the large workloads are reported beside the back-to-back ones.  A step issues
the cache write and the decode as one pkv_decode_step call.  The roofline entry times
the decode kernels alone (main kernel + merge of split rows) in a second loop of decode
calls on the same resident caches, timed the same way.  The end-to-end entry times the
step from pinned host memory: each step's inputs go in as one copy and its output comes
back inside the timed region; back-to-back workloads pipeline those copies on a second
stream beside the neighbouring steps' kernels, as a serving loop would.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_90_gb300 import binding, workloads as wl  # noqa: E402
from paged_kv_cache_90_gb300.decode_step import DeviceStep, DeviceWorkload, prepare_step, run_decode_step  # noqa: E402

METRIC = "paged decode attention: effective KV-read GB/s (% of HBM peak), µs/step"
UNIT = "GB/s"
L2_FLUSH_BYTES = 256 << 20
DECODE_SOURCES = ["decode_core.cuh", "decode_mma.cuh", "decode_mma.cu", "decode_mma_small.cu", "decode_mma_launch.cuh", "merge.cuh",
                  "decode_dispatch.cu", "device_common.cuh", "pkv_internal.h"]
PREFILL_SOURCES = ["prefill_tc.cu", "tcgen05.cuh", "prefill_mma.cuh", "decode_mma_launch.cuh", "device_common.cuh",
                   "pkv_internal.h"]


# ---- workloads -----------------------------------------------------------------------

def make_workload(name: str, rank: int = 0) -> wl.Workload:
    seed_off = 1000 * rank
    if name == "llama3_8b_decode":
        return wl.llama3_8b_decode(seed=2 + seed_off)
    if name.startswith("long_context"):
        bs = 32 if name.endswith("bs32") else 16
        return wl.long_context(seed=3 + seed_off, block_size=bs)
    if name == "shared_prefix_cow":
        return wl.shared_prefix_cow(seed=4 + seed_off)
    m = re.fullmatch(r"continuous_batching_bs(\d+)_(bf16|e4m3)(_headscales)?", name)
    if m:   # _headscales: KV heads 2^3 apart in magnitude, one e4m3 scale each
        return wl.continuous_batching(seed=5 + seed_off, block_size=int(m.group(1)), kv_dtype=m.group(2),
                                      head_spread=3.0 if m.group(3) else 0.0)
    m = re.fullmatch(r"sliding_window(?:_bs(\d+))?", name)
    if m:   # Mistral-style 4096-position window over 8 x 32768-token contexts
        return wl.sliding_window_decode(seed=6 + seed_off, block_size=int(m.group(1) or 16))
    if name == "chunked_prefill":  # two 2048-token prompts, two 512-token chunks after 512 / 1536 cached
        return wl.chunked_prefill(seed=7 + seed_off)
    m = re.fullmatch(r"prefill_(\d+)x(\d+)", name)
    if m:   # N fresh prompts of T tokens each
        n, t = int(m.group(1)), int(m.group(2))
        return wl.chunked_prefill(seed=8 + seed_off, prefix_lens=[0] * n, chunk_lens=[t] * n)
    if name == "mha_decode":  # multi-head attention (one query head per KV head), Llama-3-8B-shaped batch
        g = torch.Generator().manual_seed(9 + seed_off)
        lens = (torch.randint(128, 2049, (64,), generator=g) + 1).tolist()
        return wl.variable_length_decode("mha_decode", 9 + seed_off, lens, 32, 32, 128, 16, "bf16")
    if name == "tiny":
        return wl.tiny(seed=1 + seed_off)
    raise SystemExit(f"unknown workload {name}")


def describe_workload(w: wl.Workload, name: str) -> str:
    L = torch.cat([st.context_lens for st in w.steps]).float()
    if w.steps[0].query_start_loc is not None:
        st = w.steps[0]
        return (f"{name}: {st.context_lens.numel()} seqs, {st.query.shape[0]} new tokens (chunks "
                f"{(st.query_start_loc[1:] - st.query_start_loc[:-1]).tolist()}), contexts "
                f"{st.context_lens.tolist()}, {w.num_heads}/{w.num_kv_heads} heads, head_dim {w.head_dim}, "
                f"{wl.DTYPE_NAMES[w.kv_dtype]} KV, block {w.block_size}")
    return (f"{name}: {w.num_seqs} seqs, {w.num_heads}/{w.num_kv_heads} heads, head_dim {w.head_dim}, "
            f"{wl.DTYPE_NAMES[w.kv_dtype]} KV, block {w.block_size}, ctx mean {L.mean():.0f} "
            f"[{int(L.min())}, {int(L.max())}], {len(w.steps)} distinct step(s)")


def decode_bytes(w: wl.Workload, st) -> int:
    """Bytes paged decode must move for one step: K and V of every attended token of
    every KV head (with a sliding window, the last W positions), queries in, outputs
    out, the table entries of the blocks holding those tokens, and lengths."""
    elt = w.key_cache.element_size()
    L = st.context_lens.long()
    W = int(getattr(w, "sliding_window", 0))
    start = (L - W).clamp(min=0) if W > 0 else torch.zeros_like(L)
    n = L - start
    kv = int(n.sum()) * w.num_kv_heads * w.head_dim * elt * 2
    q = st.query.numel() * st.query.element_size()
    first_blk = start // w.block_size
    last_blk = (L + w.block_size - 1) // w.block_size
    tbl = int((last_blk - first_blk).clamp(min=0).sum()) * 4 + 4 * L.numel()
    return kv + 2 * q + tbl


def step_bytes(w: wl.Workload, st) -> int:
    """Decode bytes plus the cache write (new K/V read, slots read, cache written)
    and the copy-on-write block copies (read + write, K and V)."""
    elt = w.key_cache.element_size()
    t = st.slot_mapping.numel()
    write = 2 * st.new_key.numel() * st.new_key.element_size() + 8 * t + 2 * t * w.num_kv_heads * w.head_dim * elt
    blk = w.num_kv_heads * w.block_size * w.head_dim * elt
    cow = st.cow_pairs.shape[0] * blk * 2 * 2 + st.cow_pairs.numel() * 8
    return decode_bytes(w, st) + write + cow


# ---- helpers -------------------------------------------------------------------------

def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def source_digest(kind: str = "decode") -> str:
    h = hashlib.sha256()
    for name in (DECODE_SOURCES if kind == "decode" else PREFILL_SOURCES):
        p = os.path.join(ROOT, "paged_kv_cache_90_gb300", "csrc", name)
        if os.path.exists(p):
            with open(p, "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kind: str = "decode"):
    """dram read+write bytes per launch of the decode call (kind "decode") or of the
    prefill kernel ("prefill") from the committed ncu summary for this workload, if it
    was taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", f"paged_{kind}_{workload}.md")
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m_src = re.search(r"kernel sources digest:\s*`?([0-9a-f]+)`?", text)
    m_tr = re.search(r"dram bytes per launch \(read \+ write\):\s*([0-9]+)", text)
    if not m_src or not m_tr or m_src.group(1) != source_digest(kind):
        return None
    return int(m_tr.group(1))


def smi_index(local: int) -> int:
    """nvidia-smi's index of this rank's GPU: entry `local` of CUDA_VISIBLE_DEVICES when
    that lists indices, else `local` itself."""
    vis = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")]
    return int(vis[local]) if local < len(vis) and vis[local].isdigit() else local


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
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
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, t0: float, t1: float):
        rows = []
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except Exception:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = [r for r in rows if t0 - 1.0 <= r[0] <= t1 + 1.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


def oracle_throughput(w: wl.Workload, budget_s: float, max_seqs=None):
    """Time the CPU oracle on whole sequences of the first step until ~budget_s of CPU
    work is done; returns (GB/s of needed bytes, threads, description)."""
    import oracle
    oracle.build()
    threads = len(os.sched_getaffinity(0))
    st = w.steps[0]
    kc, vc = w.key_cache.clone(), w.value_cache.clone()
    if st.cow_pairs.numel():
        oracle.copy_blocks(kc, st.cow_pairs)
        oracle.copy_blocks(vc, st.cow_pairs)
    oracle.reshape_and_cache(st.new_key, st.new_value, kc, vc, st.slot_mapping, w.k_scale, w.v_scale,
                             w.k_head_scales, w.v_head_scales)
    s_total = st.query.shape[0]
    n = s_total if max_seqs is None else max(1, min(s_total, max_seqs))
    done_bytes, elapsed, reps = 0, 0.0, 0
    while True:
        sub = wl.DecodeStep(st.query[:n], st.new_key[:n], st.new_value[:n], st.slot_mapping[:n],
                            st.block_tables[:n], st.context_lens[:n], st.cow_pairs[:0])
        t = time.perf_counter()
        oracle.paged_attention_decode(sub.query, kc, vc, sub.block_tables, sub.context_lens, w.scale,
                                      w.k_scale, w.v_scale, threads, w.sliding_window, w.k_head_scales,
                                      w.v_head_scales)
        elapsed += time.perf_counter() - t
        done_bytes += decode_bytes(w, sub)
        reps += 1
        if elapsed >= budget_s or reps >= 1000:
            break
    desc = f"fp64 C oracle decode of the first {n} of {s_total} sequences x {reps} repetition(s), {elapsed:.1f} s"
    return done_bytes / elapsed / 1e9, threads, desc


# ---- prefill: causal attention of new tokens, a tensor-core contraction ---------------

PREFILL_METRIC = "paged prefill attention: causal attention TFLOP/s (fp32 accumulate)"


def is_prefill(w: wl.Workload) -> bool:
    return w.steps[0].query_start_loc is not None


def prefill_flops(w: wl.Workload, st) -> int:
    """Multiply-adds of a prefill step, two flops each: every new token at position p
    scores p + 1 keys (D each) and sums p + 1 values (D each), in every query head."""
    qsl = st.query_start_loc.tolist()
    total = 0
    for s, L in enumerate(st.context_lens.tolist()):
        n = qsl[s + 1] - qsl[s]
        pairs = n * (L - n) + n * (n + 1) // 2     # sum over the new tokens of (p + 1)
        total += 4 * w.head_dim * w.num_heads * pairs
    return total


def oracle_prefill_throughput(w: wl.Workload, budget_s: float):
    """TFLOP/s of the CPU oracle's prefill on the first sequence(s) of the step."""
    import oracle
    oracle.build()
    threads = len(os.sched_getaffinity(0))
    st = w.steps[0]
    kc, vc = w.key_cache.clone(), w.value_cache.clone()
    oracle.reshape_and_cache(st.new_key, st.new_value, kc, vc, st.slot_mapping, w.k_scale, w.v_scale)
    qsl = st.query_start_loc
    done, elapsed, reps, n = 0, 0.0, 0, 1
    sub_qsl = qsl[:n + 1].clone()
    sub = wl.DecodeStep(st.query[:int(sub_qsl[-1])], st.new_key[:0], st.new_value[:0], st.slot_mapping[:0],
                        st.block_tables[:n], st.context_lens[:n], st.cow_pairs[:0], sub_qsl)
    while True:
        t = time.perf_counter()
        oracle.paged_attention_prefill(sub.query, kc, vc, sub.block_tables, sub.context_lens, sub.query_start_loc,
                                       w.scale, w.k_scale, w.v_scale, threads)
        elapsed += time.perf_counter() - t
        done += prefill_flops(w, sub)
        reps += 1
        if elapsed >= budget_s or reps >= 1000:
            break
    desc = (f"fp64 C oracle prefill of the first sequence ({int(sub_qsl[-1])} new tokens) x {reps} "
            f"repetition(s), {elapsed:.1f} s")
    return done / elapsed / 1e12, threads, desc


def staged_inputs(st, fields, dev):
    """A step's inputs packed into one pinned host buffer, with device views into one
    device buffer of the same layout (every field at a 256-byte aligned offset), so a
    step's host-to-device traffic is one copy: (host buffer, device buffer, device
    step, bytes per step)."""
    offs, off = [], 0
    for f in fields:
        t = getattr(st, f)
        offs.append(off)
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(max(off, 256), dtype=torch.uint8).pin_memory()
    devb = torch.empty(max(off, 256), dtype=torch.uint8, device=dev)
    views = {}
    for f, o in zip(fields, offs):
        t = getattr(st, f).contiguous()
        nb = t.numel() * t.element_size()
        host[o:o + nb].copy_(t.reshape(-1).view(torch.uint8))
        views[f] = devb[o:o + nb].view(t.dtype).view(t.shape)
    for f in DeviceStep.__dataclass_fields__:
        views.setdefault(f, None)
    return host, devb, DeviceStep(**views), sum(getattr(st, f).numel() * getattr(st, f).element_size()
                                                for f in fields)


def e2e_pipeline_ops(count: int) -> list:
    """The order in which the pipelined end-to-end loop issues its work, as (stream, op,
    step) with stream "copy" or "compute".  Ops: "h2d" (step k's inputs into device input
    buffer k mod nbuf), "record_in"/"wait_in" (the event after that copy, waited on by the
    compute stream), "call" (the step's library call, writing output buffer k mod 2),
    "record_done"/"wait_done" (the event after the call, waited on by the copy stream),
    "d2h" (the step's output back to the host).  Step k+1's input copy is issued before
    step k's call, and step k's output copy after it, so that each copy runs beside the
    neighbouring steps' kernels; the copy stream's order (input copy of k+1 behind the
    output copy of k-1, which waits for step k-1's call) keeps every buffer free when it
    is reused, for any even number of input buffers."""
    ops = [("copy", "h2d", 0), ("copy", "record_in", 0)]
    for k in range(count):
        if k + 1 < count:
            ops += [("copy", "h2d", k + 1), ("copy", "record_in", k + 1)]
        ops += [("compute", "wait_in", k), ("compute", "call", k), ("compute", "record_done", k),
                ("copy", "wait_done", k), ("copy", "d2h", k)]
    return ops


def run_prefill_gpu(args, world, rank, local, w, dw, dev, flush_l2, barrier):
    """Steps = the new tokens' cache write + causal prefill attention."""
    stream = torch.cuda.current_stream(dev)
    st = dw.steps[0]
    for _ in range(args.warmup):
        flush_l2()
        dw.run_step(0)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(smi_index(local))
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize(dev)
    n0 = binding.launch_count()
    t0 = time.time()
    for k in range(args.steps):
        flush_l2()
        a, c = ev[k]
        a.record(stream)
        dw.run_step(0)                 # cache write of the new tokens, then prefill attention
        c.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    launches = binding.launch_count() - n0
    total_ms = sum(a.elapsed_time(c) for a, c in ev)
    # the prefill kernel alone, for the roofline
    pre_steps = min(args.steps, 200)
    for k in range(pre_steps):
        flush_l2()
        a, c = ev[k]
        a.record(stream)
        binding.paged_attention_prefill(dw.out, st.query, dw.key_cache, dw.value_cache, st.block_tables,
                                        st.context_lens, st.query_start_loc, w.num_kv_heads, w.scale, w.block_size,
                                        w.max_blocks_per_seq)
        c.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    time.sleep(0.2)
    clocks.stop()
    pre_ms = sum(a.elapsed_time(c) for a, c in ev[:pre_steps]) / pre_steps
    flops = prefill_flops(w, w.steps[0])
    (max_ms,), (all_flops,) = reduce_over_ranks(world, dev, [total_ms], [flops * args.steps])
    value = all_flops / (max_ms * 1e-3) / 1e12
    # end to end: step inputs from pinned host memory, output back
    fields = ("query", "new_key", "new_value", "slot_mapping", "block_tables", "context_lens", "cow_pairs",
              "query_start_loc")
    hbuf, dbuf, di, h2d = staged_inputs(w.steps[0], fields, dev)
    out_host = torch.empty(dw.out.shape, dtype=dw.out.dtype).pin_memory()
    d2h = out_host.numel() * out_host.element_size()
    e_ms, e_steps = 0.0, max(5, min(args.steps, 50))
    for k in range(e_steps + 3):
        flush_l2()
        a, c = ev[k % len(ev)]
        a.record(stream)
        dbuf.copy_(hbuf, non_blocking=True)   # every input of the step, one copy
        run_decode_step(w, dw.key_cache, dw.value_cache, di, dw.out)
        out_host.copy_(dw.out, non_blocking=True)
        c.record(stream)
        c.synchronize()
        if k >= 3:
            e_ms += a.elapsed_time(c)
    (e_ms,), (e2e_flops, launches) = reduce_over_ranks(world, dev, [e_ms], [flops * e_steps, launches])
    e2e = e2e_flops / (e_ms * 1e-3) / 1e12
    if rank != 0:
        return 0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, peak_kind = float(json.load(f)["bf16_tflops"]), "measured (bf16 dense, burst)"
    except Exception:
        peak, peak_kind = 1900.0, "fallback"
    achieved = flops / (pre_ms * 1e-3) / 1e12
    cpu_base = None
    if world == 1 and not args.no_cpu_baseline:
        g, threads, desc = oracle_prefill_throughput(w, args.cpu_budget)
        cpu_base = {"value": round(g, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc}
    line = {
        "metric": PREFILL_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": describe_workload(w, args.workload),
                   "new_tokens": int(st.query.shape[0]), "flops_per_step": flops,
                   "l2": "flushed between steps (256 MiB write + 256 MiB read, untimed)", "accumulate": "f32",
                   "prefill_us": round(pre_ms * 1e3, 2), "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": profiled_traffic(args.workload, "prefill"),
                     "kernel": ("paged_prefill_kernel (mma.sync bf16)" if args.prefill_kernel == "mma_sync" else
                                "paged_prefill_tc_kernel (tcgen05, accumulators in tensor memory)"),
                     "peak_kind": peak_kind},
        "cpu_baseline": cpu_base,
        "e2e": {"value": round(e2e, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(t0, t1),
    }
    print(json.dumps(line), flush=True)
    return 0


# ---- the two arms --------------------------------------------------------------------

def reduce_over_ranks(world, dev, maxes, sums):
    """Whole-job figures of a run on `world` ranks: the max over ranks of each entry of
    `maxes` (times) and the sum of each entry of `sums` (work done, launches); every
    rank calls it at the same point.  One rank: the values as given."""
    maxes, sums = [float(x) for x in maxes], [float(x) for x in sums]
    if world == 1:
        return maxes, sums
    import torch.distributed as dist
    m = torch.tensor(maxes, dtype=torch.float64, device=dev)
    t = torch.tensor(sums, dtype=torch.float64, device=dev)
    dist.all_reduce(m, op=dist.ReduceOp.MAX)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return m.cpu().tolist(), t.cpu().tolist()


def init_dist(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl != "reference" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    w = make_workload(args.workload)
    if is_prefill(w):
        vals = []
        for i in range(args.warmup + args.steps):
            g, threads, desc = oracle_prefill_throughput(w, 120.0 / (args.warmup + args.steps))
            if i >= args.warmup:
                vals.append(g)
        value = statistics.median(vals)
        line = {"impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6), "unit": "TFLOP/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": describe_workload(w, args.workload), "l2": "n/a (host)"},
                "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                 "sample": "each step: " + desc},
                "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0
    steps = args.warmup + args.steps
    # calibrate: one sequence, then size the per-step sample to fit ~2 minutes overall
    gbs1, threads, _ = oracle_throughput(w, 0.0, max_seqs=1)
    per_seq = decode_bytes(w, w.steps[0]) / w.num_seqs / (gbs1 * 1e9)
    target = max(0.05, min(2.0, 120.0 / steps))
    n = max(1, min(w.num_seqs, int(target / max(per_seq, 1e-9))))
    vals, total = [], 0.0
    for i in range(steps):
        g, threads, desc = oracle_throughput(w, 0.0, max_seqs=n)
        if i >= args.warmup:
            vals.append(g)
    value = statistics.median(vals)
    sample = f"each step: fp64 C oracle decode of the first {n} of {w.num_seqs} sequences ({args.workload})"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe_workload(w, args.workload), "l2": "n/a (host)"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args, world, rank, local):
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the reference arm is --impl reference)")
    dev = torch.device("cuda", local)
    binding.load_library()
    binding.set_option("decode_kernel", {"auto": 0, "core": 1, "tensor": 2}[args.decode_kernel])
    binding.set_option("prefill_kernel", {"auto": 0, "mma_sync": 1, "tcgen05": 2}[args.prefill_kernel])
    w = make_workload(args.workload, rank)
    dw = DeviceWorkload(w, dev)
    nsteps = len(w.steps)
    ws_bytes = binding.decode_workspace_bytes(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                              w.max_blocks_per_seq)
    if ws_bytes:
        binding.reserve_workspace(ws_bytes)
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_sink)

    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    if is_prefill(w):
        return run_prefill_gpu(args, world, rank, local, w, dw, dev, flush_l2, barrier)

    # ---- device-resident timing (value) ----
    # Steps that read more than twice the L2 run back to back (their K/V are streamed with
    # an evict-first policy, so a step does not find the previous one's data in L2);
    # smaller ones, and steps that share blocks between sequences, flush the L2 between
    # steps outside the timed events.
    try:
        l2_bytes = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    except Exception:
        l2_bytes = 129 << 20
    joint = STEP_MODES[args.step_mode]
    if args.step_mode == "fused":
        binding.set_option("fused_append", 2)   # the write inside the decode kernel
    step0_bytes = decode_bytes(w, w.steps[0])
    back_to_back = step0_bytes > 2 * l2_bytes and not any(st.cow_pairs.numel() for st in w.steps)
    for i in range(args.warmup):
        flush_l2()
        dw.run_step(i % nsteps, joint=joint)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(smi_index(local))
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize(dev)
    def decode_call(k):
        st = dw.steps[k % nsteps]
        binding.paged_attention_decode(dw.out, st.query, dw.key_cache, dw.value_cache, st.block_tables,
                                       st.context_lens, w.num_kv_heads, w.scale, w.block_size,
                                       w.max_blocks_per_seq, w.k_scale, w.v_scale, None, w.sliding_window,
                                       dw.k_head_scales, dw.v_head_scales)

    def time_flushed(fn, count):
        """Per-call times (ms), the L2 flushed before each call, outside its events."""
        for k in range(count):
            flush_l2()
            a, _, c = ev[k]
            a.record(stream)
            fn(k)
            c.record(stream)
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(c) for a, _, c in ev[:count]]

    def time_back_to_back(fn, count):
        """Total time (ms) of `count` calls queued back to back between two events.  A
        device-side spin queued before the first event (about 0.25 ms per call, at most
        16 ms) holds the stream while the host queues the calls, so that the GPU does
        not wait inside the timed region for the host's first launches (a benchmark
        harness's "blocking kernel"); the events bracket exactly the `count` calls."""
        a, _, c = ev[0]
        torch.cuda._sleep(int(min(count, 64) * 5.0e5))
        a.record(stream)
        for k in range(count):
            fn(k)
        c.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(c)

    def step_call(k):
        dw.run_step(k % nsteps, joint=joint)  # CoW copies, then the cache write and the decode

    n0 = binding.launch_count()
    t0 = time.time()
    if back_to_back:
        total_ms = time_back_to_back(step_call, args.steps)
    else:
        total_ms = sum(time_flushed(step_call, args.steps))
    torch.cuda.synchronize(dev)
    t1 = time.time()
    launches = binding.launch_count() - n0
    # the decode kernels alone (main + merge), for the roofline: the same calls on the
    # same resident caches, timed the same way
    dec_steps = min(args.steps, 500)
    if back_to_back:
        dec_ms = [time_back_to_back(decode_call, dec_steps) / dec_steps]
        flushed_step_ms = statistics.mean(time_flushed(step_call, min(args.steps, 500)))
        flushed_dec_ms = statistics.mean(time_flushed(decode_call, dec_steps))
    else:
        dec_ms = time_flushed(decode_call, dec_steps)
    torch.cuda.synchronize(dev)
    barrier()
    time.sleep(0.2)
    clocks.stop()
    flags = binding.read_device_errors()
    if flags:
        raise SystemExit(f"device error word 0x{flags:x} during the bench")

    bytes_steps = [step_bytes(w, w.steps[k % nsteps]) for k in range(args.steps)]
    dec_bytes = [float(statistics.mean(decode_bytes(w, w.steps[k % nsteps]) for k in range(dec_steps)))]
    (max_ms,), (all_bytes,) = reduce_over_ranks(world, dev, [total_ms], [sum(bytes_steps)])
    value = all_bytes / (max_ms * 1e-3) / 1e9

    # ---- end to end through the public API from pinned host buffers (e2e) ----
    fields = ("query", "new_key", "new_value", "slot_mapping", "block_tables", "context_lens", "cow_pairs")
    e2e_steps = max(10, min(args.steps, 200))
    if back_to_back:
        # Pipelined like a serving loop: each step's inputs go in, and its output comes
        # back, on a copy stream while the neighbouring steps compute.  An even number
        # (at least two) of device input buffers and two output buffers, so that no copy
        # overwrites what a step still reads or writes.
        nbuf = nsteps if nsteps % 2 == 0 else 2 * nsteps
        staged = [staged_inputs(w.steps[j % nsteps], fields, dev) for j in range(nbuf)]
        outs = [dw.out, torch.empty_like(dw.out)]
    else:
        staged = [staged_inputs(st, fields, dev) for st in w.steps]
        outs = [dw.out]
    out_host = torch.empty(dw.out.shape, dtype=dw.out.dtype).pin_memory()
    h2d = staged[0][3]
    d2h = out_host.numel() * out_host.element_size()
    for k in range(3):
        i = k % nsteps
        staged[i][1].copy_(staged[i][0], non_blocking=True)
        run_decode_step(w, dw.key_cache, dw.value_cache, staged[i][2], dw.out, None, joint, dw.k_head_scales,
                        dw.v_head_scales)
        out_host.copy_(dw.out, non_blocking=True)
    torch.cuda.synchronize(dev)
    # each staged step's call marshalled once (the library's prepared form of the call)
    e2e_steps_fn = [prepare_step(w, dw.key_cache, dw.value_cache, staged[j][2], outs[j % len(outs)], None, joint,
                                 dw.k_head_scales, dw.v_head_scales) for j in range(len(staged))]

    if back_to_back:
        xs = torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(e2e_steps)]
        ev_done = [torch.cuda.Event() for _ in range(e2e_steps)]
        ev_last = torch.cuda.Event()

        def pipelined(count, start=None):
            """Issue e2e_pipeline_ops(count) on the compute and copy streams."""
            if start is not None:
                xs.wait_event(start)
            for _, op, k in e2e_pipeline_ops(count):
                if op == "h2d":
                    with torch.cuda.stream(xs):
                        staged[k % nbuf][1].copy_(staged[k % nbuf][0], non_blocking=True)
                elif op == "record_in":
                    ev_in[k].record(xs)
                elif op == "wait_in":
                    stream.wait_event(ev_in[k])
                elif op == "call":
                    e2e_steps_fn[k % nbuf]()
                elif op == "record_done":
                    ev_done[k].record(stream)
                elif op == "wait_done":
                    xs.wait_event(ev_done[k])
                else:   # d2h
                    with torch.cuda.stream(xs):
                        out_host.copy_(outs[k % 2], non_blocking=True)
            ev_last.record(xs)
            stream.wait_event(ev_last)

        pipelined(min(3, e2e_steps))
        torch.cuda.synchronize(dev)
        a, _, c = ev[0]
        torch.cuda._sleep(int(min(e2e_steps, 64) * 5.0e5))   # as in time_back_to_back
        a.record(stream)
        pipelined(e2e_steps, start=a)
        c.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = a.elapsed_time(c)
    else:
        def e2e_call(k):
            i = k % nsteps
            staged[i][1].copy_(staged[i][0], non_blocking=True)   # every input of the step, one copy
            e2e_steps_fn[i]()
            out_host.copy_(dw.out, non_blocking=True)             # and its result back
        e_ms = 0.0
        for k in range(e2e_steps):
            flush_l2()
            a, _, c = ev[k % len(ev)]
            a.record(stream)
            e2e_call(k)
            c.record(stream)
            c.synchronize()
            e_ms += a.elapsed_time(c)
    e2e_bytes = sum(step_bytes(w, w.steps[k % nsteps]) for k in range(e2e_steps))
    (e_ms,), (e2e_bytes, launches) = reduce_over_ranks(world, dev, [e_ms], [e2e_bytes, launches])
    e2e_value = e2e_bytes / (e_ms * 1e-3) / 1e9

    if rank != 0:
        return 0
    peak, peak_kind = load_peaks()
    dec_avg_s = sum(dec_ms) / len(dec_ms) * 1e-3
    achieved = (sum(dec_bytes) / len(dec_bytes)) / dec_avg_s / 1e9
    traffic = profiled_traffic(args.workload)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "kernel": "paged_attention_decode (main + log-sum-exp reduce)", "peak_kind": peak_kind}
    cpu_base = None
    if world == 1 and not args.no_cpu_baseline:
        g, threads, desc = oracle_throughput(w, args.cpu_budget)
        cpu_base = {"value": round(g, 4), "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.DTYPE_NAMES[w.kv_dtype], "data": "synthetic",
        "config": {"workload": describe_workload(w, args.workload),
                   "l2": (f"not flushed: steps back to back, each reading {step0_bytes / 1e6:.0f} MB, over twice the "
                          f"{l2_bytes / 2**20:.0f} MiB L2 (K/V streamed evict-first)" if back_to_back else
                          "flushed between steps (256 MiB write + 256 MiB read, untimed)"),
                   "accumulate": "f32", "step_mode": args.step_mode,
                   "us_per_step": round(max_ms / args.steps * 1e3, 2),
                   "decode_us": round(dec_avg_s * 1e6, 2),
                   **({"flushed_step_us": round(flushed_step_ms * 1e3, 2),
                       "flushed_decode_us": round(flushed_dec_ms * 1e3, 2),
                       "flushed_step_gbs": round(step_bytes(w, w.steps[0]) / (flushed_step_ms * 1e-3) / 1e9, 1)}
                      if back_to_back else {}),
                   "tokens_per_s": round(w.num_seqs * world / (max_ms / args.steps * 1e-3), 1),
                   "pct_of_8TBps": round(value / 8000 * 100, 2), "parallelism": f"replicas x{world}"},
        "roofline": roofline,
        "cpu_baseline": cpu_base,
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(t0, t1),
    }
    print(json.dumps(line), flush=True)
    return 0


STEP_MODES = {"fused": "fused", "joint": True, "split": False}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--workload", default="llama3_8b_decode",
                    help="llama3_8b_decode, long_context[_bs32], shared_prefix_cow, "
                         "continuous_batching_bs{8,16,32}_{bf16,e4m3}[_headscales], sliding_window[_bs32], "
                         "mha_decode, chunked_prefill, prefill_<N>x<T>, tiny")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle CPU time")
    ap.add_argument("--decode-kernel", choices=["auto", "tensor", "core"], default="auto",
                    help="decode kernel: chosen by the library, tensor-core, or CUDA-core")
    ap.add_argument("--prefill-kernel", choices=["auto", "tcgen05", "mma_sync"], default="auto",
                    help="prefill kernel: chosen by the library (tcgen05 where supported), or forced")
    ap.add_argument("--step-mode", choices=sorted(STEP_MODES), default="joint",
                    help="how a decode step's cache write is issued: joint (write + dependent decode "
                         "launch in one call), fused (the write inside the decode kernel), or split "
                         "(two calls)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("at least 3 warm-up steps")
    world, rank, local = init_dist(args)
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        return run_gpu(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
