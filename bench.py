"""Decode-step benchmark of the paged KV-cache path on GB300.

One step = one pass of the whole hot path over one batch: zero the blocks
the step freshly allocates, write each sequence's new token through its
slot, then paged decode attention (with the split-KV reduce when the
partitioning splits sequences).  Workload: Llama-8B-shaped GQA decode
(batch 64, 32 q / 8 kv heads, head_dim 128, bf16 KV, seq_lens uniform in
[512, 4096], 16-token blocks scattered over a pool 20% larger than needed).

Prints one JSON line.  --impl reference times the fp64 CPU oracle on the
same workload instead (a bounded sample of sequences per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import platform
import os
import re
import statistics
import subprocess
import sys
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = ("paged decode attention KV-read GB/s (% of GB300 HBM peak); "
          "seq-steps/sec")
L2_BYTES = 126 * 2**20
SEQ_LENS = {"llama8b_gqa": "uniform [512, 4096]",
            "prefix_shared": "1024 shared + uniform [32, 512]",
            "long_context": "uniform [32768, 131072]",
            "fp8_recycle": "uniform [1024, 8192]",
            "tiny_mha": "{1, 17, 33, 64}"}
FALLBACK_HBM_GBS = 6800.0
PROFILE = ROOT / "profiles" / "paged_decode_kernel_llama8b_gqa.md"
# decode workloads with a committed ncu summary of the decode kernel
# GPU clock cycles of the sleep that precedes a timed loop (about 2 ms):
# long enough for the host to queue a few dozen steps.
PRIME_CYCLES = 4_000_000

DECODE_PROFILES = {
    "llama8b_gqa": PROFILE,
    "long_context": ROOT / "profiles" / "paged_decode_kernel_long_context.md",
    "fp8_recycle": ROOT / "profiles" / "paged_decode_kernel_fp8_recycle.md",
    # (workload, partition tokens) where a partition length has its own capture
    ("long_context", 512): ROOT / "profiles" / "paged_decode_kernel_long_context_p512.md",
}
KERNEL_SOURCES = ["paged_kv_cache_48_gb300/csrc/attention_decode.cu",
                  "paged_kv_cache_48_gb300/csrc/pkv_device.cuh",
                  "paged_kv_cache_48_gb300/csrc/e4m3_encode.cuh"]
# prefill workloads with a committed ncu summary of the prefill kernel
PREFILL_PROFILES = {w: ROOT / "profiles" / f"paged_prefill_kernel_{w}.md"
                    for w in ("chunked_prefill_8k", "chunked_prefill_8k_fp8", "prefill_8k")}
PREFILL_SOURCES = ["paged_kv_cache_48_gb300/csrc/attention_prefill.cu",
                   "paged_kv_cache_48_gb300/csrc/tcgen05.cuh",
                   "paged_kv_cache_48_gb300/csrc/pkv_device.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--partition-tokens", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-seqs", type=int, default=16)
    ap.add_argument("--kernel", default="decode",
                    choices=["decode", "zero_blocks", "copy_blocks", "swap",
                             "input_prep", "prefill", "cascade"],
                    help="decode: the decode step (headline); the others time "
                         "the block-movement entry points on the workload's "
                         "pool")
    ap.add_argument("--two-call-step", action="store_true",
                    help="decode step as paged_kv_zero_and_write + "
                         "paged_attention_decode even where the step's only "
                         "writes are the new tokens (default there: one "
                         "paged_attention_decode_step call)")
    ap.add_argument("--graph", action="store_true",
                    help="replay the decode step as one captured CUDA graph")
    ap.add_argument("--workload", default="llama8b_gqa",
                    choices=["llama8b_gqa", "prefix_shared", "long_context",
                             "fp8_recycle", "tiny_mha", "prefill_8k",
                             "chunked_prefill_8k", "chunked_prefill_8k_fp8"],
                    help="decode workload (the headline metric is quoted on "
                         "llama8b_gqa, the others are reported for context); "
                         "with --kernel prefill, prefill_8k, "
                         "chunked_prefill_8k or chunked_prefill_8k_fp8")
    return ap.parse_args()


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, device=None):
    """Element-wise max of per-rank timings over the process group (the
    slowest rank sets the whole-job time); identity without one."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or \
            dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64,
                     device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_gbs(world: int, bytes_per_rank: int, ms_per_step: float) -> float:
    """Aggregate throughput: every rank moves bytes_per_rank per step and
    the job's step time is the slowest rank's."""
    return world * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


def kernel_sha(sources=None) -> str:
    h = hashlib.sha256()
    for rel in sources or KERNEL_SOURCES:
        h.update((ROOT / rel).read_bytes())
    return h.hexdigest()[:16]


def measured_tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s): the burst figure, for a kernel
    timed on its own."""
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return float(json.loads(p.read_text())["bf16_tflops"]), "measured"
        except Exception:
            pass
    return 1900.0, "fallback"


def measured_peak():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return float(json.loads(p.read_text())["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(profile=None, sources=None):
    """DRAM bytes per launch of a kernel from its committed ncu summary, if
    the summary was taken on the current kernel source (the decode kernel by
    default)."""
    profile = profile or PROFILE
    if not profile.exists():
        return None
    text = profile.read_text()
    sha = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    val = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not sha or not val or sha.group(1) != kernel_sha(sources):
        return None
    return float(val.group(1))


def packed(tensors, device=None, pinned=False):
    """One byte buffer holding copies of `tensors` at 256-byte aligned
    offsets, and a view of it per tensor (same dtype and shape): a step's
    inputs then move with one copy."""
    import torch
    offs, n = [], 0
    for t in tensors:
        offs.append(n)
        n += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(max(n, 1), dtype=torch.uint8, device=device)
    if pinned:
        buf = buf.pin_memory()
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
             for o, t in zip(offs, tensors)]
    for v, t in zip(views, tensors):
        v.copy_(t)
    return buf, views


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() in ("active", "0x1", "1"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_oracle_step(W, kc, vc, seqs, n_threads=0):
    """The oracle's decode step on the sequences `seqs` (all heads)."""
    import oracle
    o = oracle.load()
    dt = oracle.DTYPE_BF16 if W.kv_dtype == "bf16" else oracle.DTYPE_FP8_E4M3
    o.zero_blocks(kc, vc, W.block_bytes, W.fresh_blocks)
    o.kv_write(kc, vc, dt, W.block_size, W.num_kv_heads, W.head_dim,
               W.k_scale, W.v_scale, W.step_k, W.step_v, W.step_slots)
    pairs = np.array([(b, h) for b in seqs for h in range(W.num_heads)],
                     dtype=np.int32)
    out, err = o.attention_decode(W.q, kc, vc, dt, W.k_scale, W.v_scale,
                                  W.block_size, W.num_kv_heads, W.head_dim,
                                  W.block_tables, W.seq_lens, W.scale,
                                  pairs=pairs, n_threads=n_threads)
    assert err == 0
    return out


def oracle_setup(W):
    import oracle
    o = oracle.load()
    dt = oracle.DTYPE_BF16 if W.kv_dtype == "bf16" else oracle.DTYPE_FP8_E4M3
    kc, vc = W.init_key.copy(), W.init_value.copy()
    o.kv_write(kc, vc, dt, W.block_size, W.num_kv_heads, W.head_dim,
               W.k_scale, W.v_scale, W.hist_k, W.hist_v, W.hist_slots)
    return kc, vc, o.num_threads()


def time_cpu_oracle(W, n_seqs, steps, warmup=0, n_threads=0):
    """Seconds per oracle step on the first n_seqs sequences; returns
    (value GB/s, seq-steps/s, seconds per step, threads, bytes).
    n_threads = 0 uses every host core."""
    import oracle
    kc, vc, _ = oracle_setup(W)
    threads = oracle.load().num_threads(n_threads)
    seqs = list(range(min(n_seqs, W.batch)))
    kv_bytes = int(W.seq_lens[seqs].astype(np.int64).sum()) * \
        W.num_kv_heads * W.head_dim * 2 * W.elem_bytes
    for _ in range(warmup):
        cpu_oracle_step(W, kc, vc, seqs, n_threads)
    t0 = time.perf_counter()
    for _ in range(steps):
        cpu_oracle_step(W, kc, vc, seqs, n_threads)
    dt = (time.perf_counter() - t0) / max(1, steps)
    return kv_bytes / dt / 1e9, len(seqs) / dt, dt, threads, kv_bytes


def host_cpu_model():
    """The host CPU as /proc/cpuinfo names it (x86 'model name', or the Arm
    implementer / part codes), with the number of online cores."""
    name = None
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for line in info.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "model name":
                name = v.strip()
                break
        if name is None:
            fields = {}
            for line in info.splitlines():
                k, _, v = line.partition(":")
                fields.setdefault(k.strip(), v.strip())
            if "CPU part" in fields:
                name = (f"arm implementer {fields.get('CPU implementer', '?')} "
                        f"part {fields['CPU part']}")
    except OSError:
        pass
    return f"{name or platform.machine()}, {os.cpu_count()} cores"


def one_core_baseline(W, n_seqs):
    """The same oracle step on one host core (a single step of a smaller
    sample: a quarter of the sequences, at least one)."""
    gbs, _, dt, _, kvb = time_cpu_oracle(W, max(1, n_seqs // 4), steps=1,
                                         warmup=0, n_threads=1)
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1,
            "sample": f"first {max(1, min(n_seqs // 4, W.batch))} sequences, "
                      f"1 step ({kvb / 1e6:.1f} MB of KV)"}


def run_reference(args):
    world, rank, _ = dist_info()
    if rank != 0:
        return 0
    from paged_kv_cache_48_gb300 import workload as wl
    W = wl.CONFIGS[args.workload]()
    gbs, sps, dt, threads, kvb = time_cpu_oracle(W, args.cpu_sample_seqs,
                                                 args.steps, args.warmup)
    peak, kind = measured_peak()
    sample = (f"first {min(args.cpu_sample_seqs, W.batch)} of {W.batch} "
              f"sequences, all heads, per step ({kvb / 1e6:.1f} MB of KV)")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4),
        "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "seq_steps_per_s": round(sps, 3),
        "pct_of_hbm_peak": round(100 * gbs / peak, 4),
        "config": {"workload": W.name, "batch": W.batch,
                   "num_heads": W.num_heads, "num_kv_heads": W.num_kv_heads,
                   "head_dim": W.head_dim, "block_size": W.block_size,
                   "seq_lens": SEQ_LENS[W.name], "kv_dtype": W.kv_dtype,
                   "l2": "host oracle (no L2 flush)"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s",
                         "cores": threads, "kind": "oracle",
                         "sample": sample, "cpu": host_cpu_model(),
                         "one_core": one_core_baseline(W, args.cpu_sample_seqs)},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _replay(graph, ev, stream):
    """One graph replay; with `ev`, the pair brackets the whole step."""
    if ev is not None:
        ev[0].record(stream)
    graph.replay()
    if ev is not None:
        ev[1].record(stream)


def run_ours(args):
    import torch
    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from paged_kv_cache_48_gb300 import (PagedKVCache, paged_attention_decode,
                                         paged_attention_decode_step,
                                         paged_attention_partition_tokens,
                                         paged_attention_workspace_bytes,
                                         paged_kv_write, paged_kv_zero_and_write,
                                         pkv_check)
    from paged_kv_cache_48_gb300 import workload as wl

    make = wl.CONFIGS[args.workload]
    W = make() if rank == 0 else make(seed=1000 + rank)
    fp8 = W.kv_dtype == "fp8_e4m3"
    elt = torch.uint8 if fp8 else torch.bfloat16
    shape = (W.num_blocks, 16, W.num_kv_heads, W.head_dim)
    kc = torch.from_numpy(W.init_key).view(elt).reshape(shape).to(dev)
    vc = torch.from_numpy(W.init_value).view(elt).reshape(shape).to(dev)
    cache = PagedKVCache(kc, vc, W.kv_dtype, W.k_scale, W.v_scale)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16)
    chunk = 1 << 18
    for s0 in range(0, W.hist_slots.size, chunk):
        s1 = min(W.hist_slots.size, s0 + chunk)
        paged_kv_write(bf(W.hist_k[s0:s1]).to(dev), bf(W.hist_v[s0:s1]).to(dev),
                       torch.from_numpy(W.hist_slots[s0:s1]).to(dev), cache)
    q = bf(W.q).to(dev)
    tables = torch.from_numpy(W.block_tables).to(dev)
    lens = torch.from_numpy(W.seq_lens).to(dev)
    new_tokens = None if args.two_call_step else W.new_token_tail()
    if new_tokens is not None and not np.all(np.diff(new_tokens[1]) == 1):
        # Several new tokens a sequence (the fp8 workload rewrites each
        # sequence's last four or five blocks): one call was measured about
        # 1% slower than the separate write launch there, since the decode
        # warps' encoding sits on their streams' critical path.
        new_tokens = None
    if new_tokens is not None:
        # every sequence's one write is its new token, and the fresh blocks
        # are the blocks those tokens open: the step is one
        # paged_attention_decode_step call (the write inside the decode
        # kernel)
        rows, _ = new_tokens
        sk, sv = bf(W.step_k[rows]).to(dev), bf(W.step_v[rows]).to(dev)
        slots = torch.empty(0, dtype=torch.int32, device=dev)
        fresh = np.zeros(0, dtype=np.int32)
    else:
        sk, sv = bf(W.step_k).to(dev), bf(W.step_v).to(dev)
        slots = torch.from_numpy(W.step_slots).to(dev)
        fresh = W.fresh_blocks
    # the step's device inputs live in one buffer (one copy moves them)
    d_main, (q, tables, lens, sk, sv, slots) = packed((q, tables, lens, sk, sv, slots), dev)
    max_len = int(W.max_blocks * 16)  # host bound: the table width
    pt = paged_attention_partition_tokens(W.batch, W.num_heads,
                                          W.num_kv_heads, max_len,
                                          args.partition_tokens)
    ws_bytes = paged_attention_workspace_bytes(W.batch, W.num_heads,
                                               W.num_kv_heads, W.head_dim,
                                               max_len, args.partition_tokens)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    # zeroing + write (one launch, unless the decode kernel writes the new
    # tokens), the decode kernel and the merge of split sequences (when a
    # sequence can be split)
    split = -(-max_len // pt) > 1
    launches_per_step = (0 if new_tokens is not None else 1) + 1 + (1 if split else 0)
    kv_bytes = W.kv_read_bytes()
    # Workloads whose KV fits in twice the L2 are timed step by step with an
    # L2 flush (a 512 MiB write) between steps, outside the timed events.
    flush = kv_bytes < 2 * L2_BYTES
    scrub = torch.empty(512 * 2**20, dtype=torch.uint8, device=dev) if flush else None

    def step(ev=None, bufs=None):
        qq, tt, ll, kk, vv, ss, oo = bufs or (q, tables, lens, sk, sv, slots, out)
        if new_tokens is not None:
            # the new tokens' write, then attention, in the decode kernel
            if ev is not None:
                ev[0].record(stream)
            paged_attention_decode_step(qq, kk, vv, cache, tt, ll, W.scale, max_len,
                                        out=oo, partition_tokens=args.partition_tokens,
                                        workspace=ws)
            if ev is not None:
                ev[1].record(stream)
            return
        if fresh.size or ss.numel():
            # zeroing of the step's fresh blocks and the write of its
            # tokens, in one launch
            paged_kv_zero_and_write(kk, vv, ss, cache, fresh)
        if ev is not None:
            ev[0].record(stream)
        paged_attention_decode(qq, cache, tt, ll, W.scale, max_len,
                               out=oo, partition_tokens=args.partition_tokens,
                               workspace=ws)
        if ev is not None:
            ev[1].record(stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def timed_loop(n, body):
        """Device time of n calls of body(): one event pair around the loop,
        or per call with an L2 flush in between when flushing.  The GPU
        first runs a sleep that touches no memory, outside the events, so
        that the host has queued the first steps when the start event is
        reached: the device time then holds the steps, not the host's
        latency to its first launch (which is several steps' worth when K
        is small)."""
        if not flush:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(PRIME_CYCLES)
            a.record(stream)
            for i in range(n):
                body(i)
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b)
        pairs = [(torch.cuda.Event(enable_timing=True),
                  torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            scrub.zero_()
            pairs[i][0].record(stream)
            body(i)
            pairs[i][1].record(stream)
        torch.cuda.synchronize()
        return sum(x.elapsed_time(y) for x, y in pairs)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, detail = pkv_check()
    if st != 0:
        raise RuntimeError(f"device error {st} at {detail} during warm-up")

    run_step = step
    if args.graph:
        # The whole step as one CUDA graph (zeroing ids ride in the captured
        # launch parameters), replayed once per step.
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                step()
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        run_step = lambda ev=None: _replay(graph, ev, stream)
        for _ in range(args.warmup):
            run_step()
        torch.cuda.synchronize()

    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with ClockSampler(dev.index) as clocks:
        barrier()
        torch.cuda.synchronize()
        # the headline: K steps with events only around the loop (an event
        # between two kernels would cut their programmatic launch overlap)
        elapsed_ms = timed_loop(K, lambda i: run_step())
        barrier()
        warm_ms = None
        if flush:
            # The same steps without the flush (KV left in L2 by the
            # previous step), reported beside the cold headline.  Each step
            # is timed on its own as in the cold loop; a GPU sleep that
            # touches no memory takes the flush's place, so the host has
            # queued the step before the GPU reaches it.
            torch.cuda.synchronize()
            wpairs = [(torch.cuda.Event(enable_timing=True),
                       torch.cuda.Event(enable_timing=True)) for _ in range(K)]
            for i in range(K):
                torch.cuda._sleep(100000)
                wpairs[i][0].record(stream)
                run_step()
                wpairs[i][1].record(stream)
            torch.cuda.synchronize()
            warm_ms = sum(x.elapsed_time(y) for x, y in wpairs)
            barrier()
        # the dominant launch's duration for the roofline: the same K steps
        # again with an event pair around each decode call (+ merge)
        torch.cuda.synchronize()
        timed_loop(K, lambda i: run_step(evs[i]))
        barrier()

        # End to end: every step uploads all of its inputs from pinned host
        # memory and reads its output back.  As a serving loop does, the
        # copies run on their own streams into two alternating device
        # buffer sets, so step i's upload overlaps step i-1's compute and
        # step i's download overlaps step i+1's compute.
        ins = (q, tables, lens, sk, sv, slots)
        h_pack, h_in = packed([t.cpu() for t in ins], pinned=True)
        h_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        packs = [packed(ins, dev) for _ in range(2)]
        sets = [views + [torch.empty_like(out)] for _, views in packs]
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_back = [torch.cuda.Event() for _ in range(2)]
        h2d = sum(h.numel() * h.element_size() for h in h_in) + fresh.nbytes
        d2h = h_out[0].numel() * h_out[0].element_size()
        K2 = max(10, K // 2)   # timed end-to-end steps
        E2E_WARM = 4           # untimed: both buffer sets used twice

        def e2e_step(i):
            b = i % 2
            if i >= 2:
                up.wait_event(ev_back[b])      # set b free: step i-2 read back
            with torch.cuda.stream(up):
                packs[b][0].copy_(h_pack, non_blocking=True)  # all inputs, one copy
                ev_in[b].record(up)
            stream.wait_event(ev_in[b])
            if args.graph:
                # the captured graph reads and writes the fixed buffers
                d_main.copy_(packs[b][0], non_blocking=True)
                run_step()
                sets[b][6].copy_(out, non_blocking=True)
            else:
                run_step(bufs=sets[b])
            ev_done[b].record(stream)
            down.wait_event(ev_done[b])
            with torch.cuda.stream(down):
                h_out[b].copy_(sets[b][6], non_blocking=True)
                ev_back[b].record(down)

        for i in range(E2E_WARM):
            e2e_step(i)
        stream.wait_stream(down)
        barrier()
        torch.cuda.synchronize()
        e_a = torch.cuda.Event(enable_timing=True)
        e_b = torch.cuda.Event(enable_timing=True)
        e_a.record(stream)
        for i in range(E2E_WARM, E2E_WARM + K2):
            e2e_step(i)
        stream.wait_stream(down)               # the last read-back is inside
        e_b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e_a.elapsed_time(e_b)
        barrier()
    st, detail = pkv_check()
    if st != 0:
        raise RuntimeError(f"device error {st} at {detail} in the timed region")

    # per-step event pairs: the decode call alone, or the whole replayed
    # step with --graph
    attn_ms = statistics.fmean(a.elapsed_time(b) for a, b in evs)
    elapsed_ms, e2e_ms, attn_ms = max_over_ranks([elapsed_ms, e2e_ms, attn_ms],
                                                 device=dev)
    if warm_ms is not None:
        warm_ms = max_over_ranks([warm_ms], device=dev)[0]

    ms_per_step = elapsed_ms / K
    value = whole_job_gbs(world, kv_bytes, ms_per_step)
    e2e_value = whole_job_gbs(world, kv_bytes, e2e_ms / K2)
    peak, peak_kind = measured_peak()
    # The dominant launches are the decode kernel and its merge.  When a
    # step is one paged_attention_decode_step call (eager), the headline
    # loop holds nothing else, so its time per step is their average
    # duration back to back; otherwise (a separate write launch in the step,
    # or a replayed graph) the per-call event pairs of the second loop,
    # which also cut the programmatic overlap between calls.
    pair_only = new_tokens is not None and not args.graph
    roof_ms = ms_per_step if pair_only else attn_ms
    achieved = kv_bytes / (roof_ms * 1e-3) / 1e9
    prof = DECODE_PROFILES.get((args.workload, pt), DECODE_PROFILES.get(args.workload))
    traffic = profiled_traffic(prof) if prof is not None else None
    l2 = (f"L2 flushed between steps ({kv_bytes / 1e6:.1f} MB of KV per step)"
          if flush else
          f"inputs larger than L2 ({kv_bytes / 1e9:.2f} GB of KV read per step, "
          "L2 126 MB)")

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3 KV, f16 mma, fp32 accumulate" if fp8 else "bf16",
        "data": "synthetic",
        "pct_of_hbm_peak": round(100 * value / world / peak, 2),
        "seq_steps_per_s": round(world * W.batch / (ms_per_step * 1e-3), 1),
        "attention_seq_steps_per_s": round(world * W.batch / (attn_ms * 1e-3), 1),
        "config": {"workload": W.name, "batch": W.batch,
                   "num_heads": W.num_heads, "num_kv_heads": W.num_kv_heads,
                   "head_dim": W.head_dim, "block_size": 16,
                   "seq_lens": SEQ_LENS[W.name], "kv_dtype": W.kv_dtype,
                   "num_blocks": W.num_blocks,
                   "fresh_blocks": int(W.fresh_blocks.size),
                   "step_tokens_written": int(W.step_slots.size),
                   "step_calls": ("paged_attention_decode_step (new tokens written "
                                  "by the decode kernel)" if new_tokens is not None
                                  else "paged_kv_zero_and_write + paged_attention_decode"),
                   "partition_tokens": pt, "kv_read_bytes": kv_bytes,
                   "cuda_graph": bool(args.graph),
                   "unique_kv_read_bytes": W.unique_kv_read_bytes(),
                   "l2": l2},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2),
                     "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": peak_kind,
                     "kernel": "paged_decode_kernel + paged_decode_merge_kernel",
                     "launch_ms": round(roof_ms, 5),
                     "timed_in": ("the headline K-step loop (events around the "
                                  "loop); each step is one decode kernel, which "
                                  "also writes the new tokens, and one merge"
                                  if pair_only else
                                  "a second K-step loop, one event pair around "
                                  "each decode call and its merge"),
                     "per_call_launch_ms": round(attn_ms, 5)},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms / K2, 5), "steps": K2,
                "untimed_steps_before": E2E_WARM,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": launches_per_step * K,
        "clocks": clocks.summary(),
    }
    if warm_ms is not None:
        line["warm"] = {"value": round(whole_job_gbs(world, kv_bytes, warm_ms / K), 2),
                        "unit": "GB/s", "ms_per_step": round(warm_ms / K, 5),
                        "note": "the same steps, each timed alone, without the L2 flush"}
    if rank == 0 and not args.no_cpu_baseline:
        gbs, sps, dt, threads, kvb = time_cpu_oracle(W, args.cpu_sample_seqs,
                                                     steps=2, warmup=0)
        line["cpu_baseline"] = {
            "value": round(gbs, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": (f"first {min(args.cpu_sample_seqs, W.batch)} of "
                       f"{W.batch} sequences, all heads, 2 steps "
                       f"({kvb / 1e6:.1f} MB of KV per step)"),
            "cpu": host_cpu_model(),
            "one_core": one_core_baseline(W, args.cpu_sample_seqs)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_blocks(args):
    """Zeroing, block copy and swap on the workload's cache geometry.

    zero_blocks: 920 MiB and 53.7 MB of blocks (the sizes the vLLM v0.17.1
    notes time for prefill and decode steps), write bandwidth;
    copy_blocks: 4096 disjoint pairs, read + write bandwidth (the measured
    copy peak counts the same way);
    swap: 4096 blocks out to pinned host memory and back in, against a
    plain pinned-memory copy of the same bytes."""
    import torch
    from paged_kv_cache_48_gb300 import (PagedKVCache, paged_kv_copy_blocks,
                                         paged_kv_swap_in, paged_kv_swap_out,
                                         paged_kv_zero_blocks, pkv_check)
    from paged_kv_cache_48_gb300 import workload as wl
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    W = wl.CONFIGS[args.workload]()
    elt = torch.uint8 if W.kv_dtype == "fp8_e4m3" else torch.bfloat16
    bb = W.block_bytes                      # per cache
    NB = max(W.num_blocks, 2 * 14720, 8192)
    shape = (NB, 16, W.num_kv_heads, W.head_dim)
    cache = PagedKVCache(torch.zeros(shape, dtype=elt, device=dev),
                         torch.zeros(shape, dtype=elt, device=dev),
                         W.kv_dtype, W.k_scale, W.v_scale)
    rng = np.random.default_rng(7)
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = measured_peak()

    def time_ms(fn, reps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(PRIME_CYCLES)  # the host queues calls meanwhile
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    reps = max(10, min(args.steps, 200))
    lines = []
    if args.kernel == "zero_blocks":
        for label, total in (("920 MiB (prefill step)", 920 * 2**20),
                             ("53.7 MB (decode step)", int(30 * 1.79 * 2**20))):
            n = max(1, total // (2 * bb))
            ids = rng.permutation(NB)[:n].astype(np.int32)
            ms = time_ms(lambda: paged_kv_zero_blocks(cache, ids), reps)
            gbs = 2 * n * bb / (ms * 1e-3) / 1e9
            lines.append({"metric": f"zero fresh blocks: {label}",
                          "value": round(ms * 1e3, 2), "unit": "us",
                          "higher_is_better": False, "blocks": int(n),
                          "bytes": 2 * n * bb, "GB_per_s": round(gbs, 1),
                          "roofline": {"bound": "hbm", "achieved": round(gbs, 1),
                                       "peak": peak, "unit": "GB/s",
                                       "frac": round(gbs / peak, 4),
                                       "peak_kind": peak_kind}})
    elif args.kernel == "copy_blocks":
        perm = rng.permutation(NB).astype(np.int32)
        src, dst = perm[:4096], perm[4096:8192]
        ms = time_ms(lambda: paged_kv_copy_blocks(cache, src, dst), reps)
        moved = 2 * 2 * 4096 * bb          # K and V, read and written
        gbs = moved / (ms * 1e-3) / 1e9
        lines.append({"metric": "copy 4096 blocks (copy-on-write)",
                      "value": round(gbs, 1), "unit": "GB/s (read+write)",
                      "higher_is_better": True, "ms": round(ms, 4),
                      "roofline": {"bound": "hbm", "achieved": round(gbs, 1),
                                   "peak": peak, "unit": "GB/s",
                                   "frac": round(gbs / peak, 4),
                                   "peak_kind": peak_kind}})
    else:
        n = 4096
        ids = rng.permutation(NB)[:n].astype(np.int32)
        hk = torch.empty(n * bb, dtype=torch.uint8).pin_memory()
        hv = torch.empty(n * bb, dtype=torch.uint8).pin_memory()
        ms_out = time_ms(lambda: paged_kv_swap_out(cache, ids, hk, hv), reps)
        ms_in = time_ms(lambda: paged_kv_swap_in(cache, ids, hk, hv), reps)
        dbuf = torch.empty(2 * n * bb, dtype=torch.uint8, device=dev)
        hbuf = torch.empty(2 * n * bb, dtype=torch.uint8).pin_memory()
        ms_d2h = time_ms(lambda: hbuf.copy_(dbuf, non_blocking=True), reps)
        ms_h2d = time_ms(lambda: dbuf.copy_(hbuf, non_blocking=True), reps)
        nbytes = 2 * n * bb
        for label, ms, ref in (("swap out 4096 blocks to pinned host memory", ms_out, ms_d2h),
                               ("swap in 4096 blocks from pinned host memory", ms_in, ms_h2d)):
            gbs = nbytes / (ms * 1e-3) / 1e9
            ref_gbs = nbytes / (ref * 1e-3) / 1e9
            lines.append({"metric": label, "value": round(gbs, 1),
                          "unit": "GB/s", "higher_is_better": True,
                          "ms": round(ms, 4),
                          "roofline": {"bound": "host link",
                                       "achieved": round(gbs, 1),
                                       "peak": round(ref_gbs, 1), "unit": "GB/s",
                                       "frac": round(gbs / ref_gbs, 4),
                                       "peak_kind": "pinned cudaMemcpy of the same bytes, measured here"}})
    st, detail = pkv_check()
    if st != 0:
        raise RuntimeError(f"device error {st} at {detail}")
    for line in lines:
        line.update({"kernel": args.kernel, "n_gpus": 1, "data": "synthetic",
                     "config": {"workload": W.name, "block_bytes_per_cache": bb,
                                "kv_dtype": W.kv_dtype}})
        print(json.dumps(line), flush=True)
    return 0


def run_input_prep(args):
    """Step input preparation from a persistent state table: µs per call on
    the GPU against the oracle's host loop, for a decode batch (64 x 1
    token) and a mixed chunked-prefill batch (8 x 512 + 56 x 1 tokens)."""
    import torch
    import oracle
    from paged_kv_cache_48_gb300 import paged_prepare_inputs, pkv_check
    torch.cuda.set_device(0)
    rng = np.random.default_rng(9)
    R, MB, ML, B = 512, 256, 4096, 64
    sbt = rng.permutation(R * MB).astype(np.int32).reshape(R, MB)
    snc = rng.integers(0, 3000, R).astype(np.int32)
    tok = rng.integers(0, 151000, (R, ML)).astype(np.int32)
    idx = rng.permutation(R)[:B].astype(np.int32)
    c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    g_sbt, g_snc, g_tok, g_idx = c(sbt), c(snc), c(tok), c(idx)
    o = oracle.load()
    stream = torch.cuda.current_stream()
    for label, ns in (("decode batch, 64 x 1 token", np.ones(B, np.int32)),
                      ("chunked batch, 8 x 512 + 56 x 1 tokens",
                       np.array([512] * 8 + [1] * 56, np.int32))):
        T = int(ns.sum())
        g_ns = c(ns)
        outs = paged_prepare_inputs(g_idx, g_ns, g_sbt, g_snc, g_tok, T)
        f = lambda: paged_prepare_inputs(g_idx, g_ns, g_sbt, g_snc, g_tok, T,
                                         out=outs)
        for _ in range(max(3, args.warmup)):
            f()
        torch.cuda.synchronize()
        reps = 500

        def timed(fn):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / reps * 1e3

        eager_us = timed(f)
        # device time: the call replayed from a captured CUDA graph, as a
        # step runner that captures its whole step does
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                f()
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        us = timed(graph.replay)
        t0 = time.perf_counter()
        n_cpu = 200
        for _ in range(n_cpu):
            o.prepare_inputs(idx, ns, sbt, snc, tok, T)
        cpu_us = (time.perf_counter() - t0) / n_cpu * 1e6
        print(json.dumps({
            "kernel": "input_prep", "metric": f"step input preparation: {label}",
            "value": round(us, 2), "unit": "us", "higher_is_better": False,
            "timing": "CUDA-graph replay (device time)",
            "eager_call_us": round(eager_us, 2),
            "tokens": T, "gpu_launches_per_call": 2,
            "cpu_baseline": {"value": round(cpu_us, 2), "unit": "us", "cores": 1,
                             "kind": "oracle",
                             "sample": "the same call, host loop, 200 repetitions"},
            "data": "synthetic",
            "config": {"state_rows": R, "max_blocks": MB, "max_model_len": ML,
                       "batch": B}}), flush=True)
    st, detail = pkv_check()
    if st != 0:
        raise RuntimeError(f"device error {st} at {detail}")
    return 0


def run_prefill(args):
    """Chunked-prefill step (write the chunk's K/V, then causal attention
    over the paged cache) on the 8K-token workloads: TFLOP/s of the
    attention's algorithmic flops against the measured bf16 tensor peak,
    with the oracle timed on a bounded sample of rows."""
    import torch
    import oracle
    from paged_kv_cache_48_gb300 import (PagedKVCache, paged_attention_prefill,
                                         paged_kv_write, pkv_check)
    from paged_kv_cache_48_gb300 import workload as wl
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    name = args.workload if args.workload in wl.PREFILL_CONFIGS else \
        "chunked_prefill_8k"
    W = wl.PREFILL_CONFIGS[name]()
    shape = (W.num_blocks, 16, W.num_kv_heads, W.head_dim)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16)
    elt = torch.bfloat16 if W.kv_dtype == "bf16" else torch.uint8
    cache = PagedKVCache(
        torch.from_numpy(W.init_key).view(elt).reshape(shape).to(dev),
        torch.from_numpy(W.init_value).view(elt).reshape(shape).to(dev),
        W.kv_dtype, W.k_scale, W.v_scale)
    if W.hist_slots.size:
        paged_kv_write(bf(W.hist_k).to(dev), bf(W.hist_v).to(dev),
                       torch.from_numpy(W.hist_slots).to(dev), cache)
    q, k, v = bf(W.q).to(dev), bf(W.step_k).to(dev), bf(W.step_v).to(dev)
    slots = torch.from_numpy(W.step_slots).to(dev)
    tables = torch.from_numpy(W.block_tables).to(dev)
    lens = torch.from_numpy(W.seq_lens).to(dev)
    qsl = torch.from_numpy(W.query_start_loc).to(dev)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    flops = W.attention_flops()
    mql = W.max_query_len

    def step():
        paged_kv_write(k, v, slots, cache)
        paged_attention_prefill(q, cache, tables, lens, qsl, W.scale, mql, out=out)

    def attend():
        paged_attention_prefill(q, cache, tables, lens, qsl, W.scale, mql, out=out)

    def time_ms(fn, reps):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(PRIME_CYCLES)  # the host queues calls meanwhile
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    reps = max(10, min(args.steps, 500))
    with ClockSampler(0) as clk:
        step_ms = time_ms(step, reps)
        attn_ms = time_ms(attend, reps)
    st, detail = pkv_check()
    if st != 0:
        raise RuntimeError(f"device error {st} at {detail}")

    # End to end: every step uploads q, the chunk's K/V and slots from
    # pinned host memory and reads the output back.  The copies run on an
    # upload and a download stream into two alternating device buffer sets,
    # so they overlap the neighbouring steps' compute.
    h_in = [bf(W.q).pin_memory(), bf(W.step_k).pin_memory(), bf(W.step_v).pin_memory(),
            torch.from_numpy(W.step_slots).pin_memory()]
    h_out = [torch.empty(out.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    sets = [[torch.empty_like(t) for t in (q, k, v, slots, out)] for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_back = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = i % 2
        dq, dk, dv, ds, do = sets[b]
        if i >= 2:
            up.wait_event(ev_back[b])
        with torch.cuda.stream(up):
            for h, d in zip(h_in, (dq, dk, dv, ds)):
                d.copy_(h, non_blocking=True)
            ev_in[b].record(up)
        stream.wait_event(ev_in[b])
        paged_kv_write(dk, dv, ds, cache)
        paged_attention_prefill(dq, cache, tables, lens, qsl, W.scale, mql, out=do)
        ev_done[b].record(stream)
        down.wait_event(ev_done[b])
        with torch.cuda.stream(down):
            h_out[b].copy_(do, non_blocking=True)
            ev_back[b].record(down)

    n_e2e = max(10, reps // 4)
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e_a = torch.cuda.Event(enable_timing=True)
    e_b = torch.cuda.Event(enable_timing=True)
    e_a.record(stream)
    for i in range(n_e2e):
        e2e_step(i)
    stream.wait_stream(down)
    e_b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e_a.elapsed_time(e_b) / n_e2e
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = h_out[0].numel() * h_out[0].element_size()

    peak, peak_kind = measured_tensor_peak()
    tflops = flops / (step_ms * 1e-3) / 1e12
    attn_tflops = flops / (attn_ms * 1e-3) / 1e12
    line = {
        "kernel": "prefill", "metric": f"chunked-prefill attention TFLOP/s ({name})",
        "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": reps, "warmup": max(3, args.warmup),
        "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if W.kv_dtype == "bf16" else "f16 MMA on e4m3 KV",
        "data": "synthetic",
        "config": {"workload": name, "batch": W.batch, "num_tokens": W.num_tokens,
                   "kv_dtype": W.kv_dtype,
                   "history": [int(x) for x in W.history],
                   "chunk": [int(x) for x in W.chunk],
                   "num_heads": W.num_heads, "num_kv_heads": W.num_kv_heads,
                   "head_dim": W.head_dim, "block_size": 16,
                   "l2": "inputs larger than L2 (queries + pool)"},
        "attention_flops": flops,
        "roofline": {"bound": "tensor", "achieved": round(attn_tflops, 2),
                     "peak": peak, "unit": "TFLOP/s",
                     "frac": round(attn_tflops / peak, 4),
                     "traffic": profiled_traffic(PREFILL_PROFILES[name], PREFILL_SOURCES)
                     if name in PREFILL_PROFILES else None,
                     "peak_kind": peak_kind + " bf16 burst",
                     "kernel_ms": round(attn_ms, 4)},
        "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 2),
                "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * reps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        kc, vc = W.init_key.copy(), W.init_value.copy()
        o = oracle.load()
        odt = oracle.DTYPE_BF16 if W.kv_dtype == "bf16" else oracle.DTYPE_FP8_E4M3
        for kk, vv, sl in ((W.hist_k, W.hist_v, W.hist_slots),
                           (W.step_k, W.step_v, W.step_slots)):
            o.kv_write(kc, vc, odt, 16, W.num_kv_heads, W.head_dim, W.k_scale,
                       W.v_scale, kk, vv, sl)
        rng = np.random.default_rng(1)
        toks = rng.choice(W.num_tokens, size=128, replace=False)
        rows = np.array([[t, h] for t in toks for h in range(W.num_heads)],
                        np.int32)
        qsl_h = W.query_start_loc
        seq = np.searchsorted(qsl_h, toks, side="right") - 1
        keys = (W.history[seq] + (toks - qsl_h[seq]) + 1).astype(np.int64)
        sample_flops = int(keys.sum()) * W.num_heads * 4 * W.head_dim
        t0 = time.perf_counter()
        o.attention_prefill(W.q, kc, vc, odt, W.k_scale, W.v_scale, 16,
                            W.num_kv_heads, W.head_dim, W.block_tables,
                            W.seq_lens, qsl_h, W.scale, rows=rows)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {
            "value": round(sample_flops / dt / 1e12, 6), "unit": "TFLOP/s",
            "cores": o.num_threads(0), "kind": "oracle",
            "sample": f"{rows.shape[0]} (token, head) rows of 128 random tokens, "
                      f"{dt:.1f} s"}
    print(json.dumps(line), flush=True)
    return 0


def run_cascade(args):
    """Shared-prefix decode on the prefix-sharing workload (256 sequences,
    16 groups sharing 1024 tokens): the cascade path against plain decode on
    the same cache, as unique and logical KV bytes per second."""
    import torch
    import oracle
    from paged_kv_cache_48_gb300 import (PagedKVCache, paged_attention_decode,
                                         paged_attention_decode_cascade,
                                         paged_kv_write, paged_kv_zero_blocks,
                                         pkv_check)
    from paged_kv_cache_48_gb300 import workload as wl
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    W = wl.prefix_shared()
    shape = (W.num_blocks, 16, W.num_kv_heads, W.head_dim)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16)
    cache = PagedKVCache(
        torch.from_numpy(W.init_key).view(torch.bfloat16).reshape(shape).to(dev),
        torch.from_numpy(W.init_value).view(torch.bfloat16).reshape(shape).to(dev),
        "bf16")
    paged_kv_write(bf(W.hist_k).to(dev), bf(W.hist_v).to(dev),
                   torch.from_numpy(W.hist_slots).to(dev), cache)
    if W.fresh_blocks.size:
        paged_kv_zero_blocks(cache, W.fresh_blocks)
    paged_kv_write(bf(W.step_k).to(dev), bf(W.step_v).to(dev),
                   torch.from_numpy(W.step_slots).to(dev), cache)
    q = bf(W.q).to(dev)
    tables = torch.from_numpy(W.block_tables).to(dev)
    lens = torch.from_numpy(W.seq_lens).to(dev)
    per = len(W.groups[0]["members"])
    gs = torch.tensor([g["members"][0] for g in W.groups] + [W.batch],
                      dtype=torch.int32, device=dev)
    plen_h = [16 * len(g["prefix_blocks"]) for g in W.groups]
    plen = torch.tensor(plen_h, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)

    def cascade():
        paged_attention_decode_cascade(q, cache, tables, lens, gs, plen, W.scale,
                                       W.max_seq_len, per, max(plen_h), out=out)

    def plain():
        paged_attention_decode(q, cache, tables, lens, W.scale, W.max_seq_len,
                               out=out)

    def time_ms(fn, reps):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(PRIME_CYCLES)  # the host queues calls meanwhile
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    reps = max(10, min(args.steps, 2000))
    with ClockSampler(0) as clk:
        c_ms = time_ms(cascade, reps)
        p_ms = time_ms(plain, reps)
    st, detail = pkv_check()
    if st != 0:
        raise RuntimeError(f"device error {st} at {detail}")
    unique, logical = W.unique_kv_read_bytes(), W.kv_read_bytes()
    peak, peak_kind = measured_peak()
    gbs = unique / (c_ms * 1e-3) / 1e9
    line = {
        "kernel": "cascade",
        "metric": "shared-prefix decode, unique KV-read GB/s (prefix_shared)",
        "value": round(gbs, 1), "unit": "GB/s", "higher_is_better": True,
        "ms_per_call": round(c_ms, 4), "steps": reps,
        "logical_GB_per_s": round(logical / (c_ms * 1e-3) / 1e9, 1),
        "plain_decode_ms": round(p_ms, 4),
        "plain_decode_logical_GB_per_s": round(logical / (p_ms * 1e-3) / 1e9, 1),
        "speedup_vs_plain_decode": round(p_ms / c_ms, 3),
        "unique_kv_bytes": unique, "logical_kv_bytes": logical,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(gbs / peak, 4), "traffic": None,
                     "peak_kind": peak_kind},
        "gpu_launches_per_call": 3, "clocks": clk.summary(), "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "prefix_shared", "batch": W.batch, "groups": len(W.groups),
                   "prefix_tokens": max(plen_h), "num_heads": W.num_heads,
                   "num_kv_heads": W.num_kv_heads, "head_dim": W.head_dim,
                   "l2": "unique KV bytes larger than L2"},
    }
    if not args.no_cpu_baseline:
        kc, vc = W.init_key.copy(), W.init_value.copy()
        o = oracle.load()
        o.kv_write(kc, vc, oracle.DTYPE_BF16, 16, W.num_kv_heads, W.head_dim,
                   1.0, 1.0, W.hist_k, W.hist_v, W.hist_slots)
        seqs = list(range(0, W.batch, max(1, W.batch // args.cpu_sample_seqs)))
        t0 = time.perf_counter()
        cpu_oracle_step(W, kc, vc, seqs)
        dt = time.perf_counter() - t0
        sample = int(W.seq_lens[seqs].astype(np.int64).sum()) * W.num_kv_heads * \
            W.head_dim * 4
        line["cpu_baseline"] = {"value": round(sample / dt / 1e9, 3), "unit": "GB/s",
                                "cores": o.num_threads(0), "kind": "oracle",
                                "sample": f"{len(seqs)} sequences, logical bytes, {dt:.1f} s"}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.kernel == "input_prep":
        return run_input_prep(args)
    if args.kernel == "prefill":
        return run_prefill(args)
    if args.kernel == "cascade":
        return run_cascade(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.kernel != "decode":
        return run_blocks(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
