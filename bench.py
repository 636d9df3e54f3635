"""Benchmark of the paged LATENT attention operator on one node.

One step = one pass of the whole operator over one synthetic batch: the
write phase (RoPE + paged scatter of the new latent rows), the decode phase
(split-KV attention + log-sum-exp combine) and, for mixed batches, the
prefill phase. The headline workload is DeepSeek-V3-style absorbed MLA
decode (bf16, H=128, latent 576 / value 512 / rotary 64 at offset 512,
batch 64, one new token per sequence, context 4096, bs=64), the largest
decode configuration; the same JSON line carries DeepSeek-V3-style chunked
prefill (4 x 4096 new tokens, tensor-bound), GLM-style decode and the mixed
fp16 serving batch under "extras", each timed the same way.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--extras A,B,...|none] [--impl reference] [--portable]

Timing: W untimed eager steps, then the step is captured in a CUDA graph
and K graph replays are timed, bracketed by a barrier and a device
synchronise; each replay is timed with CUDA events on the launching stream
and L2 is flushed (a write of 2x the L2 size) before every replay, outside
the events. A second loop replays one graph per (non-empty) phase for the
breakdown and the dominant call's duration. Under torchrun each rank runs
its own seeded batch (weak scaling, no collective on the data path) and the
max over ranks is reported. `value` is algorithmic latent-cache bytes per
second (TB/s) of the headline workload; `e2e` is the same metric through the
operator object with the step's inputs copied host->device from pinned
memory and the output copied back inside the timed region. `--impl
reference` times the CPU oracle on the same workload instead (rank 0 only).
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("paged-MLA decode latent-cache TB/s & TFLOP/s vs roofline; prefill TFLOP/s "
          "(1 GB300)")
UNIT = "TB/s"


# ---------------------------------------------------------------------------
# DRAM traffic of the dominant kernel, from ncu
# ---------------------------------------------------------------------------

# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the dominant
# attention kernel, from `ncu --set full` captures of that kernel on the
# named workload, with the SHA-256 of the tensor-core kernel sources they
# were taken on. Once those sources change the figure no longer describes
# the kernel and the roofline reports null traffic until a new capture
# replaces it.
KERNEL_SOURCES = {
    "tc_attn_kernel": ("pa_tc_attn.cuh", "pa_tc_common.cuh", "pa_tc.cu", "pa_tc_glm.cu",
                       "pa_tc_fp8.cu"),
    "tc_pair_kernel": ("pa_tc_pair.cu", "pa_tc_cluster.cuh", "pa_tc_common.cuh"),
    "tc_gqa_kernel": ("pa_gqa.cu", "pa_tc_common.cuh"),
}
# workload -> (kernel, bytes per launch, source digest, how the figure was taken)
NCU_TRAFFIC = {
    "dsv3_decode": ("tc_pair_kernel", 315103744, "73ef4a7681d71ef4", "measured on this workload"),
    # traffic grows with the tokens (query in, output out, each sequence's
    # cache rows): the quarter-size capture times four
    "dsv3_prefill": ("tc_pair_kernel", 4 * 1096469504, "73ef4a7681d71ef4",
                     "dsv3_prefill_small (4 x 1024 tokens) scaled by 4"),
    "glm_decode": ("tc_attn_kernel", 54154496, "05afb7237f0565c4", "measured on this workload"),
    "mixed_serving": ("tc_attn_kernel", 99269120, "05afb7237f0565c4", "measured on this workload"),
    "gqa_decode": ("tc_gqa_kernel", 579862272, "50f50be27473339b", "measured on this workload"),
    "glm_decode_fp8": ("tc_attn_kernel", 25967872, "05afb7237f0565c4", "measured on this workload"),
}


def kernel_source_digest(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "paged_latent_attention_cache_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """(bytes, kernel, note) of the dominant kernel's DRAM traffic per
    launch, or Nones once its sources have changed since the capture."""
    entry = NCU_TRAFFIC.get(workload)
    if entry is None or entry[2] != kernel_source_digest(entry[0]):
        return None, None, None
    return entry[1], entry[0], entry[3]


# ---------------------------------------------------------------------------
# Algorithmic work of a workload (each visible cache row counted once)
# ---------------------------------------------------------------------------

def algorithmic_work(w, seqs=None, tokens=None, include_write=True):
    """Bytes and FLOPs of the operator on a workload, counting each cache
    row a sequence's queries can see once, plus Q, O, the cos/sin rows, the
    block-table entries, the key rows read and the cache rows written.
    FLOPs = (2*hs + 2*vhs) per (visible key, head). ``seqs`` restricts the
    read phase to those sequences, ``tokens`` to those tokens. A cache row is
    hs bytes in an FP8 cache, 2*hs otherwise."""
    el = 2
    el_c = 1 if getattr(w, "cache_dtype", None) == "e4m3" else 2
    H, hs, vhs, bs = w.num_heads, w.head_size, w.v_head_size, w.block_size
    # SEPARATE layout: a visible position is kvH key rows and kvH value rows
    kvh = getattr(w, "kv_num_heads", None)
    row_bytes = kvh * (hs + vhs) * el if kvh else hs * el_c
    win = w.local_window_size
    cs = w.cumseq.tolist()
    seqs = range(w.num_seqs) if seqs is None else seqs
    tok_set = None if tokens is None else set(int(t) for t in tokens)
    cache_rows = flops = q_rows = bt_entries = 0
    for b in seqs:
        lo_t, hi_t = cs[b], cs[b + 1]
        toks = [t for t in range(lo_t, hi_t) if tok_set is None or t in tok_set]
        if not toks:
            continue
        P = w.past_lens[b]
        first_lo = None
        last_pos = None
        for t in toks:
            pos = P + t - lo_t
            lo = 0 if win < 0 else max(0, pos - win)
            flops += (pos + 1 - lo) * H * (2 * hs + 2 * vhs)
            first_lo = lo if first_lo is None else min(first_lo, lo)
            last_pos = pos if last_pos is None else max(last_pos, pos)
        span = last_pos + 1 - first_lo
        cache_rows += span
        bt_entries += last_pos // bs - first_lo // bs + 1
        q_rows += len(toks)
    read_bytes = (cache_rows * row_bytes + q_rows * H * hs * el + q_rows * H * vhs * el +
                  q_rows * w.rotary_dim * el + bt_entries * 4)
    write_bytes = 0
    if include_write:
        n_written = int((w.slot_mapping >= 0).sum())
        new_row = kvh * (hs + vhs) * el if kvh else hs * el
        write_bytes = (w.num_tokens * new_row + n_written * row_bytes +
                       w.num_tokens * (w.rotary_dim * el + 4))
    return dict(bytes=read_bytes + write_bytes, read_bytes=read_bytes, flops=flops,
                cache_rows=cache_rows, tokens=q_rows)


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int, path: str):
        self.path = path
        self.proc = None
        try:
            self.f = open(path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        return parse_clocks(self.path)


def parse_clocks(path: str):
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    try:
        lines = open(path).read().strip().splitlines()
    except Exception:
        return None
    for ln in lines:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            mx.append(float(parts[2]))
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
            "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# Multi-rank helpers (also exercised on CPU with gloo in the tests)
# ---------------------------------------------------------------------------

def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own independent batch (weak scaling)."""
    return base_seed + 1000 * rank


def reduce_max(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# Oracle timing (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------

def oracle_session(w):
    """The CPU oracle's write phase over the whole batch, then a function
    that runs its read phase for one token (rounded to the output dtype):
    LATENT with a 16-bit or E4M3 cache, or the SEPARATE layout."""
    from oracle import pa_oracle as O
    from paged_latent_attention_cache_gb300 import workloads as W
    cumseq, past, bt = w.cumseq.numpy(), w.past.numpy(), w.block_table.numpy()
    if hasattr(w, "kv_num_heads"):
        p = W.separate_oracle_params(w)
        dt, hs, kvh = p["dtype"], w.head_size, w.kv_num_heads
        vhs = p["v_head_size"] or hs
        kc = O.BitsCache(W.to_bits(w.key_cache).reshape(-1, hs), dt)
        vc = O.BitsCache(W.to_bits(w.value_cache).reshape(-1, vhs), dt)
        cos_t = O.bits_to_f64(W.to_bits(w.cos_cache), dt)
        sin_t = O.bits_to_f64(W.to_bits(w.sin_cache), dt)
        opt = lambda x: None if x is None else O.bits_to_f64(W.to_bits(x), dt)  # noqa: E731
        kn, qn, sink = opt(w.k_norm_weight), opt(w.q_norm_weight), opt(w.head_sink)
        kb, vb, qb = W.to_bits(w.key), W.to_bits(w.value), W.to_bits(w.query)
        O.separate_write(lambda t: O.bits_to_f64(kb[t], dt).reshape(kvh, hs),
                         lambda t: O.bits_to_f64(vb[t], dt).reshape(kvh, vhs), cos_t, sin_t,
                         w.slot_mapping.numpy(), cumseq, past, kc, vc, p, kn)

        def read(t):
            out = O.separate_attend_token(t, O.bits_to_f64(qb[t], dt), kc, vc, cos_t, sin_t,
                                          cumseq, past, bt, p, sink, qn)
            return O.round_f64_to_bits(out, dt)
        return read
    p = W.oracle_params(w)
    dt, hs = p["dtype"], w.head_size
    if p.get("cache_dtype") == O.E4M3:
        cache = O.E4M3Cache(W.to_bits(w.key_cache).reshape(-1, hs), p["k_scale"])
    else:
        cache = O.BitsCache(W.to_bits(w.key_cache).reshape(-1, hs), dt)
    cos_t = O.bits_to_f64(W.to_bits(w.cos_cache), dt)
    sin_t = O.bits_to_f64(W.to_bits(w.sin_cache), dt)
    kb, qb = W.to_bits(w.key), W.to_bits(w.query)
    O.latent_write(lambda t: O.bits_to_f64(kb[t], dt), cos_t, sin_t, w.slot_mapping.numpy(),
                   cumseq, past, cache, p)

    def read(t):
        out = O.latent_attend_token(t, O.bits_to_f64(qb[t], dt), cache, cos_t, sin_t, cumseq,
                                    past, bt, p)
        return O.round_f64_to_bits(out, dt)
    return read


def time_oracle(w, budget_s: float, tokens_order=None):
    """Runs the CPU oracle's read phase token by token (after its write phase
    over the whole batch) until ``budget_s`` of wall time is used. Returns
    (seconds, algorithmic bytes of the sampled work, tokens done)."""
    t0 = time.perf_counter()
    read = oracle_session(w)
    done = []
    order = list(range(w.num_tokens)) if tokens_order is None else tokens_order
    for t in order:
        read(t)
        done.append(t)
        if time.perf_counter() - t0 >= budget_s:
            break
    sec = time.perf_counter() - t0
    work = algorithmic_work(w, tokens=done)
    return sec, work, len(done)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def build_workload(name: str, seed_offset: int):
    from paged_latent_attention_cache_gb300 import workloads as W
    fn = W.WORKLOADS[name]
    import inspect
    default_seed = inspect.signature(fn).parameters["seed"].default
    return fn(seed=default_seed + seed_offset)


def make_graph(fn, keep=False):
    """Captures fn() into a CUDA graph; with keep=True the cudaGraph_t is kept
    so its nodes can be inspected (falls back to a plain graph)."""
    import torch
    g = None
    if keep:
        try:
            g = torch.cuda.CUDAGraph(keep_graph=True)
        except TypeError:
            g = None
    if g is None:
        g = torch.cuda.CUDAGraph()
        keep = False
    with torch.cuda.graph(g):
        fn()
    if keep:
        g.instantiate()
    return g, keep


def graph_kernel_nodes(g):
    """Kernel nodes in a captured graph (the launches of one replay), read
    through the driver API; None if unavailable."""
    import ctypes
    try:
        cu = ctypes.CDLL("libcuda.so.1")
        h = ctypes.c_void_p(g.raw_cuda_graph())
        n = ctypes.c_size_t(0)
        if cu.cuGraphGetNodes(h, None, ctypes.byref(n)) != 0:
            return None
        nodes = (ctypes.c_void_p * n.value)()
        if cu.cuGraphGetNodes(h, nodes, ctypes.byref(n)) != 0:
            return None
        cnt = 0
        for nd in nodes:
            t = ctypes.c_int(-1)
            cu.cuGraphNodeGetType(ctypes.c_void_p(nd), ctypes.byref(t))
            cnt += 1 if t.value == 0 else 0   # CU_GRAPH_NODE_TYPE_KERNEL
        return cnt
    except Exception:
        return None


def measure_workload(args, name, rank, world, device, steps, warmup, flush, e2e=True):
    """Times one workload: K graph replays of the whole step (write, decode,
    prefill; empty phases are not launched), then K replays of the per-phase
    graphs, optionally the end-to-end path. Returns a dict of results."""
    import torch
    from paged_latent_attention_cache_gb300.api import PagedLatentAttention

    w = build_workload(name, rank_seed(0, rank) if world > 1 else 0)
    d = w.to(device)
    out = torch.empty(w.num_tokens, w.num_heads * w.v_head_size, dtype=w.dtype, device=device)
    cache = d.key_cache
    nd = w.num_decode_seqs
    stream = torch.cuda.current_stream(device)
    separate = hasattr(w, "kv_num_heads")
    if separate:
        from paged_latent_attention_cache_gb300 import binding as B
        from paged_latent_attention_cache_gb300.api import SeparateAttention
        op = SeparateAttention.from_workload(w, device=device)
        vcache = d.value_cache

        def write():
            B.pa_separate_write(op.params, d.key, d.value, d.cos_cache, d.sin_cache,
                                d.k_norm_weight, d.slot_mapping, d.cumseq, d.past, cache, vcache,
                                op.err_flags)

        def decode():
            B.pa_separate_decode(op.params_after_write, d.query, cache, vcache, d.cos_cache,
                                 d.sin_cache, d.q_norm_weight, d.head_sink, d.cumseq, d.past,
                                 d.block_table, out, 0, nd, op.workspace, op.err_flags)

        def prefill():
            B.pa_separate_prefill(op.params_after_write if nd == 0 else op.params, d.query,
                                  cache, vcache, d.cos_cache, d.sin_cache, d.q_norm_weight,
                                  d.head_sink, d.cumseq, d.past, d.block_table, out, nd,
                                  w.num_seqs, op.workspace, op.err_flags)
    else:
        op = PagedLatentAttention.from_workload(w, device=device, portable=args.portable)

        def write():
            op.write(d.key, d.cos_cache, d.sin_cache, d.slot_mapping, d.cumseq, d.past, cache)

        def decode():
            op.decode(d.query, cache, d.cos_cache, d.sin_cache, d.cumseq, d.past,
                      d.block_table, out, 0, nd, after_write=True)

        def prefill():
            op.prefill(d.query, cache, d.cos_cache, d.sin_cache, d.cumseq, d.past,
                       d.block_table, out, nd, w.num_seqs, after_write=nd == 0)

        def mixed():
            op.mixed(d.query, cache, d.cos_cache, d.sin_cache, d.cumseq, d.past, d.block_table,
                     out, nd, after_write=True)

    if not separate and 0 < nd < w.num_seqs:
        # a mixed batch: one read call (one grid for decode and prefill work)
        phases = [("write", write), ("read", mixed)]
    else:
        phases = [("write", write), ("decode", decode if nd > 0 else None),
                  ("prefill", prefill if nd < w.num_seqs else None)]

    def step():
        for _, f in phases:
            if f is not None:
                f()

    for _ in range(max(warmup, 3)):   # eager warm-up (also configures kernels)
        flush.zero_()
        step()
    torch.cuda.synchronize(device)
    if op.error_flags() != 0:
        raise RuntimeError(f"{name}: device error flags {op.error_flags():#x}")
    # One graph for the whole step (the timed unit) and one per non-empty
    # phase (the breakdown and the dominant call's duration).
    g_step, kept = make_graph(step, keep=True)
    launches_per_step = graph_kernel_nodes(g_step) if kept else None
    g_phase = [(n, make_graph(f)[0]) for n, f in phases if f is not None]
    for _ in range(3):
        flush.zero_()
        g_step.replay()
        for _, gp in g_phase:
            gp.replay()
    torch.cuda.synchronize(device)

    K = steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    gpu_index = device.index
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_index = int(vis.split(",")[device.index])
        except ValueError:
            pass
    # the raw clock samples of the timed region (the JSON line carries their summary)
    clock_dir = os.environ.get("PA_BENCH_CLOCK_DIR", os.path.join(ROOT, "bench_out"))
    os.makedirs(clock_dir, exist_ok=True)
    sampler = ClockSampler(gpu_index, os.path.join(clock_dir, f"clocks_{name}_r{rank}.csv"))
    time.sleep(0.3)
    barrier(device)
    torch.cuda.synchronize(device)
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        evs[i][0].record(stream)
        g_step.replay()
        evs[i][1].record(stream)
    torch.cuda.synchronize(device)
    barrier(device)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    # per-phase breakdown (separate loop, same flushing)
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(g_phase) + 1)]
           for _ in range(K)]
    for i in range(K):
        flush.zero_()
        pev[i][0].record(stream)
        for j, (_, gp) in enumerate(g_phase):
            gp.replay()
            pev[i][j + 1].record(stream)
    torch.cuda.synchronize(device)

    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    phase_ms = {n: 0.0 for n, _ in phases}
    for j, (n, _) in enumerate(g_phase):
        phase_ms[n] = statistics.mean(e[j].elapsed_time(e[j + 1]) for e in pev)
    ms_per_step = reduce_max(sum(step_ms) / K, device)
    q = statistics.quantiles(step_ms, n=10) if K >= 2 else [step_ms[0]] * 9
    dist = {"median": round(statistics.median(step_ms), 5), "p10": round(q[0], 5),
            "p90": round(q[-1], 5)}

    e2e_ms = h2d = d2h = None
    if e2e:
        # End to end through the operator object: H2D of the step's inputs
        # from pinned memory, the phases, D2H of the output.
        names = ("query", "key") + (("value",) if separate else ()) + \
            ("cumseq", "past", "block_table", "slot_mapping")
        host = {k: getattr(w, k).pin_memory() for k in names}
        dev_in = {k: torch.empty_like(v, device=device) for k, v in host.items()}
        out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = out_host.numel() * out_host.element_size()

        def e2e_step():
            for k, v in host.items():
                dev_in[k].copy_(v, non_blocking=True)
            if separate:
                op.forward(dev_in["query"], dev_in["key"], dev_in["value"], cache, vcache,
                           d.cos_cache, d.sin_cache, dev_in["cumseq"], dev_in["past"],
                           dev_in["block_table"], dev_in["slot_mapping"], nd,
                           head_sink=d.head_sink, q_norm_weight=d.q_norm_weight,
                           k_norm_weight=d.k_norm_weight, out=out)
            else:
                op.forward(dev_in["query"], dev_in["key"], cache, d.cos_cache, d.sin_cache,
                           dev_in["cumseq"], dev_in["past"], dev_in["block_table"],
                           dev_in["slot_mapping"], nd, out=out)
            out_host.copy_(out, non_blocking=True)

        for _ in range(3):
            flush.zero_()
            e2e_step()
        torch.cuda.synchronize(device)
        e2e_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        barrier(device)
        for i in range(K):
            flush.zero_()
            e2e_evs[i][0].record(stream)
            e2e_step()
            e2e_evs[i][1].record(stream)
        torch.cuda.synchronize(device)
        e2e_ms = reduce_max(sum(a.elapsed_time(b) for a, b in e2e_evs) / K, device)
    if op.error_flags() != 0:
        raise RuntimeError(f"{name}: device error flags {op.error_flags():#x}")

    work = algorithmic_work(w)
    dec_work = algorithmic_work(w, seqs=range(nd), include_write=False)
    pre_work = algorithmic_work(w, seqs=range(nd, w.num_seqs), include_write=False)
    res = dict(w=w, work=work, dec_work=dec_work, pre_work=pre_work,
               value=work["bytes"] * world / (ms_per_step * 1e-3) / 1e12,
               tflops=work["flops"] * world / (ms_per_step * 1e-3) / 1e12,
               ms_per_step=ms_per_step, dist=dist, e2e_ms=e2e_ms, h2d=h2d, d2h=d2h,
               clocks=clocks, wall=wall, launches=launches_per_step, phase_ms=phase_ms,
               family=(1, 1) if separate else (op.kernel_family(0), op.kernel_family(1)),
               steps=K)
    return res


PROBE_WORKLOADS = ("glm_decode", "dsv3_decode")


def run_probe(args, device, flush, peaks):
    """Sweeps pa_latent_gather_probe (every visible cache row of a decode
    batch gathered through the block table by the decode kernels' TMA boxes,
    no arithmetic) over tile size, stages and CTAs per SM on the decode
    workloads' caches; one JSON line per workload with the visible rows'
    bytes over the CUDA-event time, against the measured copy bandwidth."""
    import torch
    from paged_latent_attention_cache_gb300 import binding as B
    from paged_latent_attention_cache_gb300 import workloads as W
    hbm = peaks[0]
    steps = min(args.steps, 200)
    names = [args.workload] if args.workload in PROBE_WORKLOADS and args.extras == "none" \
        else list(PROBE_WORKLOADS)
    for name in names:
        w = W.WORKLOADS[name]()
        d = w.to(device)
        p = B.make_params(dtype=w.dtype, num_heads=w.num_heads, head_size=w.head_size,
                          v_head_size=w.v_head_size, rotary_offset=w.rotary_offset,
                          rotary_dim=w.rotary_dim, cos_rows=w.cos_cache.shape[0],
                          block_size=w.block_size, num_blocks=w.key_cache.shape[0],
                          max_blocks_per_seq=w.block_table.shape[1], scale=w.scale)
        err = torch.zeros(1, dtype=torch.int32, device=device)
        rows = int((w.past + 1).sum())
        nbytes = rows * w.head_size * w.key_cache.element_size()
        sweep = []
        shapes = [(t, st, c) for t in (64, 128) for st in (2, 3, 4, 6, 8) for c in (1, 2, 3, 4)]
        if args.probe_config:
            shapes = [tuple(int(x) for x in args.probe_config.split(","))]
        for tile_keys, stages, ctas in shapes:
            slabs = (w.head_size + 63) // 64
            smem = stages * slabs * tile_keys * 128 + 8 * stages + 4 * (w.num_seqs + 1) + 1024
            if smem > 226 * 1024 or ctas * (smem + 1024) > 228 * 1024:
                continue

            def go():
                B.pa_latent_gather_probe(p, d.key_cache, d.past, d.block_table, tile_keys,
                                         stages, ctas, err)
            for _ in range(3):
                flush.zero_()
                go()
            torch.cuda.synchronize(device)
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
                   for _ in range(steps)]
            for e0, e1 in evs:
                flush.zero_()
                e0.record()
                go()
                e1.record()
            torch.cuda.synchronize(device)
            ms = statistics.median(a.elapsed_time(b) for a, b in evs)
            if int(err.item()) != 0:
                raise RuntimeError(f"probe {name}: device error flags {int(err.item()):#x}")
            gbs = nbytes / (ms * 1e-3) / 1e9
            sweep.append({"tile_keys": tile_keys, "stages": stages, "ctas_per_sm": ctas,
                          "us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                          "frac_of_copy": round(gbs / hbm, 3)})
        best = max(sweep, key=lambda r: r["gbs"])
        print(json.dumps({"probe": "paged gather (TMA boxes through the block table, no "
                                   "arithmetic)", "workload": name, "visible_row_bytes": nbytes,
                          "copy_peak_gbs": hbm, "peak_source": peaks[3], "steps": steps,
                          "l2": "flushed before every run", "best": best, "sweep": sweep}),
              flush=True)
    return 0


def load_peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return (float(pk["hbm_gbs"]), float(pk["bf16_tflops"]),
                float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def roofline(res, peaks):
    """Roofline of the dominant call (decode when the batch has decode
    sequences, else prefill): the bound is whichever of its algorithmic
    bytes at the measured HBM copy bandwidth and its FLOPs at the measured
    dense bf16 burst peak takes longer; `achieved` is the algorithmic work
    over the call's mean duration, timed live with CUDA events."""
    w = res["w"]
    hbm, bf16, bf16_sus, peak_src = peaks
    if "read" in res["phase_ms"]:
        dw, pw = res["dec_work"], res["pre_work"]
        dom = {"bytes": dw["bytes"] + pw["bytes"], "flops": dw["flops"] + pw["flops"]}
        dom_ms = res["phase_ms"]["read"]
        dom_name = "mixed read call (decode splits + prefill units in one grid, + combine)"
    elif w.num_decode_seqs:
        dom, dom_ms = res["dec_work"], res["phase_ms"]["decode"]
        dom_name = "decode call (split-KV attention + combine)"
    else:
        dom, dom_ms = res["pre_work"], res["phase_ms"]["prefill"]
        dom_name = "prefill call"
    t_bytes = dom["bytes"] / (hbm * 1e9)
    t_flops = dom["flops"] / (bf16 * 1e12)
    traffic, traffic_kernel, traffic_note = ncu_traffic(w.name)
    if t_flops > t_bytes:
        achieved = dom["flops"] / (dom_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": bf16,
                "unit": "TFLOP/s", "frac": round(achieved / bf16, 4),
                "peak_kind": "bf16 dense burst (of measured)",
                "frac_of_sustained": round(achieved / bf16_sus, 4),
                "sustained_peak": bf16_sus}
    else:
        achieved = dom["bytes"] / (dom_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "peak_kind": "HBM copy (of measured)"}
    roof.update({"traffic": traffic, "traffic_kernel": traffic_kernel,
                 "traffic_source": traffic_note,
                 "alg_bytes": dom["bytes"], "alg_flops": dom["flops"],
                 "kernel": dom_name, "kernel_ms": round(dom_ms, 5),
                 "peak_source": peak_src})
    return roof


def config_of(w, world):
    """The workload description both arms print."""
    extra = {}
    if hasattr(w, "kv_num_heads"):
        extra = {"layout": "SEPARATE", "kv_num_heads": w.kv_num_heads,
                 "head_sink": w.head_sink is not None, "qk_norm": w.q_norm_weight is not None}
    elif getattr(w, "cache_dtype", None):
        extra = {"cache_dtype": w.cache_dtype, "k_scale": w.k_scale}
    return {"workload": w.name, "dtype": {"torch.bfloat16": "bf16",
                                           "torch.float16": "f16"}[str(w.dtype)], **extra,
            "num_heads": w.num_heads, "head_size": w.head_size, "v_head_size": w.v_head_size,
            "rotary": [w.rotary_offset, w.rotary_dim], "block_size": w.block_size,
            "num_seqs": w.num_seqs, "num_decode_seqs": w.num_decode_seqs,
            "num_tokens": w.num_tokens, "softcap": w.softcap,
            "local_window_size": w.local_window_size,
            "l2": "flushed before every step (write of 2x L2)",
            "timing": "CUDA graph of the step, CUDA events per replay",
            "parallelism": f"replicas x{world} (independent batches per rank)"}


def summary(res, peaks, world, args):
    w = res["w"]
    return {
        "value": round(res["value"], 4), "unit": UNIT,
        "ms_per_step": round(res["ms_per_step"], 5), "step_ms": res["dist"],
        "steps": res["steps"],
        "tflops": round(res["tflops"], 3),
        "tokens_per_s": round(w.num_tokens * world / (res["ms_per_step"] * 1e-3), 1),
        "phase_ms": {k: round(v, 5) for k, v in res["phase_ms"].items()},
        "alg_bytes_per_step": res["work"]["bytes"], "alg_flops_per_step": res["work"]["flops"],
        "roofline": roofline(res, peaks),
        "kernels": "portable" if args.portable or res["family"][0] != 1 else "tcgen05",
        "clocks": res["clocks"],
        "config": config_of(w, world),
    }


EXTRA_STEPS = {"dsv3_prefill": 20}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="dsv3_decode")
    ap.add_argument("--extras",
                    default="dsv3_prefill,glm_decode,mixed_serving,glm_decode_fp8,dsv3_decode_fp8,gqa_decode",
                    help="comma-separated workloads timed after the headline one "
                         "('none' to skip)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--portable", action="store_true",
                    help="force the portable CUDA-core attention kernels")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--probe", action="store_true",
                    help="instead of the operator: sweep the paged streaming probe "
                         "(pa_latent_gather_probe) over the decode workloads' caches")
    ap.add_argument("--probe-config", default="",
                    help="with --probe: one TILE_KEYS,STAGES,CTAS_PER_SM shape instead of the sweep")
    args = ap.parse_args(argv)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import torch.distributed as dist
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    from paged_latent_attention_cache_gb300 import build as _build
    _build.build()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush = torch.empty(2 * max(l2, 64 << 20), dtype=torch.uint8, device=device)
    peaks = load_peaks()
    if args.probe:
        return run_probe(args, device, flush, peaks)
    res = measure_workload(args, args.workload, rank, world, device, args.steps, args.warmup,
                           flush)
    extras = [] if args.extras in ("", "none") else \
        [x for x in args.extras.split(",") if x and x != args.workload]
    extra_res = {}
    for name in extras:
        k = min(args.steps, EXTRA_STEPS.get(name, args.steps))
        r = measure_workload(args, name, rank, world, device, k, args.warmup, flush, e2e=False)
        extra_res[name] = summary(r, peaks, world, args)
        del r
        torch.cuda.empty_cache()
    if rank == 0:
        w = res["w"]
        head = summary(res, peaks, world, args)
        line = {
            "metric": METRIC,
            "value": head["value"],
            "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": max(args.warmup, 3),
            "ms_per_step": head["ms_per_step"],
            "step_ms": head["step_ms"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": head["config"]["dtype"],
            "data": "synthetic (seeded N(0,0.5^2) latent rows, shuffled block pool)",
            "config": head["config"],
            "kernels": head["kernels"],
            "tflops": head["tflops"],
            "tokens_per_s": head["tokens_per_s"],
            "phase_ms": head["phase_ms"],
            "alg_bytes_per_step": head["alg_bytes_per_step"],
            "alg_flops_per_step": head["alg_flops_per_step"],
            "roofline": head["roofline"],
            "e2e": {"value": round(res["work"]["bytes"] * world / (res["e2e_ms"] * 1e-3) / 1e12,
                               4),
                    "unit": UNIT, "ms_per_step": round(res["e2e_ms"], 5),
                    "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"]},
            "gpu_launches": None if res["launches"] is None else res["launches"] * args.steps,
            "clocks": head["clocks"],
            "extras": extra_res,
        }
        if world == 1:
            sec, work, n = time_oracle(w, args.cpu_budget)
            line["cpu_baseline"] = {
                "value": work["bytes"] / sec / 1e12, "unit": UNIT,
                "cores": os.cpu_count(), "kind": "oracle",
                "sample": f"oracle write phase over all {w.num_tokens} tokens + read phase of "
                          f"the first {n} tokens ({sec:.1f} s, numpy float64, BLAS threads = "
                          f"host cores)"}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_reference(args, rank, world):
    """The oracle arm: rank 0 times the CPU oracle on the same workload and
    metric; each step is the oracle on one token's read phase (cycling
    through the batch) after its write phase."""
    if rank != 0:
        return 0
    from paged_latent_attention_cache_gb300 import workloads as W
    w = build_workload(args.workload, 0)
    one = oracle_session(w)
    T = w.num_tokens
    # keep the whole run within a few minutes
    per_step_budget = max(0.02, 120.0 / max(1, args.steps + args.warmup))

    for i in range(max(args.warmup, 3)):
        one(i % T)
    total_s, total_bytes, done = 0.0, 0, 0
    for i in range(args.steps):
        t = i % T
        t0 = time.perf_counter()
        one(t)
        total_s += time.perf_counter() - t0
        total_bytes += algorithmic_work(w, tokens=[t], include_write=False)["bytes"]
        done += 1
        if total_s > per_step_budget * args.steps:
            break
    value = total_bytes / total_s / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": done, "warmup": max(args.warmup, 3),
            "ms_per_step": 1e3 * total_s / done, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": W.dtype_tag(w.dtype), "data": "synthetic",
            "config": config_of(w, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": "one token's read phase per step, cycling through the "
                                       "batch, after one write phase over all tokens"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
