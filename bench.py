"""Benchmark: decode query-tokens/s and achieved HBM GB/s of the dynamic
sparse attention step (indexer -> radix top-k -> sparse GQA attention) at a
131,072-token context with top_k = 2,048, on synthetic data.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl libdsa|reference]
                    [--workload NAME] [--no-graph] [--op step|append|rope [--q-len S]]

One JSON line on stdout (rank 0). A step is one call of the whole decode path
(dsa_sparse_attn_decode) over one batch of query tokens with inputs resident
in HBM; L2 is flushed (a 256 MiB write) before every timed step, and each
step is timed with CUDA events on the stream the kernels run on. By default
the step is replayed from a CUDA graph captured around the C-ABI call; `e2e`
times the same call eagerly with the step's inputs copied from pinned host
memory and its output copied back. Under torchrun every rank runs its own
replica of the workload (the path shards by sequence with no exchange:
weak scaling); the slowest rank's time is reported.

By default the run also measures, in the same process and the same way, the
other four workloads (decode_4k, grouped_decode_32k, prefill_8k_on_32k,
decode_256k_int8) and reports each under "configs" with its own step time,
throughput, e2e, roofline (prefill: the indexer and the attention against the
bf16 tensor peak, with the attention's gather rate), per-kernel split, CPU
oracle baseline and clocks (--no-all-configs: the named workload only).

--op append times dsa_cache_append alone (the cache write before the step) on
the workload's shape and reports its HBM GB/s; --op rope does the same for
dsa_rmsnorm_rotary on the workload's query and key heads.

--impl reference times the float64 CPU oracle on the same workload (rank 0
only) -- a deliberately slow baseline, not the optimisation target.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode query-tokens/s and achieved HBM GB/s (% of peak) at L=128K, top_k=2048"
UNIT = "query-tokens/s"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ measured traffic
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one indexer
# launch per workload, from an ncu capture of that launch at full size (see
# profiles/). They hold for the indexer source they were taken on: the
# indexer's own file, the device headers it includes, and the part of the
# shared internal header it compiles against (its parameters and the cache
# addressing). When any of that changes, the figure is dropped (null) until it
# is measured again.
TRAFFIC_SOURCES = ["indexer.cu", "sm100_ptx.cuh", "dsa_common.cuh"]
TRAFFIC_SOURCE_SHA = "58e783604f49e682"
INDEXER_TRAFFIC = {"decode_4k": 580608, "grouped_decode_32k": 16910848, "decode_128k": 16834304,
                   "decode_256k_int8": 33632512}


def indexer_source_hash():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "top_sparse_attention_chunked_gb300", "csrc")
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    with open(os.path.join(csrc, "dsa_internal.h"), "rb") as fh:
        text = fh.read()
    # from the indexer's constants through its parameter block
    a = text.index(b"constexpr int kChunk")
    b = text.index(b"};", text.index(b"struct IndexerParams")) + 2
    h.update(text[a:b])
    return h.hexdigest()[:16]


def indexer_traffic(name):
    if indexer_source_hash() != TRAFFIC_SOURCE_SHA:
        return None
    return INDEXER_TRAFFIC.get(name)


# ------------------------------------------------------------------ algorithmic bytes
def algorithmic_bytes(wl, idx_np=None):
    """Bytes the method itself must move per step (DRAM), excluding work the
    sparse method avoids: every visible index key once, the fp32 scores
    written and read back, the unique selected K/V rows (with their scales),
    q, qI, w, the index rows and the output."""
    import numpy as np
    B, S = wl.batch, wl.q_len
    kv_elem = 1 if wl.kv_dtype == "int8" else 2
    row_kv = wl.num_kv_heads * (128 * kv_elem + (4 if wl.kv_dtype == "int8" else 0))
    n_vis = [[wl.total_len - S + s + 1 for s in range(S)] for _ in range(B)]
    kI = B * wl.total_len * 64 * 2
    scores = sum(sum(r) for r in n_vis) * 4 * 2
    if idx_np is not None:
        uniq = sum(len(np.unique(idx_np[b][idx_np[b] >= 0])) for b in range(B))
    else:
        uniq = B * min(wl.top_k, wl.total_len)
    kv = uniq * row_kv * 2
    small = B * S * (16 * 64 * 2 + 16 * 4 + wl.num_q_heads * 128 * 2 * 2 + wl.top_k * 4 * 2)
    indexer = kI + scores // 2 + B * S * (16 * 64 * 2 + 16 * 4)
    return {"step": kI + scores + kv + small, "indexer": indexer, "kv": kv}


def indexer_flops(wl):
    """2 * 16 heads * 64 dims per (query token, visible key)."""
    S, T = wl.q_len, wl.total_len
    vis = sum(T - S + s + 1 for s in range(S))
    return wl.batch * vis * 2 * 16 * 64


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm = [float(r[0]) for r in self.rows if len(r) >= 8 and r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if len(r) >= 8 and r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            if len(r) < 8:
                continue
            for i, n in enumerate(names):
                if r[4 + i].lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle leg
def oracle_rows(wl, max_rows=32):
    """Query rows the oracle leg times: all of them for decode-sized batches, a
    seeded sample (first and last included) when there are many."""
    import numpy as np
    rows = [(b, s) for b in range(wl.batch) for s in range(wl.q_len)]
    if len(rows) <= max_rows:
        return None, len(rows)
    rng = np.random.default_rng(0)
    pick = sorted({0, len(rows) - 1, *rng.choice(len(rows), max_rows - 2, replace=False).tolist()})
    return [rows[i] for i in pick], len(pick)


def oracle_step_time(wl, cpu, budget_s=10.0, max_reps=50):
    """Time the float64 oracle on steps of the workload (bounded). Returns
    (seconds per step, query tokens per step)."""
    import numpy as np
    import oracle.dsa_oracle as O
    from dsa_inputs import to_f64
    f = {k: to_f64(v) if hasattr(v, "numpy") else v for k, v in cpu.items()}
    f["total_len"] = cpu["total_len"].numpy().astype(np.int64)
    rows, ntok = oracle_rows(wl)
    times = []
    t_end = time.perf_counter() + budget_s
    while len(times) < max_reps and (not times or time.perf_counter() < t_end):
        t0 = time.perf_counter()
        O.sparse_attention_step(f, wl.num_kv_heads, wl.top_k, rows=rows)
        times.append(time.perf_counter() - t0)
    return times, ntok


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ reference arm
def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from dsa_inputs import make_inputs
    cpu = make_inputs(wl)
    for _ in range(args.warmup):
        oracle_step_time(wl, cpu, budget_s=0.0, max_reps=1)
    times = []
    for _ in range(args.steps):
        t, ntok = oracle_step_time(wl, cpu, budget_s=0.0, max_reps=1)
        times += t
    ms = 1e3 * statistics.mean(times)
    value = ntok / (ms / 1e3)
    sample = (f"{ntok} of {wl.query_tokens} query tokens of {wl.name} per timed step"
              if ntok < wl.query_tokens else
              f"full {wl.name} step ({wl.query_tokens} query tokens) per timed step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl, graph=False),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(wl, graph):
    return {"workload": wl.name, "batch": wl.batch, "q_len": wl.q_len,
            "context": wl.total_len, "top_k": wl.top_k, "q_heads": wl.num_q_heads,
            "kv_heads": wl.num_kv_heads, "head_dim": 128, "index_heads": 16, "index_dim": 64,
            "q_dtype": wl.q_dtype, "kv_dtype": wl.kv_dtype,
            "l2": "flushed before every timed step (256 MiB write)",
            "cuda_graph": bool(graph)}


def to_paged(dev, wl, block_size, spare, seed):
    """The workload's dense caches scattered over a shuffled pool of
    block_size-token blocks (the blocks that hold visible tokens plus `spare`
    unused ones), and the device block table [B, cap / block_size]."""
    import torch
    B, cap = wl.batch, wl.cap
    if cap % block_size:
        raise SystemExit(f"--paged {block_size}: the cache capacity {cap} is not a multiple")
    per_seq = cap // block_size
    used = -(-wl.total_len // block_size)
    nblocks = B * used + spare
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(nblocks, generator=g)[:B * used].view(B, used)
    table = torch.full((B, per_seq), -1, dtype=torch.int32)
    table[:, :used] = perm.to(torch.int32)
    table_d = table.cuda()
    src = perm.reshape(-1).cuda()
    pools = {}
    for name in ("kI", "k", "v", "k_scale", "v_scale"):
        d = dev.get(name)
        if d is None:
            pools[name] = None
            continue
        tail = tuple(d.shape[2:])
        pool = torch.zeros((nblocks, block_size) + tail, dtype=d.dtype, device="cuda")
        blocks = d[:, :used * block_size].reshape((B * used, block_size) + tail)
        pool[src] = blocks
        pools[name] = pool.view((nblocks * block_size,) + tail)
    return pools, table_d, nblocks


# ------------------------------------------------------------------ replicas
# Multi-GPU runs are independent replicas of the workload (the method has no
# exchange step): one process per GPU, each with its own seeded inputs; the
# job's time is the slowest rank's and its throughput counts every rank.
def replica_seed(wl, rank):
    return wl.seed + 7919 * rank


def slowest_rank_ms(ms, world, device=None):
    """The largest per-step time over all ranks (every rank receives it)."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world, query_tokens, ms):
    """Query tokens per second processed by all ranks together."""
    return world * query_tokens / (ms / 1e3)


# ------------------------------------------------------------------ libdsa arm
# The four workloads reported beside the headline (decode_128k) in the same
# JSON line, under "configs".
OTHER_WORKLOADS = ["decode_4k", "grouped_decode_32k", "prefill_8k_on_32k", "decode_256k_int8"]


def attention_flops_bytes(wl, idx_np):
    """Prefill attention's algorithmic work: 2 * 2 * Hq * 128 flop (QK^T and
    PV) per (query row, selected key), and its gather traffic (the selected K
    and V rows of every query row, Hkv * 128 16-bit values each)."""
    import numpy as np
    sel = int((idx_np >= 0).sum())
    flops = sel * 2 * 2 * wl.num_q_heads * 128
    elem = 1 if wl.kv_dtype == "int8" else 2
    gather = sel * wl.num_kv_heads * 128 * elem * 2
    return flops, gather


def measure_workload(args, wl, world, rank, dev_index, cpu_budget):
    """One workload: the graph-replayed step (L2 flushed before each), the
    roofline of its dominant kernels, the per-kernel split, the end-to-end
    call with host copies and (rank 0, N = 1) the CPU oracle. Returns the
    fields of its JSON entry."""
    import numpy as np
    import torch
    import torch.distributed as dist

    from dsa_inputs import make_inputs
    from top_sparse_attention_chunked_gb300 import dsa as D

    cpu = make_inputs(wl, seed=replica_seed(wl, rank))   # an independent replica per rank
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in cpu.items()}
    p = D.problem_for(wl)
    ws = D.alloc_workspace(p, D.DSA_OP_PREFILL if wl.q_len > 16 else D.DSA_OP_DECODE)
    out = torch.empty(wl.batch, wl.q_len, wl.num_q_heads, 128, dtype=D._TORCH_DT[p.out_dtype],
                      device="cuda")
    idx = torch.empty(wl.batch, wl.q_len, wl.top_k, dtype=torch.int32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    prefill = wl.q_len > 16
    call = D.dsa_sparse_attn_prefill if prefill else D.dsa_sparse_attn_decode
    caches = {k: dev[k] for k in ("kI", "k", "v", "k_scale", "v_scale")}
    pages = None
    if args.paged:
        # the same caches in a paged pool (13 spare blocks: the 256K layout's
        # 1,037 blocks of 256 tokens)
        pools, table_d, nblocks = to_paged(dev, wl, args.paged, 13, seed=wl.seed)
        pages = D.make_pages(table_d, args.paged, nblocks)
        caches = pools
        for k in ("kI", "k", "v", "k_scale", "v_scale"):
            dev[k] = None   # only the pool stays resident
        torch.cuda.empty_cache()

    def step():
        call(p, dev["q"], dev["qI"], dev["w"], caches["kI"], caches["k"], caches["v"],
             caches["k_scale"], caches["v_scale"], idx, out, ws, pages=pages)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert D.dsa_read_device_status(ws) == 0
    kernels_per_step = D.dsa_last_launches()   # what one call enqueues
    graph = None

    def capture():
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        return g

    def run_once():
        if graph is not None:
            graph.replay()
        else:
            step()

    def timed_loop(kernel_timing):
        """K steps, L2 flushed before each, CUDA events on the launching stream
        around every step (and, with kernel_timing, the library's events
        around one kernel launch)."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        kern_ms = []
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            run_once()
            evs[i][1].record(stream)
            torch.cuda.synchronize()
            if kernel_timing:
                kern_ms.append(D.dsa_timing_read())
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        return [a.elapsed_time(b) for a, b in evs], kern_ms

    # the headline loop: the step exactly as a caller runs it (no extra events
    # inside the step, so consecutive kernels keep their launch overlap)
    D.dsa_timing_select(-1)
    graph = capture() if args.graph else None
    clocks = ClockSampler(dev_index)
    clocks.start()
    step_ms, _ = timed_loop(False)
    clk = clocks.stop()
    ms = slowest_rank_ms(statistics.mean(step_ms), world, device="cuda")
    # the roofline loops: the same steps with events recorded around the
    # indexer launch (and, for prefill, around the attention launch)
    D.dsa_timing_select(D.DSA_KERNEL_INDEXER)
    graph = capture() if args.graph else None
    step_ms_t, idx_ms = timed_loop(True)
    attn_ms = []
    if prefill:
        D.dsa_timing_select(D.DSA_KERNEL_ATTENTION)
        graph = capture() if args.graph else None
        _, attn_ms = timed_loop(True)
    D.dsa_timing_select(-1)
    graph = None
    idx_np = idx.cpu().numpy()
    ab = algorithmic_bytes(wl, idx_np)
    hbm, bf16, peak_kind = peaks()
    value = whole_job_value(world, wl.query_tokens, ms)

    # ---------------- per-kernel breakdown (separate short eager loop)
    per_kernel = {}
    kinds = [("indexer", D.DSA_KERNEL_INDEXER),
             ("topk_row", D.DSA_KERNEL_TOPK_ROW) if prefill else ("topk_select", D.DSA_KERNEL_TOPK_SELECT),
             ("attention", D.DSA_KERNEL_ATTENTION)]
    for name, kind in kinds:
        D.dsa_timing_select(kind)
        vals = []
        for _ in range(10):
            flush.zero_()
            step()
            torch.cuda.synchronize()
            vals.append(D.dsa_timing_read())
        per_kernel[name] = round(1e3 * statistics.median(vals), 2)
    D.dsa_timing_select(-1)

    # ---------------- end to end through the C ABI with host buffers
    # The step's inputs (q, qI, w) live in one pinned host buffer and one
    # device buffer (256-byte aligned slices viewed as the tensors), so each
    # step copies them in with one host-to-device copy.
    names = ("q", "qI", "w")
    offs, nbytes = {}, 0
    for k2 in names:
        offs[k2] = nbytes
        nbytes += (cpu[k2].numel() * cpu[k2].element_size() + 255) // 256 * 256
    pin_buf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    for k2 in names:
        n2 = cpu[k2].numel() * cpu[k2].element_size()
        pin_buf[offs[k2]:offs[k2] + n2].copy_(cpu[k2].contiguous().view(-1).view(torch.uint8))
        dev[k2] = dev_buf[offs[k2]:offs[k2] + n2].view(cpu[k2].dtype).view(cpu[k2].shape)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = nbytes
    d2h = out_h.numel() * out_h.element_size()
    for _ in range(3):
        dev_buf.copy_(pin_buf, non_blocking=True)
        step()
        out_h.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dev_buf.copy_(pin_buf, non_blocking=True)
        step()
        out_h.copy_(out, non_blocking=True)
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    e2e = whole_job_value(world, wl.query_tokens,
                          slowest_rank_ms(statistics.mean(e2e_ms), world, device="cuda"))

    # ---------------- CPU oracle baseline (rank 0, N = 1 only)
    cpu_base = None
    if rank == 0 and world == 1:
        times, ntok = oracle_step_time(wl, cpu, budget_s=cpu_budget)
        what = (f"{ntok} sampled query rows of" if ntok < wl.query_tokens else "full")
        cpu_base = {"value": ntok / statistics.mean(times), "unit": UNIT,
                    "cores": cores(), "kind": "oracle",
                    "sample": f"{len(times)} x {what} {wl.name} step ({ntok} query "
                              f"token(s) each) in float64 NumPy"}
        if ntok < wl.query_tokens:
            cpu_base["extrapolated_step_s"] = round(statistics.mean(times) * wl.query_tokens / ntok, 3)

    idx_us = 1e3 * statistics.mean(idx_ms)
    step_gbs = ab["step"] / (ms * 1e-3) / 1e9
    if prefill:
        # the dense causal indexer contraction is tensor-bound
        flops = indexer_flops(wl)
        achieved = flops / (idx_us * 1e-6) / 1e12
        roof = {"kernel": "indexer_tc_kernel", "bound": "tensor", "achieved": round(achieved, 1),
                "peak": bf16, "unit": "TFLOP/s", "frac": round(achieved / bf16, 4),
                "peak_kind": peak_kind, "traffic": None, "algorithmic_flops": flops,
                "launch_us_events": round(idx_us, 2)}
        attn_us = 1e3 * statistics.mean(attn_ms)
        aflops, gbytes = attention_flops_bytes(wl, idx_np)
        a_tf = aflops / (attn_us * 1e-6) / 1e12
        roof_attn = {"kernel": "sparse_attn_prefill_tc_kernel", "bound": "tensor",
                     "achieved": round(a_tf, 1), "peak": bf16, "unit": "TFLOP/s",
                     "frac": round(a_tf / bf16, 4), "peak_kind": peak_kind,
                     "algorithmic_flops": aflops, "launch_us_events": round(attn_us, 2),
                     # the selected rows are gathered from the L2-resident cache:
                     # the rate it moves them at is the kernel's practical bound
                     "gather_bytes": gbytes,
                     "gather_gbs": round(gbytes / (attn_us * 1e-6) / 1e9, 1)}
    else:
        achieved = ab["indexer"] / (idx_us * 1e-6) / 1e9
        roof = {"kernel": "indexer_tc_kernel", "bound": "hbm", "achieved": round(achieved, 1),
                "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "peak_kind": peak_kind, "traffic": indexer_traffic(wl.name),
                "algorithmic_bytes": ab["indexer"],
                # events around the launch inside the graph break its overlap with
                # the kernel before it, so this time includes that gap
                "launch_us_events": round(idx_us, 2)}
        roof_attn = None
    res = {
        "ms_per_step": ms, "value": value,
        "config": dict(config_of(wl, args.graph),
                       **({"paged": {"block_size": args.paged, "num_blocks": pages.num_blocks}}
                          if pages is not None else {})),
        "hbm_gbs_step": round(step_gbs, 1),
        "hbm_frac_step": round(step_gbs / hbm, 4),
        "hbm_frac_step_of_8tbs": round(step_gbs / 8000.0, 4),
        "algorithmic_bytes_step": ab["step"],
        "roofline": roof,
        "per_kernel_us": per_kernel,
        "ms_per_step_with_indexer_events": statistics.mean(step_ms_t),
        "cpu_baseline": cpu_base,
        "e2e": {"value": e2e, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": statistics.mean(e2e_ms)},
        # the library's own count of the kernels one call enqueues, times the
        # timed steps of the headline loop
        "gpu_launches": len(kernels_per_step) * args.steps,
        "kernels_per_step": kernels_per_step,
        "clocks": clk,
    }
    if roof_attn is not None:
        res["roofline_attention"] = roof_attn
    del dev, caches, ws, out, idx, flush
    torch.cuda.empty_cache()
    return res


def run_libdsa(args, wl):
    import torch
    import torch.distributed as dist

    from dsa_inputs import WORKLOADS, make_inputs
    from top_sparse_attention_chunked_gb300 import build_lib
    from top_sparse_attention_chunked_gb300 import dsa as D

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build_lib.build()
    D.load_library()
    dev_index = torch.cuda.current_device()

    if args.profile_calls:
        # untimed calls only, for an ncu capture of the step's kernels
        cpu = make_inputs(wl, seed=replica_seed(wl, rank))
        dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in cpu.items()}
        p = D.problem_for(wl)
        ws = D.alloc_workspace(p, D.DSA_OP_PREFILL if wl.q_len > 16 else D.DSA_OP_DECODE)
        out = torch.empty(wl.batch, wl.q_len, wl.num_q_heads, 128, dtype=D._TORCH_DT[p.out_dtype],
                          device="cuda")
        idx = torch.empty(wl.batch, wl.q_len, wl.top_k, dtype=torch.int32, device="cuda")
        call = D.dsa_sparse_attn_prefill if wl.q_len > 16 else D.dsa_sparse_attn_decode
        for _ in range(args.profile_calls):
            call(p, dev["q"], dev["qI"], dev["w"], dev["kI"], dev["k"], dev["v"],
                 dev["k_scale"], dev["v_scale"], idx, out, ws)
        torch.cuda.synchronize()
        assert D.dsa_read_device_status(ws) == 0
        if rank == 0:
            print(json.dumps({"profile_calls": args.profile_calls, "workload": wl.name,
                              "kernels_per_step": D.dsa_last_launches()}), flush=True)
        return

    head = measure_workload(args, wl, world, rank, dev_index, args.cpu_budget)
    others = {}
    if args.all_configs:
        for name in OTHER_WORKLOADS:
            if name == wl.name:
                continue
            r = measure_workload(args, WORKLOADS[name], world, rank, dev_index,
                                 min(args.cpu_budget, 5.0))
            others[name] = r
    if rank == 0:
        line = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16",
                "data": "synthetic (seeded N(0,1) / U(0,1) tensors, see dsa_inputs.py)"}
        line.update({k: v for k, v in head.items() if k not in ("value", "ms_per_step")})
        # every launch of the measured runs counts, the other workloads' included
        line["gpu_launches"] = head["gpu_launches"] + sum(r["gpu_launches"] for r in others.values())
        if others:
            line["configs"] = others
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def append_bytes(batch, q_len, num_kv_heads, q_dtype, kv_dtype):
    """Algorithmic bytes of one cache append: every new-token byte read once
    and every cache byte it produces written once (index key 64 bf16; K and V
    rows of 128 elements per KV head; INT8 adds a 4-byte scale per row)."""
    tokens = batch * q_len
    read = tokens * (64 * 2 + 2 * num_kv_heads * 128 * 2)
    row_out = 128 + 4 if kv_dtype == "int8" else 256
    write = tokens * (64 * 2 + 2 * num_kv_heads * row_out)
    return read + write


def run_append_bench(args, wl):
    """--op append: dsa_cache_append alone on the workload's shape (batch,
    KV heads, dtypes; --q-len new tokens per sequence, default the
    workload's), timed per call with CUDA events after an L2 flush."""
    import torch

    from dsa_inputs import make_append_inputs
    from top_sparse_attention_chunked_gb300 import build_lib
    from top_sparse_attention_chunked_gb300 import dsa as D

    build_lib.build()
    D.load_library()
    S = args.q_len or wl.q_len
    T = max(wl.total_len, S)
    cap = T
    cpu = make_append_inputs(wl.batch, S, wl.num_kv_heads, cap, [T] * wl.batch, wl.q_dtype,
                             wl.kv_dtype, seed=wl.seed, specials=False)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in cpu.items()}
    p = D.make_problem(batch=wl.batch, q_len=S, total_len=[T] * wl.batch, top_k=1,
                       num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                       cache_capacity=cap, q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        D.dsa_cache_append(p, dev["kI_new"], dev["k_new"], dev["v_new"], dev["kI"], dev["k"],
                           dev["v"], dev["k_scale"], dev["v_scale"])

    if args.profile_calls:
        for _ in range(args.profile_calls):
            step()
        torch.cuda.synchronize()
        print(json.dumps({"profile_calls": args.profile_calls, "op": "append",
                          "kernels_per_step": D.dsa_last_launches()}), flush=True)
        return
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    kernels = D.dsa_last_launches()

    def graph_of():
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        return g

    def timed(g, kernel_events):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        kern = []
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            g.replay()
            evs[i][1].record(stream)
            if kernel_events:
                torch.cuda.synchronize()
                kern.append(D.dsa_timing_read())
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evs), kern

    # the step as a caller replays it (graph), then the kernel alone (events
    # recorded by the library around its launch, captured in the graph)
    D.dsa_timing_select(-1)
    g = graph_of()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    ms, _ = timed(g, False)
    clk = clocks.stop()
    D.dsa_timing_select(D.DSA_KERNEL_APPEND)
    g = graph_of()
    _, kern_ms = timed(g, True)
    D.dsa_timing_select(-1)
    kms = statistics.mean(kern_ms)
    nbytes = append_bytes(wl.batch, S, wl.num_kv_heads, wl.q_dtype, wl.kv_dtype)
    gbs = nbytes / (ms * 1e-3) / 1e9
    kgbs = nbytes / (kms * 1e-3) / 1e9
    hbm, _, peak_kind = peaks()
    print(json.dumps({
        "metric": "cache append achieved HBM GB/s", "value": round(gbs, 1), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": f"{wl.q_dtype}->{wl.kv_dtype}",
        "data": "synthetic (seeded N(0,1) rows of magnitude 10^U(-3,3), see dsa_inputs.py)",
        "config": {"workload": f"cache append of {S} tokens x {wl.batch} sequence(s), "
                               f"{wl.num_kv_heads} KV heads, {wl.q_dtype} -> {wl.kv_dtype}",
                   "l2": "flushed (256 MiB write) before every step", "graph": True},
        "tokens_per_s": wl.batch * S / (ms * 1e-3),
        "roofline": {"kernel": "cache_append_kernel", "bound": "hbm", "achieved": round(kgbs, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(kgbs / hbm, 4),
                     "peak_kind": peak_kind, "traffic": None, "algorithmic_bytes": nbytes,
                     "launch_us": round(kms * 1e3, 2)},
        "gpu_launches": len(kernels) * args.steps, "kernels_per_step": kernels,
        "clocks": clk}), flush=True)


def run_rope_bench(args, wl):
    """--op rope: dsa_rmsnorm_rotary alone on the query and key heads of the
    workload's new tokens (--q-len tokens, default the workload's; head dim
    128, full rotary width, FP32 cos / sin cache), timed per call."""
    import torch

    from dsa_inputs import make_rope_inputs
    from top_sparse_attention_chunked_gb300 import build_lib
    from top_sparse_attention_chunked_gb300 import dsa as D

    build_lib.build()
    D.load_library()
    N = args.q_len or wl.q_len
    H = wl.num_q_heads + wl.num_kv_heads
    r = 128
    max_pos = wl.total_len
    inp = make_rope_inputs(N, H, 128, r, max_pos, wl.q_dtype, "fp32", seed=wl.seed,
                           first_pos=max(0, wl.total_len - N))
    x = inp["x"].cuda()
    y = torch.empty_like(x)
    g, c, sn, pos = (inp[k].cuda() for k in ("gamma", "cos", "sin", "positions"))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        D.dsa_rmsnorm_rotary(x, g, y, eps=1e-6, cos_cache=c, sin_cache=sn, positions=pos,
                             rotary_dim=r)

    if args.profile_calls:
        for _ in range(args.profile_calls):
            step()
        torch.cuda.synchronize()
        print(json.dumps({"profile_calls": args.profile_calls, "op": "rope",
                          "kernels_per_step": D.dsa_last_launches()}), flush=True)
        return
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    kernels = D.dsa_last_launches()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        graph.replay()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    # every x element read and every y element written once, plus each
    # token's cos / sin row
    nbytes = N * H * 128 * 2 * 2 + N * (r // 2) * 4 * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    hbm, _, peak_kind = peaks()
    print(json.dumps({
        "metric": "RMSNorm + rotary embedding achieved HBM GB/s", "value": round(gbs, 1),
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "f32 arithmetic, bf16 in/out",
        "data": "synthetic (seeded, see dsa_inputs.make_rope_inputs)",
        "config": {"workload": f"RMSNorm + RoPE of {N} tokens x {H} heads x 128 "
                               f"(query and key heads of {wl.name})",
                   "l2": "flushed (256 MiB write) before every step", "graph": True},
        "roofline": {"kernel": "rmsnorm_rotary_kernel", "bound": "hbm", "achieved": round(gbs, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                     "peak_kind": peak_kind, "traffic": None, "algorithmic_bytes": nbytes},
        "gpu_launches": len(kernels) * args.steps, "kernels_per_step": kernels,
        "clocks": clk}), flush=True)


def run_layer_bench(args, wl):
    """--op layer: one decoding layer's step built from the library's calls,
    replayed from one CUDA graph: RMSNorm + RoPE of q, qI, the new k and kI
    (positions T - S + s), the cache append of kI, k, v, then the decode."""
    import torch

    from dsa_inputs import make_append_inputs, make_inputs, make_rope_inputs
    from top_sparse_attention_chunked_gb300 import build_lib
    from top_sparse_attention_chunked_gb300 import dsa as D

    build_lib.build()
    D.load_library()
    B, S, Hq, Hkv, cap = wl.batch, wl.q_len, wl.num_q_heads, wl.num_kv_heads, wl.cap
    cpu = make_inputs(wl)
    app = make_append_inputs(B, S, Hkv, 1, [1] * B, wl.q_dtype, wl.kv_dtype, seed=wl.seed + 1,
                             specials=False)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in cpu.items()}
    new = {k: app[k].cuda() for k in ("kI_new", "k_new", "v_new")}
    p = D.problem_for(wl)
    ws = D.alloc_workspace(p, D.DSA_OP_DECODE)
    out = torch.empty(B, S, Hq, 128, dtype=D._TORCH_DT[p.out_dtype], device="cuda")
    idx = torch.empty(B, S, wl.top_k, dtype=torch.int32, device="cuda")
    rope = {}
    for name, H, Dh in (("q", Hq, 128), ("qI", 16, 64), ("k", Hkv, 128), ("kI", 1, 64)):
        r = make_rope_inputs(B * S, H, Dh, Dh, cap, wl.q_dtype, "fp32", seed=wl.seed + H)
        r["positions"] = torch.tensor([wl.total_len - S + s for _ in range(B) for s in range(S)],
                                      dtype=torch.int32)
        rope[name] = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in r.items()}
    views = {"q": dev["q"].view(B * S, Hq, 128), "qI": dev["qI"].view(B * S, 16, 64),
             "k": new["k_new"].view(B * S, Hkv, 128), "kI": new["kI_new"].view(B * S, 1, 64)}
    raw = {n: views[n].clone() for n in views}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step_chain():
        for n in ("q", "qI", "k", "kI"):
            r = rope[n]
            D.dsa_rmsnorm_rotary(raw[n], r["gamma"], views[n], eps=1e-6, cos_cache=r["cos"],
                                 sin_cache=r["sin"], positions=r["positions"])
        D.dsa_cache_append(p, new["kI_new"], new["k_new"], new["v_new"], dev["kI"], dev["k"],
                           dev["v"], dev["k_scale"], dev["v_scale"])
        D.dsa_sparse_attn_decode(p, dev["q"], dev["qI"], dev["w"], dev["kI"], dev["k"], dev["v"],
                                 dev["k_scale"], dev["v_scale"], idx, out, ws)

    def step_fused():
        # (q and qI are rotated in place: each replay renormalises them again)
        D.dsa_rope_append(p, dev["q"], dev["qI"], new["k_new"], new["kI_new"], new["v_new"],
                          dev["kI"], dev["k"], dev["v"], dev["k_scale"], dev["v_scale"],
                          rope["q"]["gamma"], rope["k"]["gamma"], rope["qI"]["gamma"],
                          rope["kI"]["gamma"], eps=1e-6, cos=rope["q"]["cos"], sin=rope["q"]["sin"],
                          cos_index=rope["qI"]["cos"], sin_index=rope["qI"]["sin"])
        D.dsa_sparse_attn_decode(p, dev["q"], dev["qI"], dev["w"], dev["kI"], dev["k"], dev["v"],
                                 dev["k_scale"], dev["v_scale"], idx, out, ws)

    step = step_fused if args.fused else step_chain

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert D.dsa_read_device_status(ws) == 0
    # four RMSNorm + RoPE launches and the append (or the one fused launch),
    # then the decode's kernels
    kernels = ((["rope_append_kernel"] if args.fused
                else ["rmsnorm_rotary_kernel"] * 4 + ["cache_append_kernel"]) + D.dsa_last_launches())
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        graph.replay()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    print(json.dumps({
        "metric": "decoding layer step (RMSNorm+RoPE, cache append, sparse attention) query-tokens/s",
        "value": wl.query_tokens / (ms * 1e-3), "unit": "query-tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic (seeded, see dsa_inputs.py)",
        "config": dict(config_of(wl, True), op="layer", fused_prologue=bool(args.fused)),
        "gpu_launches": len(kernels) * args.steps, "kernels_per_step": kernels,
        "clocks": clk}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="libdsa", choices=["libdsa", "reference"])
    ap.add_argument("--workload", default="decode_128k")
    ap.add_argument("--no-all-configs", dest="all_configs", action="store_false",
                    help="measure only --workload (by default the headline run also measures "
                         "the other four workloads and reports them under \"configs\")")
    ap.add_argument("--no-graph", dest="graph", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--profile-calls", type=int, default=0,
                    help="run this many untimed calls and exit (for ncu captures)")
    ap.add_argument("--fused", action="store_true",
                    help="with --op layer: RMSNorm+RoPE and the append as one launch")
    ap.add_argument("--paged", type=int, default=0,
                    help="run the step on a paged cache with blocks of this many tokens")
    ap.add_argument("--op", default="step", choices=["step", "append", "rope", "layer"],
                    help="append: time dsa_cache_append alone on the workload's shape; "
                         "rope: time dsa_rmsnorm_rotary on its query and key heads; "
                         "layer: RMSNorm+RoPE, append and decode as one graph")
    ap.add_argument("--q-len", type=int, default=0,
                    help="with --profile-calls: query tokens per sequence of a reduced case; "
                         "with --op append: new tokens per sequence")
    ap.add_argument("--context", type=int, default=0,
                    help="with --profile-calls: cache length of a reduced case")
    args = ap.parse_args()
    if args.workload != "decode_128k" or args.paged:
        args.all_configs = False
    if args.warmup < 3:
        args.warmup = 3
    from dsa_inputs import WORKLOADS
    wl = WORKLOADS[args.workload]
    if args.op == "append":
        run_append_bench(args, wl)
        return
    if args.op == "rope":
        run_rope_bench(args, wl)
        return
    if args.op == "layer":
        run_layer_bench(args, wl)
        return
    if args.profile_calls and (args.q_len or args.context):
        # a reduced case of the same structure (heads, top_k, dtypes)
        from dsa_inputs import small_workload
        wl = small_workload(name=f"{wl.name}_reduced", batch=wl.batch,
                            q_len=args.q_len or wl.q_len, total_len=args.context or wl.total_len,
                            num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                            top_k=wl.top_k, q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype,
                            bias_frac=wl.bias_frac, seed=wl.seed)
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_libdsa(args, wl)


if __name__ == "__main__":
    main()
