#!/usr/bin/env python
"""Benchmark of the MSA hot path on GB300.

One step = one pass of the sparse-prefill hot path over the S=32768
workload (batch 1, 32 query / 8 KV heads, d=128, 8 proxy heads of 64, one
shared proxy K head, 128-token pages, topk=16, identity page table,
bf16 N(0,1) inputs): msa_proxy_maxscore -> msa_topk_select ->
msa_sparse_attn.  The JSON line reports tokens/s of that step (value),
the attention kernel's TFLOP/s counted on the selected blocks against the
tensor roofline, the FP8 paged decode's HBM GB/s (32 sequences x 131072
keys, 64/8 heads, e4m3 K/V), an end-to-end figure through host buffers,
and the fp64 oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs its own replica of the workload (the path
needs no exchange between GPUs); value = all ranks' tokens / the slowest
rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-prefill tokens/s & TFLOP/s (selected blocks) at S=32K; decode HBM GB/s"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# dram bytes of one attention-forward launch at the 32K prefill workload from
# an ncu capture, valid only for the kernel source it was taken on.
# Captured on S=16384 (15424 selected tile-blocks: 244.9 MB read + 108.7 MB
# written) and scaled by selected tile-blocks to the S=32768 launch (31808).
NCU_TRAFFIC = {
    # (DRAM bytes read + written) of one launch of the small S=16384 capture and the
    # (tile, group, block) selections it processed; scaled to a launch by selections.
    "attn_fwd.cu": {"src": "ddc78d865d0567a3", "bytes": 244076288 + 108070400, "sel": 15424},
    "attn_fwd.cu:fp8": {"src": "ddc78d865d0567a3", "bytes": 180636416 + 101585152, "sel": 15424},
}


def ncu_traffic(key, n_sel):
    """DRAM traffic of one launch from the committed ncu capture, or None when
    the kernel source has changed since the counters were taken."""
    t = NCU_TRAFFIC.get(key)
    if not t or t["src"] != src_hash(key.split(":")[0]):
        return None
    return int(t["bytes"] * n_sel / t["sel"])


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def src_hash(name):
    """Hash of a kernel source's code: comments and whitespace are dropped, so
    a comment edit keeps the counters taken on that code."""
    with open(os.path.join(ROOT, "block_sparse_long_proxy_gb300", "csrc", name)) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()[:16]


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out = ""
        else:
            self.out = ""

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


class L2Flush:
    """Evicts L2 between timed steps, outside the timed region: a 256 MiB
    write followed by a 256 MiB read of a second buffer, so that the dirty
    lines of the write are written back before the next step starts and the
    step finds L2 holding only clean, unrelated lines."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def dist_setup(args):
    """One process per GPU under torchrun; NCCL on GPUs, gloo on a host-only run."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if torch.cuda.is_available():
        torch.cuda.set_device(local if world > 1 else 0)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def _reduce(x, world, op):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def allreduce_max(x, world):
    import torch.distributed as dist
    return _reduce(x, world, dist.ReduceOp.MAX if world > 1 else None)


def allreduce_sum(x, world):
    import torch.distributed as dist
    return _reduce(x, world, dist.ReduceOp.SUM if world > 1 else None)


def job_throughput(units_local, ms_local, world):
    """Whole-job throughput of independent replicas: the units every rank
    processed divided by the slowest rank's time.  Returns (units/s, max ms)."""
    ms = allreduce_max(ms_local, world)
    units = allreduce_sum(units_local, world)
    return units / (ms / 1e3), ms


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------ oracle (CPU)

def oracle_inputs(inp_cpu):
    """The bit patterns the oracle reads, decoded once per run."""
    from block_sparse_long_proxy_gb300 import synth
    return {k: synth.bits(inp_cpu[k]) for k in ("pq", "pk_pages", "q", "k_pages", "v_pages")}


def oracle_sample(case, inp_cpu, n_tiles_sample, seed=0, bits=None):
    """Run the fp64 oracle's whole chain (proxy max-score, top-k, attention)
    on a seeded sample of tiles; returns (query rows processed, seconds)."""
    import numpy as np
    from oracle import msa_oracle as O
    tiles = O.tiles_of(case.qo_lens, case.kv_lens)
    rng = np.random.default_rng(seed)
    ids = sorted(rng.choice(len(tiles), size=min(n_tiles_sample, len(tiles)), replace=False).tolist())
    table = inp_cpu["kv_indices"].numpy()
    nvp = O.num_valid_pages(case.qo_lens, case.kv_lens)
    if bits is None:
        bits = oracle_inputs(inp_cpu)
    t0 = time.perf_counter()
    ms = O.proxy_max_score(bits["pq"], bits["pk_pages"], table, case.qo_lens, case.kv_lens, tile_ids=ids)
    idx = np.full((len(tiles), case.hkv, case.topk), -1, np.int32)
    idx[ids] = O.topk_select(ms[ids], case.topk, nvp[ids])
    kw = {}
    if case.kv_dtype != "bf16":
        kw = dict(k_scale=inp_cpu["k_scale"].numpy(), v_scale=inp_cpu["v_scale"].numpy())
    O.sparse_attention(bits["q"], bits["k_pages"], bits["v_pages"], table, idx, case.qo_lens, case.kv_lens,
                       tile_ids=ids, **kw)
    dt = time.perf_counter() - t0
    rows = sum(tiles[i].q_end - tiles[i].q_begin for i in ids)
    return rows, dt, ids


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def bench_config(case, world):
    """The workload of the JSON line, the same for both arms."""
    return {"workload": case.name, "batch": 1, "seq_len": 32768, "heads": "32q/8kv", "head_dim": 128,
            "proxy_heads": 8, "proxy_dim": 64, "topk": 16, "page_size": 128,
            "parallelism": "replicas" if world > 1 else "single",
            "l2": "flushed between timed steps (256 MiB write, then 256 MiB read)"}


def run_reference(args):
    """The oracle, as it stands, on the host cores, on the same workload."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from block_sparse_long_proxy_gb300 import synth
    case = synth.prefill_32k()
    inp = synth.make_inputs(case, device="cpu")
    bits = oracle_inputs(inp)
    # a step is a bounded sample: two tiles, or one when many steps are asked
    # for, so that the run stays within minutes
    per_step_tiles = 2 if args.steps <= 100 else 1
    for w in range(args.warmup):
        oracle_sample(case, inp, per_step_tiles, seed=1000 + w, bits=bits)
    rows = 0
    secs = 0.0
    for k in range(args.steps):
        r, dt, _ = oracle_sample(case, inp, per_step_tiles, seed=k, bits=bits)
        rows += r
        secs += dt
    value = rows / secs
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(case, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": "%d random query tiles of 128 rows per step through the whole oracle chain "
                                       "(proxy max-score, top-k, attention)" % per_step_tiles},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------- ours (GPU)

def selected_flops(idx_cpu, case):
    """4*T*B*d per (tile, head, selected block), counting whole blocks."""
    n_sel = int((idx_cpu >= 0).sum())             # (tile, group, block) triples
    return n_sel * (case.hq // case.hkv) * 4.0 * 128 * 128 * case.d, n_sel


def visible_pair_flops(idx_cpu, case):
    """4*d per visible (query, key) pair of the selected blocks, per head: the
    exact count, in which the diagonal block counts about half."""
    import numpy as np
    total = 0
    t = 0
    for ql, kl in zip(case.qo_lens, case.kv_lens):
        off = kl - ql
        for r0 in range(0, ql, 128):
            rows = np.arange(r0, min(r0 + 128, ql)) + off           # absolute query positions
            sel = idx_cpu[t][idx_cpu[t] >= 0]                      # [groups x blocks] selected
            for j in np.unique(sel):
                cnt = int((sel == j).sum())                        # groups that selected block j
                k0, k1 = 128 * int(j), min(128 * int(j) + 128, kl)
                vis = np.clip(np.minimum(rows + 1, k1) - k0, 0, None).sum()
                total += cnt * int(vis)
            t += 1
    return total * (case.hq // case.hkv) * 4.0 * case.d


def run_ours(args):
    import torch
    world, rank, local = dist_setup(args)
    from block_sparse_long_proxy_gb300 import msa, synth
    dev = torch.device("cuda", torch.cuda.current_device())
    pk_info, peak_kind = peaks()
    case = synth.prefill_32k()
    case.seed = rank
    inp = synth.make_inputs(case, device=dev)
    plan = msa.Plan(case.qo_lens, case.kv_lens, case.hq, case.hkv, case.hp, case.d, case.dp, case.topk,
                    num_pages=inp["k_pages"].shape[0])
    ms = torch.empty((plan.n_tiles, case.hp, plan.max_blocks), dtype=torch.float32, device=dev)
    idx = torch.empty((plan.n_tiles, case.hkv, case.topk), dtype=torch.int32, device=dev)
    out = torch.empty_like(inp["q"])
    lse = torch.empty((plan.total_q, case.hq), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"], out=ms)
        if ev:
            ev[1].record(stream)
        msa.topk_select(ms, case.topk, plan.num_valid_pages, out=idx)
        if ev:
            ev[2].record(stream)
        plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx, out=out, lse=lse)
        if ev:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    plan.check_errors()
    flops, n_sel = selected_flops(idx.cpu().numpy(), case)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for k in range(args.steps):
            flush()                            # evict L2 between timed steps (untimed)
            step(evs[k])
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    plan.check_errors()
    st = [[evs[k][i].elapsed_time(evs[k][i + 1]) for i in range(3)] for k in range(args.steps)]
    step_ms = [sum(s) for s in st]
    value, total_ms = job_throughput(case.total_q * args.steps, sum(step_ms), world)
    proxy_ms = statistics.mean(s[0] for s in st)
    topk_ms = statistics.mean(s[1] for s in st)
    attn_ms = statistics.mean(s[2] for s in st)

    # the fused proxy + top-k call (msa_proxy_topk), timed the same way
    # outside the headline step, which keeps the two separate calls (faster
    # here: the fused selection lengthens every proxy CTA's tail)
    fused_ms = []
    for _ in range(args.steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        plan.proxy_topk(inp["pq"], inp["pk_pages"], inp["kv_indices"], out=idx)
        b.record(stream)
        torch.cuda.synchronize()
        fused_ms.append(a.elapsed_time(b))
    plan.check_errors()

    # proxy FLOPs: causal lower triangle of 128x128 blocks per proxy head
    proxy_flops = sum(t.nvp for t in plan_tiles(case)) * case.hp * 2.0 * 128 * 128 * case.dp
    attn_tflops = flops / (attn_ms / 1e3) / 1e12
    proxy_tflops = proxy_flops / (proxy_ms / 1e3) / 1e12
    peak_bf16 = pk_info.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    traffic = ncu_traffic("attn_fwd.cu", n_sel)
    roofline = {"bound": "tensor", "kernel": "attn_fwd_kernel<128> (msa_sparse_attn)", "achieved": attn_tflops,
                "peak": peak_bf16, "unit": "TFLOP/s", "frac": attn_tflops / peak_bf16,
                "traffic": traffic,
                "peak_kind": "%s bf16 dense burst (cuBLAS)" % peak_kind,
                "flops_per_launch": flops, "selected_blocks": n_sel,
                "visible_pair_flops": visible_pair_flops(idx.cpu().numpy(), case),
                "nominal_frac": attn_tflops / 2250.0}

    # End to end through host buffers: every step copies all of its inputs
    # host -> device from pinned memory, runs the three calls, and copies out
    # device -> host.  Steps are pipelined the way a serving loop would be:
    # copies in, compute and copies out run on three streams over two sets of
    # device buffers, so step k+1's inputs and step k-1's output move while
    # step k computes.
    names = ["q", "k_pages", "v_pages", "pq", "pk_pages", "kv_indices"]
    host = {n: inp[n].cpu().pin_memory() for n in names}
    out_host = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = out_host[0].numel() * out_host[0].element_size()
    dev_in = [inp, {n: torch.empty_like(inp[n]) for n in names}]
    dev_out = [out, torch.empty_like(out)]
    s_in, s_cmp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    e2e_steps = max(4, min(args.steps, 10))

    def e2e_step(k, ev):
        b = k % 2
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(ev["cmp"][b])           # buffers of step k-2 no longer read
            for n in names:
                dev_in[b][n].copy_(host[n], non_blocking=True)
            ev["in"][b].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev["in"][b])
            if k >= 2:
                s_cmp.wait_event(ev["out"][b])          # out of step k-2 copied to the host
            x = dev_in[b]
            plan.proxy_maxscore(x["pq"], x["pk_pages"], x["kv_indices"], out=ms, stream=s_cmp)
            msa.topk_select(ms, case.topk, plan.num_valid_pages, out=idx, stream=s_cmp)
            plan.sparse_attn(x["q"], x["k_pages"], x["v_pages"], x["kv_indices"], idx, out=dev_out[b], lse=lse,
                             stream=s_cmp)
            ev["cmp"][b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["cmp"][b])
            out_host[b].copy_(dev_out[b], non_blocking=True)
            ev["out"][b].record(s_out)

    def new_events():
        return {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "cmp", "out")}
    torch.cuda.synchronize()
    ev = new_events()
    for k in range(2):                                  # warm the streams
        e2e_step(k, ev)
    torch.cuda.synchronize()
    barrier(world)
    ev = new_events()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_cmp.wait_event(e0)
    s_out.wait_event(e0)
    for k in range(e2e_steps):
        e2e_step(k, ev)
    s_in.wait_stream(s_out)
    s_in.wait_stream(s_cmp)
    e1.record(s_in)
    torch.cuda.synchronize()
    plan.check_errors()
    e2e_value, e2e_ms = job_throughput(case.total_q * e2e_steps, e0.elapsed_time(e1), world)

    decode = bench_decode(args, dev, pk_info, peak_kind, world)
    train = bench_train(args, dev, pk_info, peak_kind)
    fp8_prefill = bench_prefill_fp8(args, dev, pk_info, peak_kind, attn_tflops)
    varlen = bench_varlen(args, dev, pk_info, peak_kind)

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": bench_config(case, world),
            "stages_ms": {"proxy_maxscore": proxy_ms, "topk_select": topk_ms, "sparse_attn": attn_ms},
            "proxy_topk_fused_ms": statistics.median(fused_ms),
            "tflops_selected": attn_tflops, "proxy_tflops": proxy_tflops,
            "roofline": roofline,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps,
                    "pipelining": "H2D of every input from pinned memory, the three calls and D2H of out on three "
                                  "streams over two device buffer sets"},
            "gpu_launches": 3 * args.steps,
            "clocks": clk.summary(),
            "wall_s": t_wall}
    if fp8_prefill:
        line["prefill_fp8"] = fp8_prefill
    if varlen:
        line["varlen_paged"] = varlen
    if decode:
        line["decode"] = decode
    if train:
        line["training"] = train
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _tiles_nvp(case):
    """num_valid_pages of every tile (bottom-right causal, 128-row tiles)."""
    out = []
    for ql, kl in zip(case.qo_lens, case.kv_lens):
        off = kl - ql
        for t in range((ql + 127) // 128):
            r1 = min((t + 1) * 128, ql)
            out.append((off + r1 - 1) // 128 + 1)
    return out


class _T:
    def __init__(self, nvp):
        self.nvp = nvp


def plan_tiles(case):
    return [_T(n) for n in _tiles_nvp(case)]


def cpu_baseline(case):
    import torch
    from block_sparse_long_proxy_gb300 import synth
    inp = synth.make_inputs(case, device="cpu")
    rows, dt, ids = oracle_sample(case, inp, 1, seed=123)      # calibrate
    n = max(1, min(64, int(15.0 / max(dt, 1e-3))))
    rows, dt, ids = oracle_sample(case, inp, n, seed=7)
    return {"value": rows / dt, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": "%d random 128-row query tiles of the same workload through the whole fp64 oracle chain "
                      "(proxy max-score, top-k, attention), %.1f s" % (len(ids), dt)}


def bench_prefill_fp8(args, dev, pk_info, peak_kind, bf16_tflops):
    """The S=32768 prefill attention with e4m3 K/V (per-KV-head scales):
    msa_sparse_attn on the selections of its own proxy and top-k, TFLOP/s
    counted on the selected blocks, beside the bf16 figure."""
    import torch
    from block_sparse_long_proxy_gb300 import msa, synth
    case = synth.prefill_32k()
    case.kv_dtype = "e4m3"
    inp = synth.make_inputs(case, device=dev)
    plan = msa.Plan(case.qo_lens, case.kv_lens, case.hq, case.hkv, case.hp, case.d, case.dp, case.topk,
                    num_pages=inp["k_pages"].shape[0], kv_dtype="e4m3")
    ms = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    idx = msa.topk_select(ms, case.topk, plan.num_valid_pages)
    out = torch.empty_like(inp["q"])
    lse = torch.empty((plan.total_q, case.hq), dtype=torch.float32, device=dev)

    def attn():
        plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx,
                         k_scale=inp["k_scale"], v_scale=inp["v_scale"], out=out, lse=lse)
    for _ in range(max(3, args.warmup)):
        attn()
    torch.cuda.synchronize()
    plan.check_errors()
    flops, n_sel = selected_flops(idx.cpu().numpy(), case)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(max(10, min(args.steps, 200))):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        attn()
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    plan.check_errors()
    ms_ = statistics.mean(a.elapsed_time(b) for a, b in times)
    tf = flops / (ms_ / 1e3) / 1e12
    peak = pk_info.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    del inp
    return {"workload": "sparse prefill S=32768, e4m3 K/V", "sparse_attn_ms": ms_, "tflops_selected": tf,
            "vs_bf16": tf / bf16_tflops,
            "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel<128, fp8> (msa_sparse_attn)", "achieved": tf,
                         "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                         "peak_kind": "%s bf16 dense burst (cuBLAS); the MMAs run f16 at the same rate" % peak_kind,
                         "traffic": ncu_traffic("attn_fwd.cu:fp8", n_sel)},
            "kv_bytes_read": n_sel * 2 * 128 * case.d}


def bench_decode(args, dev, pk_info, peak_kind, world):
    """FP8 paged sparse decode: HBM GB/s of msa_sparse_attn on its selected
    K/V blocks (32 x 131072 keys, 64/8 heads, topk 16)."""
    import torch
    from block_sparse_long_proxy_gb300 import msa, synth
    case = synth.paged_decode()
    inp = synth.make_inputs(case, device=dev)
    plan = msa.Plan(case.qo_lens, case.kv_lens, case.hq, case.hkv, case.hp, case.d, case.dp, case.topk,
                    num_pages=inp["k_pages"].shape[0], kv_dtype="e4m3")
    try:
        ms = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
        idx = msa.topk_select(ms, case.topk, plan.num_valid_pages)
        out = torch.empty_like(inp["q"])
        lse = torch.empty((plan.total_q, case.hq), dtype=torch.float32, device=dev)

        def attn():
            plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx,
                             k_scale=inp["k_scale"], v_scale=inp["v_scale"], out=out, lse=lse)
        attn()
    except msa.MsaError as e:
        return {"unavailable": str(e)}
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    n_sel = int((idx >= 0).sum().item())
    kv_bytes = n_sel * 2 * 128 * case.d          # e4m3 K and V of each selected (seq, group, block)
    io_bytes = 2 * out.numel() * 2 + lse.numel() * 4
    # The event clock ticks in ~2 us steps, as long as a third of a decode
    # launch, so each kernel is timed as T(N x [flush, kernel]) - T(N x
    # [flush]) over N launches (events around each batch, L2 flushed before
    # every launch), the median of 5 such differences.
    n_batch = max(10, min(args.steps, 50))

    def batch(kernel):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record(stream)
        for _ in range(n_batch):
            flush()
            if kernel is not None:
                kernel()
        ev[1].record(stream)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1])

    def per_launch_s(kernel):
        for _ in range(3):
            kernel()
        diffs = [(batch(kernel) - batch(None)) / n_batch for _ in range(5)]
        return statistics.median(diffs) / 1e3

    t = per_launch_s(attn)
    tp = per_launch_s(lambda: plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"], out=ms))
    # the same scan over the e4m3 proxy K (msa_proxy_maxscore_fp8)
    tp8 = per_launch_s(lambda: plan.proxy_maxscore_fp8(inp["pq"], inp["pk_pages_e4m3"], inp["pk_scale"],
                                                       inp["kv_indices"], out=ms))
    # ... and over the NVFP4 proxy K, the FP4 block-score indexer (msa_proxy_maxscore_nvfp4)
    tp4 = per_launch_s(lambda: plan.proxy_maxscore_nvfp4(inp["pq"], inp["pk_fp4_codes"], inp["pk_fp4_scales"],
                                                         inp["pk_fp4_global"], inp["kv_indices"], out=ms))
    plan.check_errors()
    gbs = (kv_bytes + io_bytes) / t / 1e9
    proxy_bytes = sum((k + 127) // 128 for k in case.kv_lens) * 128 * case.dp * 2
    hbm = pk_info.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    return {"workload": case.name, "sparse_attn_us": t * 1e6, "hbm_gbs": gbs, "bytes": kv_bytes + io_bytes,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                         "peak_kind": "%s HBM copy" % peak_kind, "nominal_frac": gbs / 8000.0},
            "proxy_scan_us": tp * 1e6, "proxy_scan_gbs": proxy_bytes / tp / 1e9,
            "proxy_scan_frac": proxy_bytes / tp / 1e9 / hbm,
            "proxy_scan_fp8_us": tp8 * 1e6, "proxy_scan_fp8_gbs": proxy_bytes / 2 / tp8 / 1e9,
            "proxy_scan_fp8_frac": proxy_bytes / 2 / tp8 / 1e9 / hbm,
            # NVFP4: 32 code bytes and 4 scale bytes per key at dp = 64
            "proxy_scan_nvfp4_us": tp4 * 1e6, "proxy_scan_nvfp4_gbs": proxy_bytes * 9 / 32 / tp4 / 1e9,
            "proxy_scan_nvfp4_frac": proxy_bytes * 9 / 32 / tp4 / 1e9 / hbm,
            "timing": "per launch = (T(N x [L2 flush, kernel]) - T(N x [L2 flush])) / N, N = %d, median of 5" % n_batch}


def run_ncu_case(args):
    """A small case of one kernel for profiler captures (no JSON line):
    inputs above the 129 MB L2 but a few hundred MB on the device.
      attn / proxy / topk: sparse prefill S=16384 (32q/8kv, d=128, topk 16)
      attn_fp8: the same with e4m3 K/V
      decode: FP8 paged decode, 32 sequences x 16384 keys
      bwd: the KL-coupled backward of the S=16384 prefill."""
    import torch
    from block_sparse_long_proxy_gb300 import msa, synth
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    if args.ncu_case == "decode":
        case = synth.Case("decode 32x16384 fp8", [1] * 32, [16384] * 32, 64, 8, 128, 8, 64, 16, kv_dtype="e4m3",
                          page_perm_seed=1)
    elif args.ncu_case == "attn_fp8":
        case = synth.Case("prefill S=16384 fp8", [16384], [16384], 32, 8, 128, 8, 64, 16, kv_dtype="e4m3")
    else:
        case = synth.Case("prefill S=16384", [16384], [16384], 32, 8, 128, 8, 64, 16)
    inp = synth.make_inputs(case, device=dev, with_dout=args.ncu_case == "bwd")
    plan = msa.Plan(case.qo_lens, case.kv_lens, case.hq, case.hkv, case.hp, case.d, case.dp, case.topk,
                    num_pages=inp["k_pages"].shape[0], kv_dtype=case.kv_dtype)
    ms = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    idx = msa.topk_select(ms, case.topk, plan.num_valid_pages)
    kw = {}
    if case.kv_dtype != "bf16":
        kw = dict(k_scale=inp["k_scale"], v_scale=inp["v_scale"])
    if args.ncu_case == "bwd":
        out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx)
    for _ in range(args.steps):
        if args.ncu_case == "bwd":
            plan.sparse_attn_bwd(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx, out, lse,
                                 inp["dout"], inp["pq"], inp["pk_pages"])
        if args.ncu_case in ("proxy", "decode"):
            plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"], out=ms)
        if args.ncu_case == "decode":
            plan.proxy_maxscore_fp8(inp["pq"], inp["pk_pages_e4m3"], inp["pk_scale"], inp["kv_indices"], out=ms)
            plan.proxy_maxscore_nvfp4(inp["pq"], inp["pk_fp4_codes"], inp["pk_fp4_scales"], inp["pk_fp4_global"],
                                      inp["kv_indices"], out=ms)
        if args.ncu_case == "topk":
            msa.topk_select(ms, case.topk, plan.num_valid_pages, out=idx)
        if args.ncu_case in ("attn", "attn_fp8", "decode"):
            plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx, **kw)
    torch.cuda.synchronize()
    plan.check_errors()
    print("ncu case %s done: %d launches" % (args.ncu_case, args.steps))


def bench_varlen(args, dev, pk_info, peak_kind):
    """Varlen paged prefill (4 packed sequences of 8192/16384/32768/131072
    tokens, pages under a random permutation, planted block signal): the
    step proxy -> top-k -> attention, with the L2 flushed before each timed
    step; tokens/s and the two tensor-core stages' TFLOP/s (proxy on the
    causal lower triangle of blocks, attention on the selected blocks)."""
    import torch
    from block_sparse_long_proxy_gb300 import msa, synth
    case = synth.varlen_paged()
    inp = synth.make_inputs(case, device=dev)
    plan = msa.Plan(case.qo_lens, case.kv_lens, case.hq, case.hkv, case.hp, case.d, case.dp, case.topk,
                    num_pages=inp["k_pages"].shape[0])
    ms = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    idx = msa.topk_select(ms, case.topk, plan.num_valid_pages)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    for _ in range(3):
        plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"], out=ms)
        msa.topk_select(ms, case.topk, plan.num_valid_pages, out=idx)
        plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx, out=out, lse=lse)
    torch.cuda.synchronize()
    plan.check_errors()
    t_step, t_proxy, t_attn = [], [], []
    for _ in range(max(3, min(args.steps, 8))):
        flush()
        a, b, c, d = (torch.cuda.Event(enable_timing=True) for _ in range(4))
        a.record(stream)
        plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"], out=ms)
        b.record(stream)
        msa.topk_select(ms, case.topk, plan.num_valid_pages, out=idx)
        c.record(stream)
        plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx, out=out, lse=lse)
        d.record(stream)
        torch.cuda.synchronize()
        t_step.append(a.elapsed_time(d))
        t_proxy.append(a.elapsed_time(b))
        t_attn.append(c.elapsed_time(d))
    plan.check_errors()
    step_ms, proxy_ms, attn_ms = (statistics.median(v) for v in (t_step, t_proxy, t_attn))
    flops, n_sel = selected_flops(idx.cpu().numpy(), case)
    proxy_flops = sum(t.nvp for t in plan_tiles(case)) * case.hp * 2.0 * 128 * 128 * case.dp
    peak = pk_info.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    at, pt = flops / (attn_ms / 1e3) / 1e12, proxy_flops / (proxy_ms / 1e3) / 1e12
    return {"workload": case.name, "tokens": case.total_q, "ms_per_step": step_ms,
            "tokens_per_s": case.total_q / (step_ms / 1e3), "proxy_ms": proxy_ms, "sparse_attn_ms": attn_ms,
            "proxy_tflops": pt, "attn_tflops_selected": at, "proxy_frac": pt / peak, "attn_frac": at / peak,
            "peak_kind": "%s bf16 dense burst" % peak_kind}


def bench_train(args, dev, pk_info, peak_kind):
    """Training step at S=65536 (32q/8kv, d=128, 8 proxy heads x 64, topk
    16): forward (proxy, top-k, attention with LSE) and the KL-coupled
    backward, each timed with CUDA events; FLOPs counted on the selected
    blocks (forward 4*T*B*d, backward 10*T*B*d per tile, head and block) plus
    the KL products (proxy logits twice, p.pk and p^T.pq: 8*T*B*dp per tile,
    group and block)."""
    import torch
    from block_sparse_long_proxy_gb300 import msa, synth
    case = synth.training_64k()
    inp = synth.make_inputs(case, device=dev, with_dout=True)
    plan = msa.Plan(case.qo_lens, case.kv_lens, case.hq, case.hkv, case.hp, case.d, case.dp, case.topk,
                    num_pages=inp["k_pages"].shape[0])
    ms = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    idx = msa.topk_select(ms, case.topk, plan.num_valid_pages)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx)
    grads = dict(dq=torch.empty(inp["q"].shape, dtype=torch.float32, device=dev),
                 dk=torch.zeros(inp["k_pages"].shape, dtype=torch.float32, device=dev),
                 dv=torch.zeros(inp["v_pages"].shape, dtype=torch.float32, device=dev),
                 dpq=torch.empty(inp["pq"].shape, dtype=torch.float32, device=dev),
                 dpk=torch.zeros(inp["pk_pages"].shape, dtype=torch.float32, device=dev))
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)

    def fwd():
        plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"], out=ms)
        msa.topk_select(ms, case.topk, plan.num_valid_pages, out=idx)
        plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx, out=out, lse=lse)

    def bwd():
        plan.sparse_attn_bwd(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx, out, lse, inp["dout"],
                             inp["pq"], inp["pk_pages"], kl_weight=1.0, grads=grads)
    for _ in range(3):
        fwd()
        bwd()
    torch.cuda.synchronize()
    plan.check_errors()
    n_sel = int((idx >= 0).sum().item())
    grp = case.hq // case.hkv
    f_fwd = n_sel * grp * 4.0 * 128 * 128 * case.d
    f_bwd = n_sel * grp * 10.0 * 128 * 128 * case.d + n_sel * 8.0 * 128 * 128 * case.dp
    tf, tb = [], []
    for _ in range(max(3, min(args.steps, 10))):
        flush()
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record(stream)
        fwd()
        b.record(stream)
        bwd()
        c.record(stream)
        torch.cuda.synchronize()
        tf.append(a.elapsed_time(b))
        tb.append(b.elapsed_time(c))
    fms, bms = statistics.median(tf), statistics.median(tb)
    peak = pk_info.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    bt = f_bwd / (bms / 1e3) / 1e12
    return {"workload": case.name, "fwd_ms": fms, "bwd_ms": bms, "tokens_per_s": case.total_q / ((fms + bms) / 1e3),
            "fwd_sparse_flops": f_fwd, "bwd_flops": f_bwd, "bwd_tflops": bt,
            "roofline_bwd": {"bound": "tensor", "achieved": bt, "peak": peak, "unit": "TFLOP/s", "frac": bt / peak,
                             "peak_kind": "%s bf16 dense burst" % peak_kind}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--ncu-case", choices=["attn", "attn_fp8", "proxy", "topk", "decode", "bwd"], default=None,
                    help="run a small case of one kernel for a profiler capture and exit")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.ncu_case:
        run_ncu_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
