"""Benchmark: one DCP decode step on one GB300 (or N independent replicas).

A step is one pass of the whole hot path over one batch: slot mapping and
cache write of the batch's new tokens into their owners' paged slots, then the
partial attention of every virtual rank with the exact LSE merge fused in.

Workload (default): MLA, 128 heads sharing one 576-wide latent (512 values),
FP8-e4m3 cache, bf16 queries, 16 requests with mixed contexts (lognormal,
median 67K, clipped to [4K, 200K]), N = 8 virtual ranks, interleave 1,
block 64.  The KV bytes (~0.75 GB) exceed L2 (129 MB), so no flush is needed
between steps.  Other workloads: --workload <name> (dcp_workloads.CONFIGS).

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle instead.
"""

import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dcp_workloads import config, make_workload  # noqa: E402

METRIC = "decode-attn tokens/s and KV-read TB/s vs roofline (MLA 128h, 64K ctx, 1 GB300)"
DEFAULT_WORKLOAD = "mla_fp8_mixed"
ESIZE = {"f32": 4, "bf16": 2, "fp8": 1}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# DRAM bytes per cached KV token of the attention kernel, from one ncu capture
# each (dram__bytes_read.sum + dram__bytes_write.sum of one launch divided by
# the launch's cached tokens; summaries and commands under profiles/).  Valid
# only for the kernel source they were taken on: a changed source gives null.
MEASURED_TRAFFIC = {
    ("mla_tcgen05", "fp8"): ("attn_mla_pair.cu", "6ac87a4a8535bfa083190d7c2022c347b6d9b360423382eb90936f588f2a8cb3",
                             (219.794688e6 + 4.131584e6) / 376734),
    ("mla_tcgen05", "bf16"): ("attn_mla_pair.cu", "6ac87a4a8535bfa083190d7c2022c347b6d9b360423382eb90936f588f2a8cb3",
                              (308.545280e6 + 5.903872e6) / 262144),
    ("gqa_mma", "bf16"): ("attn_gqa_mma.cu", "67755412d54aa3ba8046b17584b4ccddeaf57333dc06d2d86f49ad71f0006772",
                          (268.675840e6 + 2.791168e6) / 65536),
    # per table entry (N B max_blocks) of the block-transfer listing
    ("transfer_blocks", "entry"): ("transfer.cu", "ba69fc5af5bf509387a4668d62e0fd322f75cc04daf9e1105750d478aee93893",
                                   (161.792e3 + 0.0) / (8 * 16 * 284)),
    # per request of the prefill workload's shape (2K chunk on a 64K context)
    ("prefill", "request"): ("attn_prefill_tc.cu", "8ae5abb4749b2662aa5b93bbdca6bf9d2ec024c60d9065d7701a84ca0bcd33e2",
                             294.982912e6 + 112.019968e6),
}


def measured_traffic(kernel, kv_dtype, tokens):
    import hashlib
    entry = MEASURED_TRAFFIC.get((kernel, kv_dtype))
    if entry is None:
        return None
    fname, sha, per_token = entry
    path = os.path.join(ROOT, "context_decode_attention_gb300", "csrc", fname)
    if not os.path.exists(path) or hashlib.sha256(open(path, "rb").read()).hexdigest() != sha:
        return None
    return per_token * tokens


def algorithmic(wl):
    """Algorithmic bytes and FLOPs of one attention launch (every KV byte read once)."""
    c = wl.cfg
    B, Tq, Hq, Hkv, Dk, Dv = (int(c[k]) for k in ("B", "Tq", "Hq", "Hkv", "Dk", "Dv"))
    L = wl.seq_lens.astype(np.int64)
    kv_row = Dk * ESIZE[c["kv_dtype"]] * Hkv + (0 if c["layout"] == "mla" else Dv * ESIZE[c["kv_dtype"]] * Hkv)
    kv_bytes = int(L.sum()) * kv_row
    q_bytes = B * Tq * Hq * Dk * ESIZE[c["q_dtype"]]
    out_bytes = B * Tq * Hq * (Dv * ESIZE[c["out_dtype"]] + 4)
    # every query row t sees L - Tq + t + 1 tokens
    vis = sum(int(l) * Tq - Tq * (Tq - 1) // 2 for l in L)
    flops = 2 * vis * Hq * (Dk + Dv)
    return dict(kv_bytes=kv_bytes, bytes=kv_bytes + q_bytes + out_bytes, flops=flops)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms (best effort)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in out.strip().splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxs.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return None
        return {"sm_mhz": float(np.median(sms)), "sm_max_mhz": float(max(maxs)), "reasons": sorted(reasons),
                "samples": len(sms)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(values, world):
    """Max over ranks of a list of floats (gloo, host tensors; no GPU collective)."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_oracle_sample(wl, budget_s=20.0):
    """Time the oracle on a bounded sample: query rows of the median-length request.

    Returns (tokens_per_s scaled to the whole workload, description, threads)."""
    import oracle
    c = wl.cfg
    B, Tq, Hq = int(c["B"]), int(c["Tq"]), int(c["Hq"])
    L = wl.seq_lens.astype(np.int64)
    b = int(np.argsort(L)[len(L) // 2])
    threads = oracle.threads()
    # probe with a few rows, then size the sample to ~budget_s
    rows_all = np.array([(b * Tq + t) * Hq + h for t in range(Tq) for h in range(Hq)], dtype=np.int64)
    n = min(len(rows_all), max(threads, 8))
    t0 = time.perf_counter()
    oracle.attention(wl, rows=rows_all[:n], nthreads=threads)
    dt = time.perf_counter() - t0
    per_row = dt / n
    n2 = int(min(len(rows_all), max(n, budget_s / max(per_row, 1e-9))))
    if n2 > n:
        t0 = time.perf_counter()
        oracle.attention(wl, rows=rows_all[:n2], nthreads=threads)
        dt = time.perf_counter() - t0
        n = n2
    # seconds for the whole workload: scale by rows and by each request's context
    rows_total = B * Tq * Hq
    sec_workload = dt / n * rows_total * (float(L.mean()) / float(L[b]))
    tok_s = B * Tq / sec_workload
    desc = (f"{n} of {rows_total} query rows (request {b}, {int(L[b])} tokens), fp64 C oracle; "
            f"scaled by rows and mean/sample context length")
    return tok_s, desc, threads, dt


def run_reference(args):
    """The CPU oracle as it stands, timed on the host cores (rank 0 only).

    A step here is one bounded sample of the workload: the oracle computes a
    slice of the median-length request's query rows, sized to a few seconds.
    ms_per_step is the measured wall time of one such step; value scales each
    step's rows/s to the whole workload (rows and context length) and is
    therefore an extrapolation, which the line says in `extrapolation`."""
    rank, world, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        if rank != 0:
            dist.barrier()
            dist.destroy_process_group()
            return
    cfg = config(args.workload)
    wl = make_workload(cfg)
    budget = max(1.0, 120.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_oracle_sample(wl, budget_s=budget / 4)
    vals, step_s, sample_s, desc, threads = [], [], [], "", 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ts = time.perf_counter()
        v, desc, threads, dt = cpu_oracle_sample(wl, budget_s=budget)
        step_s.append(time.perf_counter() - ts)
        sample_s.append(dt)
        vals.append(v)
    timed_s = time.perf_counter() - t0
    value = float(np.median(vals))
    c = wl.cfg
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(step_s)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; stands in for the pages' agentic ~67K-median trace)",
        "config": workload_config(c, wl),
        "extrapolation": {
            "step": "one bounded sample of the workload (see cpu_baseline.sample), not a whole decode step",
            "timed_region_s": timed_s,
            "sample_s_median": float(np.median(sample_s)),
            "workload_s_extrapolated": int(c["B"]) * int(c["Tq"]) / value,
            "value_from": "each sample's rows/s scaled by rows and by mean/sample context length; median over steps",
        },
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def workload_config(c, wl, l2="inputs larger than L2 (no flush)"):
    return {
        "workload": c["name"], "layout": c["layout"], "batch": int(c["B"]), "query_tokens": int(c["Tq"]),
        "q_heads": int(c["Hq"]), "kv_heads": int(c["Hkv"]), "key_width": int(c["Dk"]), "value_width": int(c["Dv"]),
        "context_tokens_total": int(wl.seq_lens.sum()), "context_median": int(np.median(wl.seq_lens)),
        "dcp_ranks": int(c["N"]), "interleave": int(c["I"]), "block_size": int(c["block_size"]),
        "kv_dtype": c["kv_dtype"], "q_dtype": c["q_dtype"], "out_dtype": c["out_dtype"],
        "global_batch": int(c["B"]) * int(c["Tq"]), "parallelism": "replicas (virtual DCP ranks on one GPU)",
        "l2": l2,
    }


TRANSFER_METRIC = "PD block-transfer listing: requests/s (per-rank non-empty blocks and fills, 1 GB300)"


def run_transfer(args):
    """Time the block-transfer listing (dcp_transfer_blocks) on the workload's
    block tables: the blocks each rank moves under prefill-decode
    disaggregation, their token counts and the batch's fill.  The inputs are a
    few MB, so L2 is flushed (a 256 MB write) between timed launches and each
    launch is timed alone with CUDA events."""
    import torch
    import context_decode_attention_gb300 as dcp
    from context_decode_attention_gb300.harness import DeviceWorkload

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    over = {"B": args.batch} if args.batch else {}
    if args.context:
        over["L"] = args.context
    cfg = config(args.workload, **over)
    wl = make_workload(cfg, seed=int(cfg["index"]) + 1000 * rank)
    dw = DeviceWorkload(wl, device=dev, populate=False)
    stream = dw.stream
    N, B, M = (int(x) for x in dw.block_tables.shape)
    bs = int(cfg["block_size"])
    counts = torch.empty((N, B), dtype=torch.int32, device=dev)
    blocks = torch.empty((N, B, M), dtype=torch.int32, device=dev)
    fills = torch.empty((N, B, M), dtype=torch.int32, device=dev)
    totals = torch.empty(2, dtype=torch.int64, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    peaks = load_peaks()

    def launch():
        dcp.dcp_transfer_blocks(dw.params, dw.seq_lens, dw.block_tables, dw.num_blocks, counts, blocks, fills,
                                totals, workspace=dw.workspace, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            launch()
    torch.cuda.synchronize()
    if dw.error_bits() != 0:
        raise SystemExit("device error bits set during warm-up")
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    launches0 = dcp.dcp_launch_count()
    with torch.cuda.stream(stream):
        for k in range(K):
            flush.fill_(k & 255)
            ev[k][0].record(stream)
            launch()
            ev[k][1].record(stream)
    torch.cuda.synchronize()
    launches = dcp.dcp_launch_count() - launches0
    barrier(world)
    clk = clocks.stop()
    if dw.error_bits() != 0:
        raise SystemExit("device error bits set during the timed region")
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    # context for a latency-bound launch: the same event bracket around a
    # one-element fill (a trivial kernel), after the same L2 flush
    one = torch.zeros(1, dtype=torch.int32, device=dev)
    fl = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with torch.cuda.stream(stream):
        for k in range(K):
            flush.fill_(k & 255)
            fl[k][0].record(stream)
            one.fill_(k)
            fl[k][1].record(stream)
    torch.cuda.synchronize()
    floor_ms = float(np.mean([a.elapsed_time(b) for a, b in fl]))

    # algorithmic bytes of one launch: the lengths and the listed table
    # entries read once; counts, blocks, fills and totals written once (the
    # listing's bit-exact parity with the oracle is a test's job, not the bench's)
    listed = int(counts.sum().item())
    alg_bytes = 4 * B + 4 * listed + 4 * N * B + 2 * 4 * N * B * M + 16

    e2e = None
    if not args.no_e2e:
        sl_h = dw.seq_lens.cpu().pin_memory()
        bt_h = dw.block_tables.cpu().pin_memory()
        outs_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (counts, blocks, fills, totals)]
        h2d = sl_h.numel() * 4 + bt_h.numel() * 4
        d2h = sum(t.numel() * t.element_size() for t in outs_h)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(K):
                dw.seq_lens.copy_(sl_h, non_blocking=True)
                dw.block_tables.copy_(bt_h, non_blocking=True)
                launch()
                for h, d in zip(outs_h, (counts, blocks, fills, totals)):
                    h.copy_(d, non_blocking=True)
            e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max([e0.elapsed_time(e1) / K], world)[0]
        e2e = {"value": world * B / (e2e_ms / 1e3), "unit": "requests/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms}

    ms = reduce_max([ms], world)[0]
    achieved = alg_bytes / (ms / 1e3) / 1e9
    tot = totals.cpu().numpy()  # slots and tokens moved, as the listing reports them
    line = {
        "metric": TRANSFER_METRIC, "value": world * B / (ms / 1e3), "unit": "requests/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32", "data": "synthetic (seeded block tables of the workload)",
        "config": dict(workload_config(cfg, wl), op="transfer-blocks", max_blocks=M,
                       l2="flushed (256 MB write) before every timed launch"),
        "blocks_listed": listed, "slots_moved": int(tot[0]), "tokens_moved": int(tot[1]),
        "transfer_fill": float(tot[1]) / max(1, int(tot[0])),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": measured_traffic("transfer_blocks", "entry", N * B * M),
                     "traffic_note": "ncu DRAM bytes per table entry of one capture (profiles/), scaled to this launch",
                     "algorithmic_bytes": alg_bytes,
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json, burst)",
                     "kernel": "transfer_blocks_kernel"},
        "trivial_launch_ms": floor_ms,
        "gpu_launches": int(launches), "clocks": clk, "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 2.0 or reps < 3:
            oracle.transfer_blocks(N, int(cfg["I"]), bs, wl.seq_lens, dw.block_tables_host, dw.num_blocks)
            reps += 1
        dt = (time.perf_counter() - t0) / reps
        line["cpu_baseline"] = {"value": B / dt, "unit": "requests/s", "cores": 1, "kind": "oracle",
                                "sample": f"the whole batch, {reps} repetitions, token-by-token enumeration in C"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


PREFILL_METRIC = "PCP prefill: chunk tokens/s and tensor roofline (head-tail partition + causal prefill over DCP shards, 1 GB300)"


def prefill_flops(wl):
    """FLOPs of one prefill pass: every new token t of request b sees the
    positions 0..p (p = L - Tq + t), 2 (Dk + Dv) per key and query head."""
    c = wl.cfg
    Tq, Hq, Dk, Dv = (int(c[k]) for k in ("Tq", "Hq", "Dk", "Dv"))
    vis = sum(int(L) * Tq - Tq * (Tq - 1) // 2 for L in wl.seq_lens.astype(np.int64))
    return 2 * vis * Hq * (Dk + Dv)


def run_prefill(args):
    """Time one PCP prefill step: the chunk's cache write, the head-tail
    partition, causal prefill attention of the gathered rows over every
    virtual rank's shard, and the LSE merge.  The KV (~0.55 GB) exceeds L2."""
    import torch
    import context_decode_attention_gb300 as dcp
    from context_decode_attention_gb300.harness import DeviceWorkload

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    name = args.workload if args.workload != DEFAULT_WORKLOAD else "gqa_prefill_64k"
    over = {"B": args.batch} if args.batch else {}
    if args.context:
        over["L"] = args.context
    cfg = config(name, **over)
    wl = make_workload(cfg, seed=int(cfg["index"]) + 1000 * rank)
    dw = DeviceWorkload(wl, device=dev, workspace_bytes=256)
    K = int(cfg.get("pcp", 4))
    dw.prefill_setup(K)
    stream = dw.stream
    peaks = load_peaks()
    flops = prefill_flops(wl)
    B, Tq = int(cfg["B"]), int(cfg["Tq"])

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            dw.write_new_tokens()
            dw.prefill()
    torch.cuda.synchronize()
    if dw.error_bits() != 0:
        raise SystemExit("device error bits set during warm-up")
    steps = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    launches0 = dcp.dcp_launch_count()
    with torch.cuda.stream(stream):
        for k in range(steps):
            ev[k][0].record(stream)
            dw.write_new_tokens()
            ev[k][1].record(stream)
            dw.prefill()
            ev[k][2].record(stream)
    torch.cuda.synchronize()
    launches = dcp.dcp_launch_count() - launches0
    barrier(world)
    clk = clocks.stop()
    if dw.error_bits() != 0:
        raise SystemExit("device error bits set during the timed region")
    step_ms = float(np.mean([e[0].elapsed_time(e[2]) for e in ev]))
    attn_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in ev]))
    write_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))

    e2e = None
    if not args.no_e2e:
        qg_h = dw.q_gathered.cpu().pin_memory()
        nk_h, nv_h = dw.new_k.cpu().pin_memory(), dw.new_v.cpu().pin_memory()
        out_h = torch.empty(dw.g_out.shape, dtype=dw.g_out.dtype).pin_memory()
        lse_h = torch.empty(dw.g_lse.shape, dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (qg_h, nk_h, nv_h))
        d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * 4
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                dw.q_gathered.copy_(qg_h, non_blocking=True)
                dw.new_k.copy_(nk_h, non_blocking=True)
                dw.new_v.copy_(nv_h, non_blocking=True)
                dw.write_new_tokens()
                dw.prefill()
                out_h.copy_(dw.g_out, non_blocking=True)
                lse_h.copy_(dw.g_lse, non_blocking=True)
            e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max([e0.elapsed_time(e1) / steps], world)[0]
        e2e = {"value": world * B * Tq / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms}

    step_ms, attn_ms, write_ms = reduce_max([step_ms, attn_ms, write_ms], world)
    achieved = flops / (attn_ms / 1e3) / 1e12
    roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops"],
            "traffic": measured_traffic("prefill", "request", B) if name == "gqa_prefill_64k" and not args.context else None,
            "traffic_note": "ncu DRAM bytes of one request's launch (profiles/), times the requests",
            "algorithmic_flops": flops,
            "peak_source": peaks["source"] + " (MEASURED_PEAKS.json, burst; bf16 tcgen05 kind::f16)",
            "kernel": "prefill_tc_kernel" if int(cfg["Dk"]) == 128 else "prefill_partial_kernel", "attn_ms": attn_ms,
            "roofline_ms": 1e3 * flops / (peaks["bf16_tflops"] * 1e12)}
    line = {
        "metric": PREFILL_METRIC, "value": world * B * Tq / (step_ms / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; a 2K-token chunk on a 64K cached context)",
        "config": dict(workload_config(cfg, wl), op="prefill", pcp_ranks=K, chunk_tokens=Tq),
        "cache_write_ms": write_ms, "roofline": roof, "gpu_launches": int(launches), "clocks": clk, "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        c = wl.cfg
        Hq = int(c["Hq"])
        rows = np.arange(0, Hq * 8, dtype=np.int64) + (Tq - 8) * Hq  # the last 8 query tokens of request 0
        threads = oracle.threads()
        t0 = time.perf_counter()
        oracle.attention(wl, rows=rows, nthreads=threads)
        dt = time.perf_counter() - t0
        per_flop = dt / (2 * len(rows) * int(wl.seq_lens[0]) * (int(c["Dk"]) + int(c["Dv"])))
        line["cpu_baseline"] = {"value": B * Tq / (per_flop * flops), "unit": "tokens/s", "cores": threads,
                                "kind": "oracle",
                                "sample": f"{len(rows)} query rows (the last 8 tokens x {Hq} heads of request 0), "
                                          "fp64 C oracle, scaled by FLOPs to the whole step"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


SPARSE_METRIC = "DCP-localised sparse MLA decode: query tokens/s and tensor roofline (top-2048 candidates, 1 GB300)"


def run_sparse(args):
    """Time one sparse decode pass: localisation of every query row's
    candidates to their ranks, staging, the rank partials on the dense MLA
    kernels and the merge."""
    import torch
    import context_decode_attention_gb300 as dcp
    from context_decode_attention_gb300.harness import DeviceWorkload
    from dcp_workloads import sparse_candidates

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    name = args.workload if args.workload != DEFAULT_WORKLOAD else "mla_fp8_sparse_2k"
    over = {"B": args.batch} if args.batch else {}
    cfg = config(name, **over)
    wl = make_workload(cfg, seed=int(cfg["index"]) + 1000 * rank)
    k = int(cfg.get("topk", 2048))
    params = dcp.params_from_config(cfg, wl.kv_scale)
    B, Tq, Hq, Dk, Dv = (int(cfg[x]) for x in ("B", "Tq", "Hq", "Dk", "Dv"))
    dw = DeviceWorkload(wl, device=dev, workspace_bytes=dcp.dcp_sparse_workspace_size(params, B, k))
    cand_h = sparse_candidates(wl, k, seed=1)
    cand = torch.from_numpy(cand_h).to(dev)
    out = torch.empty_like(dw.out)
    lse = torch.empty_like(dw.lse)
    stream = dw.stream
    peaks = load_peaks()
    nc = int((cand_h >= 0).sum())
    flops = 2 * nc * Hq * (Dk + Dv)
    kv_bytes = nc * Dk * ESIZE[cfg["kv_dtype"]]
    alg_bytes = kv_bytes + B * Tq * Hq * (Dk * 2 + Dv * 2 + 4)

    def step():
        dcp.dcp_sparse_decode_attention(dw.params, dw.q, cand, dw.k_pool, dw.num_blocks, dw.block_tables,
                                        dw.seq_lens, out, lse, workspace=dw.workspace, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    if dw.error_bits() != 0:
        raise SystemExit("device error bits set during warm-up")
    steps = args.steps
    # the candidates' rows (~75 MB) fit in L2: flush it before every timed step
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    launches0 = dcp.dcp_launch_count()
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.fill_(i & 255)
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    launches = dcp.dcp_launch_count() - launches0
    barrier(world)
    clk = clocks.stop()
    if dw.error_bits() != 0:
        raise SystemExit("device error bits set during the timed region")
    ms = reduce_max([float(np.mean([a.elapsed_time(b) for a, b in ev]))], world)[0]

    e2e = None
    if not args.no_e2e:
        q_h = dw.q.cpu().pin_memory()
        c_h = cand.cpu().pin_memory()
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                dw.q.copy_(q_h, non_blocking=True)
                cand.copy_(c_h, non_blocking=True)
                step()
                out_h.copy_(out, non_blocking=True)
                lse_h.copy_(lse, non_blocking=True)
            e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max([e0.elapsed_time(e1) / steps], world)[0]
        e2e = {"value": world * B * Tq / (e2e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": int(q_h.numel() * 2 + c_h.numel() * 4),
               "d2h_bytes_per_step": int(out_h.numel() * out_h.element_size() + lse_h.numel() * 4),
               "ms_per_step": e2e_ms}

    t = ms / 1e3
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    t_mem = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    if t_tc >= t_mem:
        roof = {"bound": "tensor", "achieved": flops / t / 1e12, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": alg_bytes / t / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof.update({"frac": roof["achieved"] / roof["peak"], "traffic": None, "algorithmic_flops": flops,
                 "algorithmic_bytes": alg_bytes, "roofline_ms": 1e3 * max(t_tc, t_mem),
                 "peak_source": peaks["source"] + " (MEASURED_PEAKS.json, burst)",
                 "kernel": "sparse localise + stage + mla_tcgen05 (one virtual rank) + merges", "step_ms": ms})
    line = {
        "metric": SPARSE_METRIC, "value": world * B * Tq / t, "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3" if cfg["kv_dtype"] == "fp8" else "bf16",
        "data": "synthetic (seeded; candidates from a synthetic top-k indexer)",
        "config": dict(workload_config(cfg, wl), op="sparse", topk=k, candidates=nc,
                       l2="flushed (256 MB write) before every timed step"),
        "roofline": roof, "gpu_launches": int(launches), "clocks": clk, "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        sample = np.full_like(cand_h, -1)
        sample[:2] = cand_h[:2]
        t0 = time.perf_counter()
        oracle.sparse_attention(wl, sample)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": 2 / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": "2 query rows (x 128 heads x 2048 candidates), fp64 numpy oracle"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def roofline(alg, attn_ms, peaks, kernel, kv_dtype, tokens):
    """Roofline entry of one attention launch: achieved algorithmic bytes or
    FLOPs per second against the measured peak of its bound."""
    t_attn = attn_ms / 1e3
    t_mem = alg["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = alg["flops"] / (peaks["bf16_tflops"] * 1e12)
    if t_tc > t_mem:
        roof = {"bound": "tensor", "achieved": alg["flops"] / t_attn / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": alg["bytes"] / t_attn / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    # the same achieved figure against the part's nominal peaks (8 TB/s HBM3e,
    # 2.25 PFLOP/s dense bf16), which the metric's wording also asks for
    nominal = 8000.0 if roof["bound"] == "hbm" else 2250.0
    roof["nominal"] = {"peak": nominal, "unit": roof["unit"], "frac": roof["achieved"] / nominal}
    roof["traffic"] = measured_traffic(kernel, kv_dtype, tokens)
    roof["traffic_note"] = "ncu DRAM bytes per cached token of one capture (profiles/), scaled to this launch's tokens"
    roof["algorithmic_bytes"] = alg["bytes"]
    roof["peak_source"] = peaks["source"] + " (MEASURED_PEAKS.json, burst)"
    roof["kernel"] = kernel
    roof["roofline_ms"] = 1e3 * max(t_mem, t_tc)
    roof["attn_ms"] = attn_ms
    return roof


# The other decode configs, measured after the headline workload in the same
# run (attention time, roofline fraction, traffic ratio), so that every
# config's figure comes from the same box and the same clock record.
OTHER_CONFIGS = ("gqa_llama8b", "mla_bf16_32k", "mla_fp8_1m")


def measure_config(name, dev, steps, warmup, peaks):
    """One decode workload at its full size: `steps` timed steps (cache write
    + attention) after `warmup`, CUDA events on the launching stream."""
    import torch
    import context_decode_attention_gb300 as dcp
    from context_decode_attention_gb300.harness import DeviceWorkload
    cfg = config(name)
    wl = make_workload(cfg, seed=int(cfg["index"]))
    dw = DeviceWorkload(wl, device=dev)
    alg = algorithmic(wl)
    kernel = dcp.dcp_attention_kernel(dw.params)
    stream = dw.stream
    for _ in range(warmup):
        dw.step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    clocks = ClockSampler(dev.index)
    with torch.cuda.stream(stream):
        for k in range(steps):
            ev[k][0].record(stream)
            dw.plan_and_write()  # the plan on a second stream beside the cache write
            ev[k][1].record(stream)
            dw.decode_planned()
            ev[k][2].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    bits = dw.error_bits()
    attn_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in ev]))
    step_ms = float(np.mean([e[0].elapsed_time(e[2]) for e in ev]))
    roof = roofline(alg, attn_ms, peaks, kernel, cfg["kv_dtype"], int(wl.seq_lens.sum()))
    entry = {
        "workload": name, "kernel": kernel, "steps": steps, "warmup": warmup,
        "attn_ms": attn_ms, "step_ms": step_ms,
        "tokens_per_s": int(cfg["B"]) * int(cfg["Tq"]) / (step_ms / 1e3),
        "kv_read_tbps": alg["kv_bytes"] / (attn_ms / 1e3) / 1e12,
        "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac", "roofline_ms")},
        "roofline_nominal_frac": roof["nominal"]["frac"],
        "traffic_ratio": None if roof["traffic"] is None else roof["traffic"] / roof["algorithmic_bytes"],
        "clocks": clk, "device_error_bits": int(bits),
    }
    del dw, wl
    torch.cuda.empty_cache()
    return entry


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="dcp", choices=["dcp", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other decode configs' block")
    ap.add_argument("--batch", type=int, default=0, help="override the batch (profiling a smaller case)")
    ap.add_argument("--context", type=int, default=0, help="override to one fixed context length")
    ap.add_argument("--op", default="decode", choices=["decode", "transfer-blocks", "prefill", "sparse"],
                    help="decode: the decode step (default); transfer-blocks: the PD block-transfer listing; "
                         "prefill: the PCP prefill step; sparse: DCP-localised top-k sparse decode")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        return run_reference(args)
    if args.op == "transfer-blocks":
        return run_transfer(args)
    if args.op == "prefill":
        return run_prefill(args)
    if args.op == "sparse":
        return run_sparse(args)

    import torch
    import context_decode_attention_gb300 as dcp
    from context_decode_attention_gb300.harness import DeviceWorkload, raw_to_torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    over = {}
    if args.batch:
        over["B"] = args.batch
    if args.context:
        over["L"] = args.context
    cfg = config(args.workload, **over)
    wl = make_workload(cfg, seed=int(cfg["index"]) + 1000 * rank)  # replicas: same shape, own data
    dw = DeviceWorkload(wl, device=dev)
    stream = dw.stream
    kernel = dcp.dcp_attention_kernel(dw.params)
    alg = algorithmic(wl)
    peaks = load_peaks()
    # Consecutive steps must not find the KV in L2.  The decode workloads' KV
    # exceeds it; a smaller one (the toy, a --batch override) gets L2 flushed
    # before every timed step, outside the step's events.
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or (129 << 20)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if alg["kv_bytes"] <= l2_bytes else None
    l2_note = ("inputs larger than L2 (no flush)" if flush is None
               else "flushed (256 MB write) before every timed step, outside its events")

    for _ in range(args.warmup):
        dw.step()
    torch.cuda.synchronize()
    if dw.error_bits() != 0:
        raise SystemExit("device error bits set during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    launches0 = dcp.dcp_launch_count()
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for k in range(K):
            if flush is not None:
                flush.fill_(k & 255)
            ev[k][0].record(stream)
            dw.plan_and_write()  # the plan on a second stream beside the cache write
            ev[k][1].record(stream)
            dw.decode_planned()
            ev[k][2].record(stream)
        t_end.record(stream)
    torch.cuda.synchronize()
    launches = dcp.dcp_launch_count() - launches0
    barrier(world)
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    if flush is not None:  # the flushes lie between the steps: count the steps only
        total_ms = float(sum(e[0].elapsed_time(e[2]) for e in ev))
    attn_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in ev]))
    write_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    if dw.error_bits() != 0:
        raise SystemExit("device error bits set during the timed region")

    # ---- end to end through the public API: host buffers in, host results out
    e2e = None
    if not args.no_e2e:
        q_h = raw_to_torch(wl.q, cfg["q_dtype"]).pin_memory()
        nk_h = dw.new_k.cpu().pin_memory()
        nv_h = None if dw.new_v is None else dw.new_v.cpu().pin_memory()
        req_h, pos_h = dw.new_req.cpu().pin_memory(), dw.new_pos.cpu().pin_memory()
        sl_h = dw.seq_lens.cpu().pin_memory()
        out_h = torch.empty(dw.out.shape, dtype=dw.out.dtype).pin_memory()
        lse_h = torch.empty(dw.lse.shape, dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in [q_h, nk_h, req_h, pos_h, sl_h] + ([nv_h] if nv_h is not None else []))
        d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * 4
        for _ in range(2):
            dw.step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        ee = ([(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
              if flush is not None else None)
        barrier(world)
        names = ("q", "new_k", "new_v", "new_req", "new_pos", "seq_lens", "out", "lse")
        host_in = {"q": q_h, "new_k": nk_h, "new_v": nv_h, "new_req": req_h, "new_pos": pos_h, "seq_lens": sl_h}
        if ee is not None:
            # a workload that fits in L2: L2 is flushed before every step, so the
            # steps run one after the other, each with its copies, timed one by one
            with torch.cuda.stream(stream):
                for k in range(K):
                    flush.fill_(k & 255)
                    ee[k][0].record(stream)
                    for n in names[:6]:
                        if host_in[n] is not None:
                            getattr(dw, n).copy_(host_in[n], non_blocking=True)
                    dw.step()
                    out_h.copy_(dw.out, non_blocking=True)
                    lse_h.copy_(dw.lse, non_blocking=True)
                    ee[k][1].record(stream)
            torch.cuda.synchronize()
            step_ms = float(np.mean([a.elapsed_time(b) for a, b in ee]))
            pipelined = False
        else:
            # As a serving loop runs: the inputs and results of two steps are
            # double-buffered on the device, and two copy streams (one per
            # direction, so that an input copy never queues behind a result copy
            # that waits for its step) move step k + 1's inputs in and step k's
            # results out while step k computes.  Every step still copies its own
            # inputs and reads back its own results inside the timed region.
            bufs = [{n: getattr(dw, n) for n in names}]
            bufs.append({n: (None if t is None else torch.empty_like(t)) for n, t in bufs[0].items()})
            outs_h = [(out_h, lse_h), (torch.empty_like(out_h).pin_memory(), torch.empty_like(lse_h).pin_memory())]
            hs, ds = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
            ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("h2d", "done", "d2h")}

            def run(nsteps, t0=None, t1=None):
                if t0 is not None:
                    t0.record(stream)
                hs.wait_stream(stream)
                ds.wait_stream(stream)
                for k in range(nsteps):
                    i = k & 1
                    bset = bufs[i]
                    with torch.cuda.stream(hs):
                        if k >= 2:
                            hs.wait_event(ev["done"][i])  # step k - 2 is done with this buffer set
                        for n in names[:6]:
                            if host_in[n] is not None:
                                bset[n].copy_(host_in[n], non_blocking=True)
                        ev["h2d"][i].record(hs)
                    with torch.cuda.stream(stream):
                        stream.wait_event(ev["h2d"][i])
                        if k >= 2:
                            stream.wait_event(ev["d2h"][i])  # step k - 2's results have left this set
                        for n in names:
                            setattr(dw, n, bset[n])
                        dw.step()
                        ev["done"][i].record(stream)
                    with torch.cuda.stream(ds):
                        ds.wait_event(ev["done"][i])
                        outs_h[i][0].copy_(bset["out"], non_blocking=True)
                        outs_h[i][1].copy_(bset["lse"], non_blocking=True)
                        ev["d2h"][i].record(ds)
                stream.wait_stream(hs)
                stream.wait_stream(ds)
                if t1 is not None:
                    t1.record(stream)

            run(4)
            torch.cuda.synchronize()
            run(K, e0, e1)
            torch.cuda.synchronize()
            for n in names:
                setattr(dw, n, bufs[0][n])
            step_ms = e0.elapsed_time(e1) / K
            pipelined = True
        e2e_ms = reduce_max([step_ms], world)[0]
        e2e = {"value": world * int(cfg["B"]) * int(cfg["Tq"]) / (e2e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
               "copies": ("double-buffered: step k+1's inputs in and step k's results out on two copy streams "
                          "while step k computes" if pipelined else "in line with each step (L2 flushed between steps)")}

    total_ms, attn_ms, write_ms = reduce_max([total_ms, attn_ms, write_ms], world)
    write_bytes = sum(t.numel() * t.element_size() for t in (dw.new_k, dw.new_v) if t is not None)
    ms_per_step = total_ms / K
    tokens_per_step = int(cfg["B"]) * int(cfg["Tq"])
    value = world * tokens_per_step / (ms_per_step / 1e3)

    # roofline of the dominant kernel: the attention launches (their plan was made on a
    # second stream beside the cache write, inside the step but off this interval)
    roof = roofline(alg, attn_ms, peaks, kernel, cfg["kv_dtype"], int(wl.seq_lens.sum()))
    t_attn = attn_ms / 1e3

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        # the operand type of the dominant kernel's products (accumulation is fp32 throughout):
        # bf16 tensor-core MMAs, e4m3 (kind::f8f6f4, two-term query and P) on the fp8 cache,
        # fp32 on the CUDA-core path
        "dtype": ("e4m3" if cfg["kv_dtype"] == "fp8" else "bf16") if kernel == "mla_tcgen05"
                 else ("bf16" if kernel == "gqa_mma" else "f32"),
        "data": "synthetic (seeded; stands in for the pages' agentic ~67K-median trace)",
        "config": workload_config(cfg, wl, l2=l2_note),
        "kv_read_tbps": alg["kv_bytes"] / t_attn / 1e12,
        "cache_write_ms": write_ms,
        "cache_write_note": "the cache write, with the attention's plan made beside it on a second stream",
        # the step's new K/V rows scattered into the paged cache (slot mapping + write)
        "cache_write_bytes": int(write_bytes),
        "cache_write_gbps": write_bytes / (write_ms / 1e3) / 1e9,
        "roofline": roof,
        "gpu_launches": int(launches),
        "clocks": clk,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc, threads, _ = cpu_oracle_sample(wl)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": desc}
    if (world == 1 and not args.no_configs and args.workload == DEFAULT_WORKLOAD and not args.batch
            and not args.context):
        del dw
        torch.cuda.empty_cache()
        line["other_configs"] = [measure_config(n, dev, max(20, min(100, K)), args.warmup, peaks)
                                 for n in OTHER_CONFIGS]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
