"""Benchmark of one paged decode step on GB300: copy-on-write copies (if any), the
append of one new token per sequence, and decode attention through block tables.

Prints ONE JSON line (rank 0).  `value` is the KV bytes decode attends per step
divided by the device time of a step (GB/s), inputs resident in HBM.  The dominant
kernel (decode, split-K partitions + merge) is also reported against the HBM
roofline; `e2e` repeats the step with each step's inputs copied from pinned host
memory and the output copied back inside the timed region; `cpu_baseline` times
the float64 oracle on the host's cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 2] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "paged decode attention: KV GB/s, seq-tokens/s, fraction of GB300 HBM peak"
FALLBACK_HBM_GBS = 6800.0
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=2, choices=sorted(workloads.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default="auto", choices=["auto", "cuda_core", "tensor_core"])
    ap.add_argument("--partition", type=int, default=0, help="split-K partition tokens (0 = auto)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill", action="store_true", help="measure causal multi-token (prefill) attention instead")
    ap.add_argument("--block-size", type=int, default=0, help="override the workload's block size (8/16/32/64)")
    ap.add_argument("--head-dim", type=int, default=0, help="override the workload's head_dim (64/128)")
    ap.add_argument("--num-q-heads", type=int, default=0,
                    help="override the workload's query heads (a multiple of its KV heads: another group size)")
    ap.add_argument("--dtype", default="", choices=["", "f32", "f16", "bf16"],
                    help="override the workload's cache dtype")
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="override the workload's batch size (workloads 2, 3 and 5; a smaller profiling case)")
    ap.add_argument("--identity-tables", action="store_true",
                    help="physical blocks in logical order (contiguous sequences): the indirection A/B")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip the decode-call timing of workloads 3, 4 and 5 on the default line")
    return ap.parse_args()


KERNEL_SOURCES = {"tensor_core": ["common.cuh", "decode_tc.cu", "launch.h", "tc_util.cuh", "tcgen05.cuh"],
                  "tensor_core_f32": ["common.cuh", "decode_tc32.cu", "launch.h", "tc_util.cuh", "tcgen05.cuh"],
                  "cuda_core": ["common.cuh", "decode_simt.cu", "launch.h"],
                  "prefill": ["common.cuh", "prefill_tc.cu", "launch.h", "tc_util.cuh", "tcgen05.cuh"]}


PREFILL_WORKLOAD = "chunked prefill: 32 seqs, contexts U[1024,4096], last 512 tokens new, 64/8 heads, D128, bf16, bs16"


def recorded_traffic(path_name, workload, partition):
    """DRAM bytes per launch from a committed ncu capture of the same kernel sources,
    workload and partition size (profiles/traffic.json), else None."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            entries = json.load(f)["entries"]
        h = hashlib.sha256()
        for name in KERNEL_SOURCES[path_name]:
            with open(os.path.join(ROOT, "paged_kv_cache_310_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        sha = h.hexdigest()
    except (OSError, KeyError, ValueError):
        return None
    for e in entries:
        if (e.get("path") == path_name and e.get("workload") == workload and e.get("partition_tokens") == partition
                and e.get("sources_sha256") == sha):
            return e["dram_bytes_per_launch"]
    return None


def max_over_ranks(x, dist, device):
    """The largest of every rank's x (the slowest rank sets a whole-job time); x itself
    when there is no process group."""
    if dist is None:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def whole_job_rate(world, bytes_per_rank, ms):
    """Bytes per second of all ranks together, in GB/s: every rank moves bytes_per_rank
    in ms (the max over ranks)."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def elem(dtype):
    return torch.empty((), dtype=dtype).element_size()


def roofline_bytes(w, out_elem):
    """Algorithmic bytes of one decode: K+V once, q, out, block-table entries, lengths."""
    e = elem(w.dtype)
    lens = w.context_lens.to(torch.int64)
    kv = int(lens.sum()) * 2 * w.num_kv_heads * w.head_dim * e
    S = w.num_seqs
    qo = S * w.num_q_heads * w.head_dim * (e + out_elem)
    table = 4 * int(((lens + w.block_size - 1) // w.block_size).sum()) + 4 * S
    return kv, kv + qo + table


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while it runs."""

    def __init__(self, index):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [[x.strip() for x in ln.split(",")] for ln in out.splitlines() if ln.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        loaded = [x for x in sm if mx and x >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


DECODE_CALLS_MIN = 200


def decode_call_ms(call, stream, n):
    """Mean device time of one decode call: each of n calls bracketed by CUDA events
    on the stream it is launched on."""
    k0 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    k1 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for i in range(n):
        k0[i].record(stream)
        call()
        k1[i].record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in zip(k0, k1))


def traffic_path(plan_path, dtype):
    """Key of the kernel sources a decode plan runs (profiles/traffic.json)."""
    if plan_path == 2:
        return "tensor_core_f32" if dtype == torch.float32 else "tensor_core"
    return "cuda_core"


def measure_config(pkv, cfg, dev, path, partition, n_calls):
    """Decode-call roofline of workload `cfg` (its step's copies and append done once
    first, as the step does), inputs resident in HBM."""
    w = workloads.make_workload(cfg, canary=False, pool_device=dev)
    g = w.to(dev)
    S, Hq, D = g.q.shape
    out = torch.empty((S, Hq, D), dtype=w.dtype, device=dev)
    maxL = w.max_context_len
    stream = torch.cuda.current_stream(dev)
    if g.cow_pairs.numel():
        pkv.paged_block_copy(g.cow_pairs, g.k_cache, g.v_cache, host_pairs=w.cow_pairs.cpu())
    pkv.paged_kv_append(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)

    def call():
        pkv.paged_attention_decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, w.scale, out,
                                   max_context_len=maxL, path=path, partition_tokens=partition)

    for _ in range(5):
        call()
    torch.cuda.synchronize()
    if pkv.device_error() != 0:
        raise SystemExit(f"device error flag set on workload {cfg}")
    ms = decode_call_ms(call, stream, n_calls)
    if pkv.device_error() != 0:
        raise SystemExit(f"device error flag set on workload {cfg}")
    plan = pkv.paged_attention_plan(S, Hq, maxL, g.k_cache, path=path, partition_tokens=partition)
    path_name = {1: "cuda_core", 2: "tensor_core"}[plan["path"]]
    kv, algo = roofline_bytes(w, elem(out.dtype))
    sources = traffic_path(plan["path"], w.dtype)
    peak, peak_kind = peaks()
    achieved = algo / (ms * 1e-3) / 1e9
    entry = {"workload": w.name, "path": path_name, "partition_tokens": plan["partition_tokens"],
             "partitions": plan["max_partitions"], "calls": n_calls, "ms_per_call": ms,
             "kv_gbs": kv / (ms * 1e-3) / 1e9, "seq_tokens_per_s": int(w.context_lens.sum()) / (ms * 1e-3),
             "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                          "frac": achieved / peak, "peak_source": peak_kind,
                          "traffic": recorded_traffic(sources, w.name, plan["partition_tokens"]),
                          "algorithmic_bytes_per_launch": algo}}
    if cfg == 4:
        e = elem(w.dtype)
        unique = w.unique_blocks * w.block_size * 2 * w.num_kv_heads * w.head_dim * e
        entry["l2"] = ("the shared prefix and beam prompts are read by several sequences per call and "
                       "mostly hit L2: logical bytes can exceed the HBM peak")
        entry["unique_kv_bytes"] = unique
    else:
        entry["l2"] = f"inputs larger than L2 (KV {kv / 1e9:.2f} GB > 129 MB): no flush"
    del g, out, w
    torch.cuda.empty_cache()
    return entry


def cpu_baseline(w, budget_s):
    """The float64 oracle on this host's cores over the same step, repeated within a budget."""
    import oracle

    kc, vc = w.k_cache.cpu(), w.v_cache.cpu()
    wc = w.to("cpu")
    oracle.block_copy(wc.cow_pairs, kc, vc)
    oracle.kv_append(wc.k_new, wc.v_new, wc.slot_mapping, kc, vc)
    kv_bytes, _ = roofline_bytes(wc, elem(w.dtype))
    # bounded sample: sequences in order until the first call takes ~budget/3
    S = wc.num_seqs
    n = S
    t0 = time.perf_counter()
    oracle.attention_decode(wc.q[:1], kc, vc, wc.block_tables[:1], wc.context_lens[:1], wc.scale)
    one = max(time.perf_counter() - t0, 1e-4)
    n = max(1, min(S, int((budget_s / 3) / one)))
    sel = slice(0, n)
    times = []
    t_end = time.perf_counter() + budget_s
    while len(times) < 3 or (time.perf_counter() < t_end and len(times) < 50):
        t0 = time.perf_counter()
        oracle.attention_decode(wc.q[sel], kc, vc, wc.block_tables[sel], wc.context_lens[sel], wc.scale)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() > t_end and len(times) >= 3:
            break
    sample_lens = wc.context_lens[sel].to(torch.int64)
    sample_kv = int(sample_lens.sum()) * 2 * w.num_kv_heads * w.head_dim * elem(w.dtype)
    t = statistics.median(times)
    return {"value": sample_kv / t / 1e9, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{n} of {S} sequences ({int(sample_lens.sum())} tokens), median of {len(times)} calls",
            "seq_tokens_per_s": int(sample_lens.sum()) / t, "seconds_per_call": t, "_kv_bytes": kv_bytes}


def run_reference(args):
    """--impl reference: the float64 oracle timed on the host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workloads.make_workload(args.config, canary=False)
    import oracle

    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    oracle.block_copy(w.cow_pairs, kc, vc)
    oracle.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    t0 = time.perf_counter()
    oracle.attention_decode(w.q[:1], kc, vc, w.block_tables[:1], w.context_lens[:1], w.scale)
    one = max(time.perf_counter() - t0, 1e-4)
    # each step: a bounded sample of sequences, sized so the whole run takes ~1-2 minutes
    per_step = 60.0 / max(1, args.steps + args.warmup)
    n = max(1, min(w.num_seqs, int(per_step / one)))
    sel = slice(0, n)

    def step():
        oracle.attention_decode(w.q[sel], kc, vc, w.block_tables[sel], w.context_lens[sel], w.scale)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    lens = w.context_lens[sel].to(torch.int64)
    kv = int(lens.sum()) * 2 * w.num_kv_heads * w.head_dim * elem(w.dtype)
    value = kv / dt / 1e9
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample_sequences": n, "num_seqs": w.num_seqs},
            "seq_tokens_per_s": int(lens.sum()) / dt,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"{n} of {w.num_seqs} sequences per step"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_prefill(args):
    """--prefill: causal multi-token attention (chunked prefill) on tensor cores.

    Workload: 32 sequences with contexts uniform in [1024, 4096], each bringing its last
    512 tokens as new queries, 64 query / 8 KV heads, head_dim 128, bf16, block size 16.
    Algorithmic flops: 4 * Hq * D * (p + 1) per new token at position p (QK and PV,
    causal); the kernel's hi/lo probability split doubles the PV MMAs, which is not
    counted.
    """
    import paged_kv_cache_310_gb300 as pkv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    nq = 512
    w, q, qs = workloads.prefill_workload(310_990, num_seqs=32, max_len=4096, min_len=1024, num_q_heads=64,
                                          num_kv_heads=8, block_size=16, dtype="bf16",
                                          new_tokens=lambda s, L: nq, canary=False, pool_device=dev)
    g = w.to(dev)
    qd, qsd = q.to(dev), qs.to(dev)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        pkv.paged_attention_prefill(qd, g.k_cache, g.v_cache, g.block_tables, g.context_lens, qsd, w.scale, out,
                                    max_context_len=w.max_context_len)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if pkv.device_error() != 0:
        raise SystemExit("device error flag set during warm-up")
    clocks = ClockSampler(dev.index or 0)
    time.sleep(0.3)
    steps = min(args.steps, 500)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / steps
    if pkv.device_error() != 0:
        raise SystemExit("device error flag set in the timed region")
    lens = w.context_lens.tolist()
    Hq, D = w.num_q_heads, w.head_dim
    flops = sum(4 * Hq * D * (L - nq + i + 1) for L in lens for i in range(nq))

    # End to end: each step's queries (and query_start) go up from pinned host memory and
    # its output comes back, on their own streams, double-buffered so that step i's
    # upload and step i - 1's download overlap the kernels (every copy in the timed region).
    q_host = q.contiguous().pin_memory()
    out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    qs_host = qs.contiguous().pin_memory()
    q_dev = [torch.empty_like(qd) for _ in range(2)]
    qs_dev = [torch.empty_like(qsd) for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n_e2e = max(3, min(args.e2e_steps, 100))

    def e2e_run(n):
        uploaded, consumed, fetched = [None, None], [None, None], [None, None]
        t0 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        up.wait_event(t0)

        def upload(i):
            b = i % 2
            with torch.cuda.stream(up):
                if consumed[b] is not None:
                    up.wait_event(consumed[b])
                q_dev[b].copy_(q_host, non_blocking=True)
                qs_dev[b].copy_(qs_host, non_blocking=True)
                uploaded[b] = torch.cuda.Event()
                uploaded[b].record(up)

        upload(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                upload(i + 1)
            stream.wait_event(uploaded[b])
            if fetched[b] is not None:
                stream.wait_event(fetched[b])
            pkv.paged_attention_prefill(q_dev[b], g.k_cache, g.v_cache, g.block_tables, g.context_lens, qs_dev[b],
                                        w.scale, outs[b], max_context_len=w.max_context_len)
            consumed[b] = torch.cuda.Event()
            consumed[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(consumed[b])
                out_host[b].copy_(outs[b], non_blocking=True)
                fetched[b] = torch.cuda.Event()
                fetched[b].record(down)
        for f in fetched:
            if f is not None:
                stream.wait_event(f)
        t1 = torch.cuda.Event(enable_timing=True)
        t1.record(stream)
        return t0, t1

    e2e_run(2)
    torch.cuda.synchronize()
    t0, t1 = e2e_run(n_e2e)
    torch.cuda.synchronize()
    e2e_ms = t0.elapsed_time(t1) / n_e2e
    if not torch.equal(out_host[(n_e2e - 1) % 2], out.cpu()):
        raise SystemExit("end-to-end output differs from the device-timed output")
    h2d = q_host.numel() * q_host.element_size() + qs_host.numel() * qs_host.element_size()
    d2h = out_host[0].numel() * out_host[0].element_size()

    # CPU baseline: the float64 oracle on one sequence's new tokens, timed on the host cores
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        kc, vc = w.k_cache.cpu(), w.v_cache.cpu()
        tables, lh = w.block_tables.cpu(), w.context_lens.cpu()
        rows = slice(int(qs[0]), int(qs[1]))
        t_start = time.perf_counter()
        oracle.attention_prefill(q[rows], kc, vc, tables[0:1], lh[0:1], torch.tensor([0, nq], dtype=torch.int32),
                                 w.scale)
        dt = time.perf_counter() - t_start
        f0 = sum(4 * Hq * D * (lens[0] - nq + i + 1) for i in range(nq))
        cpu = {"value": f0 / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"1 of {len(lens)} sequences ({nq} new tokens, context {lens[0]}), one call",
               "seconds_per_call": dt}
    kv = sum(lens) * 2 * w.num_kv_heads * D * 2
    qo = 2 * int(qs[-1]) * Hq * D * 2
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tpeak, tkind = float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        tpeak, tkind = 1900.0, "fallback"
    hpeak, hkind = peaks()
    tflops = flops / (ms * 1e-3) / 1e12
    line = {"metric": "paged prefill attention (causal): TFLOP/s, new tokens/s", "value": tflops, "unit": "TFLOP/s",
            "n_gpus": 1, "steps": steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": PREFILL_WORKLOAD, "new_tokens": int(qs[-1])},
            "tokens_per_s": int(qs[-1]) / (ms * 1e-3),
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": tpeak, "unit": "TFLOP/s",
                         "frac": tflops / tpeak, "peak_source": tkind,
                         "traffic": recorded_traffic("prefill", PREFILL_WORKLOAD, 0),
                         "kernel": "paged_attention_prefill (work list + prefill_tc)",
                         "algorithmic_flops_per_launch": flops},
            "hbm": {"algorithmic_bytes_per_launch": kv + qo, "achieved_gbs": (kv + qo) / (ms * 1e-3) / 1e9,
                    "peak": hpeak, "peak_source": hkind},
            "gpu_launches": 2 * steps, "clocks": clk,
            "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}}
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.prefill:
        run_prefill(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU fallback)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    import paged_kv_cache_310_gb300 as pkv

    path = {"auto": pkv.PATH_AUTO, "cuda_core": pkv.PATH_CUDA_CORE, "tensor_core": pkv.PATH_TENSOR_CORE}[args.path]
    # every rank decodes its own batch of the same workload shape (independent replicas)
    overrides = {k: v for k, v in (("block_size", args.block_size), ("head_dim", args.head_dim),
                                   ("num_q_heads", args.num_q_heads), ("dtype", args.dtype),
                                   ("num_seqs", args.num_seqs)) if v}
    w = workloads.make_workload(args.config, canary=False, pool_device=dev, shuffle=not args.identity_tables,
                                **overrides)
    g = w.to(dev)
    S, Hq, D = g.q.shape
    out = torch.empty((S, Hq, D), dtype=w.dtype, device=dev)
    maxL = w.max_context_len
    host_pairs = w.cow_pairs.cpu()
    stream = torch.cuda.current_stream(dev)

    # A step is the library's three calls, each prepared once (arguments checked and
    # marshalled) and then replayed on the stream, as a serving loop over fixed buffers
    # would: copy-on-write copies, the append, decode.
    def step_calls(q, kn, vn, slots, tables, lens, o):
        calls = []
        if g.cow_pairs.numel():
            calls.append(pkv.prepare_block_copy(g.cow_pairs, g.k_cache, g.v_cache))
        calls.append(pkv.prepare_kv_append(kn, vn, slots, g.k_cache, g.v_cache))
        calls.append(pkv.prepare_attention_decode(q, g.k_cache, g.v_cache, tables, lens, w.scale, o,
                                                  max_context_len=maxL, path=path,
                                                  partition_tokens=args.partition))
        return calls

    handle = stream.cuda_stream
    resident = step_calls(g.q, g.k_new, g.v_new, g.slot_mapping, g.block_tables, g.context_lens, out)

    def step(calls=resident):
        for call in calls:
            call(handle)

    if g.cow_pairs.numel():  # validate the pairs once on the host
        pkv.paged_block_copy(g.cow_pairs, g.k_cache, g.v_cache, host_pairs=host_pairs)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if pkv.device_error() != 0:
        raise SystemExit("device error flag set during warm-up")

    plan = pkv.paged_attention_plan(S, Hq, maxL, g.k_cache, path=path, partition_tokens=args.partition)
    launches_per_step = (1 if g.cow_pairs.numel() else 0) + 1 + plan["kernel_launches"]

    # ---------------- device-timed region ----------------
    clocks = ClockSampler(local)
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    # Events bracket the whole run only: an event between a step's kernels would keep
    # the work list from overlapping the append (dependent launch).
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_begin.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    total_ms = t_begin.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, dist, dev)
    if pkv.device_error() != 0:
        raise SystemExit("device error flag set in the timed region")
    ms_per_step = total_ms / args.steps
    # The decode call alone (work list + decode kernel, + merge when split), each launch
    # bracketed by events on its stream: the roofline's kernel time.
    n_k = max(DECODE_CALLS_MIN, min(args.steps, 1000))
    decode_ms = decode_call_ms(lambda: resident[-1](handle), stream, n_k)
    # The other decode workloads the method is measured on, each timed the same way
    # (only on the default workload, without overrides, so the line stays one run)
    per_config = None
    if args.config == 2 and not overrides and not args.identity_tables and args.per_config:
        per_config = {str(c): measure_config(pkv, c, dev, path, args.partition, n_k) for c in (3, 4, 5)}
    torch.cuda.synchronize()
    clk = clocks.stop()

    # ---------------- end to end: host inputs in, host output out ----------------
    # The step's inputs sit in one pinned staging buffer (each tensor 256-byte aligned)
    # and travel in one copy per step.  As a serving loop would, the copies run on their
    # own streams and overlap the previous step's kernels: staging and output are
    # double-buffered, step i's inputs go up while step i - 1 computes, and step i's
    # output comes down while step i + 1 computes.  Every copy is inside the timed region.
    host_in = [t.cpu().contiguous() for t in (w.q, w.k_new, w.v_new, w.slot_mapping, w.block_tables,
                                               w.context_lens)]
    offs, total = [], 0
    for t in host_in:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    stage_host = torch.empty(total, dtype=torch.uint8).pin_memory()
    for t, o in zip(host_in, offs):
        nb = t.numel() * t.element_size()
        stage_host[o:o + nb].copy_(t.view(-1).view(torch.uint8))
    stage_dev = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    dev_in = [[sd[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(host_in, offs)]
              for sd in stage_dev]
    outs = [torch.empty_like(out) for _ in range(2)]
    out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = out_host[0].numel() * out_host[0].element_size()
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n_e2e = max(3, args.e2e_steps)
    e2e_calls = [step_calls(*dev_in[b], outs[b]) for b in range(2)]
    # per buffer b: its inputs are on the device / its kernels are done with it / its
    # output is back on the host (events re-recorded each step)
    uploaded = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    fetched = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n):
        e0 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up.wait_event(e0)

        def upload(i):
            b = i % 2
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(consumed[b])
                stage_dev[b].copy_(stage_host, non_blocking=True)
                uploaded[b].record(up)

        upload(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                upload(i + 1)
            stream.wait_event(uploaded[b])
            if i >= 2:
                stream.wait_event(fetched[b])
            step(e2e_calls[b])
            consumed[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(consumed[b])
                out_host[b].copy_(outs[b], non_blocking=True)
                fetched[b].record(down)
        for i in range(max(0, n - 2), n):
            stream.wait_event(fetched[i % 2])
        e1 = torch.cuda.Event(enable_timing=True)
        e1.record(stream)
        return e0, e1

    e2e_run(3)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = e2e_run(n_e2e)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / n_e2e
    if not torch.equal(out_host[(n_e2e - 1) % 2], out.cpu()):
        raise SystemExit("end-to-end output differs from the device-timed output")
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)

    kv_bytes, algo_bytes = roofline_bytes(w, elem(out.dtype))
    peak, peak_kind = peaks()
    tokens = int(w.context_lens.sum())
    value = whole_job_rate(world, kv_bytes, ms_per_step)
    achieved = algo_bytes / (decode_ms * 1e-3) / 1e9
    result = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": workloads.DTYPE_NAMES[w.dtype], "data": "synthetic",
        "config": {"workload": w.name, "num_seqs": S, "num_q_heads": Hq, "num_kv_heads": w.num_kv_heads,
                   "head_dim": D, "block_size": w.block_size, "sum_context_tokens": tokens,
                   "kv_bytes_per_step": kv_bytes, "path": {1: "cuda_core", 2: "tensor_core"}[plan["path"]],
                   "partition_tokens": plan["partition_tokens"], "partitions": plan["max_partitions"],
                   "kv_heads_per_item": plan["kv_heads_per_item"],
                   "l2": f"inputs larger than L2 (KV {kv_bytes / 1e9:.2f} GB > 129 MB): no flush",
                   "parallelism": f"replicas x{world}", "block_tables": "identity" if args.identity_tables
                   else "shuffled"},
        "seq_tokens_per_s": world * tokens / (ms_per_step * 1e-3),
        "hbm_frac_step": (algo_bytes / (ms_per_step * 1e-3) / 1e9) / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "traffic": recorded_traffic(traffic_path(plan["path"], w.dtype), w.name,
                                                 plan["partition_tokens"]),
                     "kernel": {"tensor_core": "paged_attention_decode (work list + decode_tc, + merge when split)",
                                "tensor_core_f32": "paged_attention_decode (work list + decode_tc32, + merge when "
                                                   "split)",
                                "cuda_core": "paged_attention_decode (decode_simt, + merge when split)"}[
                         traffic_path(plan["path"], w.dtype)],
                     "algorithmic_bytes_per_launch": algo_bytes, "ms_per_launch": decode_ms},
        "e2e": {"value": whole_job_rate(world, kv_bytes, e2e_ms), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if per_config is not None:
        result["per_config"] = per_config
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(w, args.cpu_seconds)
        cb.pop("_kv_bytes", None)
        result["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
