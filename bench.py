"""Benchmark of the hybrid-batch step: one Mistral-7B-shaped decoder layer plus
its 32000-entry LM head at token budget tau = 512 -- a 448-token prefill chunk
at start positions 0, 512 and 1536 (cycled) with 64 piggybacked decodes whose
contexts are uniform in [128, 4096].

Prints one JSON line.  ``value`` is hybrid-batch tokens/s (rows of the
stacked batch per second) over the timed steps with inputs resident in HBM,
each case's step replayed from a captured CUDA graph (``--no-graph``: launched
kernel by kernel);
``e2e`` is the same metric through the host-buffer C entry point with the
host<->device copies inside the timed region.  ``--impl reference`` times the
CPU oracle on a bounded sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

TAU, BD, STARTS = 512, 64, (0, 512, 1536)
PAGE = 16
METRIC = "hybrid-step tokens/s at tau=512 (Mistral-7B-shaped layer + LM head)"
UNIT = "tokens/s"
WORKLOAD = ("Mistral-7B-shaped layer (H=4096, 32q/8kv heads x 128, FFN 14336) + final norm + "
            "LM head 32000; Lp=448 chunk at start {0,512,1536} (cycled) + Bd=64 decodes, "
            "ctx U[128,4096]; bf16 weights N(0,0.02), random N(0,1) KV pages")


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# Replicas only: every rank runs its own model on its own GPU (the step does
# not shard), the ranks meet at barriers around the timed region, the slowest
# rank's time is the job's, and the job's value counts every rank's rows.

def max_over_ranks(x: float, world: int) -> float:
    """The largest of every rank's x (the job's time is the slowest rank's)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(rows_per_rank: int, world: int, seconds: float) -> float:
    """Rows of every rank over the job's (slowest rank's) time."""
    return rows_per_rank * world / seconds


def config_block(n):
    return {"workload": WORKLOAD, "layers": 1, "tau": TAU, "lp": TAU - BD, "bd": BD,
            "starts": list(STARTS), "page_size": PAGE, "parallelism": f"replicas x{n}",
            "l2": "inputs larger than L2 (weights 436 MB + LM head 262 MB + KV ~0.55 GB per step)"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        # sampling every 5 ms; the timed region starts once the first sample has
        # arrived, so every later sample falls inside it (or just after it ends)
        import threading
        self.lines, self.first = [], threading.Event()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "5"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except OSError:
            self.proc = None
            return self

        def reader():
            for line in self.proc.stdout:
                self.lines.append(line)
                self.first.set()
            self.first.set()

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        self.first.wait(timeout=10)
        self.skip = len(self.lines)  # samples taken before the timed region
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            self.thread.join(timeout=5)
            self.out = "".join(self.lines[self.skip:])

    def summary(self):
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sms.append(float(f[0]))
                maxs.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sms.sort()
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(maxs), "reasons": sorted(reasons),
                "samples": len(sms)}


# ------------------------------------------------------------------ peaks

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ our arm

def setup_gpu(seed=0, storage=None):
    import torch

    import chunked_prefill_hybrid_sar_gb300 as sar
    from chunked_prefill_hybrid_sar_gb300 import harness

    dims = synth.MISTRAL_LAYER
    gen = synth.generator(seed, "cuda")
    layers = [synth.layer_weights(gen, dims, torch.bfloat16, "cuda")]
    head = synth.head_weights(gen, dims, torch.bfloat16, "cuda")
    m = harness.load_model(dims, layers, head, max_tokens=TAU, max_decodes=BD,
                           storage=sar.SAR_STORAGE_F16 if storage is None else storage)
    del layers, head
    cg = synth.generator(seed + 1)
    ctxs = synth.uniform_int(cg, BD, 128, 4096)
    need = sum(math.ceil((c + 1) / PAGE) for c in ctxs) + len(STARTS) * (2048 // PAGE)
    kv = sar.KVCache(m, PAGE, need)
    # random N(0,1) key/value histories everywhere; prompt pages get rewritten by the prior chunks
    for kind in (0, 1):
        pv = harness.page_view(kv, 0, kind, dims)
        pv.copy_(torch.randn(pv.shape, generator=gen, device="cuda", dtype=torch.float32).to(torch.bfloat16))
    alloc = harness.PageAllocator(range(need))
    dec_bt = [alloc.take(math.ceil((c + 1) / PAGE)) for c in ctxs]
    decs = [(100 + i, c, dec_bt[i]) for i, c in enumerate(ctxs)]
    lp = TAU - BD
    cases = []
    for s in STARTS:
        bt = alloc.take(2048 // PAGE)
        prompt = synth.normal(gen, (s + lp, dims.hidden), dtype=torch.bfloat16, device="cuda")
        for s0 in range(0, s, 512):  # the prompt's earlier chunks
            m.step(kv, sar.Batch((s, s0, 512, bt), []), prompt[s0:s0 + 512].contiguous())
        dec_in = synth.normal(gen, (BD, dims.hidden), dtype=torch.bfloat16, device="cuda")
        x = torch.cat([prompt[s:s + lp], dec_in]).contiguous()
        cases.append((sar.Batch((s, s, lp, bt), decs), x))
    torch.cuda.synchronize()
    m.sync_status()
    return dims, m, kv, cases, ctxs


def decode_attention_bytes(dims, ctxs):
    """Algorithmic HBM bytes of one decode-attention launch: every key and value
    of every decode's context (ctx + 1 keys incl. the new one) once, plus its
    query and output rows."""
    kv = sum(c + 1 for c in ctxs) * dims.n_kv_heads * dims.head_dim * 2 * 2
    qo = len(ctxs) * dims.q_dim * 2 * 2
    return kv + qo


def chunk_attention_flops(dims, lp, start):
    """Algorithmic flops of the chunk's causal attention: each query at
    position start + i scores and sums start + i + 1 keys (2 d flops each for
    q.k and for p.v) in every query head."""
    keys = lp * start + lp * (lp + 1) // 2
    return 4 * dims.head_dim * dims.n_q_heads * keys


# DRAM bytes read + written per launch (dram__bytes_read.sum +
# dram__bytes_write.sum) from one ncu capture on this workload, with the
# source files of the kernel they were taken on and those files' SHA-256
# prefix: a figure whose kernel source has changed since is reported as null.
TRAFFIC = {
    "decode_attn": {"bytes": 521.6e6, "files": ("csrc/attn_decode.cu",), "sha": "073943615c60a19e",
                    "capture": "profiles/decode_attn_mistral_layer.md"},
}


def source_sha(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "chunked_prefill_hybrid_sar_gb300", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_of(kernel):
    t = TRAFFIC.get(kernel)
    if not t:
        return None, "no capture of this kernel"
    cur = source_sha(t["files"])
    if cur != t["sha"]:
        return None, f"kernel source changed since the capture in {t['capture']} (sha {cur})"
    return t["bytes"], f"ncu capture, {t['capture']} (kernel source sha {cur})"


def step_roofline(dims, ctxs, hbm, tf):
    """Per-operator max(T_math, T_mem) summed over the step, and the
    concurrent-overlap bound max(sum T_math, sum T_mem), at peaks (hbm GB/s,
    tf TFLOP/s).  Chunk attention is averaged over the three chunk starts."""
    wb = 2 * dims.hidden
    lp = TAU - BD
    ops = {  # name: (flops, bytes)
        "gemm_qkv": (gemm_flops(dims, TAU)["gemm_qkv"], wb * (dims.q_dim + 2 * dims.kv_dim) + TAU * wb),
        "gemm_o": (gemm_flops(dims, TAU)["gemm_o"], wb * dims.q_dim + TAU * dims.q_dim * 2 + TAU * dims.hidden * 8),
        "gemm_gateup": (gemm_flops(dims, TAU)["gemm_gateup"], wb * 2 * dims.ffn + TAU * wb + TAU * dims.ffn * 2),
        "gemm_down": (gemm_flops(dims, TAU)["gemm_down"], 2 * dims.ffn * dims.hidden + TAU * dims.ffn * 2
                      + TAU * dims.hidden * 8),
        "chunk_attn": (sum(chunk_attention_flops(dims, lp, s) for s in STARTS) / len(STARTS),
                       sum((s + lp) for s in STARTS) / len(STARTS) * dims.kv_dim * 2 * 2),
        "decode_attn": (sum(4 * dims.head_dim * dims.n_q_heads * (c + 1) for c in ctxs),
                        decode_attention_bytes(dims, ctxs)),
        "gemm_head": (2 * (BD + 1) * dims.hidden * dims.vocab, dims.vocab * dims.hidden * 2),
        # four row passes: input + first norm, second norm, final norm (sampled rows), each reading
        # fp32 rows and writing 16-bit rows; counted as full passes over the stacked rows
        "norms": (0, 3 * TAU * dims.hidden * (4 + 2)),
    }
    t = {k: max(f / (tf * 1e12), b / (hbm * 1e9)) for k, (f, b) in ops.items()}
    t_math = sum(f for f, _ in ops.values()) / (tf * 1e12)
    t_mem = sum(b for _, b in ops.values()) / (hbm * 1e9)
    return sum(t.values()), max(t_math, t_mem), t, t_math, t_mem


def gemm_flops(dims, rows):
    return {"gemm_qkv": 2 * rows * dims.hidden * (dims.q_dim + 2 * dims.kv_dim),
            "gemm_o": 2 * rows * dims.q_dim * dims.hidden,
            "gemm_gateup": 2 * rows * dims.hidden * 2 * dims.ffn,
            "gemm_down": 2 * rows * dims.ffn * dims.hidden}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import chunked_prefill_hybrid_sar_gb300 as sar

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dims, m, kv, cases, ctxs = setup_gpu()
    if args.overlap:
        m.set_overlap(True)
    hid = torch.empty(TAU, dims.hidden, dtype=torch.float32, device="cuda")
    logits = torch.empty(BD + 1, dims.vocab, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    graphs, graph_launches = None, 0

    def step(i):
        if graphs:
            graphs[i % len(cases)].launch()
            return
        b, x = cases[i % len(cases)]
        m.step(kv, b, x, hidden_out=hid, logits_out=logits)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    m.sync_status()
    if args.graph:
        # one captured step per case (the cases repeat unchanged)
        l0 = sar.launch_count()
        graphs = [sar.StepGraph(m, kv, b, x, hidden_out=hid, logits_out=logits) for b, x in cases]
        graph_launches = (sar.launch_count() - l0) / len(cases)
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # timed region: device events on the launching stream
    launches0 = sar.launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        t0 = time.perf_counter()
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
        barrier()
        wall = time.perf_counter() - t0
    launches = sar.launch_count() - launches0
    graph_set = graphs
    if graphs:
        launches = int(graph_launches * args.steps)  # kernels inside the replayed graphs
        graphs = None  # the per-kernel pass launches kernel by kernel
    ms = ev0.elapsed_time(ev1)
    m.sync_status()
    ms = max_over_ranks(ms, world)
    value = whole_job_rate(TAU * args.steps, world, ms / 1e3)

    # per-kernel times: the same steps again with an event pair around every kernel
    m.profile(True)
    for i in range(args.steps):
        step(i)
    prof = m.profile_read()
    m.profile(False)
    hbm, tf_burst, tf_sust, peak_src = peaks()
    total = sum(v[0] for v in prof.values()) or 1.0
    kernels = {}
    for k, (t, n) in prof.items():
        if n:
            kernels[k] = {"ms_per_launch": t / n, "share": t / total, "launches": n}
    flops = gemm_flops(dims, TAU)
    for k, f in flops.items():
        if k in kernels:
            kernels[k]["tflops"] = f / (kernels[k]["ms_per_launch"] * 1e-3) / 1e12
    dab = decode_attention_bytes(dims, ctxs)
    if "decode_attn" in kernels:
        kernels["decode_attn"]["gbs"] = dab / (kernels["decode_attn"]["ms_per_launch"] * 1e-3) / 1e9
    head_bytes = dims.vocab * dims.hidden * 2
    if "gemm_head" in kernels:
        kernels["gemm_head"]["gbs"] = head_bytes / (kernels["gemm_head"]["ms_per_launch"] * 1e-3) / 1e9
    dom = max(kernels, key=lambda k: kernels[k]["share"])
    traffic, traffic_src = traffic_of(dom)
    # the timed region lasts milliseconds at full clocks: the burst peak applies
    if dom in flops:
        ach = kernels[dom]["tflops"]
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": tf_burst, "unit": "TFLOP/s",
                "frac": ach / tf_burst, "traffic": traffic, "traffic_source": traffic_src,
                "peak_source": f"{peak_src} bf16 burst", "algorithmic_per_launch": flops[dom]}
    else:
        byts = dab if dom == "decode_attn" else head_bytes
        ach = byts / (kernels[dom]["ms_per_launch"] * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm, "traffic": traffic, "traffic_source": traffic_src,
                "peak_source": f"{peak_src} HBM copy", "algorithmic_per_launch": byts}

    # step roofline: per-operator max(T_math, T_mem) summed, and the overlap
    # bound, at the burst peak (the timed region is milliseconds long at full
    # clocks) and at the sustained one
    step_ms = ms / args.steps
    t_roof, t_overlap, t_ops, t_math, t_mem = step_roofline(dims, ctxs, hbm, tf_burst)
    t_roof_s, t_overlap_s, _, _, _ = step_roofline(dims, ctxs, hbm, tf_sust)
    roof_step = {"per_op_sum_ms": t_roof * 1e3, "per_op_frac": t_roof * 1e3 / step_ms,
                 "overlap_bound_ms": t_overlap * 1e3, "overlap_frac": t_overlap * 1e3 / step_ms,
                 "sum_t_math_ms": t_math * 1e3, "sum_t_mem_ms": t_mem * 1e3,
                 "per_op_ms": {k: v * 1e3 for k, v in t_ops.items()},
                 "peaks": f"{peak_src}: bf16 burst {tf_burst} TFLOP/s, HBM {hbm} GB/s",
                 "sustained_peak": {"per_op_sum_ms": t_roof_s * 1e3, "per_op_frac": t_roof_s * 1e3 / step_ms,
                                    "overlap_bound_ms": t_overlap_s * 1e3,
                                    "overlap_frac": t_overlap_s * 1e3 / step_ms, "tflops": tf_sust}}

    # end to end: host buffers through the host entry points, one step at a
    # time (each step's input rows in from pinned memory, its result back,
    # then the next step).  With the captured graph of each case the result is
    # every sampled row's greedy token id, picked on the device
    # (sar_graph_launch_host_tokens: the serving loop's round trip); the same
    # loop reading back the whole logits rows instead (sar_graph_launch_host)
    # is reported beside it.  With --no-graph: the planning entry point
    # (sar_step_host), logits back.
    pin_in = [x.cpu().pin_memory() for _, x in cases]
    h_log = torch.empty(BD + 1, dims.vocab, dtype=torch.float32).pin_memory()
    h_tok = torch.empty(BD + 1, dtype=torch.int32).pin_memory()

    def e2e_run(step_fn):
        for i in range(3):
            step_fn(i)
        barrier()
        t0 = time.perf_counter()
        for i in range(args.steps):
            step_fn(i)
        barrier()
        return max_over_ranks(time.perf_counter() - t0, world)

    def logits_step(i):
        if graph_set:
            graph_set[i % 3].launch_host(pin_in[i % 3], logits_out=h_log)
        else:
            m.step_host(kv, cases[i % 3][0], pin_in[i % 3], logits_out=h_log)

    def tokens_step(i):
        graph_set[i % 3].launch_host_tokens(pin_in[i % 3], h_tok)

    def replanned_tokens_step(i):
        # the serving loop's step: plan the batch on the host and re-point the
        # captured graph at it (sar_graph_update), then run it with host buffers
        graph_set[i % 3].update(cases[i % 3][0])
        graph_set[i % 3].launch_host_tokens(pin_in[i % 3], h_tok)

    def planned_logits_step(i):
        m.step_host(kv, cases[i % 3][0], pin_in[i % 3], logits_out=h_log)

    h2d = TAU * dims.hidden * 2
    e2e_log_s = e2e_run(logits_step)
    e2e_logits = {"value": whole_job_rate(TAU * args.steps, world, e2e_log_s), "unit": UNIT,
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": (BD + 1) * dims.vocab * 4,
                  "api": "sar_graph_launch_host" if graph_set else "sar_step_host"}
    e2e_eager_s = e2e_run(planned_logits_step)
    e2e_eager = {"value": whole_job_rate(TAU * args.steps, world, e2e_eager_s), "unit": UNIT,
                 "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": (BD + 1) * dims.vocab * 4,
                 "api": "sar_step_host (host planning, kernel-by-kernel launch, logits back)"}
    e2e_fixed = None
    e2e_pipe = None
    if graph_set:
        e2e_s = e2e_run(replanned_tokens_step)
        e2e = {"value": whole_job_rate(TAU * args.steps, world, e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": (BD + 1) * 4,
               "api": "sar_graph_update (the step planned on the host) + sar_graph_launch_host_tokens "
                      "(greedy token ids of the 65 sampled rows back)"}
        # the same serving loop with step i+1 planned (sar_graph_update) and
        # enqueued -- its input copied on the graph's own copy stream -- while
        # step i runs, and step i's token ids waited for after that
        toks = [torch.empty(BD + 1, dtype=torch.int32).pin_memory() for _ in range(3)]

        def pipelined(n):
            prev = None
            for i in range(n):
                g = graph_set[i % 3]
                g.update(cases[i % 3][0])
                g.enqueue_host_tokens(pin_in[i % 3], toks[i % 3])
                if prev is not None:
                    prev.wait()
                prev = g
            prev.wait()

        pipelined(3)
        barrier()
        t0 = time.perf_counter()
        pipelined(args.steps)
        barrier()
        e2e_pipe_s = max_over_ranks(time.perf_counter() - t0, world)
        e2e_pipe = {"value": whole_job_rate(TAU * args.steps, world, e2e_pipe_s), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": (BD + 1) * 4,
                    "api": "sar_graph_update + sar_graph_enqueue_host_tokens, sar_graph_wait one step late "
                           "(the next step planned and its input copied while the current one runs)"}
        e2e_fixed_s = e2e_run(tokens_step)
        e2e_fixed = {"value": whole_job_rate(TAU * args.steps, world, e2e_fixed_s), "unit": UNIT,
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": (BD + 1) * 4,
                     "api": "sar_graph_launch_host_tokens without replanning"}
    else:
        e2e = e2e_eager

    # the same workload with bf16 storage of weights, activations and KV
    bf16 = None
    if not args.no_bf16:
        for g in graph_set or []:
            g.close()
        graph_set = None
        bf16 = bf16_storage_line(args, world)

    out = None
    if rank == 0:
        cpu = cpu_baseline(args) if (world == 1 and not args.no_cpu) else None
        out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None,
               "dtype": "f16 storage (bf16 weights converted exactly), fp32 accumulate and residual",
               "data": "synthetic (seeded random-init weights and KV histories)",
               "config": dict(config_block(world), attn_streams=2 if args.overlap else 1,
                              launch="cuda graph per case" if args.graph else "kernel by kernel"),
               "e2e": e2e, "e2e_pipelined": e2e_pipe, "e2e_no_replan": e2e_fixed,
               "e2e_logits_readback": e2e_logits,
               "e2e_eager_planned": e2e_eager, "gpu_launches": launches,
               "roofline": roof, "step_roofline_ms": t_roof * 1e3,
               "step_roofline_frac": (t_roof * 1e3) / step_ms, "step_roofline": roof_step,
               "bf16_storage": bf16,
               "kernels": kernels, "clocks": clk.summary(), "wall_s": wall, "cpu_baseline": cpu}
        print(json.dumps(out))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return out


def bf16_storage_line(args, world):
    """The step of the same workload on a model that stores weights,
    activations and KV in bf16 (fp32 accumulation and residual), each case
    replayed from its captured graph; device-timed like the main line."""
    import torch

    import chunked_prefill_hybrid_sar_gb300 as sar

    dims, m, kv, cases, _ = setup_gpu(storage=sar.SAR_STORAGE_BF16)
    hid = torch.empty(TAU, dims.hidden, dtype=torch.float32, device="cuda")
    logits = torch.empty(BD + 1, dims.vocab, dtype=torch.float32, device="cuda")
    graphs = [sar.StepGraph(m, kv, b, x, hidden_out=hid, logits_out=logits) for b, x in cases]
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        graphs[i % 3].launch()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        graphs[i % 3].launch()
    ev1.record(stream)
    torch.cuda.synchronize()
    m.sync_status()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    for g in graphs:
        g.close()
    m.close()
    kv.close()
    return {"value": whole_job_rate(TAU * args.steps, world, ms / 1e3), "unit": UNIT,
            "ms_per_step": ms / args.steps, "dtype": "bf16 storage, fp32 accumulate and residual",
            "launch": "cuda graph per case",
            "parity": "bf16 storage meets the per-layer bars on the tiny layer; on this layer bf16 "
                      "rounding of the activations alone exceeds max-abs 3e-2, hence fp16 storage for the "
                      "main line"}


# ------------------------------------------------------------------ oracle arm

def oracle_cases(seed=3, dtype="float64"):
    """The workload's cases for the CPU oracle: per chunk start (0, 512,
    1536) one hybrid step of the 448-token chunk and all 64 decodes (contexts
    uniform in [128, 4096], random K/V histories), drawn by the same recipe
    as the GPU cases with another seed, as arrays of ``dtype`` (the oracle
    computes in the type of its inputs).  Returns (dims, weights, head, the
    steps' parts, rows per step)."""
    import numpy as np

    from oracle import model as om

    dt = np.dtype(dtype)
    case = synth.mistral_layer_case(seed, n_decode=BD, tau=TAU, starts=synth.MISTRAL_STARTS)
    dims = case["dims"]
    w = om.layer_weights_np(case["layers"][0], dt)
    head = om.layer_weights_np(case["head"], dt)
    decs = []
    for i, c in enumerate(case["ctxs"]):
        k, v = case["histories"][i]
        decs.append(om.Part(x=om.to_np(case["decode_inputs"][i:i + 1], dt), lo=c,
                            given=[om.LayerCache(om.to_np(k, dt), om.to_np(v, dt))]))
    steps = [[om.Part(x=om.to_np(case["prompts"][s], dt), lo=s, is_prefill=True)] + decs
             for s in synth.MISTRAL_STARTS]
    return dims, w, head, steps, case["lp"] + BD


def oracle_sample_text(n_steps, dt, dtype="float64"):
    starts = synth.MISTRAL_STARTS[:min(n_steps, len(synth.MISTRAL_STARTS))]
    return (f"{n_steps} oracle hybrid steps ({dtype} NumPy) of the workload itself, the chunk at start "
            f"{'/'.join(str(s) for s in starts)} in turn with all {BD} decodes "
            f"({TAU} rows each; {dt:.1f} s; the oracle computes a chunk by running its prompt prefix)")


def oracle_leg(dtype="float64", min_s=10.0, max_passes=4):
    """Times the oracle on the workload's cases in turn (start 0 first), whole
    passes over the three cases until at least ``min_s`` seconds of work (at
    most ``max_passes``); with ``max_passes`` 0, steps until ``min_s`` (at
    least one).  Returns (tokens/s, steps, seconds)."""
    from oracle import model as om

    dims, w, head, steps, rows = oracle_cases(dtype=dtype)
    n = 0
    t0 = time.perf_counter()
    if max_passes:
        while n < max_passes * len(steps) and (n % len(steps) or n == 0 or time.perf_counter() - t0 < min_s):
            om.hybrid_step([w], head, dims, steps[n % len(steps)])
            n += 1
    else:
        while n == 0 or time.perf_counter() - t0 < min_s:
            om.hybrid_step([w], head, dims, steps[n % len(steps)])
            n += 1
    dt = time.perf_counter() - t0
    return rows * n / dt, n, dt


def cpu_leg_subprocess(dtype, threads, min_s):
    """One oracle leg in a fresh interpreter whose BLAS and OpenMP pools are
    limited to ``threads`` (set before NumPy loads); returns its JSON."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-leg", dtype, "--cpu-leg-min-s", str(min_s)],
                       env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout).strip().splitlines()[-1:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(args):
    """The oracle as it stands (float64) on all the host's cores, with the
    fp32 oracle on all cores and on one thread beside it."""
    value, n, dt = oracle_leg("float64")
    cores = len(os.sched_getaffinity(0))
    out = {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": oracle_sample_text(n, dt)}
    f32_all = cpu_leg_subprocess("float32", cores, 5.0)
    f32_one = cpu_leg_subprocess("float32", 1, 5.0)
    out["variants"] = {
        "float32_all_cores": dict(f32_all, cores=cores),
        "float32_one_thread": dict(f32_one, cores=1),
    }
    return out


def run_cpu_leg(args):
    value, n, dt = oracle_leg(args.cpu_leg, min_s=args.cpu_leg_min_s, max_passes=0)
    print(json.dumps({"value": value, "unit": UNIT, "kind": "oracle",
                      "sample": oracle_sample_text(n, dt, args.cpu_leg)}))


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    from oracle import model as om

    dims, w, head, steps, rows = oracle_cases()
    for i in range(min(args.warmup, 1)):
        om.hybrid_step([w], head, dims, steps[i % len(steps)])
    t0 = time.perf_counter()
    for i in range(args.steps):  # the cases in turn, as the GPU arm cycles them
        om.hybrid_step([w], head, dims, steps[i % len(steps)])
    dt = time.perf_counter() - t0
    value = rows * args.steps / dt
    cores = len(os.sched_getaffinity(0))
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": config_block(world),
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                            "sample": oracle_sample_text(args.steps, dt)},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))
    return out


# ------------------------------------------------------------------ tile sweep

SWEEP_ROWS = synth.SWEEP_ROWS
SWEEP_DECODE_ONLY = (1, 8, 32, 64)


def run_sweep(args):
    """Tile-quantisation and budget sweep on the Mistral-shaped layer: per GEMM
    and tiling, device time with L2 flushed between launches; then the full
    hybrid step at each row count (Bd = 32 decodes at context 2048, the rest
    one chunk); then the decode-only linear cost per token relative to 2048-row
    steps.  Prints one JSON line."""
    import torch

    import chunked_prefill_hybrid_sar_gb300 as sar
    from chunked_prefill_hybrid_sar_gb300 import harness

    dims = synth.MISTRAL_LAYER
    gen = synth.generator(0, "cuda")
    w = synth.layer_weights(gen, dims, torch.bfloat16, "cuda")
    f16 = {k: v.to(torch.float16) for k, v in w.items()}
    wqkv = torch.cat([f16["wq"], f16["wk"], f16["wv"]])
    wgu = torch.stack([f16["wg"].view(-1, 64, dims.hidden), f16["wu"].view(-1, 64, dims.hidden)], 1)
    wgu = wgu.reshape(2 * dims.ffn, dims.hidden)
    shapes = {"qkv": (wqkv, sar.SAR_EPI_STORE), "o": (f16["wo"], sar.SAR_EPI_RESIDUAL),
              "gateup": (wgu, sar.SAR_EPI_SWIGLU), "down": (f16["wd"], sar.SAR_EPI_RESIDUAL)}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    variants = {"m128n128": sar.SAR_GEMM_M128_N128, "m128n256": sar.SAR_GEMM_M128_N256,
                "m256n128": sar.SAR_GEMM_M256_N128, "swap": sar.SAR_GEMM_SWAP, "auto": sar.SAR_GEMM_AUTO}
    # CTA-pair tilings and stream-K on request only (not in the default sweep)
    extra_variants = {"pair256": sar.SAR_GEMM_PAIR_N256, "pair128": sar.SAR_GEMM_PAIR_N128,
                      "pair192": sar.SAR_GEMM_PAIR_N192, "pair256_sk": sar.SAR_GEMM_PAIR_N256 | sar.SAR_GEMM_STREAM_K}
    _, _, tf_sust, _ = peaks()
    lin_flops = 2 * (dims.hidden * (dims.q_dim + 2 * dims.kv_dim) + dims.q_dim * dims.hidden
                     + 3 * dims.hidden * dims.ffn)

    rows_list = [int(r) for r in args.rows.split(",")] if args.rows else list(SWEEP_ROWS)
    if args.variants:
        variants = {k: {**variants, **extra_variants}[k] for k in args.variants.split(",")}
    reps_default = args.reps

    def time_gemm(M, name, variant, reps=None):
        reps = reps_default if reps is None else reps
        wt, epi = shapes[name]
        K = wt.shape[1]
        a = torch.randn(M, K, device="cuda").to(torch.float16)
        if epi == sar.SAR_EPI_SWIGLU:
            c = torch.empty(M, wt.shape[0] // 2, dtype=torch.float16, device="cuda")
        elif epi == sar.SAR_EPI_RESIDUAL:
            c = torch.zeros(M, wt.shape[0], dtype=torch.float32, device="cuda")
        else:
            c = torch.empty(M, wt.shape[0], dtype=torch.float16, device="cuda")
        r = c if epi == sar.SAR_EPI_RESIDUAL else None
        ts = []
        for _ in range(reps + 1):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            sar.gemm(a, wt, c, residual=r, epilogue=epi, variant=variant)
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        ts = sorted(ts[1:])
        return ts[len(ts) // 2]

    gemm = {}
    for M in rows_list:
        gemm[M] = {}
        for vn, v in variants.items():
            if vn == "swap" and M > 256:
                continue
            row = {}
            for name in shapes:
                try:
                    row[name] = time_gemm(M, name, v)
                except sar.SarError:
                    row[name] = None
            if all(x is not None for x in row.values()):
                row["linear_ms"] = sum(row[n] for n in shapes)
                row["tflops"] = M * lin_flops / (row["linear_ms"] * 1e-3) / 1e12
                row["frac_of_sustained_peak"] = row["tflops"] / tf_sust
            gemm[M][vn] = row
    if args.gemm_only:
        out = {"mode": "sweep", "workload": "Mistral-7B-shaped layer projections, rows " + str(rows_list) +
               "; f16 storage; L2 flushed (256 MB write) before every timed launch", "gemm_ms": gemm}
        print(json.dumps(out))
        return out
    per_tok_2048 = gemm[2048]["auto"]["linear_ms"] / 2048
    equiv = {}
    for bd in SWEEP_DECODE_ONLY:
        t = sum(time_gemm(bd, n, sar.SAR_GEMM_AUTO) for n in shapes)
        equiv[bd] = {"linear_ms": t, "per_token_ms": t / bd,
                     "prefill_token_equivalents": (t / bd) / per_tok_2048}
    m = harness.load_model(dims, [w], None, max_tokens=2048, max_decodes=64)
    bd = 32
    need = bd * (2048 // PAGE + 1) + 2048 // PAGE + 8
    kv = sar.KVCache(m, PAGE, need)
    for kind in (0, 1):
        pv = harness.page_view(kv, 0, kind, dims)
        pv.copy_(torch.randn(pv.shape, generator=gen, device="cuda").to(pv.dtype))
    alloc = harness.PageAllocator(range(need))
    dec = [(i, 2048, alloc.take(2048 // PAGE + 1)) for i in range(bd)]
    pbt = alloc.take(2048 // PAGE)
    step = {}
    for M in SWEEP_ROWS:
        b = sar.Batch((99, 0, M - bd, pbt), dec)
        x = torch.randn(M, dims.hidden, device="cuda").to(torch.bfloat16)
        for _ in range(3):
            m.step(kv, b, x)
        torch.cuda.synchronize()
        m.profile(True)
        for _ in range(5):
            flush.zero_()
            m.step(kv, b, x)
        prof = m.profile_read()
        m.profile(False)
        step[M] = {k: v[0] / v[1] for k, v in prof.items() if v[1]}
        step[M]["linear_ms"] = sum(step[M].get(k, 0.0) for k in ("gemm_qkv", "gemm_o", "gemm_gateup", "gemm_down"))
    m.sync_status()
    out = {"mode": "sweep", "workload": "Mistral-7B-shaped layer, rows Lp+Bd in " + str(list(SWEEP_ROWS)) +
           ", Bd=32 decodes at ctx 2048; f16 storage; L2 flushed (256 MB write) before every timed launch",
           "gemm_ms": gemm, "decode_only_equivalence": equiv, "step_kernel_ms": step}
    print(json.dumps(out))
    return out


# ------------------------------------------------------------------ serving trace

def run_trace_mode(args):
    """The 32-layer Mistral-7B shape served from a request trace (256 requests,
    Poisson arrivals at 4 req/s by default, lognormal prompt / output lengths) by the
    stall-free scheduler at each token budget, arrivals on the wall clock.
    One JSON line with tokens/s, step latency and TTFT / TBT percentiles per
    budget."""
    import torch

    import chunked_prefill_hybrid_sar_gb300 as sar
    from chunked_prefill_hybrid_sar_gb300 import harness, serve

    taus = [int(t) for t in args.taus.split(",")]
    dims = dataclasses.replace(synth.MISTRAL_7B, sliding_window=args.window)
    m, _ = harness.load_synthetic_model(0, dims, max_tokens=max(taus), max_decodes=256)
    free, _ = torch.cuda.mem_get_info()
    page_bytes = dims.n_layers * 2 * dims.kv_dim * PAGE * 2
    n_pages = int(free * 0.8) // page_bytes
    kv = sar.KVCache(m, PAGE, n_pages)
    trace = synth.request_trace(0, args.requests, rate=args.rate, prompt_median=1024, prompt_clip=(64, 8192),
                                out_median=256, out_clip=(16, 1024))
    toks = synth.prompt_tokens(1, trace, dims.vocab)
    runs = {}
    for tau in taus:
        res = serve.run_trace(m, kv, trace, toks, tau=tau, keep_batches=False, max_chunks=args.max_chunks)
        m.sync_status()
        st = sorted(res.step_ms)
        summ = res.summary()
        summ["step_ms_p50"] = st[len(st) // 2] if st else None
        summ["step_ms_p90"] = st[int(0.9 * (len(st) - 1))] if st else None
        summ["rows_per_step"] = res.rows / max(1, len(st))
        summ["tokens_per_s_wall"] = res.rows / res.wall_s
        runs[tau] = summ
    attn = f"sliding window {dims.sliding_window}" if dims.sliding_window else "full causal"
    adm = "one chunk per batch" if args.max_chunks == 1 else (
        f"at most {args.max_chunks} chunks per batch" if args.max_chunks else "Algorithm 3 admission loop")
    out = {"mode": "trace", "workload": f"Mistral-7B shape, 32 layers + 32000 head, {attn}, f16 storage, {adm}; "
           f"{args.requests} requests, Poisson {args.rate:g} req/s, prompt lognormal(median 1024, sigma 1, clip 64-8192), "
           f"output lognormal(median 256, sigma 1, clip 16-1024), greedy sampling, wall-clock arrivals",
           "kv_pages": n_pages, "page_size": PAGE, "per_tau": runs}
    print(json.dumps(out))
    return out


# ------------------------------------------------------------------ throughput vs batch

FIG3_PREFILL_B = (1, 2, 4, 8)
FIG3_DECODE_B = (1, 2, 4, 8, 16, 32, 64, 128, 256)


def run_batch_sweep(args):
    """Prefill and decode throughput against batch size on the 32-layer
    Mistral-7B shape at prompt length 1024 (the pages' motivating
    measurement: prefill saturates the GPU at small batches, decode throughput
    keeps growing with the batch).  Prefill: one step over B whole 1024-token
    prompts (B chunks, B x 1024 rows); decode: one step of B decodes whose
    contexts hold 1024 tokens (random KV), token inputs.  Each step is replayed
    from a captured graph and device-timed; tokens/s counts the step's rows."""
    import torch

    import chunked_prefill_hybrid_sar_gb300 as sar
    from chunked_prefill_hybrid_sar_gb300 import harness

    dims = synth.MISTRAL_7B
    plen = 1024
    max_rows = max(FIG3_PREFILL_B) * plen
    m, _ = harness.load_synthetic_model(0, dims, max_tokens=max_rows, max_decodes=max(FIG3_DECODE_B))
    pages_per = plen // PAGE + 1
    n_pages = max(max(FIG3_PREFILL_B), max(FIG3_DECODE_B)) * pages_per + 8
    kv = sar.KVCache(m, PAGE, n_pages)
    gen = synth.generator(2, "cuda")
    for l in range(dims.n_layers):
        for kind in (0, 1):
            pv = harness.page_view(kv, l, kind, dims)
            pv.copy_(torch.randn(pv.shape, generator=gen, device="cuda").to(pv.dtype))
    tables = [list(range(i * pages_per, (i + 1) * pages_per)) for i in range(n_pages // pages_per)]
    stream = torch.cuda.current_stream()

    def time_step(batch, inp, logits_rows):
        logits = torch.empty(logits_rows, dims.vocab, dtype=torch.float32, device="cuda")
        g = sar.StepGraph(m, kv, batch, inp, logits_out=logits)
        for _ in range(3):
            g.launch()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(3, args.steps // 10)
        e0.record(stream)
        for _ in range(reps):
            g.launch()
        e1.record(stream)
        torch.cuda.synchronize()
        g.close()
        return e0.elapsed_time(e1) / reps

    tok = torch.randint(0, dims.vocab, (max_rows,), generator=synth.generator(3), dtype=torch.int32).cuda()
    prefill, decode = {}, {}
    for B in FIG3_PREFILL_B:
        b = sar.Batch([(i, 0, plen, tables[i]) for i in range(B)], [], in_kind=sar.SAR_IN_TOKENS)
        ms = time_step(b, tok[:B * plen].contiguous(), B)
        prefill[B] = {"ms_per_step": ms, "tokens_per_s": B * plen / (ms * 1e-3)}
    for B in FIG3_DECODE_B:
        b = sar.Batch(None, [(i, plen, tables[i]) for i in range(B)], in_kind=sar.SAR_IN_TOKENS)
        ms = time_step(b, tok[:B].contiguous(), B)
        decode[B] = {"ms_per_step": ms, "tokens_per_s": B / (ms * 1e-3)}
    m.sync_status()
    out = {"mode": "batch-sweep", "workload": "Mistral-7B shape, 32 layers + 32000 head, f16 storage; prompt 1024: "
           "prefill steps of B whole prompts, decode steps of B decodes at context 1024 (random KV); "
           "captured graph per step, device-timed", "prefill": prefill, "decode": decode}
    print(json.dumps(out))
    return out


# ------------------------------------------------------------------ long prompt

def run_decode_graph(args):
    """The 32-layer Mistral-7B shape taking decode-only steps (64 decodes,
    contexts uniform in [128, 4096], random KV): the step launched kernel by
    kernel against the same step replayed as a captured CUDA graph, each
    device-timed over the steps and host-timed per step with the sampled
    logits read back (the serving loop's pattern)."""
    import torch

    import chunked_prefill_hybrid_sar_gb300 as sar
    from chunked_prefill_hybrid_sar_gb300 import harness

    dims = synth.MISTRAL_7B
    n_dec = 64
    m, _ = harness.load_synthetic_model(0, dims, max_tokens=n_dec, max_decodes=n_dec)
    ctxs = synth.uniform_int(synth.generator(1), n_dec, 128, 4096)
    n_pages = sum(c // PAGE + 1 for c in ctxs) + 8
    kv = sar.KVCache(m, PAGE, n_pages)
    gen = synth.generator(2, "cuda")
    for l in range(dims.n_layers):
        for kind in (0, 1):
            pv = harness.page_view(kv, l, kind, dims)
            pv.copy_(torch.randn(pv.shape, generator=gen, device="cuda").to(pv.dtype))
    alloc = harness.PageAllocator(range(n_pages))
    b = sar.Batch(None, [(i, c, alloc.take(c // PAGE + 1)) for i, c in enumerate(ctxs)],
                  in_kind=sar.SAR_IN_TOKENS)
    tok = ((torch.arange(n_dec, dtype=torch.int32) * 7 + 3) % dims.vocab).cuda()
    logits = torch.empty(n_dec, dims.vocab, dtype=torch.float32, device="cuda")
    host_logits = torch.empty(n_dec, dims.vocab, dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()
    l0 = sar.launch_count()
    g = sar.StepGraph(m, kv, b, tok, logits_out=logits)
    per_step_launches = sar.launch_count() - l0

    def eager():
        m.step(kv, b, tok, logits_out=logits)

    out = {}
    for name, fn in (("kernel_by_kernel", eager), ("graph", g.launch)):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        dev_ms = e0.elapsed_time(e1) / args.steps
        host = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            fn()
            host_logits.copy_(logits, non_blocking=True)
            stream.synchronize()
            host.append((time.perf_counter() - t0) * 1e3)
        host.sort()
        out[name] = {"device_ms_per_step": dev_ms, "host_ms_per_step_p50": host[len(host) // 2],
                     "host_ms_per_step_min": host[0]}
    m.sync_status()
    g.close()
    res = {"mode": "decode-graph", "workload": f"Mistral-7B shape, 32 layers + 32000 head, f16 storage; "
           f"decode-only steps of {n_dec} decodes (ctx U[128,4096], random KV), token inputs, logits read back",
           "kernels_per_step": per_step_launches, "steps": args.steps, "per_launch": out}
    print(json.dumps(res))
    return res


def run_long_prompt(args):
    """The Yi-34B shape (60 layers, 64000 head; or the 32-layer Mistral-7B
    shape with ``--model mistral7b``) prefilling one 16384-token prompt in
    chunks of C tokens, each step carrying 128 decodes (contexts uniform in
    [512, 8192], random KV): per chunk size the prefill time, the
    chunk-attention time and the prior-chunk KV re-read the chunking implies
    (N(N-1)/2 chunk loads per layer with full causal attention; with a
    sliding window of W keys a chunk starting at s reads back only the
    positions [s - W + 1, s))."""
    import torch

    import chunked_prefill_hybrid_sar_gb300 as sar
    from chunked_prefill_hybrid_sar_gb300 import harness

    chunks = [int(c) for c in args.chunks.split(",")]
    dims = synth.MISTRAL_7B if args.model == "mistral7b" else synth.YI_34B
    dims = dataclasses.replace(dims, sliding_window=args.window)
    if args.layers:
        dims = dataclasses.replace(dims, n_layers=args.layers)
    plen, n_dec = 16384, 128
    m, _ = harness.load_synthetic_model(0, dims, max_tokens=max(chunks) + n_dec, max_decodes=n_dec)
    m.set_chunk_split(args.chunk_split)
    tokens, ctxs = synth.long_prompt_case(0, dims, prompt_len=plen, n_decode=n_dec, ctx_range=(512, 8192))
    n_pages = plen // PAGE + sum(c // PAGE + 1 for c in ctxs) + 8
    kv = sar.KVCache(m, PAGE, n_pages)
    gen = synth.generator(2, "cuda")
    for l in range(dims.n_layers):
        for kind in (0, 1):
            pv = harness.page_view(kv, l, kind, dims)
            pv.copy_(torch.randn(pv.shape, generator=gen, device="cuda").to(pv.dtype))
    alloc = harness.PageAllocator(range(n_pages))
    pbt = alloc.take(plen // PAGE)
    decs = [(100 + i, c, alloc.take(c // PAGE + 1)) for i, c in enumerate(ctxs)]
    tok = tokens.cuda()
    dec_tok = (torch.arange(n_dec, dtype=torch.int32, device="cuda") * 7 + 3) % dims.vocab
    logits = torch.empty(1 + n_dec, dims.vocab, dtype=torch.float32, device="cuda")
    xs = {C: [torch.cat([tok[s:s + C], dec_tok]).contiguous() for s in range(0, plen, C)] for C in chunks}
    stream = torch.cuda.current_stream()

    def prefill(C, events=None):
        for i, s in enumerate(range(0, plen, C)):
            if events is not None:
                events[i][0].record(stream)
            m.step(kv, sar.Batch((0, s, C, pbt), decs, in_kind=sar.SAR_IN_TOKENS), xs[C][i], logits_out=logits)
            if events is not None:
                events[i][1].record(stream)

    if not args.no_warmup:
        prefill(max(chunks))
    torch.cuda.synchronize()
    kv_tok = dims.n_layers * 2 * dims.kv_dim * 2  # K and V bytes of one token over all layers
    per_c = {}
    for C in chunks:
        n = plen // C
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        prefill(C, ev)
        torch.cuda.synchronize()
        step_ms = [a.elapsed_time(b) for a, b in ev]
        m.profile(True)
        prefill(C)
        prof = m.profile_read()
        m.profile(False)
        ca_ms = prof["chunk_attn"][0]
        W = dims.sliding_window
        reread = sum(s - max(0, s - W + 1) if W > 0 else s for s in range(0, plen, C)) * kv_tok
        own = n * C * kv_tok
        per_c[C] = {"steps": n, "prefill_ms": sum(step_ms), "step_ms_mean": sum(step_ms) / n,
                    "step_ms_first": step_ms[0], "step_ms_last": step_ms[-1],
                    "prompt_tokens_per_s": plen / (sum(step_ms) * 1e-3),
                    "hybrid_tokens_per_s": n * (C + n_dec) / (sum(step_ms) * 1e-3),
                    "chunk_attn_ms": ca_ms, "decode_attn_ms": prof["decode_attn"][0],
                    "prior_chunk_kv_bytes": reread, "own_chunk_kv_bytes": own,
                    "chunk_attn_kv_gbs": (reread + own) / (ca_ms * 1e-3) / 1e9 if ca_ms else None,
                    "kernel_ms": {k: v[0] for k, v in prof.items() if v[1]}}
    m.sync_status()
    name = "Mistral-7B" if args.model == "mistral7b" else "Yi-34B"
    attn = f"sliding window {dims.sliding_window}" if dims.sliding_window else "full causal"
    out = {"mode": "long-prompt", "workload": f"{name} shape ({dims.n_layers} layers, H {dims.hidden}, "
           f"{dims.n_q_heads}q/{dims.n_kv_heads}kv x {dims.head_dim}, FFN {dims.ffn}, head {dims.vocab}, "
           f"{attn}), f16 storage; one {plen}-token prompt in chunks of C with {n_dec} decodes "
           f"per step (ctx U[512,8192], random KV)", "sliding_window": dims.sliding_window,
           "chunk_split": bool(args.chunk_split), "per_chunk": per_c}
    print(json.dumps(out))
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=6)
    ap.add_argument("--impl", choices=["sar", "reference"], default="sar")
    ap.add_argument("--no-cpu", action="store_true", help="skip the cpu_baseline leg")
    ap.add_argument("--mode", choices=["step", "sweep", "trace", "long-prompt", "decode-graph", "batch-sweep"],
                    default="step",
                    help="step: the tau=512 hybrid step (default); sweep: tile-quantisation sweep; "
                         "trace: 32-layer serving trace; long-prompt: 60-layer chunked 16k prefill; "
                         "decode-graph: 32-layer decode-only steps, kernel by kernel vs CUDA graph; "
                         "batch-sweep: 32-layer prefill and decode tokens/s against batch size at prompt 1024")
    ap.add_argument("--taus", default="256,512,1024", help="trace mode: token budgets")
    ap.add_argument("--requests", type=int, default=256, help="trace mode: requests of the trace")
    ap.add_argument("--chunks", default="256,512,1024", help="long-prompt mode: chunk sizes")
    ap.add_argument("--layers", type=int, default=0, help="long-prompt mode: fewer layers (profiling)")
    ap.add_argument("--no-warmup", action="store_true", help="long-prompt mode: no untimed prefill first")
    ap.add_argument("--model", choices=["yi34b", "mistral7b"], default="yi34b", help="long-prompt mode: model shape")
    ap.add_argument("--rate", type=float, default=4.0, help="trace mode: Poisson arrival rate (requests/s)")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="step mode: launch kernel by kernel in the timed region instead of replaying each "
                         "case's captured CUDA graph")
    ap.add_argument("--overlap", action="store_true",
                    help="step mode: chunk attention on a second stream, concurrent with decode attention")
    ap.add_argument("--max-chunks", type=int, default=0,
                    help="trace mode: prefill chunks per batch (0 = Algorithm 3's admission loop, 1 = one chunk)")
    ap.add_argument("--chunk-split", action="store_true",
                    help="long-prompt mode: key-range splits of chunk-attention tiles that leave SMs idle")
    ap.add_argument("--window", type=int, default=0,
                    help="long-prompt and trace modes: sliding-window attention of W keys (0 = full causal)")
    ap.add_argument("--rows", default="", help="sweep mode: stacked row counts (default: the configured list)")
    ap.add_argument("--variants", default="", help="sweep mode: tilings (m128n128, m128n256, m256n128, swap, auto)")
    ap.add_argument("--reps", type=int, default=5, help="sweep mode: timed launches per GEMM")
    ap.add_argument("--gemm-only", action="store_true", help="sweep mode: the per-GEMM part only")
    ap.add_argument("--cpu-leg", choices=["float64", "float32"], default=None,
                    help="internal: time one oracle leg on this process's threads and print its JSON")
    ap.add_argument("--cpu-leg-min-s", type=float, default=5.0)
    ap.add_argument("--no-bf16", action="store_true", help="step mode: skip the bf16-storage line")
    args = ap.parse_args()
    if args.cpu_leg:
        run_cpu_leg(args)
        return
    if args.mode == "sweep":
        run_sweep(args)
        return
    if args.mode == "trace":
        run_trace_mode(args)
        return
    if args.mode == "long-prompt":
        run_long_prompt(args)
        return
    if args.mode == "decode-graph":
        run_decode_graph(args)
        return
    if args.mode == "batch-sweep":
        run_batch_sweep(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        if args.steps > 3:
            args.steps = 3  # each oracle step takes seconds
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
