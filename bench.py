#!/usr/bin/env python
"""Benchmark: one IndexShare group step of DSA sparse attention on B300.

A step is one pass of the whole hot path over one batch: the indexer scores
every cached position, the top-2048 are selected, and 4 sparse MLA layers
attend over them (MTP drafting: one indexer pass + 7 draft steps).  The
default workload is decode over a 1M-token context (B = 8 sequences, one
query token each).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Prints one JSON line on rank 0.  Under torchrun every rank runs its own batch
(weak scaling, no collective on the data path); the step time is the max over
ranks.  After the headline workload the same run measures the other
configurations (128K decode, chunked prefill, MTP drafting, the tiny decode
and multi-token verification) and reports each under "workloads"
(--only-headline skips them).  Every workload carries its step time, the
roofline of its dominant kernel, each kernel of the path timed alone
("kernels"), the end-to-end rate through the C ABI with host buffers and the
clock record of its timed window.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from long_context_sparse_26_b300 import workloads as wl  # noqa: E402

METRIC = "4-layer IndexShare group decode tokens/s @1M ctx; % of HBM roofline"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = wl.DECODE_1M.name
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0


# --------------------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1400.0, "fallback"


def algorithmic_bytes(w: wl.Workload, B: int, fp8_keys: bool = False, fp8_kv: bool = False) -> dict:
    """Indexer keys read once per group + gathered latent rows (576 bf16) per layer or draft step.
    FP8 keys: 128 bytes and one fp32 scale per key.  FP8 latent rows: 656 bytes."""
    key_bytes = B * w.T * (wl.IDX_DIM + 4 if fp8_keys else wl.IDX_DIM * 2)
    uses = w.mtp_steps if w.kind == "mtp" else w.n_layers
    gather = uses * B * w.Q * w.topk * (wl.FP8_LATENT_ROW_BYTES if fp8_kv else wl.D_QK * 2)
    return {"indexer_keys": key_bytes, "gathered_rows": gather, "total": key_bytes + gather}


def indexer_flops(w: wl.Workload, B: int) -> int:
    """Multiply-adds x2 of the indexer over the causal (query, key) pairs."""
    pos = np.arange(w.first_pos, w.first_pos + w.Q)
    pairs = int(np.minimum(pos + 1, w.T).sum()) * B
    return 2 * wl.N_IDX_HEADS * wl.IDX_DIM * pairs


class ClockSampler:
    """Samples SM clocks and clock-event reasons with nvidia-smi (read-only)
    every 100 ms in a background process, for the whole run; each timed
    window is summarised from the samples whose timestamps fall inside it."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id):
        import subprocess
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        self.rows = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={device_id}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None and self.rows is None:
            self.proc.terminate()
            self.proc.wait()
            self.f.close()
            import datetime
            self.rows = []
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) < 10:
                        continue
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    except ValueError:
                        continue
                    self.rows.append([ts] + parts[1:])
            os.unlink(self.path)

    def summary(self, t0: float, t1: float) -> dict:
        """Samples taken between wall times t0 and t1 (time.time()); the
        nearest sample when none falls inside (windows shorter than 100 ms).
        Read after stop(), once every window has been run."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = self.rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = [r for r in rows if t0 <= r[0] <= t1]
        if not inside:
            mid = 0.5 * (t0 + t1)
            inside = [min(rows, key=lambda r: abs(r[0] - mid))]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        mhz = [v for v in (num(r[2]) for r in inside) if v is not None]
        power = [v for v in (num(r[4]) for r in inside) if v is not None]
        reasons = set()
        for r in inside:
            for name, val in (("hw_slowdown", r[6]), ("hw_thermal_slowdown", r[7]), ("sw_thermal_slowdown", r[8]),
                              ("sw_power_cap", r[9])):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": num(rows[0][3]),
                "reasons": sorted(reasons), "samples": len(inside), "power_w_max": max(power) if power else None}


def count_graph_kernels(graph) -> int | None:
    """Kernel nodes in a captured CUDA graph (every kernel in it is libdsa's)."""
    try:
        from cuda.bindings import runtime as rt
        g = rt.cudaGraph_t(init_value=graph.raw_cuda_graph())
        err, _, n = rt.cudaGraphGetNodes(g, 0)
        err, nodes, n = rt.cudaGraphGetNodes(g, n)
        if err != rt.cudaError_t.cudaSuccess:
            return None
        count = 0
        for node in nodes[:n]:
            err, ty = rt.cudaGraphNodeGetType(node)
            if ty == rt.cudaGraphNodeType.cudaGraphNodeTypeKernel:
                count += 1
        return count
    except Exception:
        return None


def kernel_source_hash(name: str) -> str:
    with open(os.path.join(ROOT, "long_context_sparse_26_b300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:12]


def profiled_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 4 and parts[0] == kernel_file and parts[1] == workload:
                    if parts[2] == kernel_source_hash(kernel_file):
                        return float(parts[3])
    except OSError:
        pass
    return None


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------- CPU oracle sample

def _bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_sample(w: wl.Workload, inp: wl.Inputs, b: int, t: int) -> float:
    """Times the oracle on one query token of sequence b: the full indexer row,
    the stable sort, and every attention layer (or draft step).  Returns the
    seconds of oracle arithmetic only: the inputs are copied to the host
    before the clock starts, and the latent rows the oracle's own index set
    names are fetched from the device between the two timed parts (the 1M
    caches never fit the host), outside the clock."""
    import oracle
    qi = oracle.bf16_bits_to_f64(_bits(inp.q_idx[b, t]))
    kk = oracle.bf16_bits_to_f64(_bits(inp.k_idx[b]))
    wv = inp.w[b, t].detach().cpu().double().numpy()
    pos = int(inp.q_pos[b, t])
    if w.kind == "mtp":
        qs = [oracle.bf16_bits_to_f64(_bits(inp.q_steps[s, b])) for s in range(w.mtp_steps)]
        kv_seqs = [inp.kv[0][b]] * w.mtp_steps
    else:
        qs = [oracle.bf16_bits_to_f64(_bits(q[b, t])) for q in inp.q]
        kv_seqs = [kv[b] for kv in inp.kv]
    t0 = time.perf_counter()
    S = oracle.indexer_scores_row(qi, wv, kk, pos)
    idx = oracle.topk_select_row(S, pos, w.topk)
    t1 = time.perf_counter()
    valid = idx[idx >= 0]
    sel = torch.as_tensor(valid, device=inp.k_idx.device)
    rows = [oracle.bf16_bits_to_f64(_bits(kv[sel])) for kv in kv_seqs]   # untimed data copy
    local = np.arange(valid.shape[0])
    t2 = time.perf_counter()
    for q, r in zip(qs, rows):
        oracle.sparse_mla_attn_row(q, r, local, wl.SM_SCALE)
    t3 = time.perf_counter()
    return (t1 - t0) + (t3 - t2)


def cpu_info() -> dict:
    cores = len(os.sched_getaffinity(0))
    blas = None
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        blas = max((i.get("num_threads", 0) for i in info), default=None)
    except Exception:
        pass
    return {"cores": blas or cores, "host_cores": cores}


def cpu_baseline(w: wl.Workload, inp: wl.Inputs, budget_s: float = 20.0) -> dict:
    """The oracle, as it stands, on a bounded sample of the workload: query tokens
    one at a time until about `budget_s` seconds of CPU work."""
    B, Q = inp.q_idx.shape[0], inp.q_idx.shape[1]
    rows = [(b, t) for t in range(Q) for b in range(B)]
    rng = np.random.default_rng(0)
    if len(rows) > 1:
        rows = [rows[i] for i in rng.permutation(len(rows))]
    spent, n = 0.0, 0
    for (b, t) in rows:
        spent += oracle_sample(w, inp, b, t)
        n += 1
        if spent >= budget_s:
            break
    info = cpu_info()
    uses = w.mtp_steps if w.kind == "mtp" else w.n_layers
    what = "draft steps" if w.kind == "mtp" else "layers"
    return {"value": n / spent, "unit": UNIT, "cores": info["cores"], "host_cores": info["host_cores"],
            "kind": "oracle", "seconds": spent,
            "sample": f"{n} of {B * Q} query tokens of {w.name}, each: fp64 indexer over its causal keys, "
                      f"full stable sort, {uses} {what} of exact-softmax attention over its top-{w.topk}"}


# --------------------------------------------------------------------------- GPU arm

L2_BYTES = 126 * 2 ** 20
NOMINAL_HBM_GBS = 8000.0   # the "about 8 TB/s" decode yardstick of the target


def attention_flops(w: wl.Workload, B: int) -> int:
    """2 x 64 heads x (576 + 512) FLOPs per (query row, selected key) and layer or draft step."""
    uses = w.mtp_steps if w.kind == "mtp" else w.n_layers
    return uses * B * w.Q * w.topk * 2 * wl.N_HEADS * (wl.D_QK + wl.D_V)


def input_bytes(inp: wl.Inputs) -> int:
    ts = [inp.q_idx, inp.w, inp.k_idx, inp.q_pos] + list(inp.q or []) + list(inp.kv or [])
    if inp.q_steps is not None:
        ts.append(inp.q_steps)
    return sum(t.numel() * t.element_size() for t in ts if t is not None)


def read_stream_gbs(dev) -> float:
    """A read-only HBM stream, for context beside the copy peak: the best of
    several of torch's full reductions (an fp32 sum, an fp32 max and an int32
    max) over the same 4 GiB buffer, each the best of 8, timed with CUDA
    events."""
    x = torch.ones(2 ** 30, dtype=torch.float32, device=dev)
    ops = (lambda: x.sum(), lambda: x.amax(), lambda: x.view(torch.int32).amax())
    torch.cuda.synchronize()
    best = 0.0
    for op in ops:
        op()
        for _ in range(8):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            op()
            e1.record()
            e1.synchronize()
            best = max(best, x.numel() * 4 / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del x
    torch.cuda.empty_cache()
    return best


def time_launches(fn, stream, n: int) -> float:
    """Mean device time (ms) of n back-to-back launches of fn on `stream`, after 3 untimed ones."""
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(n):
            fn()
    e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) / n


def roofline_of(kernel: str, ms: float, nbytes: int, flops: int, hbm_gbs: float, tf_peak: float, peak_src: str,
                tf_src: str, traffic) -> dict:
    """The bound whose peak time is longer (bytes at the HBM peak, or FLOPs at
    the tensor peak), and the kernel's achieved rate against it."""
    t_bytes = nbytes / (hbm_gbs * 1e9)
    t_flops = flops / (tf_peak * 1e12)
    gbs = nbytes / (ms / 1e3) / 1e9
    tfs = flops / (ms / 1e3) / 1e12
    if t_flops > t_bytes:
        return {"bound": "tensor", "achieved": tfs, "peak": tf_peak, "unit": "TFLOP/s", "frac": tfs / tf_peak,
                "traffic": traffic, "kernel": kernel, "kernel_ms": ms, "algorithmic_flops": flops,
                "algorithmic_bytes": nbytes, "achieved_gbs": gbs, "peak_source": tf_src}
    return {"bound": "hbm", "achieved": gbs, "peak": hbm_gbs, "unit": "GB/s", "frac": gbs / hbm_gbs,
            "traffic": traffic, "kernel": kernel, "kernel_ms": ms, "algorithmic_bytes": nbytes,
            "algorithmic_flops": flops, "achieved_tflops": tfs, "peak_source": f"{peak_src} hbm copy"}


def run_ours(args, w: wl.Workload, world: int, rank: int, local: int, headline: bool = True) -> dict | None:
    """Measures one workload: the whole step captured in a CUDA graph and
    timed with events (max over ranks), each kernel of the path timed alone,
    the step end to end through the C ABI with host buffers, and (headline
    only) the per-layer-indexer variant and the CPU oracle."""
    from long_context_sparse_26_b300 import binding as dsa
    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    cfg = dsa.default_config(topk=w.topk)
    inp = wl.make_inputs(w, dev)
    B, Q, T = w.B, w.Q, w.T
    stream = torch.cuda.Stream(device=dev)
    n_att = w.mtp_steps if w.kind == "mtp" else w.n_layers
    ws = dsa.alloc_workspace(cfg, B, Q, T, n_att, dev)
    scores = torch.empty(B, Q, T, device=dev)
    idx = torch.empty(B, Q, w.topk, dtype=torch.int32, device=dev)
    fp8, paged = bool(args.fp8_indexer) and w.kind != "mtp", bool(args.paged) and w.kind != "mtp"
    if w.kind == "mtp":
        out = torch.empty(w.mtp_steps, B, 64, 512, dtype=torch.bfloat16, device=dev)
        outs = [out]

        def step():
            dsa.indexer_scores(cfg, inp.q_idx, inp.w, inp.k_idx, inp.q_pos, scores, stream)
            dsa.topk_select(cfg, scores, inp.q_pos, idx, ws, stream)
            dsa.mtp_draft_attn(cfg, idx, inp.q_steps, inp.kv[0], out, ws, stream)
    elif fp8:
        # FP8 (E4M3) indexer caches with one fp32 scale per row; bf16 latents,
        # or FP8 latent rows too (--fp8-kv)
        q8, q_scale = wl.to_e4m3_rows(inp.q_idx)
        k8, k_scale = wl.to_e4m3_rows(inp.k_idx)
        outs = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=dev) for _ in range(w.n_layers)]
        if args.fp8_kv:
            kv8s = [wl.to_fp8_latent(kv) for kv in inp.kv]
            inp.kv = None
            torch.cuda.empty_cache()

            def step():
                dsa.indexshare_group_forward_fp8kv(cfg, q8, q_scale, inp.w, k8, k_scale, inp.q_pos, inp.q, kv8s,
                                                   outs, idx, ws, stream)
        else:
            def step():
                dsa.indexshare_group_forward_fp8(cfg, q8, q_scale, inp.w, k8, k_scale, inp.q_pos, inp.q, inp.kv,
                                                 outs, idx, ws, stream)
    elif paged:
        # the caches laid out in pages of args.paged rows, in a random page order
        pools, table = wl.paginate([inp.k_idx] + inp.kv, args.paged, seed=w.seed)
        inp.k_idx, inp.kv = None, None
        torch.cuda.empty_cache()
        k_pool, kv_pools = pools[0], pools[1:]
        outs = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=dev) for _ in range(w.n_layers)]

        def step():
            dsa.indexshare_group_forward_paged(cfg, inp.q_idx, inp.w, k_pool, inp.q_pos, inp.q, kv_pools, table, T,
                                               outs, idx, ws, stream)
    else:
        outs = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=dev) for _ in range(w.n_layers)]

        def step():
            dsa.indexshare_group_forward(cfg, inp.q_idx, inp.w, inp.k_idx, inp.q_pos, inp.q, inp.kv, outs, idx,
                                         ws, stream)

    # inputs under two L2 sizes would be served from L2 across steps: write a
    # buffer larger than L2 between timed steps (outside the timed intervals)
    flush = None if input_bytes(inp) > 2 * L2_BYTES else torch.empty(2 * L2_BYTES // 4, dtype=torch.int32,
                                                                        device=dev)
    torch.cuda.synchronize()
    # capture one step in a CUDA graph (launch overhead off the critical path)
    with torch.cuda.stream(stream):
        step()   # attributes and tensor-map encoders initialised outside capture
    stream.synchronize()
    graph = torch.cuda.CUDAGraph(keep_graph=True)
    with torch.cuda.graph(graph, stream=stream):
        step()
    launches_per_step = count_graph_kernels(graph)
    status = dsa.get_device_error(stream)
    if status != 0:
        raise RuntimeError(f"device error before timing: {dsa.status_string(status)}")

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()
    # untimed load so the clock record holds samples taken under this load
    t_settle = time.time()
    with torch.cuda.stream(stream):
        while time.time() - t_settle < args.settle:
            for _ in range(20):
                graph.replay()
            stream.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    e_all0, e_all1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e_all0.record(stream)
        for i in range(args.steps):
            if flush is not None:
                flush.fill_(i)
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        e_all1.record(stream)
    stream.synchronize()
    t_wall1 = time.time()
    torch.cuda.synchronize()
    barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = sum(step_ms) if flush is not None else e_all0.elapsed_time(e_all1)
    total_ms = max_over_ranks(total_ms, world)
    ms_per_step = total_ms / args.steps
    status = dsa.get_device_error(stream)
    if status != 0:
        raise RuntimeError(f"device error during timing: {dsa.status_string(status)}")
    clock_window = (t_settle, t_wall1)   # summarised once the sampler has stopped

    # ---- each kernel of the path alone, timed with events on its own stream
    kst = torch.cuda.Stream(device=dev)
    n_k = max(5, min(50, args.steps))

    def indexer_alone():
        if fp8:
            dsa.indexer_scores_fp8(cfg, q8, q_scale, inp.w, k8, k_scale, inp.q_pos, scores, kst)
        elif paged:
            dsa.indexer_scores_paged(cfg, inp.q_idx, inp.w, k_pool, table, inp.q_pos, scores, kst)
        else:
            dsa.indexer_scores(cfg, inp.q_idx, inp.w, inp.k_idx, inp.q_pos, scores, kst)

    idx_ms = time_launches(indexer_alone, kst, n_k)
    topk_ms = time_launches(lambda: dsa.topk_select(cfg, scores, inp.q_pos, idx, ws, kst), kst, n_k)
    attn_ms = None
    if w.kind == "mtp":
        attn_ms = time_launches(lambda: dsa.mtp_draft_attn(cfg, idx, inp.q_steps, inp.kv[0], out, ws, kst), kst, n_k)
    elif not fp8 and not paged:
        attn_ms = time_launches(lambda: dsa.sparse_mla_attn_shared(cfg, inp.q, inp.kv, idx, outs, ws, kst), kst, n_k)
    status = dsa.get_device_error(kst)
    if status != 0:
        raise RuntimeError(f"device error in the kernel timings: {dsa.status_string(status)}")

    hbm_gbs, bf16_tf, bf16_tf_sus, peak_src = measured_peaks()
    alg = algorithmic_bytes(w, B, fp8_keys=fp8, fp8_kv=bool(args.fp8_kv))
    flops = indexer_flops(w, B)
    tokens = B * Q * world if w.kind != "mtp" else B * w.mtp_steps * world
    value = tokens / (ms_per_step / 1e3)
    # FP8 operands: the measured bf16 peak times the nominal E4M3:bf16 dense
    # ratio (4.5 / 2.25 PFLOP/s)
    mma_tf = bf16_tf * (2.0 if fp8 else 1.0)
    mma_src = f"{peak_src} bf16 burst" + (" x 2 (nominal e4m3:bf16 dense ratio)" if fp8 else "")
    qg = 1 if Q == 1 else (2 if Q == 2 else 4)
    kernels = {
        "indexer": roofline_of(f"indexer_scores_kernel<{qg}>", idx_ms, alg["indexer_keys"], flops, hbm_gbs, mma_tf,
                               peak_src, mma_src,
                               profiled_traffic("indexer.cuh", w.name + (":fp8" if fp8 else ""))),
        "topk": {"kernel": "topk (standalone call: histogram, scan and select launches)", "kernel_ms": topk_ms,
                 "note": "inside the group at one query per sequence the histogram is counted by the indexer"},
    }
    if attn_ms is not None:
        kernels["attention"] = roofline_of(
            "sparse_mla_tc_kernel + combine", attn_ms, alg["gathered_rows"], attention_flops(w, B), hbm_gbs, bf16_tf,
            peak_src, f"{peak_src} bf16 burst", profiled_traffic("sparse_mla_tc.cuh", w.name))
    dominant = max((k for k in ("indexer", "attention") if k in kernels), key=lambda k: kernels[k]["kernel_ms"])
    roof = dict(kernels[dominant])
    if roof["bound"] == "hbm":
        roof["frac_of_nominal_8tbs"] = roof["achieved"] / NOMINAL_HBM_GBS
        if args.read_peak_gbs:
            roof["read_stream_gbs"] = args.read_peak_gbs
            roof["frac_of_best_hbm_peak"] = roof["achieved"] / max(args.read_peak_gbs, hbm_gbs)
    step_gbs = alg["total"] / (ms_per_step / 1e3) / 1e9
    step_roof = {"algorithmic_bytes": alg["total"], "achieved_gbs": step_gbs,
                 "frac_of_measured_hbm": step_gbs / hbm_gbs, "frac_of_nominal_8tbs": step_gbs / NOMINAL_HBM_GBS,
                 "roofline_ms": alg["total"] / (hbm_gbs * 1e9) * 1e3}
    if args.read_peak_gbs:
        step_roof["frac_of_best_hbm_peak"] = step_gbs / max(args.read_peak_gbs, hbm_gbs)
    t_flops = flops / (mma_tf * 1e12) * 1e3
    if t_flops > step_roof["roofline_ms"]:
        step_roof["roofline_ms"] = t_flops
        step_roof["bound"] = "indexer FLOPs at the tensor peak"
    step_roof["frac_of_roofline_time"] = step_roof["roofline_ms"] / ms_per_step

    # ---- end to end through the public API with host buffers
    e2e = None if (args.no_e2e or paged or fp8) else run_e2e(args, w, cfg, inp, outs, idx, scores, ws, stream, dsa)

    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("fp8 e4m3 indexer and latent caches, bf16 attention math" if args.fp8_kv else
                  "fp8 e4m3 indexer, bf16 attention") if fp8 else "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "Q": Q, "T": T, "topk": w.topk,
                   "layers_per_group": w.n_layers if w.kind != "mtp" else 1,
                   "mtp_steps": w.mtp_steps or None, "parallelism": f"replicas x{world}",
                   "l2": ("L2 flushed between timed steps (inputs fit in L2)" if flush is not None
                          else "inputs larger than L2 (no flush needed)"),
                   "graph": "one step captured, replayed",
                   "kv_layout": f"paged, {args.paged}-row pages in random order" if paged else "contiguous",
                   "indexer_cache": "fp8 e4m3 + fp32 row scales" if fp8 else "bf16",
                   "latent_cache": "fp8 e4m3 + fp32 group scales, bf16 rope (656 B rows)" if args.fp8_kv else "bf16"},
        "roofline": roof, "step_roofline": step_roof, "kernels": kernels,
        "e2e": e2e,
        "gpu_launches": (launches_per_step or 0) * args.steps,
        "gpu_launches_per_step": launches_per_step,
        "clocks": clock_window,
        "step_ms_median": statistics.median(step_ms),
    }
    if headline and w.name == wl.DECODE_1M.name and not args.no_variant and not paged and not fp8:
        res["per_layer_indexer"] = run_per_layer_variant(args, w, cfg, inp, dev, ms_per_step, dsa)
    if headline and rank == 0 and not args.no_cpu_baseline and not paged and not fp8:
        res["cpu_baseline"] = cpu_baseline(w, inp, args.cpu_budget)
    return res


def run_e2e(args, w, cfg, inp, outs, idx, scores, ws, stream, dsa) -> dict:
    """Per step: pinned host -> device copy of the step's new inputs (query-side
    tensors; the indexer key cache and latent caches stay resident in HBM as
    the model's state), the step through the C ABI, device -> host copy of the
    outputs.  As a serving loop would, the copies run on their own streams,
    double-buffered: step i+1's inputs go up and step i-1's outputs come down
    while step i computes.  Every step's copies lie inside the timed region
    (events on the compute stream, which waits for the last download)."""
    dev = stream.device
    if w.kind == "mtp":
        dev_in0 = [inp.q_idx, inp.w, inp.q_pos, inp.q_steps]
    else:
        dev_in0 = [inp.q_idx, inp.w, inp.q_pos] + list(inp.q)
    host_in = [t.detach().cpu().pin_memory() for t in dev_in0]
    host_out = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    dev_in = [dev_in0, [torch.empty_like(t) for t in dev_in0]]
    dev_out = [outs, [torch.empty_like(o) for o in outs]]
    torch.cuda.synchronize()
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, done, out_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def upload(k, after):
        up.wait_event(after)
        with torch.cuda.stream(up):
            for d, h in zip(dev_in[k], host_in):
                d.copy_(h, non_blocking=True)
        in_ready[k].record(up)

    def compute(k):
        stream.wait_event(in_ready[k])
        stream.wait_event(out_free[k])   # the previous download of this output set
        d_in, o = dev_in[k], dev_out[k]
        if w.kind == "mtp":
            q_idx, wt, q_pos, q_steps = d_in
            dsa.indexer_scores(cfg, q_idx, wt, inp.k_idx, q_pos, scores, stream)
            dsa.topk_select(cfg, scores, q_pos, idx, ws, stream)
            dsa.mtp_draft_attn(cfg, idx, q_steps, inp.kv[0], o[0], ws, stream)
        else:
            q_idx, wt, q_pos, qs = d_in[0], d_in[1], d_in[2], d_in[3:]
            dsa.indexshare_group_forward(cfg, q_idx, wt, inp.k_idx, q_pos, qs, inp.kv, o, idx, ws, stream)
        done[k].record(stream)

    def download(k):
        down.wait_event(done[k])
        with torch.cuda.stream(down):
            for h, o in zip(host_out[k], dev_out[k]):
                h.copy_(o, non_blocking=True)
        out_free[k].record(down)

    def run(n, start_event):
        for k in range(2):
            out_free[k].record(stream)
        upload(0, start_event)
        for i in range(n):
            k = i & 1
            if i + 1 < n:
                # the other input set is free once step i-1 has computed
                upload(1 - k, done[1 - k] if i >= 1 else start_event)
            compute(k)
            download(k)
        stream.wait_event(out_free[(n - 1) & 1])
        stream.wait_event(out_free[n & 1] if n >= 2 else out_free[(n - 1) & 1])

    s0 = torch.cuda.Event()
    s0.record(stream)
    run(max(3, args.warmup), s0)
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(args.steps, e0)
    e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    tokens = w.B * w.Q if w.kind != "mtp" else w.B * w.mtp_steps
    return {"value": tokens / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "api": "long_context_sparse_26_b300.binding (C ABI via ctypes)",
            "overlap": "double-buffered: uploads and downloads on their own streams, overlapping compute"}


def run_per_layer_variant(args, w, cfg, inp, dev, group_ms, dsa) -> dict:
    """Without IndexShare: each of the 4 layers runs its own indexer + top-k."""
    idx_q, idx_w, idx_k = wl.per_layer_indexers_of(w, inp.q_idx, inp.w, inp.k_idx, dev)
    B, Q, T = w.B, w.Q, w.T
    stream = torch.cuda.Stream(device=dev)
    ws = dsa.alloc_workspace(cfg, B, Q, T, 1, dev)
    scores = torch.empty(B, Q, T, device=dev)
    idxs = [torch.empty(B, Q, w.topk, dtype=torch.int32, device=dev) for _ in range(w.n_layers)]
    outs = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=dev) for _ in range(w.n_layers)]
    # the inputs were drawn on the default stream and the buffers above may reuse
    # memory that its pending kernels still write: finish them before `stream` runs
    torch.cuda.synchronize()

    def step():
        for layer in range(w.n_layers):
            dsa.indexer_scores(cfg, idx_q[layer], idx_w[layer], idx_k[layer], inp.q_pos, scores, stream)
            dsa.topk_select(cfg, scores, inp.q_pos, idxs[layer], ws, stream)
            dsa.sparse_mla_attn(cfg, inp.q[layer], inp.kv[layer], idxs[layer], outs[layer], None, ws, stream)

    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    alg = w.n_layers * B * T * wl.IDX_DIM * 2 + w.n_layers * B * Q * w.topk * wl.D_QK * 2
    del idx_q, idx_w, idx_k
    torch.cuda.empty_cache()
    return {"ms_per_step": ms, "tokens_per_s": B * Q / (ms / 1e3), "algorithmic_bytes": alg,
            "indexshare_speedup": ms / group_ms,
            "predicted_speedup_bytes": alg / algorithmic_bytes(w, B)["total"]}


# --------------------------------------------------------------------------- reference arm (CPU oracle)

def run_reference(args, w: wl.Workload) -> dict:
    """The oracle as it stands on the host cores; each step = one query token of the workload."""
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = wl.make_inputs(w, dev, B=1)
    times = []
    for i in range(args.warmup + args.steps):
        s = oracle_sample(w, inp, 0, i % w.Q)
        if i >= args.warmup:
            times.append(s)
    per_tok = statistics.mean(times)
    tokens_per_step = w.mtp_steps if w.kind == "mtp" else 1
    value = tokens_per_step / per_tok
    info = cpu_info()
    uses = w.mtp_steps if w.kind == "mtp" else w.n_layers
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_tok * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Q": w.Q, "T": w.T, "topk": w.topk, "sample_B": 1},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": info["cores"], "host_cores": info["host_cores"],
                         "kind": "oracle",
                         "sample": f"each step: one query token of {w.name} (fp64 indexer, full stable sort, "
                                   f"{uses} attention {'steps' if w.kind == 'mtp' else 'layers'})"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def profile_kernel(args, w: wl.Workload):
    """Runs one entry point a few times on the workload (optionally a smaller
    batch) with nothing else on the GPU: the small case for ncu captures."""
    from long_context_sparse_26_b300 import binding as dsa
    from long_context_sparse_26_b300.build import build_library
    build_library()
    dev = "cuda"
    cfg = dsa.default_config(topk=w.topk)
    B, Q, T = w.B, w.Q, w.T
    first = w.first_pos
    if args.queries and args.queries < Q:  # the last query tokens of the workload only (a smaller capture)
        first += Q - args.queries
        Q = args.queries
    q_pos = torch.arange(first, first + Q, dtype=torch.int32, device=dev).repeat(B, 1).contiguous()
    n_att = w.mtp_steps if w.kind == "mtp" else w.n_layers
    ws = dsa.alloc_workspace(cfg, B, Q, T, n_att, dev)
    scores = torch.empty(B, Q, T, device=dev)
    idx = torch.empty(B, Q, w.topk, dtype=torch.int32, device=dev)
    kind = args.profile_kernel
    if kind in ("indexer", "topk", "group"):
        q_idx = wl.indexer_queries(B, Q, w.seed, dev)
        wt = wl.head_weights(B, Q, w.seed, dev)
        k_idx = wl.indexer_keys(B, T, w.seed, dev)
        if args.fp8_indexer:
            q8, q_scale = wl.to_e4m3_rows(q_idx)
            k8, k_scale = wl.to_e4m3_rows(k_idx)
    if kind == "topk":
        if args.fp8_indexer:
            dsa.indexer_scores_fp8(cfg, q8, q_scale, wt, k8, k_scale, q_pos, scores)
        else:
            dsa.indexer_scores(cfg, q_idx, wt, k_idx, q_pos, scores)
    if kind in ("attention", "group"):
        q = [wl.mla_queries(B, Q, w.seed, layer, dev) for layer in range(n_att)]
        kv = [wl.latent_cache(B, T, w.seed, layer, dev) for layer in range(n_att if w.kind != "mtp" else 1)]
        if args.fp8_kv:
            kv = [wl.to_fp8_latent(t) for t in kv]
            torch.cuda.empty_cache()
        outs = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=dev) for _ in range(n_att)]
    if kind == "attention":
        idx.copy_(torch.sort(torch.randint(0, T, (B, Q, w.topk), device=dev), dim=-1).values)
    for _ in range(args.warmup + args.steps):
        if kind == "indexer" and args.fp8_indexer:
            dsa.indexer_scores_fp8(cfg, q8, q_scale, wt, k8, k_scale, q_pos, scores)
        elif kind == "indexer":
            dsa.indexer_scores(cfg, q_idx, wt, k_idx, q_pos, scores)
        elif kind == "topk":
            dsa.topk_select(cfg, scores, q_pos, idx, ws)
        elif kind == "attention" and not args.fp8_kv and w.kind != "mtp":
            # every layer in one launch over the shared index set, as the group makes it
            dsa.sparse_mla_attn_shared(cfg, q, kv, idx, outs, ws)
        elif kind == "attention":
            for layer in range(n_att):
                attn = dsa.sparse_mla_attn_fp8 if args.fp8_kv else dsa.sparse_mla_attn
                attn(cfg, q[layer], kv[min(layer, len(kv) - 1)], idx, outs[layer], None, ws)
        else:
            dsa.indexshare_group_forward(cfg, q_idx, wt, k_idx, q_pos, q, kv, outs, idx, ws)
    torch.cuda.synchronize()
    status = dsa.get_device_error()
    print(json.dumps({"profile_kernel": kind, "workload": w.name, "B": B, "Q": Q, "first_pos": first, "T": T,
                      "launches": args.warmup + args.steps, "device_error": status}))
    if status != 0:
        sys.exit(1)


# The other configurations of the method, measured after the headline in the
# same run and reported under "workloads" (each with its own step time,
# rooflines, end-to-end rate and clock record).
EXTRA_WORKLOADS = (wl.DECODE_128K.name, wl.PREFILL.name, wl.MTP.name, wl.TINY.name, wl.VERIFY.name)


def summary_of(r: dict) -> dict:
    keep = ("value", "unit", "ms_per_step", "step_ms_median", "roofline", "step_roofline", "kernels", "e2e",
            "clocks", "gpu_launches_per_step", "config")
    return {k: r[k] for k in keep if k in r}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--only-headline", action="store_true",
                    help="measure the selected workload only (no 'workloads' entries for the other configs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-variant", action="store_true", help="skip the per-layer-indexer comparison")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--settle", type=float, default=1.0, help="seconds of untimed load before timing (clock record)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-read-peak", action="store_true", help="skip the read-only stream measurement")
    ap.add_argument("--batch", type=int, default=None, help="smaller batch (a small case for profiling)")
    ap.add_argument("--queries", type=int, default=None,
                    help="with --profile-kernel: only the workload's last N query tokens (a small case)")
    ap.add_argument("--fp8-indexer", action="store_true",
                    help="store the indexer caches as FP8 (E4M3) rows with fp32 scales (decode workloads)")
    ap.add_argument("--fp8-kv", action="store_true",
                    help="with --fp8-indexer: store the latent caches as FP8 rows too (656 bytes per position)")
    ap.add_argument("--paged", type=int, default=0, metavar="ROWS",
                    help="lay the caches out in pages of ROWS rows (a multiple of 64) and run the paged entry points")
    ap.add_argument("--profile-kernel", choices=["indexer", "topk", "attention", "group"], default=None,
                    help="only run one entry point a few times (for ncu captures) and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.fp8_kv and not args.fp8_indexer and args.profile_kernel != "attention":
        ap.error("--fp8-kv runs with --fp8-indexer (the all-FP8 cache entry point)")
    w = wl.WORKLOADS[args.workload]
    if args.batch is not None:
        import dataclasses
        w = dataclasses.replace(w, B=args.batch)
    if args.impl == "reference":
        # the oracle is a host program: rank 0 alone runs and prints it, the
        # other ranks exit without work (no process group is needed)
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps(run_reference(args, w)), flush=True)
        return
    world, rank, local = dist_env()
    if args.profile_kernel:
        profile_kernel(args, w)
        return
    from long_context_sparse_26_b300.build import build_library
    if rank == 0 or not os.path.exists(os.path.join(ROOT, "long_context_sparse_26_b300", "libdsa.so")):
        build_library()
    barrier(world)
    torch.cuda.set_device(local)
    vis = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    clocks = ClockSampler(vis[local] if local < len(vis) else local)
    args.read_peak_gbs = None if args.no_read_peak else read_stream_gbs(f"cuda:{local}")
    res = run_ours(args, w, world, rank, local, headline=True)
    extras = not (args.only_headline or args.batch is not None or args.fp8_indexer or args.paged)
    if extras:
        import gc
        settle = args.settle
        args.settle = min(settle, 0.5)
        res["workloads"] = {}
        for name in EXTRA_WORKLOADS:
            if name == w.name:
                continue
            gc.collect()
            torch.cuda.empty_cache()
            r = run_ours(args, wl.WORKLOADS[name], world, rank, local, headline=False)
            res["workloads"][name] = summary_of(r)
            del r
        args.settle = settle
    clocks.stop()
    for r in [res] + list(res.get("workloads", {}).values()):
        r["clocks"] = clocks.summary(*r["clocks"])
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
