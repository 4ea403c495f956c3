#!/usr/bin/env python
"""Throughput of batched speculative-decoding verification on one GB300.

Metric: verified draft positions per second (positions = sum over requests
of K * L_b) on the mixed batch B=256, K=8 drafts, ragged L_b in 1..8,
V=151936 bf16, T=0.7 (SpecTr-GBV multi-draft block verification; the
token-level rule on the same batch is reported beside it).  A step is one
verification call over the whole batch, inputs resident in HBM; the inputs
(about 10.6 GB) are far larger than L2, so no flush is needed between
steps.

The JSON line also carries the roofline of the dominant kernel (the node
kernel: vocabulary-row work), timed live with CUDA events recorded by the
library around those launches, the end-to-end figure through the C-ABI with
host buffers, the oracle timed on host cores, the launch count and the SM
clocks sampled during the timed region.  "next_draft_sampling" measures the
draft-token sampling step (sdv_sample_rows) on the batch's depth-0 draft
rows; "next_psd" the one-GPU emulation of batch-parallel speculative
decoding (the batch's halves alternating draft and verify phases on two
streams).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 it runs under torch.distributed (one process per GPU): every
rank verifies its own batch (weak scaling) with no collective on the data
path; the time is the maximum over ranks.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "verified draft positions/sec at V=151936, B=256; achieved HBM GB/s vs GB300 peak"
UNIT = "positions/s"
CSRC = os.path.join(ROOT, "draft_verification_row_gb300", "csrc")
# the node kernel's sources: a recorded ncu traffic figure holds only while these are unchanged
KERNEL_SRCS = [os.path.join(CSRC, f) for f in ("sdv_stream.cu", "sdv_device.cuh", "sdv_internal.h")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "node_kernel_traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", choices=["multidraft", "token", "kseq"], default="multidraft")
    ap.add_argument("--workload", default=None, help="workload name (default: the mixed B=256 batch)")
    ap.add_argument("--B", type=int, default=None, help="override the batch size (profiling runs)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-extras", action="store_true", help="skip e2e, token mode and CPU baseline")
    ap.add_argument("--cpu-requests", type=int, default=160,
                    help="requests in the oracle's timed sample (cpu_baseline; about 10 s on one core)")
    ap.add_argument("--ref-requests", type=int, default=4, help="requests per step of --impl reference")
    ap.add_argument("--sampling-only", action="store_true",
                    help="only the draft-token sampling measurement (--B sets the batch size)")
    ap.add_argument("--lm-head-only", action="store_true",
                    help="only the LM-head-fused greedy measurement (--B sets its batch size)")
    ap.add_argument("--lm-head-parts", default="fused,cublas,unfused,trie",
                    help="parts of the LM-head measurement to run (profiling runs time one part alone)")
    return ap.parse_args()


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_seed(name, rank):
    """Seed of rank `rank`'s batch: every rank verifies its own requests."""
    from draft_verification_row_gb300 import workloads as W
    cfg = W.WORKLOADS.get(name) or W.LM_HEAD_WORKLOADS[name]
    return cfg["seed"] + 7919 * rank


def trie_nodes(tokens, lengths, K):
    """(inner nodes, leaves) of the requests' draft tries: one node per
    distinct draft prefix, leaves at depth L_b.  The node kernel reads an
    inner node's target and draft rows; a leaf's target row is read only by
    its bonus draw, when the decision ends there."""
    tok = tokens.cpu().numpy()
    lens = lengths.cpu().numpy()
    inner = leaves = 0
    for b in range(tok.shape[0]):
        Lb = int(lens[b])
        for j in range(Lb + 1):
            n = len({tuple(tok[b, k, :j]) for k in range(K)})
            if j < Lb:
                inner += n
            else:
                leaves += n
    return inner, leaves


def table_rows(lengths, K, greedy=False):
    """Rows per call as the hot-path size table counts them: per request,
    the root's target and draft rows once, then each draft's own rows at
    depths 1..L_b (L_b target rows, L_b - 1 draft rows): 2 + K (2 L_b - 1);
    target rows only for greedy: 1 + K L_b."""
    n = 0
    for Lb in lengths.cpu().numpy().tolist():
        if greedy:
            n += 1 + K * Lb
        else:
            n += 1 if Lb == 0 else 2 + K * (2 * Lb - 1)
    return n


def row_bytes_of(batch, inner, leaves, greedy=False, ended_at_leaf=0):
    """Bytes per call of the method's own rows: each distinct trie node's
    target row (leaves included) and each inner node's draft row.  Greedy
    matching needs target rows only, every inner node's (its argmax decides
    the matches) and the leaves its decisions end at (their argmax is the
    correction)."""
    row = batch.V * (2 if batch.dtype == "bf16" else 4)
    if greedy:
        return (inner + ended_at_leaf) * row
    return (2 * inner + leaves) * row


def measured_bf16_peak():
    """Dense bf16 TFLOP/s: the measured burst figure (a kernel timed on its
    own), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def lm_head_bench(args, dev, stream, rank, world):
    """Greedy verification fused into the target model's LM head, on the
    mixed batch's shape with hidden size 4096: the fused call, its tensor-core
    kernel against the measured bf16 peak, cuBLAS on the same GEMM shape, and
    the unfused path (cuBLAS logits of every row to HBM, then sdv greedy)."""
    import draft_verification_row_gb300 as sdv
    from draft_verification_row_gb300 import binding, workloads as W

    lb = W.make_lm_head(W.LM_HEAD_HEADLINE, dev, seed=rank_seed(W.LM_HEAD_HEADLINE, rank), B=args.B)
    inner, leaves = trie_nodes(lb.tokens, lb.lengths, lb.K)
    rows = inner  # the main LM-head pass: one logit row per inner trie node
    out = binding.LmHeadOutputs(lb.B, lb.K, lb.L, lb.V, lb.d, dev)

    def fused():
        sdv.verify_greedy_lm_head(lb.hidden, lb.lm_head, lb.tokens, lb.lengths, out=out, stream=stream)

    parts = set(getattr(args, "lm_head_parts", "fused,cublas,unfused,trie").split(","))
    flops = 2.0 * rows * lb.V * lb.d
    positions = sum_over_ranks(lb.positions, world)
    r = {"what": "greedy verification fused into the target LM head: logits = hidden . W^T on tcgen05, each "
                 "inner trie node's row reduced to its argmax in the epilogue (logits never stored); after the "
                 "decision, a second pass over the leaves the decisions end at",
         "workload": W.LM_HEAD_HEADLINE, "rows": rows, "leaves_in_trie": leaves, "V": lb.V, "d": lb.d}
    if "fused" in parts:
        for _ in range(args.warmup):
            fused()
        total, gemm = time_calls(fused, args.steps, stream, prof=True)
        total, gemm = max_over_ranks(total, world), max_over_ranks(gemm, world)
        if int(out.device_status.item()):
            raise RuntimeError(f"fused LM head: device status {int(out.device_status.item())}")
        ms, gemm_ms = total / args.steps, gemm / args.steps
        # the leaf pass: one row per request whose decision ends at a leaf
        ended_at_leaf = int((out.accept_len == lb.lengths).sum().item())
        tflops = flops / (gemm_ms / 1000.0) / 1e12
        peak, kind = measured_bf16_peak()
        r.update({
            "leaf_rows": ended_at_leaf,
            "metric": "verified draft positions/s", "value": positions / (ms / 1000.0), "unit": "positions/s",
            "ms_per_call": ms, "lm_head_kernel_ms": gemm_ms, "gpu_launches_per_call": 8,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak, "peak_kind": f"{kind} bf16_tflops (burst)",
                         "algorithmic_flops_per_call": flops, "kernel": "lm_head_pair_kernel<ARGMAX>"}})
    if "cublas" in parts:
        # cuBLAS on the same GEMM shape (rows x V x d, bf16 logits written)
        a = torch.randn((rows, lb.d), device=dev).to(torch.bfloat16)
        c = torch.empty((rows, lb.V), dtype=torch.bfloat16, device=dev)

        def cublas():
            with torch.cuda.stream(stream):
                torch.mm(a, lb.lm_head.t(), out=c)

        for _ in range(args.warmup):
            cublas()
        t_cb, _ = time_calls(cublas, args.steps, stream)
        del a, c
        r["cublas_same_gemm"] = {"ms": t_cb / args.steps, "tflops": flops / (t_cb / args.steps / 1000.0) / 1e12}
    if "unfused" in parts:
        # unfused: logits of every row [B][K][L+1][V] to HBM, then greedy verification
        logits = torch.empty((lb.B, lb.K, lb.L + 1, lb.V), dtype=torch.bfloat16, device=dev)
        vout = binding.Outputs("greedy", lb.B, lb.K, lb.L, lb.V, dev)

        def unfused():
            with torch.cuda.stream(stream):
                torch.mm(lb.hidden.view(-1, lb.d), lb.lm_head.t(), out=logits.view(-1, lb.V))
            sdv.verify("greedy", logits, None, lb.tokens, lb.lengths, None, None, 0.0, V=lb.V, out=vout,
                       stream=stream)

        for _ in range(args.warmup):
            unfused()
        t_un, _ = time_calls(unfused, args.steps, stream)
        del logits
        r["unfused_cublas_all_rows_then_greedy"] = {
            "ms": t_un / args.steps, "rows": lb.B * lb.K * (lb.L + 1), "value": positions / (t_un / args.steps / 1000.0)}
    if "trie" in parts:
        # for the sampling rules: every trie node's row (leaves included)
        # written once in bf16 into the verification layout
        tgt = torch.empty((lb.B, lb.K, lb.L + 1, (lb.V + 7) // 8 * 8), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(binding.lm_head_workspace_bytes(lb.B, lb.K, lb.L, lb.V, lb.d), 256), dtype=torch.uint8,
                         device=dev)
        tst = torch.empty(1, dtype=torch.int32, device=dev)

        def trie():
            sdv.lm_head_trie_logits(lb.hidden, lb.lm_head, lb.tokens, lb.lengths, target=tgt, workspace=ws,
                                    device_status=tst, stream=stream)

        for _ in range(args.warmup):
            trie()
        t_tr, g_tr = time_calls(trie, args.steps, stream, prof=True)
        del tgt, ws
        trie_flops = 2.0 * (inner + leaves) * lb.V * lb.d
        r["trie_logits_for_sampling_rules"] = {
            "what": "sdv_lm_head_trie_logits: each trie node's row, leaves included, computed once and written "
                    "in bf16 into the verification layout",
            "ms": t_tr / args.steps, "rows": inner + leaves, "lm_head_kernel_ms": g_tr / args.steps,
            "tflops": trie_flops / (g_tr / args.steps / 1000.0) / 1e12}
    return r


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_sha():
    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic():
    """DRAM bytes of the node kernel per inner trie node, from a committed
    one-pass ncu capture of a smaller batch of the same workload (the
    kernel's traffic grows with the nodes it visits): (bytes per node while
    the kernel's sources are unchanged, else None; the last capture's
    figure, or None without a record)."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        last = float(d["dram_bytes_per_inner_node"])
        return (last if d.get("kernel_source_sha256") == kernel_sha() else None), last
    except (OSError, KeyError, ValueError):
        return None, None


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons (200 ms)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def time_calls(fn, steps, stream, prof=None):
    """Total ms of `steps` calls between CUDA events on `stream`, and the
    summed ms between the library's profiling events (row kernels only)."""
    import draft_verification_row_gb300 as sdv
    pairs = []
    if prof:
        for _ in range(steps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            b.record(stream)
            pairs.append((a, b))
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        if prof:
            sdv.set_profile_events(*pairs[i])
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    sdv.set_profile_events(None, None)
    total = start.elapsed_time(end)
    rows = sum(a.elapsed_time(b) for a, b in pairs) if prof else None
    return total, rows


def sample_arrays(batch, requests):
    """Host numpy copies of the given requests' inputs (bf16 logits as int16 bits)."""
    sel = torch.as_tensor(requests, dtype=torch.long, device=batch.target.device)

    def take(t):
        t = t.index_select(0, sel).cpu()
        return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t).numpy()

    return {k: take(getattr(batch, k)) for k in ("target", "draft", "tokens", "lengths", "accept_u", "sample_u")}


def oracle_sample(batch, mode, requests, arrays=None):
    """Time the oracle, as it stands, on the given requests (host copies)."""
    import oracle
    a = arrays if arrays is not None else sample_arrays(batch, requests)
    prob = oracle.Problem(a["target"], a["draft"], a["tokens"], a["lengths"], a["accept_u"], a["sample_u"],
                          batch.temperature, V=batch.V)
    positions = int(a["lengths"].astype(np.int64).sum()) * batch.K
    t0 = time.perf_counter()
    out = oracle.verify(mode, prob)
    dt = time.perf_counter() - t0
    assert out["rc"] == 0
    return positions, dt


def config_of(batch, mode, world):
    return {"workload": batch.name, "mode": mode, "B": batch.B, "K": batch.K, "L": batch.L,
            "L_b": "uniform 1..L" if batch.meta.get("ragged") else "L", "V": batch.V,
            "logits": batch.dtype, "temperature": batch.temperature, "seed": batch.meta.get("seed"),
            "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}


def numa_placement(t, dev):
    """Where a pinned host tensor's pages sit (NUMA node -> pages, from
    /proc/self/numa_maps) and the GPU's NUMA node (sysfs): reading only."""
    info = {}
    try:
        p = torch.cuda.get_device_properties(dev)
        bus = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
            info["gpu_numa_node"] = int(f.read().strip())
        info["gpu_pci"] = bus
    except (AttributeError, OSError, ValueError):
        info["gpu_numa_node"] = None
    addr = t.data_ptr()
    try:
        with open("/proc/self/numa_maps") as f:
            for line in f:
                start = int(line.split()[0], 16)
                if start <= addr < start + t.numel() * t.element_size():
                    info["buffer_pages"] = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in line.split()
                                            if kv.startswith("N") and "=" in kv}
                    info["policy"] = line.split()[1]
                    break
    except (OSError, ValueError):
        pass
    info["process_cpus"] = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else None
    return info


def host_link(src, nbytes, dev, stream, reps):
    """The host link's own rate: one cudaMemcpyAsync of nbytes from pinned
    host memory (the e2e step's input bytes) to the device, CUDA events on
    the stream, best of reps; plus where the host buffer sits."""
    flat = src.view(-1).view(torch.uint8)
    nbytes = min(int(nbytes), flat.numel())
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = None
    for _ in range(reps + 1):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        with torch.cuda.stream(stream):
            dst.copy_(flat[:nbytes], non_blocking=True)
        b.record(stream)
        b.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    del dst
    return {"what": "one pinned host-to-device cudaMemcpyAsync of the e2e step's input bytes", "bytes": nbytes,
            "ms": best, "gbs": nbytes / (best / 1000.0) / 1e9, "numa": numa_placement(src, dev)}


# The other workloads, as extras beside the headline: (workload, T, rule).
CONFIG_RUNS = [
    ("token-B4-K1-L4-V1024-f32", 1.0, "token"),
    ("token-greedy-B64-K1-L5-V32000-bf16", 1.0, "token"),
    ("token-greedy-B64-K1-L5-V32000-bf16", 0.0, "greedy"),
    ("block-B128-K1-L5-V128256-bf16", 0.7, "block"),
    ("multidraft-B32-K4-L4-V32000-f32", 0.1, "multidraft"),
    ("multidraft-B32-K4-L4-V32000-f32", 0.4, "multidraft"),
    ("multidraft-B32-K4-L4-V32000-f32", 0.7, "multidraft"),
    ("multidraft-B32-K4-L4-V32000-f32", 0.7, "token"),
    ("multidraft-B32-K4-L4-V32000-f32", 0.7, "kseq"),
]
# SpecTr-GBV against the rules it is compared with, on the multi-draft
# workload: (label, rule, drafts used)
ACCEPT_RULES = [("SpecTr-GBV K=4", "multidraft", 4), ("GBV K=1", "multidraft", 1),
                ("per-position K=4", "token", 4), ("K-SEQ K=4", "kseq", 4)]


def first_drafts(batch, K):
    """The batch with only its first K drafts (the same rows and tokens)."""
    import dataclasses
    if K == batch.K:
        return batch
    cut = lambda t: t[:, :K].contiguous()
    return dataclasses.replace(batch, K=K, target=cut(batch.target), draft=cut(batch.draft),
                               tokens=cut(batch.tokens), accept_u=cut(batch.accept_u), sample_u=cut(batch.sample_u))


def capture_graph(fn, stream):
    """fn captured in a CUDA graph (after one call outside the capture):
    a serving loop replays one graph per step instead of launching."""
    side = torch.cuda.Stream(device=stream.device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fn()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_flushed(fn, reps, stream, flush, prof=False):
    """Mean ms of fn between CUDA events on `stream`, L2 flushed (a write
    larger than L2) before every call and outside the timed pair; with prof,
    the mean ms between the library's profiling events instead."""
    import draft_verification_row_gb300 as sdv
    pairs, rows = [], []
    for _ in range(reps):
        with torch.cuda.stream(stream):
            flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if prof:
            c, d = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c.record(stream)
            d.record(stream)
            sdv.set_profile_events(c, d)
            rows.append((c, d))
        a.record(stream)
        fn()
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize()
    sdv.set_profile_events(None, None)
    use = rows if prof else pairs
    return sum(x.elapsed_time(y) for x, y in use) / reps


def config_lines(args, dev, stream, peak, rank):
    """Positions/s, the row kernel's fraction of HBM peak and the oracle
    timed on the host (one core, the whole batch) for each other workload;
    and, on the multi-draft workload, SpecTr-GBV's acceptance against the
    rules it is compared with (E[tau] and BE = E[tau] + 1, means over many
    independent draws of the uniforms, same drafts)."""
    import draft_verification_row_gb300 as sdv
    from draft_verification_row_gb300 import binding, workloads as W
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # twice the L2
    reps = max(20, args.steps)
    res = {}
    for name, T, mode in CONFIG_RUNS:
        batch = W.make(name, dev, temperature=T)
        inner, leaves = trie_nodes(batch.tokens, batch.lengths, batch.K)
        greedy = mode == "greedy" or T == 0.0
        out = binding.Outputs(mode, batch.B, batch.K, batch.L, batch.V, dev, accept_prob=False)

        def call():
            sdv.verify(mode, batch.target, batch.draft, batch.tokens, batch.lengths, batch.accept_u,
                       batch.sample_u, batch.temperature, V=batch.V, out=out, stream=stream)

        for _ in range(3):
            call()
        ms = time_flushed(call, reps, stream, flush)
        kms = time_flushed(call, reps, stream, flush, prof=True)
        if int(out.device_status.item()):
            raise RuntimeError(f"{name} {mode}: device status {int(out.device_status.item())}")
        # the same call replayed from a CUDA graph (its launches and memsets
        # captured once), on the same stream
        graph = capture_graph(lambda: sdv.verify(mode, batch.target, batch.draft, batch.tokens, batch.lengths,
                                                 batch.accept_u, batch.sample_u, batch.temperature, V=batch.V,
                                                 out=out), stream)
        with torch.cuda.stream(stream):
            gms = time_flushed(graph.replay, reps, stream, flush)
        if int(out.device_status.item()):
            raise RuntimeError(f"{name} {mode} (graph): device status {int(out.device_status.item())}")
        del graph
        nbytes = row_bytes_of(batch, inner, leaves, greedy=greedy,
                              ended_at_leaf=int((out.accept_len == batch.lengths).sum().item()))
        gbs = nbytes / (kms / 1000.0) / 1e9
        entry = {"workload": name, "rule": mode, "temperature": T, "B": batch.B, "K": batch.K, "L": batch.L,
                 "V": batch.V, "positions": batch.positions, "ms_per_call": ms,
                 "value": batch.positions / (ms / 1000.0), "unit": UNIT, "row_kernel_ms": kms,
                 "algorithmic_bytes": nbytes, "achieved_gbs": gbs, "frac": gbs / peak,
                 "size_table_bytes": table_rows(batch.lengths, batch.K, greedy) * batch.V * (
                     2 if batch.dtype == "bf16" else 4),
                 "gpu_launches_per_call": 3, "l2": "flushed before every call",
                 "graph": {"ms_per_call": gms, "value": batch.positions / (gms / 1000.0), "unit": UNIT,
                           "what": "the same call captured once in a CUDA graph and replayed"}}
        if rank == 0:
            p, dt = oracle_sample(batch, "greedy" if greedy else mode, list(range(batch.B)))
            entry["cpu_baseline"] = {"value": p / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
                                     "sample": f"all {batch.B} requests ({p} positions, {dt:.2f} s, single thread)"}
        res[f"{name} T={T} {mode}"] = entry
        del batch, out
    # acceptance on the multi-draft workload (GPU path)
    acc = {}
    draws = 64
    for T in (0.1, 0.4, 0.7):
        batch = W.make("multidraft-B32-K4-L4-V32000-f32", dev, temperature=T)
        acc[f"T={T}"] = {}
        for label, mode, K in ACCEPT_RULES:
            b = first_drafts(batch, K)
            out = binding.Outputs(mode, b.B, b.K, b.L, b.V, dev, accept_prob=False)
            g = torch.Generator(device=dev).manual_seed(11 + K)
            taus = []
            for _ in range(draws):
                au = torch.rand(b.accept_u.shape, generator=g, device=dev)
                su = torch.rand(b.sample_u.shape, generator=g, device=dev)
                sdv.verify(mode, b.target, b.draft, b.tokens, b.lengths, au, su, b.temperature, V=b.V, out=out,
                           stream=stream)
                taus.append(out.accept_len.clone())
            t = torch.stack(taus).double()
            m = float(t.mean())
            se = float((t.var(dim=0).sum() / b.B ** 2 / draws).sqrt())
            acc[f"T={T}"][label] = {"E_tau": m, "BE": m + 1.0, "stderr": se, "draws": draws * b.B}
        del batch
    res["acceptance multidraft-B32-K4-L4-V32000-f32"] = {
        "what": "mean accepted length over 64 independent draws of every request's uniforms (same drafts); "
                "BE = E[tau] + 1", **acc}
    del flush
    return res


def sampling_bench(args, batch, dev, stream, world, peak, peak_kind):
    """Draft-token sampling (sdv_sample_rows): one draw per draft from each
    request's depth-0 draft rows (B*K rows of V logits)."""
    import draft_verification_row_gb300 as sdv
    esz = 2 if batch.dtype == "bf16" else 4
    rows = batch.draft[:, :, 0, :].reshape(batch.B * batch.K, batch.stride).contiguous()
    n_rows = rows.shape[0]
    su = torch.rand((n_rows, 1), device=dev, generator=torch.Generator(device=dev).manual_seed(17))
    toks = torch.empty((n_rows, 1), dtype=torch.int32, device=dev)
    dst = torch.empty(1, dtype=torch.int32, device=dev)

    def sample_call():
        sdv.sample_rows(rows, 1, su, batch.temperature, V=batch.V, tokens=toks, device_status=dst, stream=stream)

    for _ in range(args.warmup):
        sample_call()
    ts, _ = time_calls(sample_call, args.steps, stream)
    ts = max_over_ranks(ts, world)
    ms_s = ts / args.steps
    s_bytes = n_rows * batch.V * esz
    s_gbs = s_bytes / (ms_s / 1000.0) / 1e9
    return {"metric": "sampled draft tokens/s", "value": sum_over_ranks(n_rows, world) / (ms_s / 1000.0),
            "unit": "tokens/s", "ms_per_call": ms_s, "rows": n_rows, "draws_per_row": 1, "V": batch.V,
            "gpu_launches_per_call": 1,
            "roofline": {"bound": "hbm", "achieved": s_gbs, "peak": peak, "unit": "GB/s", "frac": s_gbs / peak,
                         "peak_kind": f"{peak_kind} hbm_gbs", "algorithmic_bytes_per_call": s_bytes,
                         "kernel": "sample_rows_kernel"}}


def run_reference(args, world, rank):
    """The oracle on the host cores: each step times a bounded sample."""
    from draft_verification_row_gb300 import workloads as W
    if rank != 0:
        return
    name = args.workload or W.HEADLINE
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    batch = W.make(name, dev, B=args.B)
    n = max(1, min(args.ref_requests, batch.B))
    rng = np.random.default_rng(0)
    times, positions = [], []
    for i in range(args.warmup + args.steps):
        req = sorted(rng.choice(batch.B, size=n, replace=False).tolist())
        p, dt = oracle_sample(batch, args.mode, req)
        if i >= args.warmup:
            times.append(dt)
            positions.append(p)
    value = sum(positions) / sum(times)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(batch, args.mode, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{n} random requests of the batch per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import draft_verification_row_gb300 as sdv
    from draft_verification_row_gb300 import binding, workloads as W

    dev = torch.device(f"cuda:{local}")
    if args.lm_head_only:
        r = lm_head_bench(args, dev, torch.cuda.current_stream(dev), rank, world)
        if rank == 0:
            print(json.dumps(r), flush=True)
        return
    name = args.workload or W.HEADLINE
    seed = rank_seed(name, rank)
    batch = W.make(name, dev, seed=seed, B=args.B)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    if args.sampling_only:
        peak, peak_kind = measured_peaks()
        r = sampling_bench(args, batch, dev, stream, world, peak, peak_kind)
        if rank == 0:
            print(json.dumps(r), flush=True)
        return
    esz = 2 if batch.dtype == "bf16" else 4
    inner, leaves = trie_nodes(batch.tokens, batch.lengths, batch.K)
    positions = batch.positions
    row_b = batch.V * esz
    # algorithmic bytes per call: the method's own rows, each distinct trie
    # node's target row (leaves included) and each inner node's draft row;
    # beside it, the size table's count (per-draft rows, the root once), the
    # rows the node kernel has to read (a pair per inner node: leaves wait
    # for the decision), and a row pair per draft position (dense, no trie)
    trie_bytes = row_bytes_of(batch, inner, leaves)
    table_bytes = table_rows(batch.lengths, batch.K) * row_b
    read_bytes = 2 * inner * row_b
    dense_bytes = 2 * positions * row_b

    def make_call(mode, out):
        def call():
            sdv.verify(mode, batch.target, batch.draft, batch.tokens, batch.lengths, batch.accept_u,
                       batch.sample_u, batch.temperature, V=batch.V, out=out, stream=stream)
        return call

    # the outputs the method defines (tau, k*, the token) and the residual's
    # mass; accept_prob, every node's threshold, is a diagnostic a caller asks
    # for apart (timed below as modes["<mode> with accept_prob"])
    out = binding.Outputs(args.mode, batch.B, batch.K, batch.L, batch.V, dev, accept_prob=False)
    call = make_call(args.mode, out)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device())
    barrier(world)
    clocks.start()
    total_ms, _ = time_calls(call, args.steps, stream)
    clk = clocks.stop()
    # the node kernel's own time, from the library's profiling events (with
    # them on, the finish kernel no longer overlaps the node kernel's tail,
    # so the call itself is timed above without them)
    _, row_ms = time_calls(call, args.steps, stream, prof=True)
    st = int(out.device_status.item())
    if st:
        raise RuntimeError(f"device status {st}")
    total_ms = max_over_ranks(total_ms, world)
    row_ms = max_over_ranks(row_ms, world)
    all_positions = sum_over_ranks(positions, world)
    ms_step = total_ms / args.steps
    value = all_positions / (ms_step / 1000.0)
    launches = 3 * args.steps  # per call: prep, the node kernel, the decision and correction draw

    peak, peak_kind = measured_peaks()
    row_step_s = row_ms / args.steps / 1000.0
    gbs = lambda nbytes: nbytes / row_step_s / 1e9
    per_node, last_per_node = recorded_traffic()
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_of(batch, args.mode, world),
            "outputs": "accept_len, accept_draft, out_token, residual_mass per request (accept_prob not requested)",
            "positions_per_step": all_positions,
            "roofline": {"bound": "hbm", "achieved": gbs(trie_bytes), "peak": peak, "unit": "GB/s",
                         "frac": gbs(trie_bytes) / peak, "peak_kind": f"{peak_kind} hbm_gbs",
                         "traffic": None if per_node is None else per_node * inner,
                         "kernel": "stream_kernel",
                         "algorithmic_bytes_per_step": trie_bytes,
                         "algorithmic_bytes": "each distinct trie node's target row (leaves included) and each "
                                              "inner node's draft row",
                         "trie_rows_per_step": {"target": inner + leaves, "draft": inner},
                         "kernel_ms_per_step": row_ms / args.steps,
                         "size_table_bytes_per_step": table_bytes,
                         "size_table_frac": gbs(table_bytes) / peak,
                         "rows_read_bytes_per_step": read_bytes,
                         "rows_read_frac": gbs(read_bytes) / peak,
                         "dense_bytes_per_step": dense_bytes,
                         "dense_frac": gbs(dense_bytes) / peak,
                         "dense": "a target and a draft row per draft position, no row shared",
                         "leaves": leaves,
                         "bonus_leaf_rows_per_step": int((out.accept_len == batch.lengths).sum().item())},
            "gpu_launches": launches,
            "clocks": clk}
    if per_node is not None:
        line["roofline"]["traffic_note"] = ("dram__bytes_read.sum + dram__bytes_write.sum of one launch of a "
                                            "smaller batch of this workload, scaled by inner trie nodes")
    elif last_per_node is not None:
        # the sources changed since the capture: its figure for reference
        line["roofline"]["traffic_last_capture"] = {"bytes_per_inner_node": last_per_node,
                                                    "sources_changed_since": True}

    if not args.no_extras:
        # the other rules on the same batch: token-level (per-position
        # recursive rejection sampling) and SpecTr's K-SEQ, whose search
        # for rho SpecTr-GBV avoids (the pages' "verification overhead")
        line["modes"] = {}
        runs = [(m, False) for m in ("multidraft", "token", "kseq", "greedy") if m != args.mode]
        runs.append((args.mode, True))
        for other, with_ap in runs:
            out2 = binding.Outputs(other, batch.B, batch.K, batch.L, batch.V, dev, accept_prob=with_ap)
            call2 = make_call(other, out2)
            for _ in range(max(2, args.warmup // 2)):
                call2()
            t2, _ = time_calls(call2, args.steps, stream)
            _, r2 = time_calls(call2, args.steps, stream, prof=True)
            t2 = max_over_ranks(t2, world)
            r2 = max_over_ranks(r2, world)
            ob = row_bytes_of(batch, inner, leaves, greedy=other == "greedy",
                              ended_at_leaf=int((out2.accept_len == batch.lengths).sum().item()))
            og = ob / (r2 / args.steps / 1000.0) / 1e9
            line["modes"][other + (" with accept_prob" if with_ap else "")] = {
                                    "value": all_positions / (t2 / args.steps / 1000.0), "unit": UNIT,
                                    "ms_per_step": t2 / args.steps,
                                    "row_kernel_ms_per_step": r2 / args.steps,
                                    "algorithmic_bytes_per_step": ob, "achieved_gbs": og, "frac": og / peak}
            del out2
        # the headline call captured once in a CUDA graph and replayed (a
        # serving loop's form: no launch work on the host per step)
        graph = capture_graph(lambda: sdv.verify(args.mode, batch.target, batch.draft, batch.tokens, batch.lengths,
                                                 batch.accept_u, batch.sample_u, batch.temperature, V=batch.V,
                                                 out=out), stream)
        for _ in range(2):
            graph.replay()
        tg, _ = time_calls(graph.replay, args.steps, stream)
        tg = max_over_ranks(tg, world)
        if int(out.device_status.item()):
            raise RuntimeError(f"graph replay: device status {int(out.device_status.item())}")
        del graph
        line["graph"] = {"value": all_positions / (tg / args.steps / 1000.0), "unit": UNIT,
                         "ms_per_step": tg / args.steps,
                         "what": "the same call captured once in a CUDA graph (its memsets and 3 launches) "
                                 "and replayed each step"}
        # end to end through the C-ABI with host buffers: the host-to-device
        # copy of the inputs (of the logits, the rows verification reads,
        # sdv_copy_read_rows), the call, and the per-request results back
        names = ["target", "draft", "tokens", "lengths", "accept_u", "sample_u"]
        small = ["tokens", "lengths", "accept_u", "sample_u"]
        host = {n: getattr(batch, n).cpu().pin_memory() for n in names}
        rows_bytes = binding.read_rows_bytes(host["tokens"], host["lengths"], batch.V, batch.stride,
                                             batch.target.dtype)
        h2d = rows_bytes + sum(host[n].numel() * host[n].element_size() for n in small)
        res_host = [torch.empty(batch.B, dtype=torch.int32).pin_memory() for _ in range(3)]
        d2h = 3 * 4 * batch.B
        dev_in = {n: getattr(batch, n) for n in names}

        def e2e_step():  # the read rows copied with one cudaMemcpyAsync per range
            for n in small:
                dev_in[n].copy_(host[n], non_blocking=True)
            binding.copy_read_rows(host["target"], host["draft"], host["tokens"], host["lengths"], batch.target,
                                   batch.draft, V=batch.V, stream=stream)
            call()
            res_host[0].copy_(out.accept_len, non_blocking=True)
            res_host[1].copy_(out.accept_draft, non_blocking=True)
            res_host[2].copy_(out.out_token, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        tc, _ = time_calls(e2e_step, args.e2e_steps, stream)
        tc = max_over_ranks(tc, world)

        # the same rows gathered by the GPU from the mapped host tensors
        def e2e_gather_step():
            for n in small:
                dev_in[n].copy_(host[n], non_blocking=True)
            binding.gather_read_rows(host["target"], host["draft"], dev_in["tokens"], dev_in["lengths"],
                                     batch.target, batch.draft, V=batch.V, stream=stream)
            call()
            res_host[0].copy_(out.accept_len, non_blocking=True)
            res_host[1].copy_(out.accept_draft, non_blocking=True)
            res_host[2].copy_(out.out_token, non_blocking=True)

        e2e_gather_step()
        torch.cuda.synchronize()
        te, _ = time_calls(e2e_gather_step, args.e2e_steps, stream)
        te = max_over_ranks(te, world)

        # the inner rows gathered; the leaf rows the decisions end at read by
        # the verification call from the host tensor itself
        def e2e_inner_step():
            for n in small:
                dev_in[n].copy_(host[n], non_blocking=True)
            binding.gather_read_rows(host["target"], host["draft"], dev_in["tokens"], dev_in["lengths"],
                                     batch.target, batch.draft, V=batch.V, stream=stream, leaves=False)
            sdv.verify(args.mode, batch.target, batch.draft, batch.tokens, batch.lengths, batch.accept_u,
                       batch.sample_u, batch.temperature, V=batch.V, out=out, stream=stream, leaf_target=host["target"])
            res_host[0].copy_(out.accept_len, non_blocking=True)
            res_host[1].copy_(out.accept_draft, non_blocking=True)
            res_host[2].copy_(out.out_token, non_blocking=True)

        e2e_inner_step()
        torch.cuda.synchronize()
        ti, _ = time_calls(e2e_inner_step, args.e2e_steps, stream)
        ti = max_over_ranks(ti, world)
        row_h2d = batch.stride * esz
        ended_at_leaf = int((out.accept_len == batch.lengths).sum().item())  # one leaf row read each
        h2d_inner = 2 * inner * row_h2d + ended_at_leaf * row_h2d + sum(host[n].numel() * host[n].element_size()
                                                                       for n in small)
        link = host_link(host["target"], h2d_inner, dev, stream, args.e2e_steps)
        e2e_ms = ti / args.e2e_steps
        line["e2e"] = {"value": all_positions / (e2e_ms / 1000.0), "unit": UNIT,
                       "h2d_bytes_per_step": h2d_inner, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e2e_ms,
                       "link_frac": (h2d_inner / link["gbs"] / 1e6) / e2e_ms if link.get("gbs") else None,
                       "link": link,
                       "inputs": "pinned host tensors; of the logits, the inner trie nodes' rows are gathered by "
                                 "the GPU over the host link (sdv_gather_inner_rows) and the leaf rows the "
                                 "decisions end at are read from the host tensor by the call itself "
                                 "(sdv_verify_leaves_apart)"}
        line["e2e_all_read_rows"] = {"value": all_positions / (te / args.e2e_steps / 1000.0), "unit": UNIT,
                                     "h2d_bytes_per_step": h2d, "ms_per_step": te / args.e2e_steps,
                                     "inputs": "every row verification may read, leaves included, gathered by the "
                                               "GPU (sdv_gather_read_rows)"}
        line["e2e_copy_calls"] = {"value": all_positions / (tc / args.e2e_steps / 1000.0), "unit": UNIT,
                                  "h2d_bytes_per_step": h2d, "ms_per_step": tc / args.e2e_steps,
                                  "inputs": "the same rows, one cudaMemcpyAsync per range (sdv_copy_read_rows)"}

        # the same with the whole logit tensors copied
        def e2e_full_step():
            for n in names:
                dev_in[n].copy_(host[n], non_blocking=True)
            call()
            res_host[0].copy_(out.accept_len, non_blocking=True)
            res_host[1].copy_(out.accept_draft, non_blocking=True)
            res_host[2].copy_(out.out_token, non_blocking=True)

        e2e_full_step()
        torch.cuda.synchronize()
        tf, _ = time_calls(e2e_full_step, args.e2e_steps, stream)
        tf = max_over_ranks(tf, world)
        line["e2e_whole_tensors"] = {"value": all_positions / (tf / args.e2e_steps / 1000.0), "unit": UNIT,
                                     "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host.values()),
                                     "ms_per_step": tf / args.e2e_steps}
        del host
        # the next row of the path: draft-token sampling
        line["next_draft_sampling"] = sampling_bench(args, batch, dev, stream, world, peak, peak_kind)
        # one-GPU PSD emulation: the batch's two halves alternate drafting
        # (L sampling launches) and verification on two streams
        from draft_verification_row_gb300 import psd
        emu = psd.PsdEmulator(batch, steps=8)
        m = psd.measure(emu, reps=max(5, args.steps // 2), warmup=3)
        line["next_psd"] = {"what": "two halves of the batch alternate draft (sdv_sample_rows per depth) and "
                                    "verify (multidraft) phases on two streams of one GPU",
                            "half_batch": emu.B, **m,
                            "gpu_launches_per_step": emu.L + 3}  # L sampling launches + prep, node, finish
        del emu
        # the next row: greedy verification fused into the target LM head
        line["next_lm_head"] = lm_head_bench(args, dev, stream, rank, world) if args.B is None else None
        # the other workloads beside the headline
        if args.B is None:
            line["configs"] = config_lines(args, dev, stream, peak, rank)
        if rank == 0:
            rng = np.random.default_rng(1)
            req = sorted(rng.choice(batch.B, size=min(args.cpu_requests, batch.B), replace=False).tolist())
            arrays = sample_arrays(batch, req)
            p, dt = oracle_sample(batch, args.mode, req, arrays)
            line["cpu_baseline"] = {"value": p / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
                                    "sample": f"{len(req)} random requests of the batch ({p} positions, "
                                              f"{dt:.1f} s, single thread)"}
            # the same sample across every host core, one oracle process each
            # (an extra: without room for it, the line says why and goes on)
            from oracle import pool
            try:
                _, dta, procs = pool.verify_all_cores(arrays, args.mode, batch.temperature, batch.V)
                line["cpu_baseline_all_cores"] = {"value": p / dta, "unit": UNIT, "cores": procs, "kind": "oracle",
                                                  "sample": f"the same {len(req)} requests split over {procs} "
                                                            f"processes ({dta:.2f} s wall)"}
            except (OSError, RuntimeError, ValueError) as e:
                line["cpu_baseline_all_cores"] = {"unavailable": str(e)[:200]}
            del arrays
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
