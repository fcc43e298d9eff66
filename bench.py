#!/usr/bin/env python3
"""Benchmark: q8-KV decode attention throughput (effective KV GB/s) on GB300.

One step = one decode token of the Qwen3-VL-8B-shaped serving batch: for each
of its 36 layers, append the new token's K/V of every sequence into the paged
q8 cache (kq8_append_kv) and run exact decode attention (kq8_decode_attn)
over the ragged batch (B = 64, lengths uniform in [1K, 32K], 32 query / 8 KV
heads).  value = algorithmic KV bytes the attention reads per step (264 B per
token and KV head) / step time.  Each layer's pool (~2.3 GB) is far larger
than L2, so consecutive layers never hit in L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kq8|reference]

--impl reference times the CPU oracle on a bounded sample of the same
workload (the pages publish no GPU implementation to compare with).
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "q8-KV decode attention: effective KV GB/s and % of GB300 HBM peak"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
WORKLOADS = ("serving", "long", "sparse", "qwen2b", "prefill", "append")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kq8", choices=["kq8", "reference"])
    ap.add_argument("--workload", default="serving", choices=WORKLOADS,
                    help="serving: B=64 ragged 1K-32K, 36 layers (default); long: B=8 n=131072; "
                         "sparse: block-sparse B=16 n=65536; qwen2b: B=1 n=4059, 28 layers; "
                         "prefill: the causal prefill kernel alone (Qwen3-VL prompts, TFLOP/s); "
                         "append: the write path alone (8 x 4096 new tokens, GB/s)")
    ap.add_argument("--layers", type=int, default=36)
    ap.add_argument("--batch", type=int, default=64)
    ap.add_argument("--graph", default="auto", choices=["auto", "on", "off"],
                    help="replay the step as a captured CUDA graph (auto: for qwen2b, whose "
                         "per-layer GPU work is shorter than its host-side launch path)")
    ap.add_argument("--no-extras", action="store_true", help="skip the secondary measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", FALLBACK_HBM_GBS)), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_peak():
    """Dense bf16 tensor peak (burst) for kernels timed alone."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured bf16_tflops (burst)"
    return FALLBACK_BF16_TFLOPS, "fallback"


def max_over_ranks(ms: float, pg, device) -> float:
    """The slowest rank's elapsed time, on every rank (a no-op for one rank)."""
    if not pg:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_rate_gbs(bytes_per_step: float, steps: int, world: int, ms: float) -> float:
    """Whole-job GB/s: each of the `world` replicas processed bytes_per_step in
    each of `steps` steps within the slowest rank's `ms` (weak scaling)."""
    return bytes_per_step * steps * world / (ms * 1e-3) / 1e9


def kernel_source_hash(sources) -> str:
    """Hash of the csrc files a kernel and its launch plan are built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "query_decode_attention_gb300", "csrc")
    for f in sorted(sources):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None, None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash(e.get("sources", [])):
        return None, None
    return e.get("bytes_per_unit"), e.get("unit")


class ClockSampler:
    """nvidia-smi clock / throttle sampling.  Started before the warm-up (NVML
    start-up can stall GPU submission); only the samples taken between
    mark_start() and mark_end() -- the timed region -- are summarised."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.start = 0
        self.end = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="kq8_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < 20:
            if os.path.getsize(self.path) > 0 or self.proc.poll() is not None:
                break
            time.sleep(0.05)
        return self

    def mark_start(self):
        self.start = os.path.getsize(self.path) if self.path else 0

    def mark_end(self):
        time.sleep(0.06)  # let the sample covering the end land
        self.end = os.path.getsize(self.path) if self.path else 0

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        with open(self.path) as f:
            text = f.read()
        os.unlink(self.path)
        region = text[self.start:self.end] if self.end is not None else text[self.start:]
        sm, smax, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in region.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

class OracleSample:
    """Sequences `seqs` of layer 0 of a workload, quantised by the oracle, ready
    to time the oracle's decode over them (all query heads; block-sparse for
    the sparse workload)."""

    def __init__(self, wl, seqs, sparse=False):
        import oracle
        from query_decode_attention_gb300 import workloads as W
        oracle.build()
        self.oracle = oracle
        self.wl = wl
        self.sparse = sparse
        self.seqs = list(seqs)
        qall = W.host_q(wl)
        self.q = qall[self.seqs]
        self.k8, self.ks, self.v8, self.vs = [], [], [], []
        self.nbytes = 0
        for b in self.seqs:
            K, V = W.host_kv(wl, b, q=qall)
            k8, ks = oracle.kv_quantize_rows(K)
            v8, vs = oracle.kv_quantize_rows(V)
            self.k8.append(k8)
            self.ks.append(ks)
            self.v8.append(v8)
            self.vs.append(vs)
            self.nbytes += int(wl.seq_lens[b]) * wl.nkv * (2 * wl.hd + 8)

    def run(self, nthreads):
        """One pass; returns seconds."""
        wl = self.wl
        t0 = time.perf_counter()
        self.oracle.decode_batch(self.q, self.k8, self.ks, self.v8, self.vs, wl.scale,
                                 kv_bs=wl.kv_bs, sparse=self.sparse, block=wl.block,
                                 topk=wl.topk, probe=wl.probe, nthreads=nthreads)
        return time.perf_counter() - t0

    def describe(self):
        lens = [int(self.wl.seq_lens[b]) for b in self.seqs]
        kind = "block-sparse" if self.sparse else "exact"
        return (f"oracle {kind} decode of sequences {self.seqs[0]}..{self.seqs[-1]} of the "
                f"{self.wl.B} (n = {min(lens)}..{max(lens)}, all {self.wl.nq} query heads, "
                f"layer 0, {self.nbytes / 1e6:.0f} MB of KV), OpenMP over (sequence, head)")


def oracle_threads():
    return max(1, os.cpu_count() or 1)


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, as it stands, on a bounded sample of
    the same workload per step (value: the same exact-equivalent KV GB/s)."""
    if rank != 0:
        return
    if args.workload == "prefill":
        run_reference_prefill(args)
        return
    wl, sparse = make_workload(args, 0)
    threads = oracle_threads()
    nseq = {"serving": 4, "long": 1, "sparse": 2, "qwen2b": 1}[args.workload]
    smp = OracleSample(wl, range(min(nseq, wl.B)), sparse=sparse)
    for _ in range(args.warmup):
        smp.run(threads)
    secs = sum(smp.run(threads) for _ in range(args.steps))
    v = smp.nbytes * args.steps / secs / 1e9
    sample = smp.describe() + ", one pass per step"
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "int8xint8->int32 scores, fp32 softmax/accumulate", "data": "synthetic",
            "config": {"workload": wl.name, "sample": sample},
            "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference_prefill(args):
    """Reference arm of --workload prefill: the oracle's batched prefill of the
    last 16 tokens of the first prompt (each sees ~n tokens) per step."""
    import oracle
    from query_decode_attention_gb300 import workloads as W
    name, nq, nkv, n = PREFILL_CASES[0]
    wl = W.Workload(name, 1, nq, nkv, np.array([n], np.int32), kind="sigma", seed=2100 + n)
    K, V = W.host_kv(wl, 0)
    k8, ks = oracle.kv_quantize_rows(K)
    v8, vs = oracle.kv_quantize_rows(V)
    nb = 16
    q = np.random.default_rng(7).standard_normal((nb, nq, wl.hd)).astype(np.float32)
    run = lambda: oracle.prefill_batch(q, [nb], [k8], [ks], [v8], [vs], wl.scale,
                                       nthreads=oracle_threads())
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    secs = time.perf_counter() - t0
    v = prefill_flops(nq, n, nb) * args.steps / secs / 1e12
    sample = (f"oracle prefill of the last {nb} tokens of the {n}-token {name} prompt "
              f"(all {nq} query heads, one layer), OpenMP over (token, head), one call per step")
    cores = oracle_threads() if oracle.openmp_threads() else 1
    print(json.dumps({"impl": "reference", "metric": "q8-KV causal prefill attention TFLOP/s",
                      "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
                      "warmup": args.warmup, "higher_is_better": True, "data": "synthetic",
                      "config": {"workload": name},
                      "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores,
                                       "kind": "oracle", "sample": sample},
                      "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                              "d2h_bytes_per_step": 0}}))


def make_workload(args, rank):
    """The bench workload (each rank draws its own batch: weak scaling)."""
    from query_decode_attention_gb300 import workloads as W
    if args.workload == "serving":
        return W.serving_8b(B=args.batch, layers=args.layers, seed=3000 + rank), False
    if args.workload == "long":
        return W.long_context(seed=4000 + rank), False
    if args.workload == "sparse":
        return W.sparse_planted(65536, B=16, seed=5000 + rank), True
    return W.qwen3vl_2b(4059, seed=2000 + rank), False


def sparse_call_bytes(wl, sel):
    """Bytes one block-sparse call must read: probe rows (K row + scale) of
    every probed block plus whole 32-token tiles (K, V, scales) of the
    per-KV-head union of kept blocks; gated sequences read all of their KV."""
    total = 0
    for b in range(wl.B):
        n = int(wl.seq_lens[b])
        if n <= 2 * wl.block:
            total += -(-n // 32) * wl.nkv * 8448
            continue
        nblk = -(-n // wl.block)
        rows = sum(len(range(j * wl.block, min((j + 1) * wl.block, n), wl.block // wl.probe)[:wl.probe])
                   for j in range(nblk))
        total += rows * wl.nkv * (wl.hd + 4)
        for h in range(wl.nkv):
            blocks = set(sel[b, h * wl.G:(h + 1) * wl.G].ravel().tolist()) - {-1}
            total += sum(min(wl.block, n - j * wl.block) + 31 >> 5 for j in blocks) * 8448
    return total


class Scenario:
    """A workload resident on the device: one paged q8 pool per layer (round
    robin over fewer pools when memory is short), per-step inputs and the
    step itself -- per layer, append each sequence's new token and run decode
    attention (exact, or block-sparse for the sparse workload)."""

    def __init__(self, args, rank, dev):
        import torch
        from query_decode_attention_gb300 import kq8, paged
        from query_decode_attention_gb300 import workloads as W
        self.kq8, self.W = kq8, W
        self.wl, self.sparse = make_workload(args, rank)
        wl = self.wl
        self.dev = dev
        self.L = wl.layers
        free, _ = torch.cuda.mem_get_info(dev)
        t0 = time.time()
        self.caches = []
        n_pools, self.per_layer = self.L, None
        for layer in range(self.L):
            if self.sparse:
                q = W.host_q(wl, layer)
                Ks, Vs = zip(*[W.host_kv(wl, b, layer, q=q) for b in range(wl.B)])
                case = paged.fill_from_host(wl, list(Ks), list(Vs), dev, q_host=q)
                del Ks, Vs
            else:
                case = paged.fill_cache(wl, layer, dev)
            if self.per_layer is None:
                self.per_layer = case.cache.nbytes()
                n_pools = max(1, min(self.L, (int(free * 0.80) - 8 * self.per_layer) // self.per_layer))
            self.caches.append(case)
            if len(self.caches) >= n_pools:
                break
        torch.cuda.synchronize()
        self.setup_s = time.time() - t0
        B, nq, nkv, hd, L = wl.B, wl.nq, wl.nkv, wl.hd, self.L
        self.q_all = torch.stack([self.caches[l % len(self.caches)].q if self.sparse
                                  else W.device_q(wl, l, dev) for l in range(L)])
        g = W.device_generator(dev, 77 + rank)
        self.k_new = torch.randn((L, B, nkv, hd), generator=g, device=dev)
        self.v_new = torch.randn((L, B, nkv, hd), generator=g, device=dev)
        last = [W.slots_for(wl, self.caches[0].page_table_np, b, int(n) - 1, int(n))[0]
                for b, n in enumerate(wl.seq_lens)]
        self.slots = torch.tensor(np.array(last, np.int32), device=dev)
        self.out_all = torch.empty((L, B, nq, hd), dtype=torch.float32, device=dev)
        if self.sparse:
            nb = kq8.kq8_sparse_decode_workspace_bytes(B, nq, nkv, wl.max_seq_len, wl.block, wl.topk)
            self.chunk_tiles, self.num_chunks = kq8.kq8_sparse_decode_plan(
                B, nq, nkv, wl.max_seq_len, wl.block, wl.topk)
            self.sel = torch.empty((B, nq, wl.topk), dtype=torch.int32, device=dev)
            # append, probe (its last CTA per (sequence, KV head) selects) and the
            # bounded attention; past the 16384 counters the selection and the
            # merge run as kernels of their own
            many = B * nkv > 16384
            self.launches_per_layer = 3 + (1 if many else 0) + (1 if self._merge_kernel() else 0)
        else:
            nb = kq8.kq8_decode_workspace_bytes(B, nq, nkv, wl.max_seq_len)
            self.chunk_tiles, self.num_chunks = kq8.kq8_decode_plan(B, nq, nkv, wl.max_seq_len)
            self.sel = None
            self.launches_per_layer = 2 + (1 if self._merge_kernel() else 0)
        self.ws = kq8.new_workspace(nb, dev)

    def _merge_kernel(self):
        """The separate merge kernel runs only when chunks split a sequence and
        the batch has more (sequence, KV head) pairs than the in-kernel merge's
        16384 counters."""
        return self.num_chunks > 1 and self.wl.B * self.wl.nkv > 16384

    def decode(self, l, out, q, stream):
        wl, case = self.wl, self.caches[l % len(self.caches)]
        if self.sparse:
            self.kq8.kq8_sparse_decode_attn(out, q, case.cache, case.page_table, case.seq_lens,
                                            wl.max_seq_len, wl.scale, wl.block, wl.topk,
                                            wl.probe, self.ws, sel_blocks=self.sel, stream=stream)
        else:
            self.kq8.kq8_decode_attn(out, q, case.cache, case.page_table, case.seq_lens,
                                     wl.max_seq_len, wl.scale, self.ws, stream=stream)

    def step(self, stream, timers=None, q=None, k=None, v=None, slots=None, out=None):
        q = self.q_all if q is None else q
        k = self.k_new if k is None else k
        v = self.v_new if v is None else v
        slots = self.slots if slots is None else slots
        out = self.out_all if out is None else out
        for l in range(self.L):
            case = self.caches[l % len(self.caches)]
            self.kq8.kq8_append_kv(case.cache, k[l], v[l], slots, stream=stream)
            if timers is not None:
                timers[l][0].record(stream)
            self.decode(l, out[l], q[l], stream)
            if timers is not None:
                timers[l][1].record(stream)

    def kv_bytes_per_layer(self):
        """KV bytes exact decode reads per layer (264 B per token and KV head)."""
        return self.wl.kv_bytes_per_layer()

    def sparse_bytes_per_layer(self):
        return sparse_call_bytes(self.wl, self.sel.cpu().numpy())


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.workload == "prefill":
        run_prefill_bench(args)
        return
    if args.workload == "append":
        run_append_bench(args)
        return

    import torch
    from query_decode_attention_gb300 import build as kbuild
    kbuild.build()
    from query_decode_attention_gb300 import kq8, paged
    from query_decode_attention_gb300 import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        pg = dist

    sc = Scenario(args, rank, dev)
    wl, L = sc.wl, sc.L
    stream = torch.cuda.current_stream(dev)

    clk = ClockSampler(local).__enter__()
    for _ in range(args.warmup):
        sc.step(stream)
    torch.cuda.synchronize()
    status = kq8.kq8_read_status(sc.ws)

    use_graph = args.graph == "on" or (args.graph == "auto" and args.workload == "qwen2b")
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            sc.step(torch.cuda.current_stream(dev))
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()

    # ---- timed region
    bytes_per_step = sc.kv_bytes_per_layer() * L
    timers = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(L)] for _ in range(args.steps)]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    clk.mark_start()
    ev0.record(stream)
    for s in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            sc.step(stream, timers[s])
    ev1.record(stream)
    torch.cuda.synchronize()
    clk.mark_end()
    if pg:
        pg.barrier()
    if graph is not None:
        # per-call decode durations for the roofline: the same steps, eagerly
        for s in range(args.steps):
            sc.step(stream, timers[s])
        torch.cuda.synchronize()
    clk.__exit__(None, None, None)
    clocks = clk.summary()
    elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1), pg, dev)
    ms_per_step = elapsed_ms / args.steps
    value = job_rate_gbs(bytes_per_step, args.steps, world, elapsed_ms)
    decode_ms = [timers[s][l][0].elapsed_time(timers[s][l][1])
                 for s in range(args.steps) for l in range(L)]
    dec_avg_ms = sum(decode_ms) / len(decode_ms)
    peak, peak_kind = measured_peaks()
    status |= kq8.kq8_read_status(sc.ws)
    if sc.sparse:
        algo = sc.sparse_bytes_per_layer()
        kernel = "kq8_sparse_decode_attn call (probe + top-k + attention + merge)"
        traffic = None
    else:
        algo = sc.kv_bytes_per_layer()
        kernel = ("kq8_attn_kernel + kq8_merge_kernel (one decode call)" if sc._merge_kernel()
                  else "kq8_attn_kernel with its in-kernel chunk merge (one decode call)")
        per_unit, _ = committed_traffic("kq8_attn_kernel")
        traffic = int(per_unit * wl.total_tokens * wl.nkv) if per_unit is not None else None
    achieved = algo / (dec_avg_ms * 1e-3) / 1e9

    # ---- end to end through the public API from pinned host buffers
    e2e = e2e_measure(args, sc, stream, bytes_per_step, world, pg)

    mode = "block-sparse" if sc.sparse else "exact"
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8xint8->int32 scores, fp32 softmax/accumulate", "data": "synthetic",
        "config": {**W.describe(wl), "workload": wl.name,
                   "step": f"{L} layers x (append {wl.B} tokens + {mode} decode attention)",
                   "value_bytes": ("exact-equivalent KV bytes (264 B per token and KV head)"
                                   if sc.sparse else "KV bytes read (264 B per token and KV head)"),
                   "distinct_layer_pools": len(sc.caches),
                   "l2": f"no flush: each layer pool is {sc.per_layer / 1e9:.2f} GB (> 129 MB L2)",
                   "bytes_per_step": bytes_per_step, "parallelism": f"replicas x{world}",
                   "chunk_tiles": sc.chunk_tiles, "num_chunks": sc.num_chunks},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": kernel, "peak_kind": f"{peak_kind} hbm_gbs",
                     "bytes_per_launch": algo, "launch_ms": round(dec_avg_ms, 5),
                     "launch_ms_source": ("eager calls after the graph-replayed timed region"
                                          if graph is not None else "the timed region")},
        "e2e": e2e,
        "gpu_launches": args.steps * L * sc.launches_per_layer,
        "cuda_graph": graph is not None,
        "clocks": clocks,
        "status_word": status,
        "setup_s": round(sc.setup_s, 1),
    }
    del sc
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_extras and args.workload == "serving":
        line["extras"] = extras(dev, kq8, paged, W, peak)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, sparse=(args.workload == "sparse"))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def e2e_measure(args, sc, stream, bytes_per_step, world, pg):
    """The same step through the public API with its inputs (q, the new K/V
    token of every sequence, write slots) copied from pinned host memory every
    step and the outputs read back, all inside the timed region."""
    import torch
    h_q = sc.q_all.cpu().pin_memory()
    h_k = sc.k_new.cpu().pin_memory()
    h_v = sc.v_new.cpu().pin_memory()
    h_slots = sc.slots.cpu().pin_memory()
    h_out = torch.empty(sc.out_all.shape, dtype=torch.float32).pin_memory()
    d_q, d_k, d_v = (torch.empty_like(x, device=sc.dev) for x in (h_q, h_k, h_v))
    d_slots = torch.empty_like(h_slots, device=sc.dev)
    d_out = torch.empty_like(h_out, device=sc.dev)

    def step():
        d_q.copy_(h_q, non_blocking=True)
        d_k.copy_(h_k, non_blocking=True)
        d_v.copy_(h_v, non_blocking=True)
        d_slots.copy_(h_slots, non_blocking=True)
        sc.step(stream, q=d_q, k=d_k, v=d_v, slots=d_slots, out=d_out)
        h_out.copy_(d_out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    steps = max(1, args.steps)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(ev0.elapsed_time(ev1), pg, sc.dev)
    h2d = sum(x.numel() * x.element_size() for x in (h_q, h_k, h_v, h_slots))
    d2h = h_out.numel() * h_out.element_size()
    return {"value": round(job_rate_gbs(bytes_per_step, steps, world, ms), 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / steps, 4)}


def _time_calls(fn, reps, stream):
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


PREFILL_CASES = (
    # (name, nq, nkv, prompt tokens): whole prompts in one call -- the longest
    # Qwen3-VL-2B prompt of the prefill table and an 8K Qwen3-VL-8B prompt
    ("qwen3vl2b_prompt_n4059", 16, 8, 4059),
    ("qwen3vl8b_prompt_n8192", 32, 8, 8192),
)


def prefill_flops(nq, n, nb):
    """Algorithmic FLOPs of one causal prefill call: per (query head, new
    token, visible token) a 128-long Q.K dot and a 128-wide P.V update,
    2 * 128 FLOPs each (the kernel's bf16 hi + lo split of P is not counted)."""
    vis = nb * (n - nb) + nb * (nb + 1) // 2
    return nq * vis * 4 * 128


def prefill_measure(dev, kq8, paged, W, peak_tflops, reps=10, cases=PREFILL_CASES):
    """Causal prefill of whole prompts, one layer per call, timed alone with
    CUDA events (median of reps).  The layer's KV (<= 17 MB) stays in L2: the
    kernel is bound by the tensor and CUDA cores, not by HBM."""
    import torch
    stream = torch.cuda.current_stream(dev)
    res = {}
    for name, nq, nkv, n in cases:
        wl = W.Workload(name, 1, nq, nkv, np.array([n], np.int32), kind="sigma", seed=2100 + n)
        case = paged.fill_cache(wl, 0, dev)
        g = W.device_generator(dev, 7 + n)
        q = torch.randn((n, nq, wl.hd), generator=g, device=dev)
        out = torch.empty_like(q)
        q_off = torch.tensor([0, n], dtype=torch.int32, device=dev)
        ws = kq8.new_workspace(kq8.kq8_prefill_workspace_bytes(1, nq, nkv, n, n), dev)
        ms = _time_calls(lambda: kq8.kq8_prefill_attn(out, q, case.cache, case.page_table,
                                                      case.seq_lens, q_off, n, n, wl.scale, ws,
                                                      stream=stream), reps, stream)
        tf = prefill_flops(nq, n, n) / (ms * 1e-3) / 1e12
        res[name] = {"ms": round(ms, 4), "TFLOP/s": round(tf, 1),
                     "frac_of_bf16_peak": round(tf / peak_tflops, 4),
                     "flops": prefill_flops(nq, n, n), "status_word": kq8.kq8_read_status(ws)}
        # the block-sparse prefill of the same prompt (block 32, k 32, probe 8):
        # per token O(n / block * probe + k * block) instead of O(n)
        wss = kq8.new_workspace(kq8.kq8_sparse_prefill_workspace_bytes(n, nq, nkv, n, 32, 32), dev)
        ms_sp = _time_calls(lambda: kq8.kq8_sparse_prefill_attn(
            out, q, case.cache, case.page_table, case.seq_lens, q_off, n, n, wl.scale, 32, 32, 8,
            wss, stream=stream), reps, stream)
        res[name].update({"sparse_ms": round(ms_sp, 4),
                          "sparse_speedup_vs_exact": round(ms / ms_sp, 3),
                          "sparse_status_word": kq8.kq8_read_status(wss)})
        del wss
        del case, q, out
        torch.cuda.empty_cache()
    return res


def run_prefill_bench(args):
    """--workload prefill: the prefill kernel alone, one JSON line."""
    import torch
    from query_decode_attention_gb300 import build as kbuild
    kbuild.build()
    from query_decode_attention_gb300 import kq8, paged
    from query_decode_attention_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, kind = measured_bf16_peak()
    res = prefill_measure(dev, kq8, paged, W, peak, reps=max(3, args.steps))
    name, r = next(iter(res.items()))
    print(json.dumps({"metric": "q8-KV causal prefill attention TFLOP/s", "value": r["TFLOP/s"],
                      "unit": "TFLOP/s", "n_gpus": 1, "higher_is_better": True,
                      "dtype": "int8 codes as fp16/bf16 operands, fp32 TMEM accumulators",
                      "config": {"workload": name, "cases": list(res)},
                      "roofline": {"bound": "tensor", "achieved": r["TFLOP/s"], "peak": peak,
                                   "unit": "TFLOP/s", "frac": r["frac_of_bf16_peak"],
                                   "peak_kind": kind},
                      "cases": res}))


def _graph_step_ms(fn, dev, reps=20):
    """Capture fn() (enqueueing on the current stream) as one CUDA graph and
    time its replays: median ms per replay over reps, after 3 warm-ups."""
    import torch
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        fn()  # eager warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.synchronize()
    return _time_calls(g.replay, reps, torch.cuda.current_stream(dev))


def qwen2b_decode_steps(dev, kq8, paged, W, reps=20):
    """The pages' own decode configuration (article 10-1 Table B): Qwen3-VL-2B,
    batch 1, 28 layers, contexts 506 / 2046 / 4059; one step = per layer the
    new token's append and exact or block-sparse (block 32, k 32, probe 8)
    decode attention, replayed as one CUDA graph (its per-layer GPU work is
    shorter than the host launch path).  28 distinct layer pools (> L2 at
    n = 4059: 240 MB)."""
    import torch
    res = {}
    for n in (506, 2046, 4059):
        wl = W.qwen3vl_2b(n)
        cases = [paged.fill_cache(wl, layer, dev) for layer in range(wl.layers)]
        L, B, nq, nkv, hd = wl.layers, wl.B, wl.nq, wl.nkv, wl.hd
        g = W.device_generator(dev, 11 + n)
        kn = torch.randn((L, B, nkv, hd), generator=g, device=dev)
        vn = torch.randn((L, B, nkv, hd), generator=g, device=dev)
        slot = torch.tensor(cases[0].slots(0, n - 1, n), dtype=torch.int32, device=dev)
        out = torch.empty((L, B, nq, hd), device=dev)
        wse = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(B, nq, nkv, n), dev)
        wss = kq8.new_workspace(kq8.kq8_sparse_decode_workspace_bytes(B, nq, nkv, n, 32, 32), dev)

        def step(sparse):
            st = torch.cuda.current_stream(dev)
            for layer, c in enumerate(cases):
                kq8.kq8_append_kv(c.cache, kn[layer], vn[layer], slot, stream=st)
                if sparse:
                    kq8.kq8_sparse_decode_attn(out[layer], c.q, c.cache, c.page_table, c.seq_lens,
                                               n, wl.scale, 32, 32, 8, wss, stream=st)
                else:
                    kq8.kq8_decode_attn(out[layer], c.q, c.cache, c.page_table, c.seq_lens, n,
                                        wl.scale, wse, stream=st)
        ms_ex = _graph_step_ms(lambda: step(False), dev, reps)
        ms_sp = _graph_step_ms(lambda: step(True), dev, reps)
        kv = wl.kv_bytes_per_layer() * L
        res[f"n{n}"] = {"exact_ms_per_token": round(ms_ex, 4),
                        "sparse_k32_ms_per_token": round(ms_sp, 4),
                        "sparse_speedup_vs_exact": round(ms_ex / ms_sp, 3),
                        "exact_us_per_layer": round(1e3 * ms_ex / L, 2),
                        "exact_kv_GB/s": round(kv / (ms_ex * 1e-3) / 1e9, 1),
                        "kv_bytes_per_token": kv,
                        "status_words": [kq8.kq8_read_status(wse), kq8.kq8_read_status(wss)]}
        del cases, kn, vn, out, wse, wss
        torch.cuda.empty_cache()
    res["step"] = ("28 layers x (append 1 token + decode attention), one CUDA graph; "
                   "the pages' RK3588 figures for the same step: exact 9.7 / 48.9 / 110.7 ms, "
                   "sparse 13.4 / 39.1 / 55.4 ms (context, not a target)")
    return res


def sparse_sweep(dev, kq8, paged, W, peak, reps=10):
    """The block-sparse configuration over its context lengths (B = 16, 16/8
    heads, block 32, k 32, probe 8, 32 planted blocks per (sequence, KV head)):
    exact vs block-sparse vs shared-selection decode, one call each, timed
    alone (median of reps).  n = 64 is at the gate (the exact kernel runs).
    frac_of_peak: the union of kept tiles plus the probe rows read, per call
    time, against the measured HBM peak.  Returns the results and, for the CPU
    baseline, the host inputs of the n = 4059 case."""
    import torch
    stream = torch.cuda.current_stream(dev)
    res, keep = {}, None
    for n in (64, 506, 4059, 16384, 65536):
        wl = W.sparse_planted(n, B=16)
        q = W.host_q(wl)
        Ks, Vs = zip(*[W.host_kv(wl, b, q=q) for b in range(wl.B)])
        case = paged.fill_from_host(wl, list(Ks), list(Vs), dev, q_host=q)
        if n == 4059:
            keep = (wl, q, list(Ks), list(Vs))
        del Ks, Vs
        out = torch.empty((wl.B, wl.nq, wl.hd), device=dev)
        ws = kq8.new_workspace(kq8.kq8_sparse_decode_workspace_bytes(
            wl.B, wl.nq, wl.nkv, wl.max_seq_len, wl.block, wl.topk), dev)
        sel = torch.empty((wl.B, wl.nq, wl.topk), dtype=torch.int32, device=dev)
        wsx = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv,
                                                               wl.max_seq_len), dev)
        args = (case.q, case.cache, case.page_table, case.seq_lens, wl.max_seq_len, wl.scale)
        ms = _time_calls(lambda: kq8.kq8_sparse_decode_attn(
            out, *args, wl.block, wl.topk, wl.probe, ws, sel_blocks=sel, stream=stream),
            reps, stream)
        ms_ex = _time_calls(lambda: kq8.kq8_decode_attn(out, *args, wsx, stream=stream), reps,
                            stream)
        ms_sh = _time_calls(lambda: kq8.kq8_sparse_decode_attn_shared(
            out, *args, wl.block, wl.topk, wl.probe, ws, stream=stream), reps, stream)
        nbytes = sparse_call_bytes(wl, sel.cpu().numpy())
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[f"n{n}"] = {"sparse_ms": round(ms, 4), "exact_ms": round(ms_ex, 4),
                        "shared_selection_ms": round(ms_sh, 4),
                        "speedup_vs_exact": round(ms_ex / ms, 3),
                        "sparse_bytes_read": nbytes, "sparse_GB/s": round(gbs, 1),
                        "frac_of_peak": round(gbs / peak, 4),
                        "exact_GB/s": round(wl.kv_bytes_per_layer() / (ms_ex * 1e-3) / 1e9, 1),
                        "status_words": [kq8.kq8_read_status(ws), kq8.kq8_read_status(wsx)]}
        del case, out, ws, wsx, sel
        torch.cuda.empty_cache()
    return res, keep


def oracle_config_baselines(keep, W, seconds=4.0):
    """The CPU oracle on the pages' configurations' full inputs: the
    Qwen3-VL-2B decode step (28 layers, n = 4059, exact) and one block-sparse
    layer (B = 16, n = 4059, block 32, k 32, probe 8), OpenMP over
    (sequence, head)."""
    import oracle
    oracle.build()
    threads = oracle_threads()
    cores = threads if oracle.openmp_threads() else 1
    res = {}
    wl = W.qwen3vl_2b(4059)
    layers = []
    for layer in range(wl.layers):
        K, V = W.host_kv(wl, 0, layer)
        k8, ks = oracle.kv_quantize_rows(K)
        v8, vs = oracle.kv_quantize_rows(V)
        layers.append((W.host_q(wl, layer), k8, ks, v8, vs))

    def step():
        for q, k8, ks, v8, vs in layers:
            oracle.decode_batch(q, [k8], [ks], [v8], [vs], wl.scale, nthreads=threads)
    step()
    passes, t = 0, 0.0
    while t < seconds:
        t0 = time.perf_counter()
        step()
        t += time.perf_counter() - t0
        passes += 1
    ms = 1e3 * t / passes
    res["qwen3vl2b_n4059_28_layers"] = {
        "ms_per_token": round(ms, 3), "cores": cores,
        "GB/s": round(wl.kv_bytes_per_layer() * wl.layers / (ms * 1e-3) / 1e9, 4),
        "sample": f"the full 28-layer step, exact decode, {passes} passes"}
    if keep is not None:
        wl, q, Ks, Vs = keep
        k8s, kss, v8s, vss = [], [], [], []
        for K, V in zip(Ks, Vs):
            k8, ks = oracle.kv_quantize_rows(K)
            v8, vs = oracle.kv_quantize_rows(V)
            k8s.append(k8), kss.append(ks), v8s.append(v8), vss.append(vs)
        for sparse in (True, False):
            run = lambda: oracle.decode_batch(q, k8s, kss, v8s, vss, wl.scale, sparse=sparse,
                                              block=wl.block, topk=wl.topk, probe=wl.probe,
                                              nthreads=threads)
            run()
            passes, t = 0, 0.0
            while t < seconds / 2:
                t0 = time.perf_counter()
                run()
                t += time.perf_counter() - t0
                passes += 1
            ms = 1e3 * t / passes
            res[f"sparse_cfg_B16_n4059_{'sparse' if sparse else 'exact'}"] = {
                "ms_per_call": round(ms, 3), "cores": cores,
                "exact_equivalent_GB/s": round(wl.kv_bytes_per_layer() / (ms * 1e-3) / 1e9, 4),
                "sample": f"all 16 sequences and 16 query heads of one layer, {passes} passes"}
    return res


def append_case(dev, kq8, paged, W, T_per_seq=4096, B=8):
    """The write path of the long-context configuration: B x T_per_seq new
    tokens (fp32 K/V, 8 KV heads) quantised into a paged pool of exactly their
    pages (random page order); inputs 268 MB, far beyond L2."""
    import torch
    wl = W.custom(B, 16, 8, [T_per_seq] * B, seed=4000, name="append_8x4096")
    cache, pt = paged.new_cache(wl, device=dev)
    T = B * T_per_seq
    g = W.device_generator(dev, 99)
    kn = torch.randn((T, wl.nkv, wl.hd), generator=g, device=dev)
    vn = torch.randn((T, wl.nkv, wl.hd), generator=g, device=dev)
    sl = torch.tensor(W.all_slots(wl, pt), dtype=torch.int32, device=dev)
    nbytes = T * wl.nkv * (2 * wl.hd * 4 + 2 * wl.hd + 8)  # fp32 K+V read, codes + maxima written
    return wl, cache, kn, vn, sl, nbytes


def run_append_bench(args):
    """--workload append: kq8_append_kv alone, one JSON line (GB/s of fp32
    read plus q8 written, against the measured HBM peak)."""
    import torch
    from query_decode_attention_gb300 import build as kbuild
    kbuild.build()
    from query_decode_attention_gb300 import kq8, paged
    from query_decode_attention_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    wl, cache, kn, vn, sl, nbytes = append_case(dev, kq8, paged, W)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(max(3, args.warmup)):
        kq8.kq8_append_kv(cache, kn, vn, sl, status=st, stream=stream)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in evs:
        a.record(stream)
        kq8.kq8_append_kv(cache, kn, vn, sl, status=st, stream=stream)
        b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    peak, kind = measured_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({"metric": "q8 KV append (write path) GB/s", "value": round(gbs, 1),
                      "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "higher_is_better": True,
                      "config": {"workload": wl.name, "tokens": int(sl.numel()), "nkv": wl.nkv},
                      "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                                   "unit": "GB/s", "frac": round(gbs / peak, 4),
                                   "peak_kind": f"{kind} hbm_gbs", "bytes_per_launch": nbytes,
                                   "launch_ms": round(ms, 5)},
                      "status_word": kq8.kq8_read_status(st)}))


def extras(dev, kq8, paged, W, peak):
    """Secondary measurements: long-context exact decode, the streaming form,
    the write path and the block-sparse path (each timed alone with CUDA
    events, median of reps; every working set exceeds L2), then the causal
    prefill kernel (compute-bound; its per-layer KV stays in L2)."""
    import torch
    stream = torch.cuda.current_stream(dev)
    res = {}
    # long context: B = 8, n = 131072, Student-t K with outlier channels
    wl = W.long_context()
    case = paged.fill_cache(wl, 0, dev)
    out = torch.empty((wl.B, wl.nq, wl.hd), device=dev)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len), dev)
    ms = _time_calls(lambda: kq8.kq8_decode_attn(out, case.q, case.cache, case.page_table,
                                                 case.seq_lens, wl.max_seq_len, wl.scale, ws,
                                                 stream=stream), 10, stream)
    gbs = wl.kv_bytes_per_layer() / (ms * 1e-3) / 1e9
    res["long_context_exact"] = {"workload": wl.name, "ms": round(ms, 4), "GB/s": round(gbs, 1),
                                 "frac_of_peak": round(gbs / peak, 4)}
    # streaming form: the same cache folded into running states in 8 pieces
    pieces = 8
    state = kq8.AttnState(wl.B, wl.nq, dev)
    bounds = [torch.full((wl.B,), (wl.max_seq_len * k) // pieces, dtype=torch.int32, device=dev)
              for k in range(pieces + 1)]

    def stream_all():
        kq8.kq8_state_reset(state, stream=stream)
        for k in range(pieces):
            kq8.kq8_decode_attn_update(state, case.q, case.cache, case.page_table, bounds[k],
                                       bounds[k + 1], wl.max_seq_len, wl.scale, ws, stream=stream,
                                       max_range_len=-(-wl.max_seq_len // pieces))
        kq8.kq8_state_finalize(out, state, stream=stream)
    ms_s = _time_calls(stream_all, 10, stream)
    gbs_s = wl.kv_bytes_per_layer() / (ms_s * 1e-3) / 1e9
    res["long_context_streamed_8_pieces"] = {"ms": round(ms_s, 4), "GB/s": round(gbs_s, 1),
                                             "frac_of_peak": round(gbs_s / peak, 4),
                                             "vs_one_call": round(ms / ms_s, 3)}
    del case, out
    torch.cuda.empty_cache()
    # write path: 8 x 4096 new tokens
    _, acache, kn, vn, sl, ab = append_case(dev, kq8, paged, W)
    ms = _time_calls(lambda: kq8.kq8_append_kv(acache, kn, vn, sl, stream=stream), 20, stream)
    res["append_8x4096"] = {"ms": round(ms, 4), "GB/s": round(ab / (ms * 1e-3) / 1e9, 1),
                            "bytes": ab, "frac_of_peak": round(ab / (ms * 1e-3) / 1e9 / peak, 4)}
    del acache, kn, vn
    torch.cuda.empty_cache()
    # q4 cache: the serving shape (B = 64, ragged 1K-32K, one layer) read through
    # kq8_decode_attn_q4; per (token, KV head) 64 + 64 B of codes + 8 B of scales
    wl4 = W.serving_8b(layers=1)
    case4 = paged.fill_cache(wl4, 0, dev, bits=4)
    out4 = torch.empty((wl4.B, wl4.nq, wl4.hd), device=dev)
    ws4 = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl4.B, wl4.nq, wl4.nkv,
                                                           wl4.max_seq_len), dev)
    ms4 = _time_calls(lambda: kq8.kq8_decode_attn_q4(out4, case4.q, case4.cache, case4.page_table,
                                                     case4.seq_lens, wl4.max_seq_len, wl4.scale,
                                                     ws4, stream=stream), 10, stream)
    b4 = wl4.total_tokens * wl4.nkv * (wl4.hd + 8)
    res["q4_serving8b_B64"] = {"ms": round(ms4, 4), "GB/s": round(b4 / (ms4 * 1e-3) / 1e9, 1),
                               "frac_of_peak": round(b4 / (ms4 * 1e-3) / 1e9 / peak, 4),
                               "bytes": b4, "status_word": kq8.kq8_read_status(ws4)}
    del case4, out4, ws4
    torch.cuda.empty_cache()
    # block-sparse configuration over its context lengths, then the pages' own
    # Qwen3-VL-2B decode step, then the CPU oracle on those configurations
    sweep, keep = sparse_sweep(dev, kq8, paged, W, peak)
    res["sparse_sweep_B16"] = sweep
    res["sparse_n65536"] = {"workload": "sparse_n65536", "ms": sweep["n65536"]["sparse_ms"],
                            "exact_ms": sweep["n65536"]["exact_ms"],
                            "speedup_vs_exact": sweep["n65536"]["speedup_vs_exact"],
                            "frac_of_peak": sweep["n65536"]["frac_of_peak"]}
    res["qwen3vl2b_decode_step_B1_28_layers"] = qwen2b_decode_steps(dev, kq8, paged, W)
    res["cpu_oracle_pages_configs"] = oracle_config_baselines(keep, W)
    del keep
    # causal prefill of whole prompts on the tensor cores
    res["prefill"] = prefill_measure(dev, kq8, paged, W, measured_bf16_peak()[0])
    return res


def cpu_baseline(wl, sparse=False, seconds=10.0):
    """The oracle timed on the host cores on a bounded sample of the workload:
    up to 8 sequences of layer 0, passes repeated for about `seconds`."""
    threads = oracle_threads()
    nseq = 8 if wl.B >= 8 and int(wl.seq_lens.max()) <= 32768 else min(2, wl.B)
    smp = OracleSample(wl, range(nseq), sparse=sparse)
    smp.run(threads)
    passes, secs = 0, 0.0
    while secs < seconds and passes < 1000:
        secs += smp.run(threads)
        passes += 1
    res = {"value": round(smp.nbytes * passes / secs / 1e9, 4), "unit": UNIT, "cores": threads,
           "kind": "oracle", "sample": smp.describe() + f", {passes} passes in {secs:.1f} s"}
    # the same oracle on one core: one pass over the first sequence of the sample
    one = OracleSample(wl, range(1), sparse=sparse)
    t1 = one.run(1)
    res["single_core"] = {"value": round(one.nbytes / t1 / 1e9, 4), "unit": UNIT, "cores": 1,
                          "sample": one.describe() + f", one pass in {t1:.2f} s"}
    return res


if __name__ == "__main__":
    main()
